"""The index check that needs no scratch from its caller (ccu_conv1d_check_indices_noalloc).

Callers that cannot allocate device memory (a plugin with no handle on the host
application's allocator, a serving loop where cudaMalloc is forbidden) use this entry
point; its one-bit-per-slot bitmap is a fixed array inside the library. This test calls
it through the C-ABI and checks that it reports exactly what ccu_conv1d_check_indices
reports with a caller-provided bitmap, on two calls in a row: the first leaves bits set
in the shared array, which the second must clear before use or it would report false
duplicates. The file sorts last so that a run stopping at the first failure has already
run every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def ccu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import depthwise_causal_conv1d_gb300 as ccu

    return ccu


def _reference_status(ccu, idx_dev, S, stream):
    """Status word from the existing entry point, with a torch-allocated bitmap."""
    status = torch.zeros((1,), dtype=torch.int32, device=DEV)
    scratch = torch.empty((max(ccu.ccu_conv1d_check_indices_scratch_bytes(S) // 4, 1),),
                          dtype=torch.int32, device=DEV)
    st = ccu.ccu_conv1d_check_indices(idx_dev.data_ptr(), idx_dev.numel(), S, scratch.data_ptr(),
                                      status.data_ptr(), stream.cuda_stream)
    assert st == 0, ccu.ccu_conv1d_last_error()
    return status


def _noalloc_status(ccu, idx_dev, S, stream):
    status = torch.zeros((1,), dtype=torch.int32, device=DEV)
    st = ccu.ccu_conv1d_check_indices_noalloc(idx_dev.data_ptr(), idx_dev.numel(), S,
                                              status.data_ptr(), stream.cuda_stream)
    assert st == 0, ccu.ccu_conv1d_last_error()
    return status


def test_noalloc_matches_caller_scratch_on_two_calls_in_a_row(ccu):
    rng = np.random.default_rng(2024)
    S = 100_000
    stream = torch.cuda.Stream()
    # first call: duplicates and an out-of-range slot, leaving many bits set in the array
    first = rng.permutation(S)[:60_000].astype(np.int32)
    first[::11] = -1
    first[59_999] = first[1]  # row 1 is not a padding row: a real duplicate
    first[123] = S + 7
    # second call: a valid batch (distinct slots, some padding) drawn from the same slots
    second = rng.permutation(S)[:60_000].astype(np.int32)
    second[::7] = -1
    cases = [first, second]
    expected = []
    got = []
    for idx in cases:
        idx_dev = torch.from_numpy(idx).to(DEV)
        with torch.cuda.stream(stream):
            got.append(_noalloc_status(ccu, idx_dev, S, stream))
            expected.append(_reference_status(ccu, idx_dev, S, stream))
    torch.cuda.synchronize()
    got = [int(t.item()) for t in got]
    expected = [int(t.item()) for t in expected]
    assert got == expected
    assert got[0] == ccu.CCU_DEVERR_RANGE | ccu.CCU_DEVERR_DUPLICATE
    assert got[1] == 0


def test_noalloc_limits(ccu):
    limit = ccu.CCU_CHECK_INDICES_NOALLOC_MAX_SLOTS
    idx = torch.zeros((4,), dtype=torch.int32, device=DEV)
    status = torch.zeros((1,), dtype=torch.int32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    st = ccu.ccu_conv1d_check_indices_noalloc(idx.data_ptr(), 4, limit + 1, status.data_ptr(), stream)
    assert st == ccu.CCU_ERR_NOT_IMPLEMENTED
    assert "built-in bitmap" in ccu.ccu_conv1d_last_error()
    # the largest served cache: slots at both ends, one repeated
    vals = torch.tensor([0, limit - 1, 7, limit - 1], dtype=torch.int32, device=DEV)
    st = ccu.ccu_conv1d_check_indices_noalloc(vals.data_ptr(), 4, limit, status.data_ptr(), stream)
    assert st == 0
    torch.cuda.synchronize()
    assert int(status.item()) == ccu.CCU_DEVERR_DUPLICATE
