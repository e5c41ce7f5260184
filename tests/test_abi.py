"""The C-ABI library without a GPU: exports, typed declines, route selection.

The argument checks are host code that runs before any CUDA call, so they are tested
here through ccu_conv1d_select_route, which never launches. Calls of the launching
entry points with placeholder pointers are made only when no GPU is visible (the
launch then fails with CCU_ERR_CUDA and touches nothing).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ccu():
    import __graft_entry__ as g

    g.build()
    import depthwise_causal_conv1d_gb300 as ccu

    return ccu


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^CCU_API\s+[\w\s\*]+?\b(ccu_\w+)\s*\(", text, flags=re.M)
    return names


def test_header_declares_entry_points():
    names = declared_functions()
    for must in ("ccu_conv1d_update", "ccu_conv1d_update_checked", "ccu_conv1d_update_ex",
                 "ccu_conv1d_select_route", "ccu_conv1d_check_indices", "ccu_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(ccu):
    lib = ctypes.CDLL(ccu.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_binding_has_same_names(ccu):
    for n in declared_functions():
        assert callable(getattr(ccu, n)), n


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "ccu_conv1d.h"\nint main(void){return CCU_OK;}\n')
    import subprocess

    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-c", str(src), "-o", str(tmp_path / "t.o")], check=True)


def test_status_strings(ccu):
    assert ccu.ccu_status_string(0) == "ok"
    assert "invalid" in ccu.ccu_status_string(1)
    assert "not implemented" in ccu.ccu_status_string(2)
    assert ccu.ccu_status_string(99) == "unknown status"
    assert [ccu.ccu_route_name(r) for r in range(5)] == ["auto", "scalar", "vector", "staged", "bulk"]
    assert ccu.ccu_route_name(5) == "unknown"
    assert ccu.ccu_conv1d_abi_version() == 2
    assert ccu.ccu_conv1d_check_indices_scratch_bytes(0) == 0
    assert ccu.ccu_conv1d_check_indices_scratch_bytes(1) == 4
    assert ccu.ccu_conv1d_check_indices_scratch_bytes(32) == 4
    assert ccu.ccu_conv1d_check_indices_scratch_bytes(33) == 8


# placeholder device addresses: aligned, never dereferenced (select_route does not launch)
X, ST, WT, BS, OUT, IDX = 0x100000, 0x200000, 0x300000, 0x400000, 0x500000, 0x600000


def args(**kw):
    a = dict(x=X, ld=None, conv_state=ST, stride_s=None, stride_d=None, stride_l=None, weight=WT,
             bias=BS, act=0, indices=None, cache_seqlens=None, N=4, D=64, S=4, L=3, W=4, out=OUT)
    a.update(kw)
    if a["ld"] is None:
        a["ld"] = a["D"]
    if a["stride_s"] is None:
        a["stride_s"], a["stride_d"], a["stride_l"] = a["D"] * a["L"], a["L"], 1
    return a


def select(ccu, route=0, **kw):
    a = args(**kw)
    return ccu.ccu_conv1d_select_route(*a.values(), route)


DECLINES = [
    ("misaligned cache_seqlens", dict(cache_seqlens=0x700002), 1, "cache_seqlens must be 4-byte"),
    ("empty state", dict(W=1, L=0), 2, "empty state"),
    ("L < W-1 at width 6", dict(W=6, L=4), 1, "L must be >= W - 1"),
    ("L < W-1", dict(L=2), 1, "L must be >= W - 1"),
    ("ld < D", dict(ld=32), 1, "ld must be >= D"),
    ("padded ld not multiple of 8", dict(ld=68), 1, "multiple of 8"),
    ("act out of range", dict(act=2), 1, "act"),
    ("negative N", dict(N=-1), 1, ">= 0"),
    ("W = 0", dict(W=0), 1, "W must be >= 1"),
    ("null x", dict(x=None), 1, "NULL"),
    ("null weight", dict(weight=None), 1, "NULL"),
    ("null out", dict(out=None), 1, "NULL"),
    ("misaligned x", dict(x=X + 2), 1, "16-byte"),
    ("misaligned state", dict(conv_state=ST + 8), 1, "16-byte"),
    ("misaligned weight", dict(weight=WT + 4), 1, "16-byte"),
    ("misaligned bias", dict(bias=BS + 2), 1, "16-byte"),
    ("misaligned out", dict(out=OUT + 14), 1, "16-byte"),
    ("misaligned indices", dict(indices=IDX + 2), 1, "4-byte"),
    ("S < N without indices", dict(S=3), 1, "S must be >= N"),
    ("strides of another layout", dict(stride_s=64 * 3, stride_d=1, stride_l=128), 2, "strides"),
    ("transposed slots", dict(stride_s=3, stride_d=12, stride_l=1), 2, "strides"),
]


@pytest.mark.parametrize("name,kw,code,msg", DECLINES, ids=[d[0] for d in DECLINES])
def test_decline(ccu, name, kw, code, msg):
    st, _ = select(ccu, **kw)
    assert st == code, (name, st, ccu.ccu_conv1d_last_error())
    assert msg in ccu.ccu_conv1d_last_error()


def test_decline_from_launching_entry_points_without_gpu(ccu):
    import torch

    if torch.cuda.is_available():
        pytest.skip("launching entries are exercised with real tensors by the GPU tests")
    for name, kw, code, msg in DECLINES:
        a = args(**kw)
        assert ccu.ccu_conv1d_update(*a.values(), None) == code, name
        assert ccu.ccu_conv1d_update_checked(*a.values(), 0x800000, None) == code, name
        assert msg in ccu.ccu_conv1d_last_error()
    # a valid call cannot launch without a GPU: CUDA error, nothing else
    assert ccu.ccu_conv1d_update(*args().values(), None) == 3
    assert ccu.ccu_conv1d_update_checked(*args().values(), None, None) == 1  # NULL status word


def test_noop_sizes(ccu):
    assert select(ccu, N=0) == (0, 0)
    assert select(ccu, D=0, x=None, weight=None) == (0, 0)


def test_widths_2_and_3_are_served(ccu):
    assert select(ccu, W=3, L=2) == (0, 2)
    assert select(ccu, W=2, L=1) == (0, 2)
    assert select(ccu, W=2, L=1, D=63) == (0, 1)
    assert select(ccu, W=3, L=12) == (0, 3)
    # large compact batches take the bulk kernels, compiled for widths 2 and 3 up to L = 4
    assert select(ccu, W=3, L=2, N=1024, D=16384, S=1024) == (0, 4)
    assert select(ccu, W=3, L=2, N=4096, D=16384, S=4096) == (0, 2)  # window-only state, full batch
    assert select(ccu, W=3, L=3, N=512, D=16384, S=512) == (0, 2)
    assert select(ccu, W=3, L=3, N=4096, D=16384, S=4096) == (0, 2)
    assert select(ccu, W=2, L=2, N=4096, D=16384, S=4096) == (0, 4)
    assert select(ccu, W=2, L=4, N=4096, D=16384, S=4096) == (0, 4)
    assert select(ccu, W=2, L=1, N=4096, D=16384, S=4096) == (0, 2)  # one-entry state: vector
    assert select(ccu, W=3, L=5, N=4096, D=16384, S=4096) == (0, 2)
    assert select(ccu, route=4, W=3, L=3) == (0, 4)
    assert select(ccu, route=4, W=2, L=4) == (0, 4)
    assert select(ccu, route=4, W=3, L=5)[0] == 2
    assert select(ccu, route=4, W=3, L=2, stride_s=128, stride_d=1, stride_l=64)[0] == 2  # channel-last: width 4
    assert select(ccu, W=3, L=1)[0] == 1  # L < W - 1


def test_other_widths_run_on_the_scalar_kernel(ccu):
    # W = 1 and W > 4 are valid ("other semantically valid widths"); only the scalar kernel
    # takes them, so AUTO picks it and the 8-channel routes decline
    for W, L in [(1, 1), (1, 3), (5, 4), (6, 8), (8, 7), (16, 20)]:
        assert select(ccu, W=W, L=L) == (0, 1), (W, L)
        assert select(ccu, W=W, L=L, N=4096, D=16384, S=4096) == (0, 1), (W, L)
        assert select(ccu, W=W, L=L, cache_seqlens=0x700000) == (0, 1), (W, L)
        assert select(ccu, route=1, W=W, L=L) == (0, 1), (W, L)
        for route in (2, 3, 4):
            assert select(ccu, route=route, W=W, L=L)[0] == 2, (W, L, route)


def test_multi_and_prefill_width_declines(ccu):
    # checked before any CUDA call, so placeholder pointers are never touched
    N, D, T, S = 4, 64, 2, 4

    def multi(W, L):
        return ccu.ccu_conv1d_update_multi(X, T * D, 1, D, ST, D * L, L, 1, WT, BS, 0, None, None,
                                           N, D, T, S, L, W, OUT, T * D, 1, D, None, None, 0, None)

    def prefill(W, L):
        return ccu.ccu_causal_conv1d_fwd(X, T * D, 1, D, WT, BS, 0, None, 0, 0, 0, 1, D, T, L, W, OUT,
                                         T * D, 1, D, None, 0, 0, 0, 0, None)

    for fn in (multi, prefill):
        assert fn(1, 0) == 2 and "empty state" in ccu.ccu_conv1d_last_error()
        assert fn(6, 4) == 1 and "L must be >= W - 1" in ccu.ccu_conv1d_last_error()
        assert fn(0, 3) == 1 and "W must be >= 1" in ccu.ccu_conv1d_last_error()


def test_multi_token_bulk_route_declines(ccu):
    # The bulk-copy multi-token kernel serves width 4, the compact state at L = 3..8, T <= 8
    # and no intermediate states; a forced bulk route declines everything else before any
    # CUDA call (placeholder pointers are never touched).
    N, D = 4, 64

    def multi(T=4, L=3, W=4, layout="compact", inter=None):
        ss = (D * L, L, 1) if layout == "compact" else (L * D, 1, D)
        return ccu.ccu_conv1d_update_multi(X, T * D, 1, D, ST, *ss, WT, BS, 0, None, None,
                                           N, D, T, N, L, W, OUT, T * D, 1, D, inter, None, 4, None)

    for kw in (dict(layout="channel_last"), dict(T=9), dict(L=2, W=3), dict(W=3), dict(L=9),
               dict(inter=0x900000), dict(W=5, L=4)):
        assert multi(**kw) == 2, kw
        assert "does not serve" in ccu.ccu_conv1d_last_error()


def test_ring_buffer_state_is_served(ccu):
    assert select(ccu, cache_seqlens=0x700000) == (0, 2)
    assert select(ccu, cache_seqlens=0x700000, N=4096, D=16384, S=4096) == (0, 2)  # vector at every size
    assert select(ccu, route=4, cache_seqlens=0x700000, N=4096, D=16384, S=4096) == (0, 4)


def test_indices_allow_S_below_N(ccu):
    st, r = select(ccu, S=2, indices=IDX)
    assert st == 0 and r == 2


ROUTE_CASES = [
    ("L3 compact D%8", dict(), "vector"),
    ("L8 compact", dict(L=8), "vector"),
    ("L9 compact", dict(L=9), "staged"),
    ("L256 compact", dict(L=256), "staged"),
    ("L257 compact", dict(L=257), "scalar"),
    ("D not multiple of 8", dict(D=63), "scalar"),
    ("channel-last L3", dict(stride_s=192, stride_d=1, stride_l=64), "vector"),
    ("channel-last L12", dict(L=12, stride_s=768, stride_d=1, stride_l=64), "staged"),
    ("padded ld", dict(ld=72), "vector"),
    ("large batch compact", dict(N=4096, D=16384, S=4096), "vector"),
    ("large batch compact L4", dict(N=4096, D=16384, S=4096, L=4), "vector"),
    ("large batch compact L7", dict(N=4096, D=16384, S=4096, L=7), "bulk"),
    ("mid batch compact", dict(N=256, D=8192, S=256), "vector"),
    ("mid batch compact L7", dict(N=256, D=8192, S=256, L=7), "bulk"),
    ("below the bulk threshold", dict(N=64, D=8192, S=64), "vector"),
    ("large batch channel-last", dict(N=4096, D=16384, S=4096, stride_s=3 * 16384, stride_d=1,
                                      stride_l=16384), "vector"),
    ("mid batch channel-last", dict(N=1024, D=16384, S=1024, stride_s=3 * 16384, stride_d=1,
                                    stride_l=16384), "vector"),
    ("mid batch channel-last ring", dict(N=1024, D=16384, S=1024, stride_s=3 * 16384, stride_d=1,
                                         stride_l=16384, cache_seqlens=0x700000), "vector"),
    ("small batch channel-last", dict(N=32, D=16384, S=32, stride_s=3 * 16384, stride_d=1,
                                      stride_l=16384), "vector"),
    ("large batch L9", dict(N=4096, D=16384, S=4096, L=9), "staged"),
]


@pytest.mark.parametrize("name,kw,route", ROUTE_CASES, ids=[c[0] for c in ROUTE_CASES])
def test_auto_route(ccu, name, kw, route):
    st, r = select(ccu, **kw)
    assert st == 0, ccu.ccu_conv1d_last_error()
    assert ccu.ccu_route_name(r) == route


def test_forced_routes(ccu):
    assert select(ccu, route=1) == (0, 1)
    assert select(ccu, route=2) == (0, 2)
    assert select(ccu, route=3) == (0, 3)
    assert select(ccu, route=4) == (0, 4)
    assert select(ccu, route=4, stride_s=192, stride_d=1, stride_l=64) == (0, 4)  # both layouts
    assert select(ccu, route=4, L=9)[0] == 2  # bulk kernels are compiled for L <= 8
    assert select(ccu, route=2, D=63)[0] == 2  # vector needs D % 8 == 0
    assert select(ccu, route=2, L=9)[0] == 2   # vector is compiled for L <= 8
    assert select(ccu, route=7)[0] == 1        # unknown route


def test_check_indices_declines(ccu):
    assert ccu.ccu_conv1d_check_indices(IDX, 0, 4, None, None, None) == 0  # N == 0: no-op
    assert ccu.ccu_conv1d_check_indices(None, 4, 4, 0x900000, 0x800000, None) == 1
    assert ccu.ccu_conv1d_check_indices(IDX + 1, 4, 4, 0x900000, 0x800000, None) == 1
    assert ccu.ccu_conv1d_check_indices(IDX, -1, 4, 0x900000, 0x800000, None) == 1


def test_every_kernel_waits_for_prior_grids_first():
    """Kernels are launched as programmatic dependents: each must run
    grid_dependency_boundary() before anything else, and every launch must go through
    launch_overlapped (no triple-chevron launch that would skip the attribute)."""
    import pathlib

    csrc = pathlib.Path(ROOT) / "depthwise_causal_conv1d_gb300" / "csrc"
    kernels = 0
    for path in sorted(list(csrc.glob("*.cu")) + list(csrc.glob("*.cuh"))):
        src = path.read_text()
        assert "<<<" not in src, f"{path.name}: launch outside launch_overlapped"
        for m in re.finditer(r"__global__ void[^{;]*\{", src):
            body = src[m.end():].lstrip()
            assert body.startswith("grid_dependency_boundary();"), \
                f"{path.name}: kernel at offset {m.start()} does not wait for prior grids first"
            kernels += 1
    assert kernels >= 13


def test_auto_route_thresholds(ccu):
    """The AUTO route at the measured thresholds: linear compact batches take the bulk kernel
    from 2^20 (row, channel) elements at L = 7 and at L = 4 for widths 2 and 3; L = 3, 5, 6, 8,
    L = 1 and width 4 at L = 4 stay on the vector route at every size; width 3 with a window-only state (L = 2) takes the bulk
    kernel from 2^20 and returns to the vector kernel from 3 * 2^24; the ring state and the
    channel-last state never take the bulk kernel."""
    D = 16384
    below, at = (1 << 20) // D - 1, (1 << 20) // D  # 63 and 64 rows
    c7 = dict(L=7, stride_s=D * 7, stride_d=7, stride_l=1)
    assert select(ccu, N=below, S=below, D=D, **c7) == (0, 2)
    assert select(ccu, N=at, S=at, D=D, **c7) == (0, 4)
    for n in (below, at, 512, 513, 4096):
        assert select(ccu, N=n, S=n, D=D) == (0, 2), n
    for L in (5, 6, 8):
        for n in (at, 512, 4096):
            assert select(ccu, N=n, S=n, D=D, L=L, stride_s=D * L, stride_l=1, stride_d=L) == (0, 2), (L, n)
    assert select(ccu, N=4096, S=4096, D=D, L=7, stride_s=D * 7, stride_l=1, stride_d=7) == (0, 4)
    assert select(ccu, N=4096, S=4096, D=D, L=4, stride_s=D * 4, stride_l=1, stride_d=4) == (0, 2)
    assert select(ccu, N=4096, S=4096, D=D, W=3, L=4, stride_s=D * 4, stride_l=1, stride_d=4) == (0, 4)
    w3_below, w3_at = (3 << 24) // D - 1, (3 << 24) // D  # 3071 and 3072 rows
    assert select(ccu, N=w3_below, S=w3_below, D=D, W=3, L=2) == (0, 4)
    assert select(ccu, N=w3_at, S=w3_at, D=D, W=3, L=2) == (0, 2)
    assert select(ccu, N=512, S=512, D=D, W=3, L=3) == (0, 2)
    assert select(ccu, N=w3_at, S=w3_at, D=D, W=3, L=3) == (0, 2)
    cl = dict(stride_s=3 * D, stride_d=1, stride_l=D)
    for n in (at, 1024, w3_below, 4096):
        assert select(ccu, N=n, S=n, D=D, **cl) == (0, 2), n
        assert select(ccu, N=n, S=n, D=D, cache_seqlens=0x700000, **cl) == (0, 2), n
        assert select(ccu, N=n, S=n, D=D, cache_seqlens=0x700000) == (0, 2), n
    assert select(ccu, N=4096, S=4096, D=D, W=2, L=1) == (0, 2)


def test_checked_ex_declines(ccu):
    """The duplicate-checking update: its own argument checks run before anything is
    enqueued (placeholder pointers are never dereferenced)."""
    assert ccu.ccu_conv1d_slot_scratch_bytes(0) == 0
    assert ccu.ccu_conv1d_slot_scratch_bytes(4096) == 16384
    base = dict(x=X, ld=64, st=ST, ss=192, sd=3, sl=1, w=WT, b=None, act=0, idx=IDX, seq=None,
                N=4, D=64, S=4, L=3, W=4, out=OUT)

    def call(status, scratch, **kw):
        a = {**base, **kw}
        return ccu.ccu_conv1d_update_checked_ex(a["x"], a["ld"], a["st"], a["ss"], a["sd"], a["sl"], a["w"],
                                                a["b"], a["act"], a["idx"], a["seq"], a["N"], a["D"], a["S"],
                                                a["L"], a["W"], a["out"], status, scratch, 0, None)

    assert call(None, 0x700000) == 1            # no status word
    assert call(0x800000, None) == 1            # indices but no scratch
    assert call(0x800000, 0x700002) == 1        # scratch not 4-byte aligned
    assert call(0x800000, 0x700000, N=(1 << 31) - 1, S=(1 << 31) - 1) == 2  # rows past the row tags
    assert call(0x800000, 0x700000, N=0) == 0   # no-op
