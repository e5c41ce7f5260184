"""GPU parity: the CUDA kernels (through the C-ABI) against the CPU oracle.

Pass criteria (from the update definition on the cuDNN page "Causal Conv1d Decode
Update" and the precision reading of this library): the updated conv_state bit-exact;
the BF16 output within one BF16 ulp of the oracle (bit-exact for identity, where the
FP32 accumulation order is the same on both sides); canary guard bands around x, state
and out unchanged; unselected slots and padding rows' state untouched (part of the
full-state comparison).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import (Guarded, assert_parity, from_dev_u16, oracle_ref, ring_seqlens, run_gpu,
                      to_dev_u16)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import depthwise_causal_conv1d_gb300  # noqa: F401


def _check(inp, layout="compact", route="auto", what=""):
    want_out, want_state = oracle_ref(inp, layout)
    got_out, got_state, _, ok = run_gpu(inp, layout, route)
    assert ok, f"{what}: a guard band was overwritten"
    assert_parity(inp, got_out, got_state, want_out, want_state, what)


# ----------------------------------------------------------------------------- full workloads

@pytest.mark.parametrize("name", list(synthetic.WORKLOADS))
def test_workload_full_size(name):
    """Every workload at full size, in the launch configuration the benchmark times."""
    inp = synthetic.generate(synthetic.WORKLOADS[name])
    _check(inp, what=name)


@pytest.mark.parametrize("name", list(synthetic.WORKLOADS))
def test_workload_channel_last(name):
    wl = synthetic.WORKLOADS[name]
    if wl.N * wl.D > 4_000_000:
        wl = synthetic.variant(wl, N=256, S=max(256, wl.S // 16) if wl.indices.startswith("distinct") else 256)
    inp = synthetic.generate(wl)
    _check(inp, layout="channel_last", what=name + " channel-last")


# ----------------------------------------------------------------------------- every route

SMALL = [
    dict(N=5, D=24, L=3, S=5, act="identity", bias_std=None, indices="none"),
    dict(N=7, D=264, L=4, S=9, act="silu", bias_std=0.1, indices="distinct_pad", pad_frac=0.3),
    dict(N=33, D=2056, L=3, S=33, act="silu", bias_std=0.1, indices="perm_pad", pad_frac=0.1),
    dict(N=3, D=4104, L=8, S=3, act="identity", bias_std=None, indices="perm", ld=4112),
    dict(N=4, D=64, L=5, S=6, act="silu", bias_std=None, indices="distinct"),
    dict(N=4, D=128, L=6, S=4, act="identity", bias_std=0.1, indices="none"),
    dict(N=2, D=16, L=7, S=2, act="silu", bias_std=0.1, indices="none"),
    dict(N=6, D=520, L=9, S=8, act="silu", bias_std=0.1, indices="distinct_pad", pad_frac=0.34),
    dict(N=3, D=72, L=16, S=3, act="identity", bias_std=None, indices="perm"),
    dict(N=2, D=40, L=33, S=4, act="silu", bias_std=0.1, indices="distinct"),
]


def _small(i, **over):
    base = synthetic.WORKLOADS["decode_n8_d2048_l4_bias_silu"]
    kw = dict(SMALL[i])
    kw.setdefault("ld", kw["D"])
    kw.update(over)
    return synthetic.variant(base, name=f"small{i}", **kw)


@pytest.mark.parametrize("route", ["scalar", "vector", "staged", "bulk"])
@pytest.mark.parametrize("layout", ["compact", "channel_last"])
@pytest.mark.parametrize("i", range(len(SMALL)))
def test_routes(route, layout, i):
    wl = _small(i)
    if route in ("vector", "bulk") and wl.L > 8:
        pytest.skip("vector and bulk kernels are compiled for L <= 8")
    inp = synthetic.generate(wl, seed=100 + i)
    _check(inp, layout=layout, route=route, what=f"{wl} {route} {layout}")


# ----------------------------------------------------------------------------- sweeps

SWEEP_D = [1, 7, 8, 9, 24, 255, 256, 257, 2048, 2050, 2056, 4104]
SWEEP_N = [1, 2, 3, 33]


@pytest.mark.parametrize("D", SWEEP_D)
@pytest.mark.parametrize("L", [3, 4, 5, 8, 12])
def test_sweep_channels_and_lengths(D, L):
    # rotate N, act, bias, indices and layout with the case so all combinations appear
    k = SWEEP_D.index(D) + L
    N = SWEEP_N[k % 4]
    act = ["identity", "silu"][k % 2]
    bias = [None, 0.1][(k // 2) % 2]
    ind = ["none", "perm_pad", "distinct", "distinct_pad"][(k // 3) % 4]
    S = N if ind.startswith("perm") or ind == "none" else N + 3
    wl = synthetic.variant(synthetic.WORKLOADS["decode_n8_d2048_l4_bias_silu"], name="sweep", N=N,
                           D=D, ld=D, L=L, S=S, act=act, bias_std=bias, indices=ind, pad_frac=0.34)
    inp = synthetic.generate(wl, seed=1000 + D + L)
    for layout in ("compact", "channel_last"):
        _check(inp, layout=layout, what=f"sweep D={D} L={L} N={N} {layout}")


@pytest.mark.parametrize("D,ld", [(8, 16), (24, 32), (2050, 2056), (6144, 6152), (7, 8), (1, 8)])
def test_padded_row_stride(D, ld):
    wl = synthetic.variant(synthetic.WORKLOADS["strided_n64_d6144_ld6152_l8_perm_identity"],
                           name="ld", N=9, S=9, D=D, ld=ld)
    inp = synthetic.generate(wl, seed=7)
    assert np.all(inp.x[:, D:] == synthetic.BF16_NAN_BITS)  # canaries that must never be read
    _check(inp, what=f"ld D={D} ld={ld}")


# ----------------------------------------------------------------------------- edge cases

def test_all_rows_padding():
    wl = synthetic.variant(synthetic.WORKLOADS["paged_n256_d8192_l3_s1024_pad10_silu"], name="allpad",
                           N=16, D=512, S=64, indices="distinct_pad", pad_frac=1.0)
    inp = synthetic.generate(wl)
    assert np.all(inp.indices == -1)
    want_out, want_state = oracle_ref(inp)
    assert np.array_equal(want_state, inp.conv_state)
    got_out, got_state, _, ok = run_gpu(inp)
    assert ok and np.all(got_out == 0) and np.array_equal(got_state, inp.conv_state)


def test_empty_batch_is_a_noop():
    import depthwise_causal_conv1d_gb300 as ccu

    x = torch.zeros((0, 64), dtype=torch.bfloat16, device=DEV)
    st = torch.randn((4, 64, 3), device=DEV).to(torch.bfloat16)
    before = st.clone()
    w = torch.randn((64, 4), device=DEV).to(torch.bfloat16)
    out = ccu.causal_conv1d_update(x, st, w)
    torch.cuda.synchronize()
    assert out.shape == (0, 64) and torch.equal(st, before)
    x = torch.zeros((3, 0), dtype=torch.bfloat16, device=DEV)
    st = torch.zeros((3, 0, 3), dtype=torch.bfloat16, device=DEV)
    out = ccu.causal_conv1d_update(x, st, torch.zeros((0, 4), dtype=torch.bfloat16, device=DEV))
    assert out.shape == (3, 0)


def test_unselected_slots_untouched_large_cache():
    wl = synthetic.variant(synthetic.WORKLOADS["paged_n256_d8192_l3_s1024_pad10_silu"], name="cache",
                           N=20, D=1024, S=500)
    inp = synthetic.generate(wl, seed=3)
    _check(inp, what="S >> N")


def test_extreme_values():
    """Large magnitudes: SiLU saturates (-0/+0 and x), identity keeps big sums exact."""
    wl = synthetic.variant(synthetic.WORKLOADS["decode_n8_d2048_l4_bias_silu"], name="extreme",
                           x_dist=("normal", 60.0), w_dist=("normal", 4.0))
    for act in ("silu", "identity"):
        inp = synthetic.generate(dataclasses.replace(wl, act=act), seed=11)
        _check(inp, what=f"extreme {act}")


def _every_finite_bf16():
    bits = np.arange(1 << 16, dtype=np.uint32)
    return bits[((bits >> 7) & 0xFF) != 0xFF].astype(np.uint16)  # 65280 values, +-0 included


@pytest.mark.parametrize("path", ["scalar", "vector", "staged", "bulk", "multi", "multi_bulk",
                                  "prefill_vector", "prefill_bulk"])
def test_silu_every_finite_bf16_input(path):
    """SiLU of every finite BF16 value (subnormals, +-0, both tails) through each kernel
    family: weights (0, 0, 0, 1), a zero state and no bias make the accumulator equal x, so
    out = silu(x); within 1 BF16 ulp of the oracle's double-precision SiLU."""
    import depthwise_causal_conv1d_gb300 as ccu
    from oracle_pins import bf16_ulp_distance

    vals = _every_finite_bf16()
    D = vals.size
    weight = np.zeros((D, 4), np.uint16)
    weight[:, 3] = 0x3F80  # 1.0
    want = oracle.conv1d_update(vals.reshape(1, D), D, np.zeros((1, D, 3), np.uint16), (3 * D, 3, 1),
                                weight, None, "silu", None, 1, D, 1, 3, 4)[0]
    w = to_dev_u16(weight, DEV)
    x2 = np.stack([vals, vals[::-1]])  # two tokens / two rows
    want2 = np.stack([want, want[::-1]])
    if path in ("scalar", "vector", "staged", "bulk"):
        st = torch.zeros((2, D, 3), dtype=torch.bfloat16, device=DEV)
        got = ccu.causal_conv1d_update(to_dev_u16(x2, DEV), st, w, None, "silu", route=path)
    elif path in ("multi", "multi_bulk"):
        st = torch.zeros((1, D, 3), dtype=torch.bfloat16, device=DEV)
        got = ccu.causal_conv1d_update(to_dev_u16(x2[None], DEV).permute(0, 2, 1), st, w, None, "silu",
                                       route="bulk" if path == "multi_bulk" else "auto")
        got = got.permute(0, 2, 1)[0]
    else:
        x = to_dev_u16(x2[None], DEV).permute(0, 2, 1)  # [1, D, 2], token-major memory
        got = ccu.causal_conv1d_fwd(x, w, None, "silu", route=path.split("_")[1])
        got = got.permute(0, 2, 1)[0]
    torch.cuda.synchronize()
    dist = bf16_ulp_distance(from_dev_u16(got), want2)
    assert dist.max() <= 1, vals[np.argmax(dist.max(axis=0))]



@pytest.mark.parametrize("L,act,layout", [(3, "identity", "compact"), (3, "silu", "channel_last"),
                                          (4, "silu", "compact"), (8, "identity", "channel_last"),
                                          (10, "silu", "compact")])
def test_chained_decode_equals_full_convolution(L, act, layout):
    """T GPU updates from a seeded state equal one full causal convolution of the sequence."""
    import depthwise_causal_conv1d_gb300 as ccu

    rng = np.random.default_rng(L)
    T, D = 16, 264
    x_seq = synthetic.f64_to_bf16_bits(rng.standard_normal((T, D)))
    weight = synthetic.f64_to_bf16_bits(rng.standard_normal((D, 4)) * 0.5)
    bias = synthetic.f64_to_bf16_bits(rng.standard_normal(D) * 0.1)
    init = synthetic.f64_to_bf16_bits(rng.standard_normal((D, L)))
    want_y, want_state = oracle.full_causal_conv(x_seq, weight, bias, act, init, L)
    w, b = to_dev_u16(weight, DEV), to_dev_u16(bias, DEV)
    if layout == "compact":
        st = to_dev_u16(init.reshape(1, D, L), DEV)
    else:
        st = to_dev_u16(np.ascontiguousarray(init.T).reshape(1, L, D), DEV).permute(0, 2, 1)
    ys = []
    for t in range(T):
        xt = to_dev_u16(x_seq[t:t + 1], DEV)
        ys.append(from_dev_u16(ccu.causal_conv1d_update(xt, st, w, b, act)))
    got_y = np.concatenate(ys)
    got_state = from_dev_u16(st.contiguous())[0]
    assert np.array_equal(got_state, want_state)
    from oracle_pins import bf16_ulp_distance

    assert bf16_ulp_distance(got_y, want_y).max() <= (0 if act == "identity" else 1)


# ----------------------------------------------------------------------------- behaviour

def test_deterministic():
    inp = synthetic.generate(synthetic.WORKLOADS["paged_n256_d8192_l3_s1024_pad10_silu"])
    a = run_gpu(inp)
    b = run_gpu(inp)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_side_stream_with_default_stream_parked():
    """The op runs on the ambient stream: with the default stream busy, a side stream's
    result is complete when that side stream alone is synchronized."""
    import depthwise_causal_conv1d_gb300 as ccu

    inp = synthetic.generate(synthetic.WORKLOADS["paged_n256_d8192_l3_s1024_pad10_silu"])
    want_out, want_state = oracle_ref(inp)
    x, st = to_dev_u16(inp.x, DEV), to_dev_u16(inp.conv_state, DEV)
    w, b = to_dev_u16(inp.weight, DEV), to_dev_u16(inp.bias, DEV)
    idx = torch.from_numpy(inp.indices).to(DEV)
    out = torch.empty((inp.wl.N, inp.wl.D), dtype=torch.bfloat16, device=DEV)
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    host_state = torch.empty(st.shape, dtype=st.dtype, pin_memory=True)
    side = torch.cuda.Stream()
    # A process's first call of a kernel loads its module and sets its attributes, which may
    # synchronize the device: make that call (on copies) before the default stream is parked.
    warm_out, warm_st = torch.empty_like(out), st.clone()
    with torch.cuda.stream(side):
        ccu.causal_conv1d_update(x, warm_st, w, b, "silu", conv_state_indices=idx, out=warm_out)
    torch.cuda.synchronize()
    # nothing below allocates device or pinned memory, which could synchronize the device
    torch.cuda._sleep(200_000_000)  # parks the default stream for ~0.1 s (bounded spin)
    with torch.cuda.stream(side):
        ccu.causal_conv1d_update(x, st, w, b, "silu", conv_state_indices=idx, out=out)
        host_out.copy_(out, non_blocking=True)
        host_state.copy_(st, non_blocking=True)
    side.synchronize()
    default_busy = not torch.cuda.default_stream().query()
    got_out = host_out.view(torch.int16).numpy().view(np.uint16)
    got_state = host_state.view(torch.int16).numpy().view(np.uint16)
    torch.cuda.synchronize()
    assert default_busy, "the default stream finished first: the test did not park it"
    assert_parity(inp, got_out, got_state, want_out, want_state, "side stream")


def test_cuda_graph_replay_matches_eager():
    import depthwise_causal_conv1d_gb300 as ccu

    inp = synthetic.generate(synthetic.WORKLOADS["strided_n64_d6144_ld6152_l8_perm_identity"])
    wl = inp.wl

    def setup():
        x = to_dev_u16(inp.x, DEV)[:, :wl.D]
        st = to_dev_u16(inp.conv_state, DEV)
        w = to_dev_u16(inp.weight, DEV)
        idx = torch.from_numpy(inp.indices).to(DEV)
        out = torch.empty((wl.N, wl.D), dtype=torch.bfloat16, device=DEV)
        return x, st, w, idx, out

    steps = 5
    x, st, w, idx, out = setup()
    eager = []
    for _ in range(steps):
        ccu.causal_conv1d_update(x, st, w, None, "identity", conv_state_indices=idx, out=out)
        eager.append(out.clone())
    eager_state = st.clone()

    x, st, w, idx, out = setup()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm the exact signature before capture
        ccu.causal_conv1d_update(x, st, w, None, "identity", conv_state_indices=idx, out=out)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    x, st2, w, idx, out = setup()
    st.copy_(st2)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ccu.causal_conv1d_update(x, st, w, None, "identity", conv_state_indices=idx, out=out)
    graphed = []
    for _ in range(steps):
        g.replay()
        graphed.append(out.clone())
    torch.cuda.synchronize()
    for a, b in zip(eager, graphed):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(eager_state.view(torch.int16), st.view(torch.int16))


def test_cuda_graph_checked_update_with_duplicates():
    """The range- and duplicate-checked update captured in a CUDA graph: the clearing of the
    slot scratch is part of the captured work, so every replay finds the duplicate and the
    out-of-range row from a dirty scratch, and its status, outputs and state equal the
    oracle's update with the losing row (read back from the scratch) as padding."""
    import depthwise_causal_conv1d_gb300 as ccu

    wl = synthetic.variant(synthetic.WORKLOADS["paged_n256_d8192_l3_s1024_pad10_silu"], name="graph_dedup",
                           N=96, D=2048, ld=2048, S=128)
    inp = synthetic.generate(wl, seed=17)
    idx = inp.indices.copy()
    active = np.flatnonzero(idx >= 0)
    pair = [active[4], active[40]]
    idx[pair[0]] = idx[pair[1]]  # a repeated slot
    idx[active[7]] = wl.S  # out of range
    want_status = oracle.check_indices(idx, wl.N, wl.S)

    x = to_dev_u16(inp.x, DEV)[:, :wl.D]
    w = to_dev_u16(inp.weight, DEV)
    b = to_dev_u16(inp.bias, DEV)
    idx_dev = torch.from_numpy(idx).to(DEV)
    st0 = to_dev_u16(inp.conv_state, DEV)
    state = st0.clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    scratch = torch.full((wl.S,), 7, dtype=torch.int32, device=DEV)
    out = torch.empty((wl.N, wl.D), dtype=torch.bfloat16, device=DEV)

    def run():
        ccu.causal_conv1d_update(x, state, w, b, "silu", conv_state_indices=idx_dev, out=out, status=status,
                                 slot_scratch=scratch)

    def check(what):
        assert int(status.item()) == want_status, what
        owners = scratch.cpu().numpy()
        winner = owners[idx[pair[0]]] - 1
        assert winner in pair, (what, winner)
        ref_idx = idx.copy()
        ref_idx[idx >= wl.S] = -1
        ref_idx[[r for r in pair if r != winner]] = -1
        want_out, want_state = oracle_ref(dataclasses.replace(inp, indices=ref_idx))
        assert_parity(inp, from_dev_u16(out), from_dev_u16(state), want_out, want_state, what)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # the eager call, which also warms the signature before capture
        run()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    check("eager")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for k in range(3):
        state.copy_(st0)
        status.zero_()
        scratch.fill_(7)  # dirty scratch: the captured clear must run
        g.replay()
        torch.cuda.synchronize()
        check(f"replay {k}")


def test_cuda_graph_multi_token_bulk_ring():
    """Multi-token calls on the bulk-copy kernel (AUTO, compact ring state at L = 5) captured
    in a CUDA graph: each replay from the same starting state equals the eager calls bit for
    bit."""
    import depthwise_causal_conv1d_gb300 as ccu

    rng = np.random.default_rng(23)
    N, D, T, L = 384, 2048, 4, 5
    x = to_dev_u16(synthetic.f64_to_bf16_bits(rng.standard_normal((N, T, D))), DEV).permute(0, 2, 1)
    w = to_dev_u16(synthetic.f64_to_bf16_bits(rng.standard_normal((D, 4)) * 0.5), DEV)
    b = to_dev_u16(synthetic.f64_to_bf16_bits(rng.standard_normal(D) * 0.1), DEV)
    st0 = to_dev_u16(synthetic.f64_to_bf16_bits(rng.standard_normal((N, D, L))), DEV)
    idx = torch.from_numpy(rng.permutation(N).astype(np.int32)).to(DEV)
    seq = torch.from_numpy(rng.integers(0, 1000, N).astype(np.int32)).to(DEV)

    def calls(st, y0, y1):
        ccu.causal_conv1d_update(x, st, w, b, "silu", conv_state_indices=idx, cache_seqlens=seq, out=y0)
        ccu.causal_conv1d_update(x, st, w, b, "silu", conv_state_indices=idx, cache_seqlens=seq + T, out=y1)

    eager = (st0.clone(), torch.empty_like(x), torch.empty_like(x))
    calls(*eager)
    torch.cuda.synchronize()
    graphed = (st0.clone(), torch.empty_like(x), torch.empty_like(x))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # the first launch sets the kernel's shared-memory limit
        calls(*graphed)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    seq_next = seq + T  # allocated outside the capture
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ccu.causal_conv1d_update(x, graphed[0], w, b, "silu", conv_state_indices=idx, cache_seqlens=seq,
                                 out=graphed[1])
        ccu.causal_conv1d_update(x, graphed[0], w, b, "silu", conv_state_indices=idx, cache_seqlens=seq_next,
                                 out=graphed[2])
    for _ in range(3):
        graphed[0].copy_(st0)
        graphed[1].zero_()
        graphed[2].zero_()
        g.replay()
        torch.cuda.synchronize()
        for a, c in zip(eager, graphed):
            assert torch.equal(a.contiguous().view(torch.int16), c.contiguous().view(torch.int16))


def test_cuda_graph_prefill_multi_decode_sequence():
    """One CUDA graph holding a serving sequence on one state: a bulk prefill that writes the
    channel-last hand-off state, a multi-token update and a (bulk) decode step. Every replay
    restarts from the prefill's state and equals the eager sequence bit for bit."""
    import depthwise_causal_conv1d_gb300 as ccu

    rng = np.random.default_rng(21)
    B, T, D, L = 512, 16, 2048, 3
    assert B * T * D >= 1 << 20 and B * D >= 1 << 20  # prefill and decode take the bulk kernels
    x_pre = to_dev_u16(synthetic.f64_to_bf16_bits(rng.standard_normal((B, T, D))), DEV).permute(0, 2, 1)
    x_multi = to_dev_u16(synthetic.f64_to_bf16_bits(rng.standard_normal((B, 4, D))), DEV).permute(0, 2, 1)
    x_dec = to_dev_u16(synthetic.f64_to_bf16_bits(rng.standard_normal((B, D))), DEV)
    w = to_dev_u16(synthetic.f64_to_bf16_bits(rng.standard_normal((D, 4)) * 0.5), DEV)
    b = to_dev_u16(synthetic.f64_to_bf16_bits(rng.standard_normal(D) * 0.1), DEV)

    def buffers():
        return (torch.empty((B, L, D), dtype=torch.bfloat16, device=DEV).permute(0, 2, 1),
                torch.empty_like(x_pre), torch.empty_like(x_multi), torch.empty_like(x_dec))

    def sequence(fin, y0, y1, y2):
        ccu.causal_conv1d_fwd(x_pre, w, b, "silu", final_states_out=fin, out=y0)
        ccu.causal_conv1d_update(x_multi, fin, w, b, "silu", out=y1)
        ccu.causal_conv1d_update(x_dec, fin, w, b, "silu", out=y2)

    eager = buffers()
    sequence(*eager)
    torch.cuda.synchronize()

    graphed = buffers()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm the exact signatures before capture
        sequence(*graphed)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sequence(*graphed)
    for _ in range(3):
        for t in graphed:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for a, c in zip(eager, graphed):
            assert torch.equal(a.contiguous().view(torch.int16), c.contiguous().view(torch.int16))


def test_side_stream_prefill_and_multi_token():
    """Prefill (bulk) and a multi-token update issued on a side stream while the default
    stream is parked: complete and correct when the side stream alone is synchronized."""
    import depthwise_causal_conv1d_gb300 as ccu
    from oracle_pins import bf16_ulp_distance

    rng = np.random.default_rng(23)
    B, T, D, L, K = 4, 300, 1024, 3, 3
    x_all = synthetic.f64_to_bf16_bits(rng.standard_normal((B, T + K, D)))
    weight = synthetic.f64_to_bf16_bits(rng.standard_normal((D, 4)) * 0.5)
    bias = synthetic.f64_to_bf16_bits(rng.standard_normal(D) * 0.1)
    x_pre = to_dev_u16(np.ascontiguousarray(x_all[:, :T]), DEV).permute(0, 2, 1)
    x_multi = to_dev_u16(np.ascontiguousarray(x_all[:, T:]), DEV).permute(0, 2, 1)
    w, b = to_dev_u16(weight, DEV), to_dev_u16(bias, DEV)
    fin = torch.empty((B, L, D), dtype=torch.bfloat16, device=DEV).permute(0, 2, 1)
    y_pre, y_multi = torch.empty_like(x_pre), torch.empty_like(x_multi)
    h_pre = torch.empty((B, T, D), dtype=torch.bfloat16, pin_memory=True)
    h_multi = torch.empty((B, K, D), dtype=torch.bfloat16, pin_memory=True)
    side = torch.cuda.Stream()
    # first calls of these kernels (module load, attributes) before the default stream is parked
    fin_w, y_pre_w, y_multi_w = torch.empty_like(fin), torch.empty_like(y_pre), torch.empty_like(y_multi)
    with torch.cuda.stream(side):
        ccu.causal_conv1d_fwd(x_pre, w, b, "silu", final_states_out=fin_w, out=y_pre_w, route="bulk")
        ccu.causal_conv1d_update(x_multi, fin_w, w, b, "silu", out=y_multi_w)
    torch.cuda.synchronize()
    torch.cuda._sleep(200_000_000)  # parks the default stream for ~0.1 s (bounded spin)
    with torch.cuda.stream(side):
        ccu.causal_conv1d_fwd(x_pre, w, b, "silu", final_states_out=fin, out=y_pre, route="bulk")
        ccu.causal_conv1d_update(x_multi, fin, w, b, "silu", out=y_multi)
        h_pre.copy_(y_pre.permute(0, 2, 1), non_blocking=True)
        h_multi.copy_(y_multi.permute(0, 2, 1), non_blocking=True)
    side.synchronize()
    default_busy = not torch.cuda.default_stream().query()
    got = np.concatenate([h_pre.view(torch.int16).numpy().view(np.uint16),
                          h_multi.view(torch.int16).numpy().view(np.uint16)], axis=1)
    torch.cuda.synchronize()
    assert default_busy, "the default stream finished first: the test did not park it"
    for bb in range(B):
        want, _ = oracle.full_causal_conv(x_all[bb], weight, bias, "silu", None, L)
        assert bf16_ulp_distance(got[bb], want).max() <= 1, bb


# ----------------------------------------------------------------------------- checked path

@pytest.mark.parametrize("route", ["scalar", "vector", "staged", "bulk"])
def test_checked_path_flags_bad_slots_without_trapping(route):
    wl = synthetic.variant(synthetic.WORKLOADS["paged_n256_d8192_l3_s1024_pad10_silu"], name="chk",
                           N=12, D=1024, S=16, indices="distinct_pad", pad_frac=0.2)
    inp = synthetic.generate(wl, seed=5)
    bad_rows = [1, 4, 9]
    bad_vals = [-2, wl.S, 10 ** 6]
    idx = inp.indices.copy()
    for r, v in zip(bad_rows, bad_vals):
        idx[r] = v
    # the oracle's view: bad rows behave as padding rows (zero output, no state access)
    ref_idx = idx.copy()
    ref_idx[bad_rows] = -1
    want_out, want_state = oracle_ref(dataclasses.replace(inp, indices=ref_idx))
    got_out, got_state, status, ok = run_gpu(dataclasses.replace(inp, indices=idx), route=route,
                                             checked=True)
    assert ok
    assert status & 1, "range error not reported"
    assert_parity(inp, got_out, got_state, want_out, want_state, "checked")
    # the context is still usable
    got_out2, _, status2, _ = run_gpu(inp, checked=True)
    assert status2 == 0


def test_checked_path_clean_inputs_report_nothing():
    inp = synthetic.generate(synthetic.WORKLOADS["paged_n256_d8192_l3_s1024_pad10_silu"])
    want_out, want_state = oracle_ref(inp)
    got_out, got_state, status, ok = run_gpu(inp, checked=True)
    assert ok and status == 0
    assert_parity(inp, got_out, got_state, want_out, want_state, "checked clean")


DEDUP_CASES = ["valid", "duplicate", "range", "padding_only", "both"]


@pytest.mark.parametrize("case", DEDUP_CASES)
@pytest.mark.parametrize("layout", ["compact", "channel_last"])
@pytest.mark.parametrize("route", ["scalar", "vector", "staged", "bulk"])
def test_checked_update_detects_duplicates_in_the_same_launch(route, layout, case):
    """ccu_conv1d_update_checked_ex: the status bits equal the oracle's index check; a row
    whose slot is out of range or was claimed by another row behaves as a padding row; of
    the rows sharing a slot exactly one updated it (the winner, read back from the slot
    scratch), so output and state equal the oracle's update with the losers as padding."""
    wl = synthetic.variant(synthetic.WORKLOADS["paged_n256_d8192_l3_s1024_pad10_silu"], name="dedup",
                           N=40, D=1032, ld=1032, S=64, indices="distinct_pad", pad_frac=0.1)
    inp = synthetic.generate(wl, seed=31 + DEDUP_CASES.index(case))
    idx = inp.indices.copy()
    active = np.flatnonzero(idx >= 0)
    groups = []
    if case in ("duplicate", "both"):
        groups = [[active[2], active[17], active[30]], [active[5], active[6]]]
        for g in groups:
            idx[g] = idx[g[0]]
    if case in ("range", "both"):
        idx[active[9]] = -2
        idx[active[12]] = wl.S
    if case == "padding_only":
        idx[:] = -1
    want_status = oracle.check_indices(idx, wl.N, wl.S)
    scratch = torch.full((wl.S,), 12345, dtype=torch.int32, device=DEV)  # dirty: the call clears it
    got_out, got_state, status, ok = run_gpu(dataclasses.replace(inp, indices=idx), layout=layout, route=route,
                                             checked=True, slot_scratch=scratch)
    assert ok, "a guard band was overwritten"
    assert status == want_status, (status, want_status)
    owners = scratch.cpu().numpy()
    ref_idx = idx.copy()
    ref_idx[(idx < -1) | (idx >= wl.S)] = -1
    for g in groups:
        winner = owners[idx[g[0]]] - 1
        assert winner in g, (winner, g)
        ref_idx[[r for r in g if r != winner]] = -1
    for n in np.flatnonzero(ref_idx >= 0):
        assert owners[ref_idx[n]] == n + 1
    assert np.count_nonzero(owners) == np.count_nonzero(ref_idx >= 0)
    want_out, want_state = oracle_ref(dataclasses.replace(inp, indices=ref_idx), layout)
    assert_parity(inp, got_out, got_state, want_out, want_state, f"dedup {route} {layout} {case}")


@pytest.mark.parametrize("case", ["duplicate", "both"])
@pytest.mark.parametrize("route,W", [("vector", 2), ("vector", 3), ("vector", 4), ("bulk", 4)])
def test_checked_update_detects_duplicates_at_l8(route, W, case):
    """The duplicate check at L = 8, where the vector route runs one channel per lane: as
    test_checked_update_detects_duplicates_in_the_same_launch, on a ragged D (not a multiple
    of the 2048 channels a CTA covers) and a padded x row stride."""
    wl = synthetic.variant(synthetic.WORKLOADS["strided_n64_d6144_ld6152_l8_perm_identity"], name="dedup8",
                           N=40, D=2056, ld=2064, S=64, W=W, indices="distinct_pad", pad_frac=0.1,
                           act="silu", bias_std=0.1)
    inp = synthetic.generate(wl, seed=71 + W)
    idx = inp.indices.copy()
    active = np.flatnonzero(idx >= 0)
    groups = [[active[2], active[17], active[30]], [active[5], active[6]]]
    for g in groups:
        idx[g] = idx[g[0]]
    if case == "both":
        idx[active[9]] = -2
        idx[active[12]] = wl.S
    want_status = oracle.check_indices(idx, wl.N, wl.S)
    scratch = torch.full((wl.S,), 12345, dtype=torch.int32, device=DEV)
    got_out, got_state, status, ok = run_gpu(dataclasses.replace(inp, indices=idx), route=route, checked=True,
                                             slot_scratch=scratch)
    assert ok, "a guard band was overwritten"
    assert status == want_status, (status, want_status)
    owners = scratch.cpu().numpy()
    ref_idx = idx.copy()
    ref_idx[(idx < -1) | (idx >= wl.S)] = -1
    for g in groups:
        winner = owners[idx[g[0]]] - 1
        assert winner in g, (winner, g)
        ref_idx[[r for r in g if r != winner]] = -1
    want_out, want_state = oracle_ref(dataclasses.replace(inp, indices=ref_idx))
    assert_parity(inp, got_out, got_state, want_out, want_state, f"dedup L8 {route} {case} W{W}")


def _two_row_batch():
    """A row count at which the vector route's small-batch two-row form runs at D = 8192
    (1024 channels per CTA): between six and eight (row, channel block) pairs per SM, odd,
    so the last CTA holds one row."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return (7 * sms) // 4 | 1


@pytest.mark.parametrize("case", ["unchecked", "duplicate"])
def test_small_batch_two_row_form(case):
    """The two-rows-in-flight form of the vector kernel (compact linear L = 3, width 4, small
    batches): bit-exact state and 1-ulp outputs against the oracle with padding rows, and in
    the checked update the duplicate check of test_checked_update_detects_duplicates_in_the_same_launch."""
    N = _two_row_batch()
    wl = synthetic.variant(synthetic.WORKLOADS["paged_n256_d8192_l3_s1024_pad10_silu"], name="two_row", N=N)
    inp = synthetic.generate(wl, seed=91)
    if case == "unchecked":
        _check(inp, route="vector", what=f"two-row N={N}")
        return
    idx = inp.indices.copy()
    active = np.flatnonzero(idx >= 0)
    groups = [[active[3], active[len(active) // 2], active[-1]], [active[7], active[8]]]
    for g in groups:
        idx[g] = idx[g[0]]
    want_status = oracle.check_indices(idx, wl.N, wl.S)
    scratch = torch.full((wl.S,), 12345, dtype=torch.int32, device=DEV)
    got_out, got_state, status, ok = run_gpu(dataclasses.replace(inp, indices=idx), route="vector", checked=True,
                                             slot_scratch=scratch)
    assert ok, "a guard band was overwritten"
    assert status == want_status, (status, want_status)
    owners = scratch.cpu().numpy()
    ref_idx = idx.copy()
    for g in groups:
        winner = owners[idx[g[0]]] - 1
        assert winner in g, (winner, g)
        ref_idx[[r for r in g if r != winner]] = -1
    want_out, want_state = oracle_ref(dataclasses.replace(inp, indices=ref_idx))
    assert_parity(inp, got_out, got_state, want_out, want_state, f"two-row dedup N={N}")


@pytest.mark.parametrize("layout", ["compact", "channel_last"])
@pytest.mark.parametrize("route", ["vector", "bulk"])
def test_large_batch_routes_agree_bitwise(route, layout):
    """The two large-batch kernel families give bit-identical results on a multi-tile case
    with a ragged last chunk (D = 3*2048 + 264) and padding rows."""
    wl = synthetic.variant(synthetic.WORKLOADS[synthetic.BENCH_WORKLOAD], name="ragged", N=300, S=300,
                           D=6408, ld=6408)
    inp = synthetic.generate(wl, seed=21)
    _check(inp, layout=layout, route=route, what=f"ragged {route} {layout}")


def test_no_device_error_raised():
    import depthwise_causal_conv1d_gb300 as ccu

    inp = synthetic.generate(synthetic.WORKLOADS[synthetic.BENCH_WORKLOAD])
    run_gpu(inp, route="bulk", guards=False)
    st, bits = ccu.ccu_conv1d_take_device_error()
    assert st == 0 and bits == 0


@pytest.mark.parametrize("case", ["valid", "padding", "range_low", "range_high", "duplicate", "both"])
def test_check_indices_matches_oracle(case):
    import depthwise_causal_conv1d_gb300 as ccu

    rng = np.random.default_rng(["valid", "padding", "range_low", "range_high", "duplicate",
                                 "both"].index(case))
    S, N = 4099, 3000
    idx = rng.permutation(S)[:N].astype(np.int32)
    if case == "padding":
        idx[::7] = -1
    elif case == "range_low":
        idx[17] = -5
    elif case == "range_high":
        idx[100] = S
    elif case == "duplicate":
        idx[2999] = idx[0]
    elif case == "both":
        idx[5] = idx[6]
        idx[7] = S + 10
    want = oracle.check_indices(idx, N, S)
    dev_idx = torch.from_numpy(idx).to(DEV)
    status = torch.zeros((1,), dtype=torch.int32, device=DEV)
    scratch = torch.full((ccu.ccu_conv1d_check_indices_scratch_bytes(S) // 4,), -1, dtype=torch.int32,
                         device=DEV)  # dirty on purpose: the call clears it
    for _ in range(2):
        ccu.check_indices(dev_idx, S, status=status, scratch=scratch)
    assert int(status.item()) == want


# ----------------------------------------------------------------------------- declines (typed)

def test_typed_declines_through_binding():
    import depthwise_causal_conv1d_gb300 as ccu

    x = torch.randn((4, 64), device=DEV).to(torch.bfloat16)
    st = torch.randn((4, 64, 3), device=DEV).to(torch.bfloat16)
    w = torch.randn((64, 4), device=DEV).to(torch.bfloat16)
    seq = torch.zeros((4,), dtype=torch.int32, device=DEV)
    with pytest.raises(ValueError, match="cache_seqlens"):
        ccu.causal_conv1d_update(x, st, w, cache_seqlens=seq[:3])
    with pytest.raises(ValueError, match="2D"):
        ccu.causal_conv1d_update(x.view(4, 64, 1, 1), st, w)
    with pytest.raises(ValueError, match="intermediate_states"):
        ccu.causal_conv1d_update(x, st, w, intermediate_states=torch.empty((4, 1, 64, 3), dtype=torch.bfloat16, device=DEV))
    with pytest.raises(NotImplementedError, match="empty state"):
        ccu.causal_conv1d_update(x, torch.empty((4, 64, 0), device=DEV, dtype=torch.bfloat16),
                                 torch.randn((64, 1), device=DEV).to(torch.bfloat16))
    with pytest.raises(NotImplementedError, match="does not serve"):
        ccu.causal_conv1d_update(x, torch.randn((4, 64, 4), device=DEV).to(torch.bfloat16),
                                 torch.randn((64, 5), device=DEV).to(torch.bfloat16), route="vector")
    with pytest.raises(ValueError, match="L must be >= W - 1"):
        ccu.causal_conv1d_update(x, st[:, :, :2].contiguous(), w)
    base = torch.randn((4 * 72 + 8,), device=DEV).to(torch.bfloat16)
    with pytest.raises(ValueError, match="16-byte"):
        ccu.causal_conv1d_update(base[1:1 + 4 * 72].view(4, 72)[:, :64], st, w)
    with pytest.raises(ValueError, match="multiple of 8"):
        ccu.causal_conv1d_update(torch.randn((4, 68), device=DEV).to(torch.bfloat16)[:, :64], st, w)
    with pytest.raises(ValueError, match="autograd"):
        ccu.causal_conv1d_update(x.clone().requires_grad_(), st, w)
    with pytest.raises(NotImplementedError, match="strides"):
        ccu.causal_conv1d_update(x, torch.randn((64, 4, 3), device=DEV).to(torch.bfloat16).transpose(0, 1), w)
    with pytest.raises(ValueError, match="activation"):
        ccu.causal_conv1d_update(x, st, w, activation="gelu")
    with pytest.raises(ValueError, match="S must be >= N"):
        ccu.causal_conv1d_update(x, st[:3].contiguous(), w)
    # nothing was launched by any decline
    torch.cuda.synchronize()


# ----------------------------------------------------------------------------- host buffers

def test_host_resident_x_and_out():
    """x and out in pinned host memory, read and written by the kernel in place."""
    import depthwise_causal_conv1d_gb300 as ccu

    wl = synthetic.variant(synthetic.WORKLOADS[synthetic.BENCH_WORKLOAD], name="hostio", N=520, S=520)
    assert wl.N * wl.D >= 1 << 22  # large enough that device operands would take the bulk route
    inp = synthetic.generate(wl, seed=33)
    want_out, want_state = oracle_ref(inp)
    h_x = torch.from_numpy(inp.x.view(np.int16)).pin_memory()
    h_out = torch.full((wl.N, wl.D), -1, dtype=torch.int16).pin_memory()
    st = to_dev_u16(inp.conv_state, DEV)
    w, b = to_dev_u16(inp.weight, DEV), to_dev_u16(inp.bias, DEV)
    idx = torch.from_numpy(inp.indices).to(DEV)
    stream = torch.cuda.current_stream().cuda_stream
    args = (h_x.data_ptr(), wl.ld, st.data_ptr(), wl.D * wl.L, wl.L, 1, w.data_ptr(), b.data_ptr(),
            ccu.CCU_ACT_SILU, idx.data_ptr(), None, wl.N, wl.D, wl.S, wl.L, wl.W, h_out.data_ptr())
    # a forced bulk route declines host operands; nothing is launched
    assert ccu.ccu_conv1d_update_ex(*args, None, ccu.ROUTES["bulk"], stream) == ccu.CCU_ERR_NOT_IMPLEMENTED
    assert ccu.ccu_conv1d_update(*args, stream) == 0, ccu.ccu_conv1d_last_error()
    torch.cuda.synchronize()
    got_out = h_out.numpy().view(np.uint16)
    got_state = from_dev_u16(st)
    assert_parity(inp, got_out, got_state, want_out, want_state, "host x/out")


# ----------------------------------------------------------------------------- ring-buffer state

def _check_ring(inp, seq, layout="compact", route="auto", what=""):
    want_out, want_state = oracle_ref(inp, layout, cache_seqlens=seq)
    got_out, got_state, _, ok = run_gpu(inp, layout, route, cache_seqlens=seq)
    assert ok, f"{what}: a guard band was overwritten"
    assert_parity(inp, got_out, got_state, want_out, want_state, what)


@pytest.mark.parametrize("case", ["unchecked", "duplicate"])
@pytest.mark.parametrize("N", [401, 4900])
def test_ring_channel_last_two_rows(N, case):
    """The channel-last ring state on the vector kernel once the batch fills the GPU: two
    rows in flight, four (N=401) or six (N=4900) rows per CTA, a ragged last CTA and a ragged
    D; bit-exact state and 1-ulp outputs, and with the duplicate check the losing rows as
    padding."""
    wl = synthetic.variant(synthetic.RING_WORKLOADS["large_n4096_d16384_l3_perm_pad5_silu_ring_chlast"],
                           name="ring_chlast_two_rows", N=N, S=N + 3, D=6408, ld=6408,
                           indices="distinct_pad")
    inp = synthetic.generate(wl, seed=61)
    seq = ring_seqlens(np.random.default_rng(62), inp)
    if case == "unchecked":
        _check_ring(inp, seq, layout="channel_last", route="vector", what=f"ring chlast two rows N={N}")
        return
    idx = inp.indices.copy()
    active = np.flatnonzero(idx >= 0)
    pair = [active[3], active[len(active) // 2]]
    idx[pair[0]] = idx[pair[1]]
    inp = dataclasses.replace(inp, indices=idx)
    seq[pair[0]] = seq[pair[1]]
    scratch = torch.full((wl.S,), 9, dtype=torch.int32, device=DEV)
    got_out, got_state, status, ok = run_gpu(inp, "channel_last", "vector", checked=True, cache_seqlens=seq,
                                             slot_scratch=scratch)
    assert ok, "a guard band was overwritten"
    assert status == oracle.check_indices(idx, wl.N, wl.S)
    winner = scratch.cpu().numpy()[idx[pair[0]]] - 1
    assert winner in pair
    ref_idx = idx.copy()
    ref_idx[[r for r in pair if r != winner]] = -1
    want_out, want_state = oracle_ref(dataclasses.replace(inp, indices=ref_idx), "channel_last", cache_seqlens=seq)
    assert_parity(inp, got_out, got_state, want_out, want_state, f"ring chlast two rows dedup N={N}")


@pytest.mark.parametrize("route", ["scalar", "vector", "staged", "bulk"])
@pytest.mark.parametrize("layout", ["compact", "channel_last"])
@pytest.mark.parametrize("i", range(len(SMALL)))
def test_ring_routes(route, layout, i):
    wl = _small(i)
    if route in ("vector", "bulk") and wl.L > 8:
        pytest.skip("vector and bulk kernels are compiled for L <= 8")
    inp = synthetic.generate(wl, seed=200 + i)
    seq = ring_seqlens(np.random.default_rng(i), inp)
    _check_ring(inp, seq, layout, route, what=f"ring {wl} {route} {layout}")


@pytest.mark.parametrize("layout", ["compact", "channel_last"])
def test_ring_large_batch_full_size(layout):
    inp = synthetic.generate(synthetic.WORKLOADS[synthetic.BENCH_WORKLOAD])
    seq = ring_seqlens(np.random.default_rng(7), inp)
    _check_ring(inp, seq, layout, what=f"ring large {layout}")


@pytest.mark.parametrize("L,layout,route", [(3, "compact", "bulk"), (3, "channel_last", "vector"),
                                            (5, "compact", "vector"), (12, "channel_last", "staged"),
                                            (9, "compact", "scalar")])
def test_ring_chain_equals_full_convolution(L, layout, route):
    """T GPU updates of a ring fed with cache_seqlens 0..T-1 equal one full convolution."""
    import depthwise_causal_conv1d_gb300 as ccu

    rng = np.random.default_rng(100 + L)
    T, D = 13, 1032
    x_seq = synthetic.f64_to_bf16_bits(rng.standard_normal((T, D)))
    weight = synthetic.f64_to_bf16_bits(rng.standard_normal((D, 4)) * 0.5)
    bias = synthetic.f64_to_bf16_bits(rng.standard_normal(D) * 0.1)
    want_y, want_state = oracle.full_causal_conv(x_seq, weight, bias, "silu", None, L)
    w, b = to_dev_u16(weight, DEV), to_dev_u16(bias, DEV)
    if layout == "compact":
        st = torch.zeros((1, D, L), dtype=torch.bfloat16, device=DEV)
    else:
        st = torch.zeros((1, L, D), dtype=torch.bfloat16, device=DEV).permute(0, 2, 1)
    ys = []
    for t in range(T):
        xt = to_dev_u16(x_seq[t:t + 1], DEV)
        seq = torch.tensor([t], dtype=torch.int32, device=DEV)
        ys.append(from_dev_u16(ccu.causal_conv1d_update(xt, st, w, b, "silu", cache_seqlens=seq,
                                                        route=route)))
    from oracle_pins import _rotate, bf16_ulp_distance

    got_ring = from_dev_u16(st.contiguous())[0]
    assert np.array_equal(_rotate(got_ring, T % L), want_state)
    assert bf16_ulp_distance(np.concatenate(ys), want_y).max() <= 1


@pytest.mark.parametrize("route", ["scalar", "vector", "staged", "bulk"])
def test_ring_checked_negative_seqlens(route):
    wl = synthetic.variant(synthetic.WORKLOADS["paged_n256_d8192_l3_s1024_pad10_silu"], name="ringchk",
                           N=12, D=1024, S=16, indices="distinct_pad", pad_frac=0.2)
    inp = synthetic.generate(wl, seed=9)
    seq = ring_seqlens(np.random.default_rng(3), inp)
    active = np.flatnonzero(inp.indices >= 0)
    bad = active[:2]
    seq[bad] = -3
    ref_idx = inp.indices.copy()
    ref_idx[bad] = -1  # the oracle's view: those rows behave as padding
    ref_seq = seq.copy()
    ref_seq[bad] = 0
    want_out, want_state = oracle_ref(dataclasses.replace(inp, indices=ref_idx), cache_seqlens=ref_seq)
    got_out, got_state, status, ok = run_gpu(inp, route=route, checked=True, cache_seqlens=seq)
    assert ok and status & 1
    assert_parity(inp, got_out, got_state, want_out, want_state, "ring checked")


# ----------------------------------------------------------------------------- multi-token update

MULTI = [
    dict(N=6, D=264, T=4, L=3, S=8, ring=False, x_layout="tokens_major"),
    dict(N=5, D=520, T=1, L=4, S=5, ring=True, x_layout="tokens_major"),
    dict(N=7, D=64, T=7, L=4, S=9, ring=False, x_layout="channels_major"),
    dict(N=3, D=2056, T=3, L=8, S=3, ring=True, x_layout="tokens_major"),
    dict(N=4, D=37, T=5, L=5, S=6, ring=False, x_layout="tokens_major"),
    dict(N=4, D=128, T=9, L=3, S=4, ring=True, x_layout="channels_major"),
    dict(N=3, D=72, T=2, L=12, S=5, ring=False, x_layout="tokens_major"),
]


def _multi_inputs(case, seed):
    rng = np.random.default_rng(seed)
    N, D, T, L, S = case["N"], case["D"], case["T"], case["L"], case["S"]
    x_tok = synthetic.f64_to_bf16_bits(rng.standard_normal((N, T, D)))  # token-major memory
    weight = synthetic.f64_to_bf16_bits(rng.standard_normal((D, 4)) * 0.5)
    bias = synthetic.f64_to_bf16_bits(rng.standard_normal(D) * 0.1)
    state = synthetic.f64_to_bf16_bits(rng.standard_normal((S, D, L)))
    idx = rng.permutation(S)[:N].astype(np.int32)
    idx[1] = -1
    seq = rng.integers(0, 50, size=N).astype(np.int32) if case["ring"] else None
    return x_tok, weight, bias, state, idx, seq


@pytest.mark.parametrize("route", ["auto", "scalar", "vector"])
@pytest.mark.parametrize("layout", ["compact", "channel_last"])
@pytest.mark.parametrize("ci", range(len(MULTI)))
def test_multi_token(route, layout, ci):
    case = MULTI[ci]
    if route == "vector" and (case["D"] % 8 or case["L"] > 8 or case["x_layout"] != "tokens_major"):
        pytest.skip("the vector kernel needs channel-contiguous 16-byte token rows and L <= 8")
    _check_multi(case, route, layout, 300 + ci)


def _check_multi(case, route, layout, seed, with_inter=True):
    """One multi-token call against the oracle: outputs, intermediate states (when asked
    for), final state."""
    import depthwise_causal_conv1d_gb300 as ccu

    N, D, T, L, S = case["N"], case["D"], case["T"], case["L"], case["S"]
    x_tok, weight, bias, state, idx, seq = _multi_inputs(case, seed)
    # oracle on its own copies
    st_ref = state.copy() if layout == "compact" else synthetic.to_channel_last(state)
    strides = (D * L, L, 1) if layout == "compact" else (L * D, 1, D)
    want_out, want_inter = oracle.conv1d_update_multi(x_tok, (T * D, 1, D), st_ref, strides, weight, bias,
                                                      "silu", idx, seq, N, D, T, S, L, 4, with_inter=True)
    want_state = st_ref if layout == "compact" else synthetic.from_channel_last(st_ref)
    # device copies
    if case["x_layout"] == "tokens_major":
        x = to_dev_u16(x_tok, DEV).permute(0, 2, 1)  # [N, D, T] view of [N, T, D] memory
    else:
        x = to_dev_u16(np.ascontiguousarray(np.transpose(x_tok, (0, 2, 1))), DEV)  # [N, D, T] memory
    if layout == "compact":
        st = to_dev_u16(state, DEV)
    else:
        st = to_dev_u16(synthetic.to_channel_last(state), DEV).permute(0, 2, 1)
    inter = torch.zeros((N, T, D, L), dtype=torch.bfloat16, device=DEV) if with_inter else None
    out = ccu.causal_conv1d_update(x, st, to_dev_u16(weight, DEV), to_dev_u16(bias, DEV), "silu",
                                   conv_state_indices=torch.from_numpy(idx).to(DEV),
                                   cache_seqlens=None if seq is None else torch.from_numpy(seq).to(DEV),
                                   route=route, intermediate_states=inter)
    torch.cuda.synchronize()
    assert out.stride() == x.stride()
    got_out = from_dev_u16(out.permute(0, 2, 1).contiguous().permute(0, 2, 1))
    got_state = from_dev_u16(st.contiguous())
    from oracle_pins import bf16_ulp_distance

    assert np.array_equal(got_state, want_state), "final state"
    if with_inter:
        assert np.array_equal(from_dev_u16(inter), want_inter), "intermediate states"
    assert bf16_ulp_distance(got_out, want_out).max() <= 1, "outputs"


def _multi_bulk_serves(case, layout):
    return (layout == "compact" and case["D"] % 8 == 0 and 3 <= case["L"] <= 8 and 1 <= case["T"] <= 8
            and case["x_layout"] == "tokens_major")




# The vector multi-token kernel runs one wave of CTAs, each walking many rows two at a time:
# rows enough for several turns of that loop (and an odd count per CTA), more than four
# tokens (the later ones loaded per group of four), ragged D (CTAs with idle threads) and
# intermediate states, in both layouts.
MULTI_MANY_ROWS = [
    dict(N=1200, D=264, T=6, L=3, S=1300, ring=False, x_layout="tokens_major"),
    dict(N=900, D=264, T=4, L=5, S=901, ring=False, x_layout="tokens_major"),
    dict(N=700, D=2056, T=3, L=8, S=700, ring=False, x_layout="tokens_major"),
    dict(N=640, D=520, T=1, L=4, S=640, ring=False, x_layout="tokens_major"),
]


@pytest.mark.parametrize("route", ["auto", "vector"])
@pytest.mark.parametrize("layout", ["compact", "channel_last"])
@pytest.mark.parametrize("ci", range(len(MULTI_MANY_ROWS)))
def test_multi_token_many_rows_per_cta(route, layout, ci):
    _check_multi(MULTI_MANY_ROWS[ci], route, layout, 500 + ci)


# The bulk-copy multi-token kernel: the compact state at L = 3..8, up to 8 tokens, no
# intermediate states; on every other case the forced route declines.
@pytest.mark.parametrize("layout", ["compact", "channel_last"])
@pytest.mark.parametrize("ci", range(len(MULTI) + len(MULTI_MANY_ROWS)))
def test_multi_token_bulk(layout, ci):
    case = (MULTI + MULTI_MANY_ROWS)[ci]
    if not _multi_bulk_serves(case, layout):
        with pytest.raises(NotImplementedError):
            _check_multi(case, "bulk", layout, 700 + ci, with_inter=False)
        return
    _check_multi(case, "bulk", layout, 700 + ci, with_inter=False)
    with pytest.raises(NotImplementedError):  # intermediate states are the vector kernel's
        _check_multi(case, "bulk", layout, 700 + ci, with_inter=True)


@pytest.mark.parametrize("L", [4, 5, 7])
def test_multi_token_auto_ring_state(L):
    """AUTO sends the compact ring state at L = 4, 5, 7 (no intermediate states) to the
    bulk-copy kernel: parity with the oracle on a batch with padding rows and a ragged D."""
    case = dict(N=300, D=1032, T=4, L=L, S=310, ring=True, x_layout="tokens_major")
    _check_multi(case, "auto", "compact", 950 + L, with_inter=False)


@pytest.mark.parametrize("ring", [False, True])
@pytest.mark.parametrize("L,T", [(3, 4), (5, 8), (8, 2), (7, 1)])
def test_multi_token_bulk_large_batch(L, T, ring):
    """The bulk-copy multi-token kernel on a batch that gives every warp many slices (N=600,
    D=16384: 64 slices a row), with padding rows, against the oracle."""
    case = dict(N=600, D=16384, T=T, L=L, S=640, ring=ring, x_layout="tokens_major")
    _check_multi(case, "bulk", "compact", 900 + 10 * L + T, with_inter=False)


@pytest.mark.parametrize("route", ["auto", "vector"])
def test_multi_large_batch(route):
    """A large multi-token batch (N=1024, D=16384, T=4, ring state)."""
    import depthwise_causal_conv1d_gb300 as ccu

    case = dict(N=1024, D=16384, T=4, L=3, S=1024, ring=True, x_layout="tokens_major")
    N, D, T, L, S = 1024, 16384, 4, 3, 1024
    x_tok, weight, bias, state, idx, seq = _multi_inputs(case, 77)
    st_ref = state.copy()
    want_out = oracle.conv1d_update_multi(x_tok, (T * D, 1, D), st_ref, (D * L, L, 1), weight, bias,
                                          "silu", idx, seq, N, D, T, S, L, 4)
    x = to_dev_u16(x_tok, DEV).permute(0, 2, 1)
    st = to_dev_u16(state, DEV)
    out = ccu.causal_conv1d_update(x, st, to_dev_u16(weight, DEV), to_dev_u16(bias, DEV), "silu",
                                   conv_state_indices=torch.from_numpy(idx).to(DEV),
                                   cache_seqlens=torch.from_numpy(seq).to(DEV), route=route)
    torch.cuda.synchronize()
    from oracle_pins import bf16_ulp_distance

    assert np.array_equal(from_dev_u16(st), st_ref)
    assert bf16_ulp_distance(from_dev_u16(out.permute(0, 2, 1)).transpose(0, 2, 1), want_out).max() <= 1


@pytest.mark.parametrize("T", [1, 25])
def test_multi_token_vector_extremes(T):
    """The vector kernel at one token and at T = 25 (six groups of four tokens and a
    remainder of one), N = 2 rows, ring state, intermediate states."""
    import depthwise_causal_conv1d_gb300 as ccu
    from oracle_pins import bf16_ulp_distance

    case = dict(N=2, D=2048, T=T, L=3, S=3, ring=True, x_layout="tokens_major")
    N, D, L, S = case["N"], case["D"], case["L"], case["S"]
    x_tok, weight, bias, state, idx, seq = _multi_inputs(case, 60 + T)
    st_ref = state.copy()
    want_out, want_inter = oracle.conv1d_update_multi(x_tok, (T * D, 1, D), st_ref, (D * L, L, 1), weight,
                                                      bias, "silu", idx, seq, N, D, T, S, L, 4, with_inter=True)
    st = to_dev_u16(state, DEV)
    inter = torch.zeros((N, T, D, L), dtype=torch.bfloat16, device=DEV)
    args = dict(conv_state_indices=torch.from_numpy(idx).to(DEV), cache_seqlens=torch.from_numpy(seq).to(DEV))
    out = ccu.causal_conv1d_update(to_dev_u16(x_tok, DEV).permute(0, 2, 1), st, to_dev_u16(weight, DEV),
                                   to_dev_u16(bias, DEV), "silu", route="vector", intermediate_states=inter,
                                   **args)
    torch.cuda.synchronize()
    assert np.array_equal(from_dev_u16(st), st_ref)
    assert np.array_equal(from_dev_u16(inter), want_inter)
    assert bf16_ulp_distance(from_dev_u16(out.permute(0, 2, 1)).transpose(0, 2, 1), want_out).max() <= 1


@pytest.mark.parametrize("route", ["scalar", "vector", "bulk"])
def test_multi_token_checked_bad_index(route):
    """Checked multi-token call: an out-of-range slot raises CCU_DEVERR_RANGE and its row
    behaves as padding (zero outputs, no state access); the other rows are exact."""
    import depthwise_causal_conv1d_gb300 as ccu

    case = dict(N=9, D=1032, T=4, L=3, S=12, ring=False, x_layout="tokens_major")
    N, D, T, L, S = case["N"], case["D"], case["T"], case["L"], case["S"]
    x_tok, weight, bias, state, idx, _ = _multi_inputs(case, 41)
    bad = idx.copy()
    bad[4] = S + 3
    ref_idx = idx.copy()
    ref_idx[4] = -1
    st_ref = state.copy()
    want_out = oracle.conv1d_update_multi(x_tok, (T * D, 1, D), st_ref, (D * L, L, 1), weight, bias,
                                          "silu", ref_idx, None, N, D, T, S, L, 4)
    st = to_dev_u16(state, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = ccu.causal_conv1d_update(to_dev_u16(x_tok, DEV).permute(0, 2, 1), st, to_dev_u16(weight, DEV),
                                   to_dev_u16(bias, DEV), "silu",
                                   conv_state_indices=torch.from_numpy(bad).to(DEV), route=route,
                                   status=status)
    torch.cuda.synchronize()
    from oracle_pins import bf16_ulp_distance

    assert int(status.item()) & 1
    assert np.array_equal(from_dev_u16(st), st_ref)
    assert bf16_ulp_distance(from_dev_u16(out.permute(0, 2, 1)).transpose(0, 2, 1), want_out).max() <= 1


# ----------------------------------------------------------------------------- prefill

PREFILL = [
    dict(B=2, D=264, T=100, L=3, x_layout="tokens_major", init=None, fin="channel_last"),
    dict(B=3, D=64, T=1, L=3, x_layout="tokens_major", init="compact", fin="channel_last"),
    dict(B=1, D=128, T=2, L=5, x_layout="tokens_major", init="channel_last", fin="compact"),
    dict(B=4, D=40, T=37, L=4, x_layout="channels_major", init="compact", fin="compact"),
    dict(B=2, D=19, T=70, L=3, x_layout="tokens_major", init="compact", fin="channel_last"),
    dict(B=2, D=2048, T=1030, L=3, x_layout="tokens_major", init="channel_last", fin="channel_last"),
    dict(B=1, D=512, T=3, L=8, x_layout="tokens_major", init="compact", fin=None),
]


def _state_dev(arr_bdl, layout):
    """[B, D, L] numpy -> device tensor [B, D, L] in the given layout."""
    if layout == "compact":
        return to_dev_u16(arr_bdl, DEV)
    return to_dev_u16(np.ascontiguousarray(np.transpose(arr_bdl, (0, 2, 1))), DEV).permute(0, 2, 1)


@pytest.mark.parametrize("route", ["auto", "scalar", "vector", "bulk"])
@pytest.mark.parametrize("act", ["identity", "silu"])
@pytest.mark.parametrize("ci", range(len(PREFILL)))
def test_prefill(route, act, ci):
    import depthwise_causal_conv1d_gb300 as ccu

    c = PREFILL[ci]
    B, D, T, L = c["B"], c["D"], c["T"], c["L"]
    if route in ("vector", "bulk") and (D % 8 or c["x_layout"] != "tokens_major"):
        pytest.skip("the vector and bulk kernels need channel-contiguous 16-byte token rows")
    rng = np.random.default_rng(500 + ci)
    x_btd = synthetic.f64_to_bf16_bits(rng.standard_normal((B, T, D)))
    weight = synthetic.f64_to_bf16_bits(rng.standard_normal((D, 4)) * 0.5)
    bias = synthetic.f64_to_bf16_bits(rng.standard_normal(D) * 0.1)
    init = synthetic.f64_to_bf16_bits(rng.standard_normal((B, D, L))) if c["init"] else None
    want_y, want_fin = [], []
    for b in range(B):
        y, fin = oracle.full_causal_conv(x_btd[b], weight, bias, act, None if init is None else init[b], L)
        want_y.append(y.T)  # [D, T]
        want_fin.append(fin)
    want_y, want_fin = np.stack(want_y), np.stack(want_fin)
    if c["x_layout"] == "tokens_major":
        x = to_dev_u16(x_btd, DEV).permute(0, 2, 1)
    else:
        x = to_dev_u16(np.ascontiguousarray(np.transpose(x_btd, (0, 2, 1))), DEV)
    init_dev = _state_dev(init, c["init"]) if init is not None else None
    fin_dev = None
    if c["fin"] is not None:
        fin_dev = _state_dev(np.zeros((B, D, L), np.uint16), c["fin"])
    res = ccu.causal_conv1d_fwd(x, to_dev_u16(weight, DEV), to_dev_u16(bias, DEV), act,
                                initial_states=init_dev, final_states_out=fin_dev, route=route)
    out = res[0] if isinstance(res, tuple) else res
    torch.cuda.synchronize()
    from oracle_pins import bf16_ulp_distance

    got_y = from_dev_u16(out)
    assert bf16_ulp_distance(got_y, want_y).max() <= (0 if act == "identity" else 1)
    if fin_dev is not None:
        assert np.array_equal(from_dev_u16(fin_dev), want_fin)


@pytest.mark.parametrize("T", [3, 21])
def test_prefill_bulk_more_runs_than_warps(T):
    """B * D / 256 channel runs above the GPU's warp count: every warp of the bulk kernel
    walks several runs, restarting its window and weights at each (the last slice of every
    row is partial: D = 16384 + 72)."""
    import depthwise_causal_conv1d_gb300 as ccu

    rng = np.random.default_rng(77 + T)
    B, D, L = 40, 16384 + 72, 3
    x_btd = synthetic.f64_to_bf16_bits(rng.standard_normal((B, T, D)))
    weight = synthetic.f64_to_bf16_bits(rng.standard_normal((D, 4)) * 0.5)
    bias = synthetic.f64_to_bf16_bits(rng.standard_normal(D) * 0.1)
    init = synthetic.f64_to_bf16_bits(rng.standard_normal((B, D, L)))
    x = to_dev_u16(x_btd, DEV).permute(0, 2, 1)
    y, fin = ccu.causal_conv1d_fwd(x, to_dev_u16(weight, DEV), to_dev_u16(bias, DEV), "silu",
                                   initial_states=to_dev_u16(init, DEV), return_final_states=True,
                                   route="bulk")
    torch.cuda.synchronize()
    from oracle_pins import bf16_ulp_distance

    got_y, got_fin = from_dev_u16(y), from_dev_u16(fin)
    for b in range(B):
        want_y, want_fin = oracle.full_causal_conv(x_btd[b], weight, bias, "silu", init[b], L)
        assert bf16_ulp_distance(got_y[b], want_y.T).max() <= 1, b
        assert np.array_equal(got_fin[b], want_fin), b


def test_prefill_host_resident_x_and_out():
    """x and out in pinned host memory: AUTO runs the vector kernel on them in place (the
    bulk kernel's copies need device memory, and a forced bulk route declines)."""
    import depthwise_causal_conv1d_gb300 as ccu
    from oracle_pins import bf16_ulp_distance

    rng = np.random.default_rng(13)
    B, T, D, L = 2, 600, 1024, 3
    assert B * T * D >= 1 << 20  # device operands this size would take the bulk route
    x_btd = synthetic.f64_to_bf16_bits(rng.standard_normal((B, T, D)))
    weight = synthetic.f64_to_bf16_bits(rng.standard_normal((D, 4)) * 0.5)
    bias = synthetic.f64_to_bf16_bits(rng.standard_normal(D) * 0.1)
    h_x = torch.from_numpy(x_btd.view(np.int16)).pin_memory()
    h_out = torch.full((B, T, D), -1, dtype=torch.int16).pin_memory()
    w, b = to_dev_u16(weight, DEV), to_dev_u16(bias, DEV)
    fin = torch.zeros((B, L, D), dtype=torch.int16, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    args = (h_x.data_ptr(), T * D, 1, D, w.data_ptr(), b.data_ptr(), ccu.CCU_ACT_SILU, None, 0, 0, 0,
            B, D, T, L, 4, h_out.data_ptr(), T * D, 1, D, fin.data_ptr(), L * D, 1, D)
    assert ccu.ccu_causal_conv1d_fwd(*args, ccu.ROUTES["bulk"], stream) == ccu.CCU_ERR_NOT_IMPLEMENTED
    assert ccu.ccu_causal_conv1d_fwd(*args, ccu.ROUTES["auto"], stream) == 0, ccu.ccu_conv1d_last_error()
    torch.cuda.synchronize()
    got = h_out.numpy().view(np.uint16)
    got_fin = fin.cpu().numpy().view(np.uint16)
    for bb in range(B):
        want, want_fin = oracle.full_causal_conv(x_btd[bb], weight, bias, "silu", None, L)
        assert bf16_ulp_distance(got[bb], want).max() <= 1
        assert np.array_equal(got_fin[bb].T, want_fin)


def test_prefill_hands_off_to_decode():
    """Prefill T tokens, hand the channel-last L=3 final state to the decode update for K
    more tokens: the outputs equal one convolution over all T + K tokens."""
    import depthwise_causal_conv1d_gb300 as ccu

    rng = np.random.default_rng(9)
    B, D, T, K = 4, 1024, 200, 5
    x_all = synthetic.f64_to_bf16_bits(rng.standard_normal((B, T + K, D)))
    weight = synthetic.f64_to_bf16_bits(rng.standard_normal((D, 4)) * 0.5)
    bias = synthetic.f64_to_bf16_bits(rng.standard_normal(D) * 0.1)
    w, b = to_dev_u16(weight, DEV), to_dev_u16(bias, DEV)
    x_pre = to_dev_u16(np.ascontiguousarray(x_all[:, :T]), DEV).permute(0, 2, 1)
    y_pre, state = ccu.causal_conv1d_fwd(x_pre, w, b, "silu", return_final_states=True)
    assert state.stride() == (3 * D, 1, D)  # the layout the decode update takes without a copy
    ys = [from_dev_u16(y_pre)]
    for k in range(K):
        xt = to_dev_u16(np.ascontiguousarray(x_all[:, T + k]), DEV)
        ys.append(from_dev_u16(ccu.causal_conv1d_update(xt, state, w, b, "silu"))[:, :, None])
    got = np.concatenate(ys, axis=2)
    from oracle_pins import bf16_ulp_distance

    for bb in range(B):
        want, _ = oracle.full_causal_conv(x_all[bb], weight, bias, "silu", None, 3)
        assert bf16_ulp_distance(got[bb], want.T).max() <= 1


# ----------------------------------------------------------------------------- widths 2 and 3

WIDTH_CASES = [(W, L) for W in (2, 3) for L in sorted({W - 1, W, 4, 5, 9})]


@pytest.mark.parametrize("ring", [False, True])
@pytest.mark.parametrize("route", ["scalar", "vector", "staged", "bulk"])
@pytest.mark.parametrize("layout", ["compact", "channel_last"])
@pytest.mark.parametrize("W,L", WIDTH_CASES)
def test_widths(W, L, layout, route, ring):
    if route == "vector" and L > 8:
        pytest.skip("vector kernels are compiled for L <= 8")
    if route == "bulk" and (layout != "compact" or L > 4):
        pytest.skip("bulk kernels serve widths 2 and 3 in the compact layout with L <= 4")
    wl = synthetic.variant(synthetic.WORKLOADS["paged_n256_d8192_l3_s1024_pad10_silu"], name="width",
                           N=9, D=264, ld=264, S=12, W=W, L=L, pad_frac=0.25)
    inp = synthetic.generate(wl, seed=W * 100 + L)
    if ring:
        _check_ring(inp, ring_seqlens(np.random.default_rng(L), inp), layout, route,
                    what=f"W={W} L={L} ring {route} {layout}")
    else:
        _check(inp, layout=layout, route=route, what=f"W={W} L={L} {route} {layout}")


@pytest.mark.parametrize("W,L", [(2, 1), (2, 3), (3, 2), (3, 4)])
def test_widths_large_batch_auto_route(W, L):
    """Large compact batches at widths 2 and 3 take the bulk kernels (AUTO)."""
    wl = synthetic.variant(synthetic.WORKLOADS[synthetic.BENCH_WORKLOAD], name="wide", N=512, S=512, W=W, L=L)
    inp = synthetic.generate(wl, seed=W * 10 + L)
    _check(inp, what=f"W={W} L={L} large")


@pytest.mark.parametrize("W,L,T", [(2, 1, 3), (3, 2, 5), (3, 4, 2)])
def test_widths_multi_token(W, L, T):
    import depthwise_causal_conv1d_gb300 as ccu

    rng = np.random.default_rng(W + L + T)
    N, D, S = 5, 96, 6
    x_tok = synthetic.f64_to_bf16_bits(rng.standard_normal((N, T, D)))
    weight = synthetic.f64_to_bf16_bits(rng.standard_normal((D, W)))
    state = synthetic.f64_to_bf16_bits(rng.standard_normal((S, D, L)))
    idx = np.array([4, -1, 0, 2, 5], np.int32)
    st_ref = state.copy()
    want_out, want_inter = oracle.conv1d_update_multi(x_tok, (T * D, 1, D), st_ref, (D * L, L, 1), weight,
                                                      None, "silu", idx, None, N, D, T, S, L, W,
                                                      with_inter=True)
    st = to_dev_u16(state, DEV)
    inter = torch.zeros((N, T, D, L), dtype=torch.bfloat16, device=DEV)
    out = ccu.causal_conv1d_update(to_dev_u16(x_tok, DEV).permute(0, 2, 1), st, to_dev_u16(weight, DEV),
                                   None, "silu", conv_state_indices=torch.from_numpy(idx).to(DEV),
                                   intermediate_states=inter)
    torch.cuda.synchronize()
    from oracle_pins import bf16_ulp_distance

    assert np.array_equal(from_dev_u16(st), st_ref) and np.array_equal(from_dev_u16(inter), want_inter)
    assert bf16_ulp_distance(from_dev_u16(out), want_out).max() <= 1


@pytest.mark.parametrize("W", [2, 3])
def test_widths_prefill(W):
    import depthwise_causal_conv1d_gb300 as ccu

    rng = np.random.default_rng(40 + W)
    B, D, T, L = 2, 136, 50, W - 1
    x_btd = synthetic.f64_to_bf16_bits(rng.standard_normal((B, T, D)))
    weight = synthetic.f64_to_bf16_bits(rng.standard_normal((D, W)))
    bias = synthetic.f64_to_bf16_bits(rng.standard_normal(D) * 0.1)
    init = synthetic.f64_to_bf16_bits(rng.standard_normal((B, D, L)))
    out, fin = ccu.causal_conv1d_fwd(to_dev_u16(x_btd, DEV).permute(0, 2, 1), to_dev_u16(weight, DEV),
                                     to_dev_u16(bias, DEV), "silu", initial_states=to_dev_u16(init, DEV),
                                     return_final_states=True)
    torch.cuda.synchronize()
    from oracle_pins import bf16_ulp_distance

    for b in range(B):
        y, f = oracle.full_causal_conv(x_btd[b], weight, bias, "silu", init[b], L)
        assert bf16_ulp_distance(from_dev_u16(out[b]), y.T).max() <= 1
        assert np.array_equal(from_dev_u16(fin[b]), f)


# ------------------------------------------------------------------- widths 1 and wider than 4

# The page calls every width with L >= W - 1 semantically valid; widths other than 2, 3 and 4
# run on the scalar kernels (AUTO picks them).
OTHER_WIDTH_CASES = [(1, 1), (1, 3), (5, 4), (5, 9), (6, 5), (8, 7), (8, 12), (16, 15)]


@pytest.mark.parametrize("ring", [False, True])
@pytest.mark.parametrize("route", ["auto", "scalar"])
@pytest.mark.parametrize("layout", ["compact", "channel_last"])
@pytest.mark.parametrize("W,L", OTHER_WIDTH_CASES)
def test_other_widths(W, L, layout, route, ring):
    wl = synthetic.variant(synthetic.WORKLOADS["paged_n256_d8192_l3_s1024_pad10_silu"], name="width",
                           N=9, D=77, ld=80, S=12, W=W, L=L, pad_frac=0.25)
    inp = synthetic.generate(wl, seed=W * 100 + L)
    if ring:
        _check_ring(inp, ring_seqlens(np.random.default_rng(L), inp), layout, route,
                    what=f"W={W} L={L} ring {route} {layout}")
    else:
        _check(inp, layout=layout, route=route, what=f"W={W} L={L} {route} {layout}")


@pytest.mark.parametrize("layout", ["compact", "channel_last"])
@pytest.mark.parametrize("W,L", [(1, 2), (5, 4), (8, 9)])
def test_other_widths_checked_duplicates(W, L, layout):
    """The duplicate-checking update at other widths (scalar kernel): the status bits equal
    the oracle's index check, and every row but the one that claimed a shared slot (read
    back from the slot scratch) acts as padding, as do out-of-range rows."""
    wl = synthetic.variant(synthetic.WORKLOADS["paged_n256_d8192_l3_s1024_pad10_silu"], name="width_dup",
                           N=40, D=72, ld=72, S=48, W=W, L=L, indices="distinct_pad", pad_frac=0.1)
    inp = synthetic.generate(wl, seed=300 + W)
    idx = inp.indices.copy()
    active = np.flatnonzero(idx >= 0)
    groups = [[active[2], active[17], active[30]], [active[5], active[6]]]
    for g in groups:
        idx[g] = idx[g[0]]
    idx[active[9]] = -2
    idx[active[12]] = wl.S
    want_status = oracle.check_indices(idx, wl.N, wl.S)
    scratch = torch.full((wl.S,), 777, dtype=torch.int32, device=DEV)  # dirty: the call clears it
    got_out, got_state, status, ok = run_gpu(dataclasses.replace(inp, indices=idx), layout=layout,
                                             checked=True, slot_scratch=scratch)
    assert ok, "a guard band was overwritten"
    assert status == want_status, (status, want_status)
    owners = scratch.cpu().numpy()
    ref_idx = idx.copy()
    ref_idx[(idx < -1) | (idx >= wl.S)] = -1
    for g in groups:
        winner = owners[idx[g[0]]] - 1
        assert winner in g, (winner, g)
        ref_idx[[r for r in g if r != winner]] = -1
    want_out, want_state = oracle_ref(dataclasses.replace(inp, indices=ref_idx), layout)
    assert_parity(inp, got_out, got_state, want_out, want_state, f"dedup W={W} L={L} {layout}")


@pytest.mark.parametrize("W,L,T", [(1, 1, 3), (1, 3, 5), (5, 4, 4), (7, 9, 3), (8, 7, 10)])
@pytest.mark.parametrize("ring", [False, True])
@pytest.mark.parametrize("layout", ["compact", "channel_last"])
def test_other_widths_multi_token(W, L, T, ring, layout):
    import depthwise_causal_conv1d_gb300 as ccu

    rng = np.random.default_rng(W * 7 + L + T)
    N, D, S = 5, 40, 6
    x_tok = synthetic.f64_to_bf16_bits(rng.standard_normal((N, T, D)))
    weight = synthetic.f64_to_bf16_bits(rng.standard_normal((D, W)))
    bias = synthetic.f64_to_bf16_bits(rng.standard_normal(D) * 0.1)
    state = synthetic.f64_to_bf16_bits(rng.standard_normal((S, D, L)))
    idx = np.array([4, -1, 0, 2, 5], np.int32)
    seq = np.array([3, 0, L + 2, 1, 11], np.int32) if ring else None
    st_ref = state.copy()
    want_out, want_inter = oracle.conv1d_update_multi(x_tok, (T * D, 1, D), st_ref, (D * L, L, 1), weight,
                                                      bias, "silu", idx, seq, N, D, T, S, L, W,
                                                      with_inter=True)
    if layout == "compact":
        st = to_dev_u16(state, DEV)
    else:
        st = to_dev_u16(np.ascontiguousarray(state.transpose(0, 2, 1)), DEV).permute(0, 2, 1)
    inter = torch.zeros((N, T, D, L), dtype=torch.bfloat16, device=DEV)
    out = ccu.causal_conv1d_update(to_dev_u16(x_tok, DEV).permute(0, 2, 1), st, to_dev_u16(weight, DEV),
                                   to_dev_u16(bias, DEV), "silu",
                                   conv_state_indices=torch.from_numpy(idx).to(DEV),
                                   cache_seqlens=None if seq is None else torch.from_numpy(seq).to(DEV),
                                   intermediate_states=inter)
    torch.cuda.synchronize()
    from oracle_pins import bf16_ulp_distance

    assert np.array_equal(from_dev_u16(st.contiguous()), st_ref), "state"
    assert np.array_equal(from_dev_u16(inter), want_inter), "intermediate states"
    assert bf16_ulp_distance(from_dev_u16(out), want_out).max() <= 1


@pytest.mark.parametrize("route", ["auto", "scalar"])
@pytest.mark.parametrize("W,L", [(1, 1), (1, 2), (5, 4), (7, 8), (9, 8)])
def test_other_widths_prefill(W, L, route):
    import depthwise_causal_conv1d_gb300 as ccu

    rng = np.random.default_rng(60 + W + L)
    B, D, T = 2, 72, 37
    x_btd = synthetic.f64_to_bf16_bits(rng.standard_normal((B, T, D)))
    weight = synthetic.f64_to_bf16_bits(rng.standard_normal((D, W)))
    bias = synthetic.f64_to_bf16_bits(rng.standard_normal(D) * 0.1)
    init = synthetic.f64_to_bf16_bits(rng.standard_normal((B, D, L)))
    for with_init in (False, True):
        out, fin = ccu.causal_conv1d_fwd(to_dev_u16(x_btd, DEV).permute(0, 2, 1), to_dev_u16(weight, DEV),
                                         to_dev_u16(bias, DEV), "silu",
                                         initial_states=to_dev_u16(init, DEV) if with_init else None,
                                         final_state_len=L, return_final_states=True, route=route)
        torch.cuda.synchronize()
        from oracle_pins import bf16_ulp_distance

        for b in range(B):
            y, f = oracle.full_causal_conv(x_btd[b], weight, bias, "silu", init[b] if with_init else None, L)
            assert bf16_ulp_distance(from_dev_u16(out[b]), y.T).max() <= 1, (b, with_init)
            assert np.array_equal(from_dev_u16(fin[b]), f), (b, with_init)


def test_other_widths_decline_on_8_channel_routes():
    import depthwise_causal_conv1d_gb300 as ccu

    wl = synthetic.variant(synthetic.WORKLOADS["paged_n256_d8192_l3_s1024_pad10_silu"], name="width",
                           N=4, D=64, ld=64, S=8, W=5, L=4)
    inp = synthetic.generate(wl, seed=5)
    for route in ("vector", "staged", "bulk"):
        with pytest.raises(NotImplementedError):
            run_gpu(inp, "compact", route)


# ----------------------------------------------------------------------------- timed workloads

# The ring-buffer, width, multi-token and prefill workloads that the benchmark times, on
# exactly its seeded inputs and entry points, at full size, against the oracle.

@pytest.mark.parametrize("name", list(synthetic.RING_WORKLOADS) + list(synthetic.WIDTH_WORKLOADS))
def test_timed_decode_variants_full_size(name):
    wl = {**synthetic.RING_WORKLOADS, **synthetic.WIDTH_WORKLOADS}[name]
    inp = synthetic.generate(wl)
    want_out, want_state = oracle_ref(inp, wl.layout, cache_seqlens=inp.cache_seqlens)
    got_out, got_state, _, ok = run_gpu(inp, wl.layout, "auto", cache_seqlens=inp.cache_seqlens)
    assert ok, f"{name}: a guard band was overwritten"
    assert_parity(inp, got_out, got_state, want_out, want_state, name)


@pytest.mark.parametrize("name", list(synthetic.MULTI_WORKLOADS))
def test_timed_multi_token_full_size(name):
    import depthwise_causal_conv1d_gb300 as ccu
    from oracle_pins import bf16_ulp_distance

    wl = synthetic.MULTI_WORKLOADS[name]
    inp = synthetic.generate(wl)
    N, D, T, L, S = wl.N, wl.D, wl.T, wl.L, wl.S
    want_state = inp.conv_state.copy()
    want_out = oracle.conv1d_update_multi(inp.x, (T * D, 1, D), want_state, (D * L, L, 1), inp.weight,
                                          inp.bias, wl.act, inp.indices, inp.cache_seqlens, N, D, T, S, L,
                                          wl.W)
    seq = torch.from_numpy(inp.cache_seqlens).to(DEV) if inp.cache_seqlens is not None else None
    x = to_dev_u16(inp.x, DEV)  # [N, T, D] memory
    st = to_dev_u16(inp.conv_state, DEV)
    w = to_dev_u16(inp.weight, DEV)
    b = to_dev_u16(inp.bias, DEV) if inp.bias is not None else None
    idx = torch.from_numpy(inp.indices).to(DEV) if inp.indices is not None else None
    out = torch.empty((N, T, D), dtype=torch.bfloat16, device=DEV)
    act = ccu.CCU_ACT_SILU if wl.act == "silu" else ccu.CCU_ACT_IDENTITY
    stream = torch.cuda.current_stream()
    rc = ccu.lib.ccu_conv1d_update_multi(
        x.data_ptr(), T * D, 1, D, st.data_ptr(), D * L, L, 1, w.data_ptr(),
        None if b is None else b.data_ptr(), act, None if idx is None else idx.data_ptr(),
        None if seq is None else seq.data_ptr(), N, D, T, S, L, wl.W, out.data_ptr(), T * D, 1, D, None, None,
        ccu.ROUTES["auto"], stream.cuda_stream)
    assert rc == 0, ccu.ccu_conv1d_last_error()
    torch.cuda.synchronize()
    assert np.array_equal(from_dev_u16(st), want_state)
    got = from_dev_u16(out).transpose(0, 2, 1)  # [N, D, T], the oracle's order
    limit = 0 if wl.act == "identity" else 1
    assert bf16_ulp_distance(got, want_out).max() <= limit


@pytest.mark.parametrize("name", list(synthetic.PREFILL_WORKLOADS))
def test_timed_prefill_full_size(name):
    import depthwise_causal_conv1d_gb300 as ccu
    from oracle_pins import bf16_ulp_distance

    spec = synthetic.PREFILL_WORKLOADS[name]
    x_btd, weight, bias = synthetic.generate_prefill(spec)
    B, T, D, L, W = spec["B"], spec["T"], spec["D"], spec["L"], spec["W"]
    x = to_dev_u16(x_btd, DEV).permute(0, 2, 1)  # [B, D, T] view of token-major memory
    w = to_dev_u16(weight, DEV)
    b = to_dev_u16(bias, DEV) if bias is not None else None
    out = torch.empty_like(x)
    fin = torch.empty((B, L, D), dtype=torch.bfloat16, device=DEV).permute(0, 2, 1)
    act = ccu.CCU_ACT_SILU if spec["act"] == "silu" else ccu.CCU_ACT_IDENTITY
    rc = ccu.lib.ccu_causal_conv1d_fwd(
        x.data_ptr(), *x.stride(), w.data_ptr(), None if b is None else b.data_ptr(), act,
        None, 0, 0, 0, B, D, T, L, W, out.data_ptr(), *out.stride(), fin.data_ptr(), *fin.stride(),
        ccu.ROUTES["auto"], torch.cuda.current_stream().cuda_stream)
    assert rc == 0, ccu.ccu_conv1d_last_error()
    torch.cuda.synchronize()
    got_y = from_dev_u16(out.permute(0, 2, 1))  # [B, T, D]
    got_fin = from_dev_u16(fin)  # [B, D, L]
    limit = 0 if spec["act"] == "identity" else 1
    for bb in range(B):
        want_y, want_fin = oracle.full_causal_conv(x_btd[bb], weight, bias, spec["act"], None, L)
        assert np.array_equal(got_fin[bb], want_fin), f"sequence {bb}: final state differs"
        assert bf16_ulp_distance(got_y[bb], want_y).max() <= limit, f"sequence {bb}: output"


@pytest.mark.parametrize("route", ["vector", "bulk"])
def test_stream_order_with_foreign_kernels(route):
    """Calls interleaved on one stream with torch kernels that write x and a state slot
    before each call and read its output after it: every call sees the writes made before
    it and its output is complete for the read after it (the kernels are launched as
    programmatic dependents and wait for prior work before touching memory)."""
    import depthwise_causal_conv1d_gb300 as ccu
    from oracle_pins import bf16_ulp_distance

    wl = synthetic.variant(synthetic.WORKLOADS["paged_n256_d8192_l3_s1024_pad10_silu"], name="order",
                           N=256, D=8192, S=300, indices="distinct_pad", pad_frac=0.1)
    inp = synthetic.generate(wl, seed=31)
    rng = np.random.default_rng(32)
    steps = 6
    xs = [synthetic.f64_to_bf16_bits(rng.standard_normal((wl.N, wl.D))) for _ in range(steps)]
    s0 = int(inp.indices[np.flatnonzero(inp.indices >= 0)[0]])
    patch = synthetic.f64_to_bf16_bits(rng.standard_normal((wl.D, wl.L)))
    # oracle: the same sequence on the host
    state = inp.conv_state.copy()
    want = []
    for k in range(steps):
        if k % 2:
            state[s0] = patch
        want.append(oracle.conv1d_update(xs[k], wl.D, state, (wl.D * wl.L, wl.L, 1), inp.weight, inp.bias,
                                         wl.act, inp.indices, wl.N, wl.D, wl.S, wl.L, wl.W))
    # device: torch writes and reads around every call, all on one side stream
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        x_src = [to_dev_u16(a, DEV) for a in xs]
        patch_d = to_dev_u16(patch, DEV)
        x = torch.empty((wl.N, wl.D), dtype=torch.bfloat16, device=DEV)
        st = to_dev_u16(inp.conv_state, DEV)
        w = to_dev_u16(inp.weight, DEV)
        b = to_dev_u16(inp.bias, DEV)
        idx = torch.from_numpy(inp.indices).to(DEV)
        out = torch.empty((wl.N, wl.D), dtype=torch.bfloat16, device=DEV)
        got = [torch.empty_like(out) for _ in range(steps)]
        stream.synchronize()
        for k in range(steps):
            x.copy_(x_src[k])
            if k % 2:
                st[s0].copy_(patch_d)
            ccu.causal_conv1d_update(x, st, w, b, wl.act, conv_state_indices=idx, out=out, route=route)
            got[k].copy_(out)
    stream.synchronize()
    final_state = from_dev_u16(st)
    for k in range(steps):
        dist = bf16_ulp_distance(from_dev_u16(got[k]), want[k])
        assert dist.max() <= 1, f"step {k}: output off by {dist.max()} ulp"
    assert np.array_equal(final_state, state)


# ----------------------------------------------------------------------------- 64-bit offsets

BIG_D, BIG_L = 16384, 3
BIG_S = (1 << 31) // (BIG_D * BIG_L) + 48  # state of ~2.15e9 elements: the last slots lie past 2^31


def _big_state(layout):
    """A 4.3 GB BF16 state filled on the device (N(0,1)); returns (memory, logical [S, D, L])."""
    torch.manual_seed(7)
    if layout == "compact":
        mem = torch.randn((BIG_S, BIG_D, BIG_L), dtype=torch.bfloat16, device=DEV)
        return mem, mem
    mem = torch.randn((BIG_S, BIG_L, BIG_D), dtype=torch.bfloat16, device=DEV)
    return mem, mem.permute(0, 2, 1)


def _big_slots():
    """Slots past element 2^31, the one that straddles it, small ones, and padding rows."""
    first_past = (1 << 31) // (BIG_D * BIG_L) + 1
    slots = [BIG_S - 1, BIG_S - 2, first_past, first_past - 1, first_past + 7, 0, 5, 1000, -1, BIG_S - 30, -1, 12345]
    return np.array(slots, dtype=np.int32)


@pytest.mark.parametrize("layout", ["compact", "channel_last"])
@pytest.mark.parametrize("route", ["scalar", "vector", "staged", "bulk", "multi", "multi_bulk"])
def test_state_offsets_past_int32(layout, route):
    """Slots whose state starts past element 2^31 of a 4.3 GB state, on every route. The
    oracle runs on the touched slots only (a row's update reads and writes its own slot
    alone); untouched neighbours must keep their bytes."""
    import depthwise_causal_conv1d_gb300 as ccu
    from oracle_pins import bf16_ulp_distance

    D, L, W = BIG_D, BIG_L, 4
    mem, st = _big_state(layout)
    idx_np = _big_slots()
    N = len(idx_np)
    if route == "multi_bulk" and layout != "compact":
        pytest.skip("the bulk-copy multi-token kernel serves the compact state")
    T = 3 if route.startswith("multi") else 1
    rng = np.random.default_rng(8)
    x_np = synthetic.f64_to_bf16_bits(rng.standard_normal((N, T, D)))
    w_np = synthetic.f64_to_bf16_bits(rng.standard_normal((D, W)) * 0.5)
    b_np = synthetic.f64_to_bf16_bits(rng.standard_normal(D) * 0.1)
    touched = idx_np[idx_np >= 0]
    t_dev = torch.from_numpy(touched.astype(np.int64)).to(DEV)
    mini = from_dev_u16(st[t_dev])  # [k, D, L] logical, before
    neighbours = np.array([s for s in {0, 1, 4, 6, 999, 1001, int(touched.max()) - 2} if s not in set(touched)],
                          dtype=np.int64)
    nb_dev = torch.from_numpy(neighbours).to(DEV)
    nb_before = from_dev_u16(st[nb_dev])
    remap = {int(s): i for i, s in enumerate(touched)}
    idx_mini = np.array([remap[int(s)] if s >= 0 else -1 for s in idx_np], dtype=np.int32)
    w, b = to_dev_u16(w_np, DEV), to_dev_u16(b_np, DEV)
    idx = torch.from_numpy(idx_np).to(DEV)
    if route.startswith("multi"):
        want_out = oracle.conv1d_update_multi(x_np, (T * D, 1, D), mini, (D * L, L, 1), w_np, b_np, "silu",
                                              idx_mini, None, N, D, T, len(touched), L, W)
        x = to_dev_u16(x_np, DEV).permute(0, 2, 1)  # [N, D, T] view of [N, T, D] memory
        out = ccu.causal_conv1d_update(x, st, w, b, "silu", conv_state_indices=idx,
                                       route="bulk" if route == "multi_bulk" else "auto")
        got_out = from_dev_u16(out)
    else:
        x2 = np.ascontiguousarray(x_np[:, 0, :])
        want_out = oracle.conv1d_update(x2, D, mini, (D * L, L, 1), w_np, b_np, "silu", idx_mini, N, D,
                                        len(touched), L, W)
        out = torch.empty((N, D), dtype=torch.bfloat16, device=DEV)
        ccu.causal_conv1d_update(to_dev_u16(x2, DEV), st, w, b, "silu", conv_state_indices=idx, out=out,
                                 route=route)
        got_out = from_dev_u16(out)
    torch.cuda.synchronize()
    got_mini = from_dev_u16(st[t_dev])
    nb_after = from_dev_u16(st[nb_dev])
    del mem, st
    torch.cuda.empty_cache()
    assert np.array_equal(got_mini, mini), "touched slots' state differs from the oracle"
    assert np.array_equal(nb_after, nb_before), "an untouched slot changed"
    assert bf16_ulp_distance(got_out, want_out).max() <= 1


@pytest.mark.parametrize("route", ["scalar", "vector", "bulk"])
def test_prefill_offsets_past_int32(route):
    """A prefill whose x and out hold more than 2^31 elements (B=1, D=16384, T=131104,
    token-major): the first and last tokens' outputs and the final state against the
    oracle (the last window starts from the three tokens before it)."""
    import depthwise_causal_conv1d_gb300 as ccu
    from oracle_pins import bf16_ulp_distance

    D, L, W, T, K = 16384, 3, 4, 131104, 40
    assert T * D > (1 << 31)
    torch.manual_seed(9)
    x_mem = torch.randn((1, T, D), dtype=torch.bfloat16, device=DEV)
    x = x_mem.permute(0, 2, 1)
    rng = np.random.default_rng(10)
    w_np = synthetic.f64_to_bf16_bits(rng.standard_normal((D, W)) * 0.5)
    b_np = synthetic.f64_to_bf16_bits(rng.standard_normal(D) * 0.1)
    out = torch.empty_like(x)
    fin = torch.empty((1, L, D), dtype=torch.bfloat16, device=DEV).permute(0, 2, 1)
    ccu.causal_conv1d_fwd(x, to_dev_u16(w_np, DEV), to_dev_u16(b_np, DEV), "silu", final_states_out=fin,
                          out=out, route=route)
    torch.cuda.synchronize()
    head_x = from_dev_u16(x_mem[0, :K])
    tail_x = from_dev_u16(x_mem[0, T - K - L:])
    head_y = from_dev_u16(out.permute(0, 2, 1)[0, :K])
    tail_y = from_dev_u16(out.permute(0, 2, 1)[0, T - K:])
    got_fin = from_dev_u16(fin[0])
    del x_mem, x, out
    torch.cuda.empty_cache()
    want_head, _ = oracle.full_causal_conv(head_x, w_np, b_np, "silu", None, L)
    init = np.ascontiguousarray(tail_x[:L].T)  # [D, L]: the three tokens before the window
    want_tail, want_fin = oracle.full_causal_conv(tail_x[L:], w_np, b_np, "silu", init, L)
    assert bf16_ulp_distance(head_y, want_head).max() <= 1
    assert bf16_ulp_distance(tail_y, want_tail).max() <= 1
    assert np.array_equal(got_fin, want_fin)


# The vector multi-token kernel at the state lengths the cases above reach only on the
# scalar route (L = 5 to 7 with D % 8 == 0), linear and ring, both layouts.
MULTI_LONG = [
    dict(N=5, D=264, T=4, L=5, S=7, ring=False, x_layout="tokens_major"),
    dict(N=4, D=136, T=6, L=6, S=6, ring=True, x_layout="tokens_major"),
    dict(N=6, D=520, T=3, L=7, S=9, ring=False, x_layout="tokens_major"),
    dict(N=3, D=72, T=9, L=7, S=5, ring=True, x_layout="tokens_major"),
]


@pytest.mark.parametrize("layout", ["compact", "channel_last"])
@pytest.mark.parametrize("ci", range(len(MULTI_LONG)))
def test_multi_token_vector_long_states(layout, ci):
    _check_multi(MULTI_LONG[ci], "vector", layout, 400 + ci)
