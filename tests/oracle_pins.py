"""Pins that tie the CPU oracle to facts outside itself.

Each ``pin_*`` function takes a loaded oracle library (``oracle.load()`` or a
deliberately broken copy) and raises AssertionError when the oracle disagrees
with the fact it is pinned to. The facts come from the cuDNN page "Causal Conv1d
Decode Update" (the update block in its introduction, the bias/activation and
conv_state_indices paragraphs, "Semantic tensor contract") and from mathematics:

- hand-worked examples with exact values (tests/golden/);
- BF16 conversion against torch's float32 <-> bfloat16 casts (round to nearest even);
- SiLU against scipy.special.expit in float64;
- one-hot weights reproduce the input delayed by W-1-k steps (exact);
- a chain of T updates equals a direct full causal convolution;
- the full convolution equals numpy.convolve in float64 within the FP32 summation
  error bound, and rounds to within one BF16 ulp of it;
- constant input with unit weights gives W*c after W-1 steps (closed form);
- padding rows give +0 and leave every slot untouched; unselected slots unchanged;
- routing through a permutation equals the unindexed update on a permuted state;
- the channel-last (L*D, 1, D) state layout gives the same result as compact.
"""

from __future__ import annotations

import os

import numpy as np

import oracle
import synthetic

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
U24 = 2.0 ** -24  # unit roundoff of FP32


# ----------------------------------------------------------------------------- helpers

def bf16_ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in BF16 steps between two arrays of BF16 bit patterns (+0 == -0)."""
    def ordered(u):
        u = u.astype(np.int32)
        mag = u & 0x7FFF
        return np.where(u & 0x8000, -mag, mag)
    return np.abs(ordered(a) - ordered(b))


def rand_bf16(rng, shape, scale=1.0):
    return synthetic.f64_to_bf16_bits(rng.standard_normal(shape) * scale)


def f32(bits):
    return synthetic.bf16_bits_to_f32(bits).astype(np.float64)


def _parse_golden(path):
    fields = {}
    with open(path) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            fields[key] = vals
    return fields


def _bits(vals):
    return synthetic.f64_to_bf16_bits(np.array([float(v) for v in vals]))


# ----------------------------------------------------------------------------- pins

def pin_golden(lib):
    for name in sorted(os.listdir(GOLDEN_DIR)):
        if not name.startswith("worked_example"):
            continue
        g = _parse_golden(os.path.join(GOLDEN_DIR, name))
        W, L, N, D, S = (int(g[k][0]) for k in ("W", "L", "N", "D", "S"))
        x = _bits(g["x"]).reshape(N, D)
        weight = _bits(g["weight"]).reshape(D, W)
        bias = None if g["bias"] == ["none"] else _bits(g["bias"])
        state = _bits(g["state"]).reshape(S, D, L)
        idx = None if g["indices"] == ["none"] else np.array([int(v) for v in g["indices"]], np.int32)
        # the stated values must be exact in BF16 or the example is not exact
        for key in ("x", "weight", "state", "expect_out", "expect_state"):
            vals = np.array([float(v) for v in g[key]])
            assert np.array_equal(f32(_bits(g[key])), vals), f"{name}: {key} not exact in BF16"
        out = oracle.conv1d_update(x, D, state, (D * L, L, 1), weight, bias, g["act"][0], idx,
                                   N, D, S, L, W, lib=lib)
        assert np.array_equal(f32(out).ravel(), np.array([float(v) for v in g["expect_out"]])), name
        assert np.array_equal(f32(state).ravel(), np.array([float(v) for v in g["expect_state"]])), name


def pin_bf16_conversion(lib):
    import torch

    rng = np.random.default_rng(1)
    words = rng.integers(0, 2 ** 32, size=4000, dtype=np.uint64).astype(np.uint32)
    # halfway and near-halfway patterns, both parities, carries into the exponent, specials
    hi = rng.integers(0, 2 ** 16, size=500, dtype=np.uint64).astype(np.uint32) << 16
    extra = np.concatenate([hi | 0x8000, hi | 0x7FFF, hi | 0x8001, hi | 0xFFFF,
                            np.array([0x7F7FFFFF, 0x7F7F8000, 0xFF7F8000, 0x00008000, 0x80018000,
                                      0x7F800000, 0xFF800000, 0x00000000, 0x80000000,
                                      0x3F808000, 0x3F818000], dtype=np.uint32)])
    words = np.concatenate([words, extra])
    vals = words.view(np.float32)
    ref = torch.from_numpy(vals.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([lib.ccu_oracle_f32_to_bf16(float(v)) for v in vals], dtype=np.uint16)
    nan = np.isnan(vals)
    assert np.array_equal(got[~nan], ref[~nan]), "float32 -> BF16 differs from torch (RNE)"
    assert np.all((got[nan] & 0x7F80) == 0x7F80) and np.all(got[nan] & 0x007F), "NaN not kept"
    b = rng.integers(0, 2 ** 16, size=3000, dtype=np.uint64).astype(np.uint16)
    wide = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).to(torch.float32).numpy()
    got_w = np.array([lib.ccu_oracle_bf16_to_f32(int(v)) for v in b], dtype=np.float32)
    fin = np.isfinite(wide)
    assert np.array_equal(got_w[fin].view(np.uint32), wide[fin].view(np.uint32))


def pin_silu(lib):
    from scipy.special import expit

    rng = np.random.default_rng(2)
    a = np.concatenate([np.linspace(-30, 30, 1201), rng.standard_normal(2000) * 4,
                        [0.0, -0.0, 1.0, -1.0, 88.0, -88.0, 200.0, -200.0]]).astype(np.float32)
    ref = (a.astype(np.float64) * expit(a.astype(np.float64))).astype(np.float32)
    got = np.array([lib.ccu_oracle_silu(float(v)) for v in a], dtype=np.float32)
    # both are float64 evaluations rounded to float32: allow one float32 step
    ulp = np.spacing(np.maximum(np.abs(ref), np.float32(1e-30))).astype(np.float64)
    assert np.all(np.abs(got.astype(np.float64) - ref) <= ulp + 1e-45), "SiLU differs from x*expit(x)"


def _chain(lib, x_seq, weight, bias, act, init_state, L):
    """Run T single-row updates on one slot; return (outputs [T, D], final state [D, L])."""
    T, D = x_seq.shape
    W = weight.shape[1]
    state = (np.zeros((1, D, L), np.uint16) if init_state is None
             else init_state.reshape(1, D, L).copy())
    outs = []
    for t in range(T):
        outs.append(oracle.conv1d_update(x_seq[t:t + 1].copy(), D, state, (D * L, L, 1), weight,
                                         bias, act, None, 1, D, 1, L, W, lib=lib)[0])
    return np.stack(outs), state[0]


def pin_one_hot(lib):
    rng = np.random.default_rng(3)
    for L in (3, 4, 6):
        W, D, T = 4, 5, 9
        x_seq = rand_bf16(rng, (T, D))
        init = rand_bf16(rng, (D, L))
        for k in range(W):
            weight = np.zeros((D, W), np.uint16)
            weight[:, k] = 0x3F80  # 1.0
            y, _ = _chain(lib, x_seq, weight, None, "identity", init, L)
            lag = W - 1 - k
            for t in range(T):
                src = t - lag
                want = x_seq[src] if src >= 0 else init[:, L + src]
                assert np.array_equal(f32(y[t]), f32(want)), f"one-hot k={k} L={L} t={t}"


def pin_chain_vs_full(lib):
    rng = np.random.default_rng(4)
    for L, act, with_bias, with_init in [(3, "identity", False, False), (3, "silu", True, True),
                                         (4, "identity", True, True), (8, "silu", False, True),
                                         (5, "silu", True, False)]:
        W, D, T = 4, 17, 16
        x_seq = rand_bf16(rng, (T, D))
        weight = rand_bf16(rng, (D, W), 0.5)
        bias = rand_bf16(rng, (D,), 0.1) if with_bias else None
        init = rand_bf16(rng, (D, L)) if with_init else None
        y_chain, st_chain = _chain(lib, x_seq, weight, bias, act, init, L)
        y_full, st_full = oracle.full_causal_conv(x_seq, weight, bias, act, init, L, lib=lib)
        assert np.array_equal(st_chain, st_full), f"state after chain L={L}"
        assert np.all(bf16_ulp_distance(y_chain, y_full) == 0), f"chain vs full L={L} {act}"
        # after T >= L steps the state is exactly the last L inputs
        assert np.array_equal(st_chain, x_seq[T - L:].T), "state != last L inputs"


def pin_full_vs_convolve(lib):
    rng = np.random.default_rng(5)
    for L, with_bias, with_init in [(3, False, False), (3, True, True), (6, True, True)]:
        W, D, T = 4, 9, 20
        x_seq = rand_bf16(rng, (T, D))
        weight = rand_bf16(rng, (D, W), 0.5)
        bias = rand_bf16(rng, (D,), 0.1) if with_bias else None
        init = rand_bf16(rng, (D, L)) if with_init else None
        y, fin, acc = oracle.full_causal_conv(x_seq, weight, bias, "identity", init, L,
                                              with_acc=True, lib=lib)
        for d in range(D):
            prev = f32(init[d, L - (W - 1):]) if init is not None else np.zeros(W - 1)
            xx = np.concatenate([prev, f32(x_seq[:, d])])
            w_rev = f32(weight[d, ::-1])
            exact = np.convolve(xx, w_rev, mode="valid")
            mag = np.convolve(np.abs(xx), np.abs(w_rev), mode="valid")
            if bias is not None:
                exact = exact + f32(bias[d:d + 1])[0]
                mag = mag + abs(f32(bias[d:d + 1])[0])
            n_terms = W + (1 if bias is not None else 0)
            bound = (n_terms - 1) * U24 * mag * (1 + 1e-6) + 1e-45
            assert np.all(np.abs(acc[:, d].astype(np.float64) - exact) <= bound), f"d={d}"
            assert np.all(bf16_ulp_distance(y[:, d], synthetic.f64_to_bf16_bits(exact)) <= 1)
        hist = np.concatenate([init.T if init is not None else np.zeros((L, D), np.uint16), x_seq])
        assert np.array_equal(fin, hist[-L:].T), "final state != last L of the history"


def pin_closed_form(lib):
    # constant x = c, weight = 1: outputs c, 2c, 3c, then 4c for every later step
    for c in (1.5, -0.375, 3.0):
        W, D, L, T = 4, 3, 3, 7
        x_seq = np.tile(synthetic.f64_to_bf16_bits(np.array([c])), (T, D))
        weight = np.full((D, W), 0x3F80, np.uint16)
        y, _ = _chain(lib, x_seq, weight, None, "identity", None, L)
        want = [min(t + 1, W) * c for t in range(T)]
        assert np.array_equal(f32(y), np.repeat(np.array(want)[:, None], D, axis=1)), c


def pin_padding_and_untouched(lib):
    rng = np.random.default_rng(6)
    N, D, S, L, W = 6, 11, 10, 4, 4
    x = rand_bf16(rng, (N, D))
    weight = rand_bf16(rng, (D, W))
    bias = rand_bf16(rng, (D,), 0.1)
    state = rand_bf16(rng, (S, D, L))
    idx = np.array([7, -1, 2, -1, 9, -1], np.int32)
    before = state.copy()
    out = oracle.conv1d_update(x, D, state, (D * L, L, 1), weight, bias, "silu", idx,
                               N, D, S, L, W, lib=lib)
    for n in np.flatnonzero(idx == -1):
        assert np.all(out[n] == 0x0000), "padding row output must be +0"
    untouched = sorted(set(range(S)) - set(int(s) for s in idx if s >= 0))
    assert np.array_equal(state[untouched], before[untouched]), "unselected slot changed"
    for n, s in enumerate(idx):
        if s >= 0:  # a selected slot takes the row's input as its newest entry
            assert np.array_equal(state[s][:, L - 1], x[n]), "selected slot missing its input"


def pin_routing(lib):
    rng = np.random.default_rng(7)
    N, D, L, W = 7, 13, 3, 4
    x = rand_bf16(rng, (N, D))
    weight = rand_bf16(rng, (D, W))
    bias = rand_bf16(rng, (D,), 0.1)
    state = rand_bf16(rng, (N, D, L))
    perm = rng.permutation(N).astype(np.int32)
    st_idx = state.copy()
    out_idx = oracle.conv1d_update(x, D, st_idx, (D * L, L, 1), weight, bias, "silu", perm,
                                   N, D, N, L, W, lib=lib)
    st_plain = state[perm].copy()  # row n's slot moved to position n
    out_plain = oracle.conv1d_update(x, D, st_plain, (D * L, L, 1), weight, bias, "silu", None,
                                     N, D, N, L, W, lib=lib)
    assert np.array_equal(out_idx, out_plain), "routing changes the output"
    assert np.array_equal(st_idx[perm], st_plain), "routing changes the state"


def pin_layouts(lib):
    rng = np.random.default_rng(8)
    for L in (3, 5):
        N, D, W = 4, 10, 4
        x = rand_bf16(rng, (N, D))
        weight = rand_bf16(rng, (D, W))
        state = rand_bf16(rng, (N, D, L))
        st_c = state.copy()
        out_c = oracle.conv1d_update(x, D, st_c, (D * L, L, 1), weight, None, "identity", None,
                                     N, D, N, L, W, lib=lib)
        st_t = synthetic.to_channel_last(state)
        out_t = oracle.conv1d_update(x, D, st_t, (L * D, 1, D), weight, None, "identity", None,
                                     N, D, N, L, W, lib=lib)
        assert np.array_equal(out_c, out_t), "layout changes the output"
        assert np.array_equal(st_c, synthetic.from_channel_last(st_t)), "layout changes the state"


def pin_padded_ld(lib):
    # columns D..ld-1 of x hold NaN canaries: they must not reach the output
    rng = np.random.default_rng(9)
    N, D, ld, L, W = 3, 6, 16, 3, 4
    x = np.full((N, ld), synthetic.BF16_NAN_BITS, np.uint16)
    x[:, :D] = rand_bf16(rng, (N, D))
    weight = rand_bf16(rng, (D, W))
    state = rand_bf16(rng, (N, D, L))
    st_pad = state.copy()
    out_pad = oracle.conv1d_update(x, ld, st_pad, (D * L, L, 1), weight, None, "identity", None,
                                   N, D, N, L, W, lib=lib)
    st_c = state.copy()
    out_c = oracle.conv1d_update(np.ascontiguousarray(x[:, :D]), D, st_c, (D * L, L, 1), weight,
                                 None, "identity", None, N, D, N, L, W, lib=lib)
    assert np.array_equal(out_pad, out_c) and np.array_equal(st_pad, st_c)
    assert not np.any(np.isnan(f32(out_pad)))


def pin_check_indices(lib):
    assert oracle.check_indices(np.array([0, 1, 2], np.int32), 3, 3, lib=lib) == 0
    assert oracle.check_indices(np.array([-1, -1, 2], np.int32), 3, 3, lib=lib) == 0
    assert oracle.check_indices(np.array([0, 3, 1], np.int32), 3, 3, lib=lib) == oracle.IDX_RANGE
    assert oracle.check_indices(np.array([0, -2, 1], np.int32), 3, 3, lib=lib) == oracle.IDX_RANGE
    assert oracle.check_indices(np.array([1, 1, 0], np.int32), 3, 3, lib=lib) == oracle.IDX_DUPLICATE
    assert oracle.check_indices(np.array([5, 1, 1], np.int32), 3, 3, lib=lib) == (
        oracle.IDX_RANGE | oracle.IDX_DUPLICATE)


def _rotate(ring, p):
    """The linear state a ring represents when its oldest entry sits at position p."""
    L = ring.shape[-1]
    return np.ascontiguousarray(ring[..., [(p + i) % L for i in range(L)]])


def pin_circular_equals_linear_through_rotation(lib):
    # Reading the ring from p gives the linear state: the ring update must produce the
    # linear update's output, and its new ring read from p + 1 must be the linear new state.
    rng = np.random.default_rng(10)
    for L in (3, 4, 7):
        N, D, W = 5, 9, 4
        x = rand_bf16(rng, (N, D))
        weight = rand_bf16(rng, (D, W))
        bias = rand_bf16(rng, (D,), 0.1)
        ring = rand_bf16(rng, (N, D, L))
        seqlens = np.array([0, 1, L - 1, L + 2, 1000 * L + 5], np.int32)
        ring_after = ring.copy()
        out_c = oracle.conv1d_update_circular(x, D, ring_after, (D * L, L, 1), weight, bias, "silu",
                                              None, seqlens, N, D, N, L, W, lib=lib)
        lin = np.ascontiguousarray(np.stack([_rotate(ring[n], int(seqlens[n]) % L) for n in range(N)]))
        out_l = oracle.conv1d_update(x, D, lin, (D * L, L, 1), weight, bias, "silu", None,
                                     N, D, N, L, W, lib=lib)
        assert np.array_equal(out_c, out_l), f"ring output differs from the linear one (L={L})"
        for n in range(N):
            p1 = (int(seqlens[n]) + 1) % L
            assert np.array_equal(_rotate(ring_after[n], p1), lin[n]), f"ring state (L={L}, n={n})"


def pin_circular_writes_one_entry(lib):
    rng = np.random.default_rng(11)
    N, D, L, W, S = 4, 6, 5, 4, 7
    x = rand_bf16(rng, (N, D))
    weight = rand_bf16(rng, (D, W))
    ring = rand_bf16(rng, (S, D, L))
    idx = np.array([6, -1, 0, 3], np.int32)
    seqlens = np.array([2, -7, 9, 0], np.int32)  # a padding row's value is never used
    after = ring.copy()
    out = oracle.conv1d_update_circular(x, D, after, (D * L, L, 1), weight, None, "identity", idx,
                                        seqlens, N, D, S, L, W, lib=lib)
    assert np.all(out[1] == 0)
    for n, s in enumerate(idx):
        if s < 0:
            continue
        p = int(seqlens[n]) % L
        changed = np.argwhere(after[s] != ring[s])
        assert set(changed[:, 1].tolist()) <= {p}, "an entry other than the oldest changed"
        assert np.array_equal(after[s][:, p], x[n])
    untouched = [1, 2, 4, 5]
    assert np.array_equal(after[untouched], ring[untouched])


def pin_circular_chain_vs_full(lib):
    # A ring fed T inputs with cache_seqlens 0, 1, 2, ... equals the direct convolution.
    rng = np.random.default_rng(12)
    for L in (3, 6):
        W, D, T = 4, 11, 14
        x_seq = rand_bf16(rng, (T, D))
        weight = rand_bf16(rng, (D, W), 0.5)
        bias = rand_bf16(rng, (D,), 0.1)
        ring = np.zeros((1, D, L), np.uint16)
        ys = []
        for t in range(T):
            ys.append(oracle.conv1d_update_circular(x_seq[t:t + 1].copy(), D, ring, (D * L, L, 1), weight,
                                                    bias, "identity", None, np.array([t], np.int32),
                                                    1, D, 1, L, W, lib=lib)[0])
        y_full, fin = oracle.full_causal_conv(x_seq, weight, bias, "identity", None, L, lib=lib)
        assert np.array_equal(np.stack(ys), y_full), f"ring chain vs full conv (L={L})"
        assert np.array_equal(_rotate(ring[0], T % L), fin), f"ring after T steps (L={L})"


def _multi_case(rng, N, D, T, L, S, ring, pad):
    x = rand_bf16(rng, (N, T, D))  # token-major memory: x[n, d, t] at n*T*D + t*D + d
    weight = rand_bf16(rng, (D, 4), 0.5)
    bias = rand_bf16(rng, (D,), 0.1)
    state = rand_bf16(rng, (S, D, L))
    idx = rng.permutation(S)[:N].astype(np.int32)
    if pad:
        idx[::3] = -1
    seq = rng.integers(0, 5 * L, size=N).astype(np.int32) if ring else None
    return x, weight, bias, state, idx, seq


def pin_multi_equals_sequential_steps(lib):
    # One call with T tokens equals T single-token updates, token by token: outputs,
    # final state and the state after every token.
    rng = np.random.default_rng(13)
    for L, T, ring in [(3, 1, False), (3, 4, False), (4, 2, True), (6, 5, False), (3, 7, True),
                       (5, 3, True)]:
        N, D, S, W = 5, 10, 8, 4
        x, weight, bias, state, idx, seq = _multi_case(rng, N, D, T, L, S, ring, pad=True)
        st_multi = state.copy()
        out, inter = oracle.conv1d_update_multi(x, (T * D, 1, D), st_multi, (D * L, L, 1), weight, bias,
                                                "silu", idx, seq, N, D, T, S, L, W, with_inter=True,
                                                lib=lib)
        st_seq = state.copy()
        for t in range(T):
            xt = np.ascontiguousarray(x[:, t, :])
            if ring:
                o = oracle.conv1d_update_circular(xt, D, st_seq, (D * L, L, 1), weight, bias, "silu", idx,
                                                  seq + t, N, D, S, L, W, lib=lib)
            else:
                o = oracle.conv1d_update(xt, D, st_seq, (D * L, L, 1), weight, bias, "silu", idx,
                                         N, D, S, L, W, lib=lib)
            assert np.array_equal(out[:, :, t], o), f"token {t} output (L={L}, T={T}, ring={ring})"
            for n, s in enumerate(idx):
                if s >= 0:
                    assert np.array_equal(inter[n, t], st_seq[s]), f"state after token {t}"
        assert np.array_equal(st_multi, st_seq), f"final state (L={L}, T={T}, ring={ring})"


def pin_multi_x_layouts(lib):
    rng = np.random.default_rng(14)
    N, D, T, L, S, W = 4, 9, 3, 4, 4, 4
    x, weight, bias, state, idx, _ = _multi_case(rng, N, D, T, L, S, False, pad=False)
    st_a = state.copy()
    out_a = oracle.conv1d_update_multi(x, (T * D, 1, D), st_a, (D * L, L, 1), weight, bias, "identity",
                                       idx, None, N, D, T, S, L, W, lib=lib)
    x_dt = np.ascontiguousarray(np.transpose(x, (0, 2, 1)))  # [N, D, T] memory
    st_b = state.copy()
    out_b = oracle.conv1d_update_multi(x_dt, (D * T, T, 1), st_b, (D * L, L, 1), weight, bias,
                                       "identity", idx, None, N, D, T, S, L, W, lib=lib)
    assert np.array_equal(out_a, out_b) and np.array_equal(st_a, st_b)


def pin_multi_vs_full(lib):
    rng = np.random.default_rng(15)
    D, T, L, W = 7, 9, 3, 4
    x_seq = rand_bf16(rng, (T, D))
    weight = rand_bf16(rng, (D, W))
    init = rand_bf16(rng, (D, L))
    st = init.reshape(1, D, L).copy()
    out = oracle.conv1d_update_multi(np.ascontiguousarray(x_seq.reshape(1, T, D)), (T * D, 1, D), st,
                                     (D * L, L, 1), weight, None, "identity", None, None, 1, D, T, 1,
                                     L, W, lib=lib)
    y, fin = oracle.full_causal_conv(x_seq, weight, None, "identity", init, L, lib=lib)
    assert np.array_equal(out[0].T, y) and np.array_equal(st[0], fin)


def pin_widths_one_hot_and_chain(lib):
    # Widths other than 4 (the page's other "semantically valid widths": 1, 2, 3 and wider
    # ones), L from max(W - 1, 1) up: one-hot weights reproduce x delayed by W-1-k steps; a
    # chain of updates equals the direct convolution; the direct convolution equals
    # numpy.convolve within the FP32 bound.
    rng = np.random.default_rng(16)
    for W in (1, 2, 3, 5, 7):
        for L in sorted({max(W - 1, 1), W, max(5, W + 1)}):
            D, T = 6, 9
            x_seq = rand_bf16(rng, (T, D))
            init = rand_bf16(rng, (D, L))
            for k in range(W):
                weight = np.zeros((D, W), np.uint16)
                weight[:, k] = 0x3F80
                y, _ = _chain(lib, x_seq, weight, None, "identity", init, L)
                for t in range(T):
                    src = t - (W - 1 - k)
                    want = x_seq[src] if src >= 0 else init[:, L + src]
                    assert np.array_equal(f32(y[t]), f32(want)), f"one-hot W={W} L={L} k={k} t={t}"
            weight = rand_bf16(rng, (D, W), 0.5)
            bias = rand_bf16(rng, (D,), 0.1)
            y_chain, st_chain = _chain(lib, x_seq, weight, bias, "silu", init, L)
            y_full, st_full, acc = oracle.full_causal_conv(x_seq, weight, bias, "silu", init, L,
                                                           with_acc=True, lib=lib)
            assert np.array_equal(y_chain, y_full) and np.array_equal(st_chain, st_full), f"W={W} L={L}"
            for d in range(D):
                xx = np.concatenate([f32(init[d, L - (W - 1):]) if W > 1 else np.zeros(0),
                                     f32(x_seq[:, d])])
                exact = np.convolve(xx, f32(weight[d, ::-1]), mode="valid") + f32(bias[d:d + 1])[0]
                mag = np.convolve(np.abs(xx), np.abs(f32(weight[d, ::-1])), mode="valid") + abs(
                    f32(bias[d:d + 1])[0])
                assert np.all(np.abs(acc[:, d] - exact) <= W * U24 * mag * (1 + 1e-6) + 1e-45)


def pin_widths_multi_and_ring(lib):
    # The multi-token and ring forms at widths other than 4 equal the single-token linear steps.
    rng = np.random.default_rng(17)
    for W, L, T in [(2, 1, 3), (3, 2, 4), (2, 3, 2), (3, 5, 6), (1, 1, 3), (1, 4, 2), (5, 4, 5),
                    (7, 9, 3)]:
        N, D, S = 3, 5, 4
        x = rand_bf16(rng, (N, T, D))
        weight = rand_bf16(rng, (D, W))
        state = rand_bf16(rng, (S, D, L))
        idx = np.array([3, -1, 0], np.int32)
        st_multi = state.copy()
        out = oracle.conv1d_update_multi(x, (T * D, 1, D), st_multi, (D * L, L, 1), weight, None,
                                         "identity", idx, None, N, D, T, S, L, W, lib=lib)
        st_seq = state.copy()
        for t in range(T):
            o = oracle.conv1d_update(np.ascontiguousarray(x[:, t]), D, st_seq, (D * L, L, 1), weight,
                                     None, "identity", idx, N, D, S, L, W, lib=lib)
            assert np.array_equal(out[:, :, t], o), f"W={W} L={L} token {t}"
        assert np.array_equal(st_multi, st_seq)
        ring = state.copy()
        seq = np.array([L + 1, 0, 7], np.int32)
        out_r = oracle.conv1d_update_circular(np.ascontiguousarray(x[:, 0]), D, ring, (D * L, L, 1),
                                              weight, None, "identity", idx, seq, N, D, S, L, W, lib=lib)
        lin = state.copy()
        for n, s in enumerate(idx):
            if s >= 0:
                lin[s] = _rotate(state[s], int(seq[n]) % L)
        out_l = oracle.conv1d_update(np.ascontiguousarray(x[:, 0]), D, lin, (D * L, L, 1), weight, None,
                                     "identity", idx, N, D, S, L, W, lib=lib)
        assert np.array_equal(out_r, out_l), f"ring W={W} L={L}"


ALL_PINS = [pin_golden, pin_bf16_conversion, pin_silu, pin_one_hot, pin_chain_vs_full,
            pin_full_vs_convolve, pin_closed_form, pin_padding_and_untouched, pin_routing,
            pin_layouts, pin_padded_ld, pin_check_indices,
            pin_circular_equals_linear_through_rotation, pin_circular_writes_one_entry,
            pin_circular_chain_vs_full, pin_multi_equals_sequential_steps, pin_multi_x_layouts,
            pin_multi_vs_full, pin_widths_one_hot_and_chain, pin_widths_multi_and_ring]
