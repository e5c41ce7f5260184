"""Seeded synthetic inputs for the depthwise causal conv1d decode update.

This module only draws numbers and arranges them. It holds none of the
update's arithmetic (no history, no shift, no dot product, no activation), so
both sides of a parity test -- the CUDA path and the CPU oracle -- can take
their inputs from it without sharing any of the method.

Every BF16 tensor is returned as a ``numpy.uint16`` array of bit patterns.
Values are drawn in float64 from ``numpy.random.Generator(PCG64(seed))``,
rounded to float32 by numpy, then rounded to BF16 with round-to-nearest-even
on the float32 bit pattern. Tensors are drawn in a fixed order: x, weight,
conv_state, bias, indices.

The workloads are the five decode shapes this library is measured and tested
on. Their distributions follow the tensor contract of the cuDNN page "Causal
Conv1d Decode Update" (section "Semantic tensor contract"); its "Python API"
example (N=8, D=2048, W=4, L=4, SiLU) is the shape of ``decode_n8_d2048_l4``.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

BF16_NAN_BITS = 0x7FC0  # canary written into padded x columns that must never be read
_CHUNK = 1 << 24  # elements drawn per generator call; bounds host memory


@dataclasses.dataclass(frozen=True)
class Workload:
    """One decode-update workload, named by what it is."""

    name: str
    N: int  # rows in the decode batch
    D: int  # channels
    W: int  # filter width
    L: int  # conv_state length, L >= W - 1
    S: int  # cache slots in conv_state
    ld: int  # row stride of x in elements (ld == D: compact)
    x_dist: tuple  # ("normal", std) or ("uniform", lo, hi); also used for conv_state
    w_dist: tuple  # distribution of weight
    bias_std: Optional[float]  # None: no bias
    act: str  # "identity" or "silu"
    indices: str  # "none", "perm", "distinct", "perm_pad", "distinct_pad"
    pad_frac: float = 0.0  # fraction of rows set to -1 (padding)
    layout: str = "compact"  # "compact" (D*L, L, 1) or "channel_last" (L*D, 1, D)
    seed: int = 0
    ring: bool = False  # ring-buffer state: draw cache_seqlens [N]
    T: int = 1  # tokens per row; T > 1: x is drawn as [N, T, D] (token-major), ld == D

    @property
    def has_bias(self) -> bool:
        return self.bias_std is not None


WORKLOADS = {
    w.name: w
    for w in [
        Workload("decode_n8_d2048_l3_identity", N=8, D=2048, W=4, L=3, S=8, ld=2048,
                 x_dist=("normal", 1.0), w_dist=("normal", 1.0), bias_std=None,
                 act="identity", indices="none"),
        Workload("decode_n8_d2048_l4_bias_silu", N=8, D=2048, W=4, L=4, S=8, ld=2048,
                 x_dist=("normal", 1.0), w_dist=("normal", 1.0), bias_std=0.1,
                 act="silu", indices="none"),
        Workload("paged_n256_d8192_l3_s1024_pad10_silu", N=256, D=8192, W=4, L=3, S=1024,
                 ld=8192, x_dist=("normal", 1.0), w_dist=("normal", 1.0), bias_std=0.1,
                 act="silu", indices="distinct_pad", pad_frac=0.10),
        Workload("strided_n64_d6144_ld6152_l8_perm_identity", N=64, D=6144, W=4, L=8, S=64,
                 ld=6152, x_dist=("uniform", -2.0, 2.0), w_dist=("normal", 0.5),
                 bias_std=None, act="identity", indices="perm"),
        Workload("large_n4096_d16384_l3_perm_pad5_silu", N=4096, D=16384, W=4, L=3, S=4096,
                 ld=16384, x_dist=("normal", 1.0), w_dist=("normal", 1.0), bias_std=0.1,
                 act="silu", indices="perm_pad", pad_frac=0.05),
    ]
}

# Ring-buffer variants of the large-batch decode (conv_state used as a ring indexed by
# cache_seqlens), in both state layouts. Measured beside the workloads above.
RING_WORKLOADS = {
    w.name: w
    for w in [
        dataclasses.replace(WORKLOADS["large_n4096_d16384_l3_perm_pad5_silu"],
                            name="large_n4096_d16384_l3_perm_pad5_silu_ring", ring=True),
        dataclasses.replace(WORKLOADS["large_n4096_d16384_l3_perm_pad5_silu"],
                            name="large_n4096_d16384_l3_perm_pad5_silu_ring_chlast", ring=True,
                            layout="channel_last"),
    ]
}

# Other widths (the shortest state each allows, L = W - 1) on the large-batch decode.
WIDTH_WORKLOADS = {
    w.name: w
    for w in [
        dataclasses.replace(WORKLOADS["large_n4096_d16384_l3_perm_pad5_silu"],
                            name="large_n4096_d16384_w3_l2_perm_pad5_silu", W=3, L=2),
        dataclasses.replace(WORKLOADS["large_n4096_d16384_l3_perm_pad5_silu"],
                            name="large_n4096_d16384_w2_l1_perm_pad5_silu", W=2, L=1),
        # a width above the page's four (the scalar kernel)
        dataclasses.replace(WORKLOADS["large_n4096_d16384_l3_perm_pad5_silu"],
                            name="large_n4096_d16384_w5_l4_perm_pad5_silu", W=5, L=4),
    ]
}

# Multi-token update: four tokens per row in one call (x token-major [N, T, D]), at the
# width-4 window-only state (L = 3), at longer states (L = 5, 8), at width 3 (L = 2), and with
# a ring-buffer state (L = 5, cache_seqlens drawn as for RING_WORKLOADS).
_MULTI_BASE = Workload("multi_n1024_d16384_t4_l3_bias_silu", N=1024, D=16384, W=4, L=3, S=1024, ld=16384,
                       x_dist=("normal", 1.0), w_dist=("normal", 1.0), bias_std=0.1, act="silu",
                       indices="perm_pad", pad_frac=0.05, T=4)
MULTI_WORKLOADS = {
    w.name: w
    for w in [
        _MULTI_BASE,
        dataclasses.replace(_MULTI_BASE, name="multi_n1024_d16384_t4_l5_bias_silu", L=5),
        dataclasses.replace(_MULTI_BASE, name="multi_n1024_d16384_t4_l8_bias_silu", L=8),
        dataclasses.replace(_MULTI_BASE, name="multi_n1024_d16384_t4_w3_l2_bias_silu", W=3, L=2),
        dataclasses.replace(_MULTI_BASE, name="multi_n1024_d16384_t4_l5_ring_bias_silu", L=5, ring=True),
    ]
}

# Full-sequence prefill: B sequences of T tokens (x token-major [B, T, D]), final state
# L = 3 in the channel-last layout the decode update continues from.
PREFILL_WORKLOADS = {
    "prefill_b8_t4096_d4096_bias_silu": dict(B=8, T=4096, D=4096, L=3, W=4, act="silu", bias_std=0.1,
                                             seed=0),
    "prefill_b8_t4096_d4096_w3_bias_silu": dict(B=8, T=4096, D=4096, L=2, W=3, act="silu", bias_std=0.1,
                                                seed=0),
}


def generate_prefill(spec: dict):
    """x [B, T, D], weight [D, W], bias [D] as BF16 bits, drawn in that order."""
    rng = np.random.Generator(np.random.PCG64(spec["seed"]))
    x = _draw(rng, ("normal", 1.0), spec["B"] * spec["T"] * spec["D"]).reshape(spec["B"], spec["T"], spec["D"])
    weight = _draw(rng, ("normal", 1.0), spec["D"] * spec["W"]).reshape(spec["D"], spec["W"])
    bias = _draw(rng, ("normal", spec["bias_std"]), spec["D"]) if spec["bias_std"] is not None else None
    return x, weight, bias


def prefill_bytes(spec: dict) -> int:
    """x read + out write (2 B each per element), final state written, weight and bias read."""
    B, T, D, L, W = spec["B"], spec["T"], spec["D"], spec["L"], spec["W"]
    return B * T * D * 4 + B * D * L * 2 + D * W * 2 + (D * 2 if spec["bias_std"] is not None else 0)


# The workload the benchmark times: the bandwidth-bound large-batch decode.
BENCH_WORKLOAD = "large_n4096_d16384_l3_perm_pad5_silu"
# The small page-shaped case used by the smoke run.
SMOKE_WORKLOAD = "decode_n8_d2048_l4_bias_silu"


def f64_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float64 -> float32 (numpy, RNE) -> BF16 bits (RNE on the float32 pattern).

    Only finite inputs are expected; this is input preparation, not a kernel.
    """
    u = np.asarray(a, dtype=np.float64).astype(np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _draw(rng: np.random.Generator, dist: tuple, count: int) -> np.ndarray:
    """Draw ``count`` BF16 values in chunks of _CHUNK (same stream as one big draw)."""
    out = np.empty(count, dtype=np.uint16)
    for lo in range(0, count, _CHUNK):
        n = min(_CHUNK, count - lo)
        if dist[0] == "normal":
            v = rng.standard_normal(n) * dist[1]
        elif dist[0] == "uniform":
            v = rng.uniform(dist[1], dist[2], n)
        else:
            raise ValueError(f"unknown distribution {dist!r}")
        out[lo:lo + n] = f64_to_bf16_bits(v)
    return out


def make_indices(rng: np.random.Generator, kind: str, N: int, S: int, pad_frac: float):
    """int32 slot indices [N] or None.

    perm: a permutation of 0..S-1 (S == N). distinct: the first N entries of a
    permutation of 0..S-1. The *_pad kinds then set round(pad_frac*N) rows,
    chosen by a second permutation, to -1.
    """
    if kind == "none":
        return None
    if kind in ("perm", "perm_pad"):
        if S != N:
            raise ValueError("a permutation needs S == N")
        idx = rng.permutation(S).astype(np.int32)
    elif kind in ("distinct", "distinct_pad"):
        if S < N:
            raise ValueError("distinct slots need S >= N")
        idx = rng.permutation(S)[:N].astype(np.int32)
    else:
        raise ValueError(f"unknown index kind {kind!r}")
    if kind.endswith("_pad"):
        n_pad = int(round(pad_frac * N))
        rows = rng.permutation(N)[:n_pad]
        idx[rows] = -1
    return idx


def to_channel_last(state: np.ndarray) -> np.ndarray:
    """Store a logical [S, D, L] state as [S, L, D] memory: element strides (L*D, 1, D).

    Always a fresh array (a transpose with a size-1 axis would otherwise come back as a
    view sharing memory with ``state``)."""
    return np.array(np.transpose(state, (0, 2, 1)), order="C", copy=True)


def from_channel_last(storage: np.ndarray) -> np.ndarray:
    """Inverse of to_channel_last: [S, L, D] memory back to a logical [S, D, L] array (a copy)."""
    return np.array(np.transpose(storage, (0, 2, 1)), order="C", copy=True)


@dataclasses.dataclass
class Inputs:
    """Host copies of one workload's tensors (BF16 as uint16 bit patterns)."""

    wl: Workload
    x: np.ndarray  # [N, ld] (columns D..ld-1 hold NaN canaries), or [N, T, D] when T > 1
    weight: np.ndarray  # [D, W]
    conv_state: np.ndarray  # logical [S, D, L], compact
    bias: Optional[np.ndarray]  # [D] or None
    indices: Optional[np.ndarray]  # int32 [N] or None
    cache_seqlens: Optional[np.ndarray] = None  # int32 [N] for a ring-buffer state, else None


def generate(wl: Workload, seed: Optional[int] = None) -> Inputs:
    """Draw one workload's inputs from its seed (x, weight, conv_state, bias, indices, and
    for a ring-buffer state cache_seqlens: counts uniform in [0, 2^20))."""
    rng = np.random.Generator(np.random.PCG64(wl.seed if seed is None else seed))
    N, D, W, L, S, ld = wl.N, wl.D, wl.W, wl.L, wl.S, wl.ld
    if wl.T > 1:
        x = _draw(rng, wl.x_dist, N * wl.T * D).reshape(N, wl.T, D)
    else:
        x = np.full((N, ld), BF16_NAN_BITS, dtype=np.uint16)
        x[:, :D] = _draw(rng, wl.x_dist, N * D).reshape(N, D)
    weight = _draw(rng, wl.w_dist, D * W).reshape(D, W)
    conv_state = _draw(rng, wl.x_dist, S * D * L).reshape(S, D, L)
    bias = _draw(rng, ("normal", wl.bias_std), D) if wl.has_bias else None
    indices = make_indices(rng, wl.indices, N, S, wl.pad_frac)
    seqlens = rng.integers(0, 1 << 20, size=N).astype(np.int32) if wl.ring else None
    return Inputs(wl, x, weight, conv_state, bias, indices, seqlens)


def variant(base: Workload, **changes) -> Workload:
    """A copy of a workload with some fields changed (sweeps and edge cases)."""
    return dataclasses.replace(base, **changes)


def algorithmic_bytes(wl: Workload, indices: Optional[np.ndarray]) -> int:
    """Bytes the update must move at minimum, by the method's own accounting.

    Active row element: 2 B x read + 2L B state read + 2L B state write + 2 B out
    write. Padding row element: 2 B out write (per token). Plus weight (2*D*W B), bias (2*D B)
    and indices (4*N B), each read once. A ring-buffer state needs only the W-1 window
    entries read and one entry written: 2 + 2(W-1) + 2 + 2 B per active element, plus
    cache_seqlens (4*N B).
    """
    n_pad = 0 if indices is None else int(np.count_nonzero(indices == -1))
    active = wl.N - n_pad
    if wl.ring:
        per_active = 2 + 2 * (wl.W - 1) + 2 + 2
    else:
        per_active = 2 + 2 * wl.L + 2 * wl.L + 2
    if wl.T > 1:  # T tokens of x and out per row; the state is read and written once
        per_active = 4 * wl.T + (2 * (wl.W - 1) + 2 * min(wl.T, wl.L) if wl.ring else 4 * wl.L)
    total = active * wl.D * per_active + n_pad * wl.D * 2 * wl.T
    total += 2 * wl.D * wl.W
    if wl.has_bias:
        total += 2 * wl.D
    if indices is not None:
        total += 4 * wl.N
    if wl.ring:
        total += 4 * wl.N
    return total
