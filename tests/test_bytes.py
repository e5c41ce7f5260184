"""The benchmark's byte counts (the numerator of every roofline fraction), checked on CPU
against totals worked out by hand from the method's accounting:

- an active (row, channel) element reads x (2 B) and the L state entries (2L B) and writes
  the L new entries (2L B) and the output (2 B); a padding row's element only writes its
  zero output (2 B); weight (2DW B), bias (2D B) and indices (4N B) are read once;
- T tokens per row move 4T B of x and output and the state once (4L B);
- a ring-buffer state needs only the W - 1 window entries read and the newest entry (or
  min(T, L) of them) written, plus cache_seqlens (4N B);
- the prefill moves x and out (4 B per element), the final state, weight and bias.

Only the number of padding rows enters, which the index recipe fixes at round(p * N).
"""
import numpy as np
import pytest

import synthetic


def _indices(wl):
    if wl.indices == "none":
        return None
    idx = np.arange(wl.N, dtype=np.int32)
    n_pad = int(round(wl.pad_frac * wl.N))
    idx[:n_pad] = -1
    return idx


# name -> (active rows, padding rows, total bytes worked out by hand)
DECODE = {
    # 8 x 2048 x (2 + 6 + 6 + 2) + weight 2048 x 4 x 2
    "decode_n8_d2048_l3_identity": 8 * 2048 * 16 + 16384,
    # 8 x 2048 x (2 + 8 + 8 + 2) + weight + bias 2048 x 2
    "decode_n8_d2048_l4_bias_silu": 8 * 2048 * 20 + 16384 + 4096,
    # 230 active and 26 padding rows of 8192; weight 65536, bias 16384, indices 1024
    "paged_n256_d8192_l3_s1024_pad10_silu": 230 * 8192 * 16 + 26 * 8192 * 2 + 65536 + 16384 + 1024,
    # 64 rows of 6144 at L = 8: 2 + 16 + 16 + 2 = 36 B; weight 49152, indices 256
    "strided_n64_d6144_ld6152_l8_perm_identity": 64 * 6144 * 36 + 49152 + 256,
    # 3891 active and 205 padding rows of 16384; weight 131072, bias 32768, indices 16384
    "large_n4096_d16384_l3_perm_pad5_silu": 3891 * 16384 * 16 + 205 * 16384 * 2 + 131072 + 32768 + 16384,
}


@pytest.mark.parametrize("name", list(DECODE))
def test_decode_bytes(name):
    wl = synthetic.WORKLOADS[name]
    assert synthetic.algorithmic_bytes(wl, _indices(wl)) == DECODE[name]


def test_decode_bytes_match_the_published_table():
    # the per-config totals of the measurement plan (C1..C5)
    assert [DECODE[n] for n in synthetic.WORKLOADS] == [278_528, 348_160, 30_655_488, 14_205_184,
                                                        1_026_899_968]


def test_ring_and_width_bytes():
    base = 3891 * 16384
    pad = 205 * 16384 * 2
    w4 = 131072 + 32768 + 16384
    ring = synthetic.RING_WORKLOADS["large_n4096_d16384_l3_perm_pad5_silu_ring"]
    # x 2 + window 2 x 3 + one entry 2 + out 2 = 12 B; cache_seqlens 4N
    assert synthetic.algorithmic_bytes(ring, _indices(ring)) == base * 12 + pad + w4 + 4 * 4096
    w3 = synthetic.WIDTH_WORKLOADS["large_n4096_d16384_w3_l2_perm_pad5_silu"]
    # L = 2: 2 + 4 + 4 + 2 = 12 B; weight [D, 3]
    assert synthetic.algorithmic_bytes(w3, _indices(w3)) == base * 12 + pad + 16384 * 3 * 2 + 32768 + 16384
    w2 = synthetic.WIDTH_WORKLOADS["large_n4096_d16384_w2_l1_perm_pad5_silu"]
    # L = 1: 2 + 2 + 2 + 2 = 8 B; weight [D, 2]
    assert synthetic.algorithmic_bytes(w2, _indices(w2)) == base * 8 + pad + 16384 * 2 * 2 + 32768 + 16384
    w5 = synthetic.WIDTH_WORKLOADS["large_n4096_d16384_w5_l4_perm_pad5_silu"]
    # L = 4: 2 + 8 + 8 + 2 = 20 B; weight [D, 5]
    assert synthetic.algorithmic_bytes(w5, _indices(w5)) == base * 20 + pad + 16384 * 5 * 2 + 32768 + 16384


def test_multi_token_bytes():
    active = (1024 - 51) * 16384  # 51 = round(0.05 * 1024) padding rows
    pad = 51 * 16384 * 2 * 4      # their zero outputs, four tokens
    extra = 16384 * 2 + 4096      # bias, indices
    wl = synthetic.MULTI_WORKLOADS
    l3 = wl["multi_n1024_d16384_t4_l3_bias_silu"]
    assert synthetic.algorithmic_bytes(l3, _indices(l3)) == active * (16 + 12) + pad + 131072 + extra
    l5 = wl["multi_n1024_d16384_t4_l5_bias_silu"]
    assert synthetic.algorithmic_bytes(l5, _indices(l5)) == active * (16 + 20) + pad + 131072 + extra
    l8 = wl["multi_n1024_d16384_t4_l8_bias_silu"]
    assert synthetic.algorithmic_bytes(l8, _indices(l8)) == active * (16 + 32) + pad + 131072 + extra
    w3 = wl["multi_n1024_d16384_t4_w3_l2_bias_silu"]
    assert synthetic.algorithmic_bytes(w3, _indices(w3)) == active * (16 + 8) + pad + 16384 * 3 * 2 + extra
    ring = wl["multi_n1024_d16384_t4_l5_ring_bias_silu"]
    # window 2 x 3 read, min(T, L) = 4 entries written, cache_seqlens 4N
    assert synthetic.algorithmic_bytes(ring, _indices(ring)) == active * (16 + 6 + 8) + pad + 131072 + extra + 4096
    # the values the benchmark prints
    assert synthetic.algorithmic_bytes(l3, _indices(l3)) == 453_218_304
    assert synthetic.algorithmic_bytes(ring, _indices(ring)) == 485_105_664


def test_prefill_bytes():
    w4 = synthetic.PREFILL_WORKLOADS["prefill_b8_t4096_d4096_bias_silu"]
    # x and out 4 B per element, final state [8, 4096, 3], weight [4096, 4], bias
    assert synthetic.prefill_bytes(w4) == 8 * 4096 * 4096 * 4 + 8 * 4096 * 3 * 2 + 4096 * 8 + 4096 * 2
    assert synthetic.prefill_bytes(w4) == 537_108_480
    w3 = synthetic.PREFILL_WORKLOADS["prefill_b8_t4096_d4096_w3_bias_silu"]
    assert synthetic.prefill_bytes(w3) == 8 * 4096 * 4096 * 4 + 8 * 4096 * 2 * 2 + 4096 * 6 + 4096 * 2
