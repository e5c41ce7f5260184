"""The CPU oracle against the facts it is pinned to (no GPU).

See tests/oracle_pins.py for what each pin checks and where the fact comes from.
"""
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
import oracle_pins

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_oracle_declines(oracle_lib):
    x = np.zeros((2, 8), np.uint16)
    w = np.zeros((8, 4), np.uint16)
    st = np.zeros((2, 8, 3), np.uint16)
    # L < W - 1 is outside the contract ("Semantic tensor contract": L >= W - 1)
    with pytest.raises(ValueError):
        oracle.conv1d_update(x, 8, st, (16, 2, 1), w, None, "identity", None, 2, 8, 2, 2, 4,
                             lib=oracle_lib)
    # duplicate slots break the uniqueness precondition
    with pytest.raises(ValueError):
        oracle.conv1d_update(x, 8, st, (24, 3, 1), w, None, "identity",
                             np.array([1, 1], np.int32), 2, 8, 2, 3, 4, lib=oracle_lib)
    # out-of-range slot
    with pytest.raises(ValueError):
        oracle.conv1d_update(x, 8, st, (24, 3, 1), w, None, "identity",
                             np.array([0, 2], np.int32), 2, 8, 2, 3, 4, lib=oracle_lib)
    # ld < D
    with pytest.raises(ValueError):
        oracle.conv1d_update(x, 4, st, (24, 3, 1), w, None, "identity", None, 2, 8, 2, 3, 4,
                             lib=oracle_lib)


# Planted mistakes: each is a plausible slip in the oracle's source. Every one of
# them must be caught by at least one pin, or the pins do not pin the oracle.
MUTATIONS = [
    ("taps reversed in the update", "float w = ccu_oracle_bf16_to_f32(weight[d * W + j]);",
     "float w = ccu_oracle_bf16_to_f32(weight[d * W + (W - 1 - j)]);"),
    ("history window off by one", "float h = ccu_oracle_bf16_to_f32(history[(L + 1) - W + j]);",
     "float h = ccu_oracle_bf16_to_f32(history[L - W + j]);"),
    ("bias dropped in the update",
     "if (bias != NULL) acc = acc + ccu_oracle_bf16_to_f32(bias[d]);\n\n      out[n * D + d]",
     "\n\n      out[n * D + d]"),
    ("shift keeps the oldest entry", "st[l * stride_l] = history[l + 1];",
     "st[l * stride_l] = history[l];"),
    ("SiLU sign flipped", "double y = a / (1.0 + exp(-a));", "double y = a / (1.0 + exp(a));"),
    ("ties round up", "upper += (upper & 1u);", "upper += 1u;"),
    ("state stride ignored on read", "history[l] = st[l * stride_l];", "history[l] = st[l];"),
    ("padding row writes -0", "out[n * D + d] = 0x0000u;", "out[n * D + d] = 0x8000u;"),
    ("padding row mutates its slot", "continue; /* padding row", "s = 0; /* padding row"),
    ("x row stride ignored", "history[L] = x[n * ld + d];", "history[L] = x[n * D + d];"),
    ("full conv taps reversed",
     "float term = ccu_oracle_bf16_to_f32(v) * ccu_oracle_bf16_to_f32(weight[d * W + j]);",
     "float term = ccu_oracle_bf16_to_f32(v) * ccu_oracle_bf16_to_f32(weight[d * W + W - 1 - j]);"),
    ("duplicate slots accepted", "if (seen[s]) flags |= CCU_ORACLE_IDX_DUPLICATE;", ""),
    ("ring read backwards", "history[i] = ring[((p + i) % L) * stride_l];",
     "history[i] = ring[((p + L - i) % L) * stride_l];"),
    ("ring writes the newest slot", "ring[p * stride_l] = history[L];",
     "ring[((p + L - 1) % L) * stride_l] = history[L];"),
    ("ring ignores seqlens", "const int64_t p = (int64_t)cache_seqlens[n] % L;",
     "const int64_t p = 0;"),
]


def _pins_fail(lib):
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    return failed


# The same mistakes planted in the ring-buffer update (second occurrence of the line).
MUTATIONS += [
    ("ring update taps reversed", "float w = ccu_oracle_bf16_to_f32(weight[d * W + j]);",
     "float w = ccu_oracle_bf16_to_f32(weight[d * W + (W - 1 - j)]);", 2),
    ("ring update bias dropped", "if (bias != NULL) acc = acc + ccu_oracle_bf16_to_f32(bias[d]);\n\n      out[n * D + d]",
     "\n\n      out[n * D + d]", 2),
    ("ring update window off by one", "float h = ccu_oracle_bf16_to_f32(history[(L + 1) - W + j]);",
     "float h = ccu_oracle_bf16_to_f32(history[L - W + j]);", 2),
]


# Mistakes in the multi-token function.
MUTATIONS += [
    ("multi: token window off by one", "float h = ccu_oracle_bf16_to_f32(history[L + t + 1 - W + j]);",
     "float h = ccu_oracle_bf16_to_f32(history[L + t - W + j]);"),
    ("multi: final state not advanced", "st[i * stride_l] = history[T + i];",
     "st[i * stride_l] = history[i];"),
    ("multi: intermediate state one token late", "it[l] = history[t + 1 + l];",
     "it[l] = history[t + 2 + l < L + T ? t + 2 + l : L + T - 1];"),
    ("multi: ring final position", "int64_t pos = (q + T + i) % L;", "int64_t pos = (q + i) % L;"),
]


# Mistakes that only a width above four shows: the window capped at the newest four taps
# (the update, the ring update, the multi-token function, the direct convolution).
_ALL_TAPS = "for (int64_t j = 0; j < W; ++j) {"
_FOUR_TAPS = "for (int64_t j = (W > 4 ? W - 4 : 0); j < W; ++j) {"
MUTATIONS += [
    ("update: window capped at four taps", _ALL_TAPS, _FOUR_TAPS, 1),
    ("ring update: window capped at four taps", _ALL_TAPS, _FOUR_TAPS, 2),
    ("multi: window capped at four taps", _ALL_TAPS, _FOUR_TAPS, 3),
    ("full conv: window capped at four taps", _ALL_TAPS, _FOUR_TAPS, 4),
]


def _replace_nth(src, old, new, nth):
    at = -1
    for _ in range(nth):
        at = src.index(old, at + 1)
    return src[:at] + new + src[at + len(old):]


@pytest.mark.parametrize("mutation", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(mutation, tmp_path):
    name, old, new = mutation[:3]
    nth = mutation[3] if len(mutation) > 3 else 1
    src_dir = os.path.dirname(oracle.__file__)
    src = open(os.path.join(src_dir, "ccu_oracle.c")).read()
    assert src.count(old) >= nth, f"mutation anchor for {name!r} not found"
    shutil.copy(os.path.join(src_dir, "ccu_oracle.h"), tmp_path / "ccu_oracle.h")
    (tmp_path / "ccu_oracle.c").write_text(_replace_nth(src, old, new, nth))
    lib_path = str(tmp_path / "libmutant.so")
    oracle.build(src=str(tmp_path / "ccu_oracle.c"), out=lib_path)
    failed = _pins_fail(oracle.load(lib_path))
    assert failed, f"no pin caught the planted mistake: {name}"
