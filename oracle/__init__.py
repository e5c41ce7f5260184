"""ctypes wrapper around the C oracle (``ccu_oracle.c``).

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / reference leg may import this package; the
product path never does.

Arrays are numpy: BF16 tensors as ``uint16`` bit patterns, indices as ``int32``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ccu_oracle.c")
LIB_PATH = os.path.join(_HERE, "libccu_oracle.so")

ACT = {"identity": 0, "silu": 1}
IDX_RANGE = 1
IDX_DUPLICATE = 2
OK = 0
BAD_ARGS = -1
BAD_INDICES = -2

# Plain C, no fast-math, no FMA contraction: float ops happen as written.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(src: str = _SRC, out: str = LIB_PATH) -> str:
    """Compile the oracle with gcc (single file, a second or two)."""
    cmd = ["gcc", *CFLAGS, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True, cwd=_HERE)
    return out


def _stale(lib: str, src: str) -> bool:
    if not os.path.exists(lib):
        return True
    deps = [src, os.path.join(os.path.dirname(src), "ccu_oracle.h")]
    return any(os.path.getmtime(p) > os.path.getmtime(lib) for p in deps if os.path.exists(p))


_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)
_i64 = ctypes.c_int64


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    lib.ccu_oracle_conv1d_update.restype = ctypes.c_int
    lib.ccu_oracle_conv1d_update.argtypes = [
        _u16p, _i64, _u16p, _i64, _i64, _i64, _u16p, _u16p, ctypes.c_int, _i32p,
        _i64, _i64, _i64, _i64, _i64, _u16p, _f32p]
    lib.ccu_oracle_conv1d_update_circular.restype = ctypes.c_int
    lib.ccu_oracle_conv1d_update_circular.argtypes = [
        _u16p, _i64, _u16p, _i64, _i64, _i64, _u16p, _u16p, ctypes.c_int, _i32p, _i32p,
        _i64, _i64, _i64, _i64, _i64, _u16p, _f32p]
    lib.ccu_oracle_conv1d_update_multi.restype = ctypes.c_int
    lib.ccu_oracle_conv1d_update_multi.argtypes = [
        _u16p, _i64, _i64, _i64, _u16p, _i64, _i64, _i64, _u16p, _u16p, ctypes.c_int, _i32p, _i32p,
        _i64, _i64, _i64, _i64, _i64, _i64, _u16p, _i64, _i64, _i64, _u16p]
    lib.ccu_oracle_full_causal_conv.restype = ctypes.c_int
    lib.ccu_oracle_full_causal_conv.argtypes = [
        _u16p, _i64, _i64, _u16p, _u16p, ctypes.c_int, _i64, _u16p, _i64, _u16p, _u16p, _f32p]
    lib.ccu_oracle_check_indices.restype = ctypes.c_int
    lib.ccu_oracle_check_indices.argtypes = [_i32p, _i64, _i64]
    lib.ccu_oracle_bf16_to_f32.restype = ctypes.c_float
    lib.ccu_oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.ccu_oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.ccu_oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.ccu_oracle_silu.restype = ctypes.c_float
    lib.ccu_oracle_silu.argtypes = [ctypes.c_float]
    return lib


_LIB: Optional[ctypes.CDLL] = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load (building first if missing or older than its source) the oracle library."""
    global _LIB
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _LIB is None:
        if _stale(LIB_PATH, _SRC):
            build()
        _LIB = _bind(ctypes.CDLL(LIB_PATH))
    return _LIB


def _ptr(a: Optional[np.ndarray], ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def conv1d_update(x: np.ndarray, ld: int, conv_state: np.ndarray, strides, weight: np.ndarray,
                  bias: Optional[np.ndarray], act: str, indices: Optional[np.ndarray],
                  N: int, D: int, S: int, L: int, W: int, *, with_acc: bool = False,
                  lib: Optional[ctypes.CDLL] = None):
    """Run one decode update in place on ``conv_state`` (a flat-addressable uint16 array).

    ``strides`` are the element strides (s, d, l) of the logical [S, D, L] state
    inside ``conv_state``'s memory. Returns ``out`` [N, D] (uint16), plus the FP32
    accumulator [N, D] when ``with_acc``. Raises ValueError if the oracle refuses.
    """
    lib = lib or load()
    for a in (x, conv_state, weight):
        assert a.dtype == np.uint16 and a.flags["C_CONTIGUOUS"]
    if bias is not None:
        assert bias.dtype == np.uint16 and bias.flags["C_CONTIGUOUS"]
    if indices is not None:
        indices = np.ascontiguousarray(indices, dtype=np.int32)
    out = np.empty((N, D), dtype=np.uint16)
    acc = np.empty((N, D), dtype=np.float32) if with_acc else None
    rc = lib.ccu_oracle_conv1d_update(
        _ptr(x, ctypes.c_uint16), ld, _ptr(conv_state, ctypes.c_uint16),
        strides[0], strides[1], strides[2], _ptr(weight, ctypes.c_uint16),
        _ptr(bias, ctypes.c_uint16), ACT[act], _ptr(indices, ctypes.c_int32),
        N, D, S, L, W, _ptr(out, ctypes.c_uint16), _ptr(acc, ctypes.c_float))
    if rc != OK:
        raise ValueError(f"oracle refused the inputs (code {rc})")
    return (out, acc) if with_acc else out


def conv1d_update_circular(x: np.ndarray, ld: int, conv_state: np.ndarray, strides, weight: np.ndarray,
                           bias: Optional[np.ndarray], act: str, indices: Optional[np.ndarray],
                           cache_seqlens: np.ndarray, N: int, D: int, S: int, L: int, W: int, *,
                           with_acc: bool = False, lib: Optional[ctypes.CDLL] = None):
    """One ring-buffer decode update in place on ``conv_state``; returns out (and acc)."""
    lib = lib or load()
    for a in (x, conv_state, weight):
        assert a.dtype == np.uint16 and a.flags["C_CONTIGUOUS"]
    if indices is not None:
        indices = np.ascontiguousarray(indices, dtype=np.int32)
    cache_seqlens = np.ascontiguousarray(cache_seqlens, dtype=np.int32)
    out = np.empty((N, D), dtype=np.uint16)
    acc = np.empty((N, D), dtype=np.float32) if with_acc else None
    rc = lib.ccu_oracle_conv1d_update_circular(
        _ptr(x, ctypes.c_uint16), ld, _ptr(conv_state, ctypes.c_uint16),
        strides[0], strides[1], strides[2], _ptr(weight, ctypes.c_uint16),
        _ptr(bias, ctypes.c_uint16), ACT[act], _ptr(indices, ctypes.c_int32),
        _ptr(cache_seqlens, ctypes.c_int32), N, D, S, L, W, _ptr(out, ctypes.c_uint16),
        _ptr(acc, ctypes.c_float))
    if rc != OK:
        raise ValueError(f"oracle refused the inputs (code {rc})")
    return (out, acc) if with_acc else out


def conv1d_update_multi(x: np.ndarray, x_strides, conv_state: np.ndarray, strides, weight: np.ndarray,
                        bias: Optional[np.ndarray], act: str, indices: Optional[np.ndarray],
                        cache_seqlens: Optional[np.ndarray], N: int, D: int, T: int, S: int, L: int,
                        W: int, *, with_inter: bool = False, lib: Optional[ctypes.CDLL] = None):
    """T tokens per row in one call; returns out [N, D, T] (and intermediate states
    [N, T, D, L] when ``with_inter``). ``x`` is flat memory addressed with ``x_strides``
    (element strides of n, d, t)."""
    lib = lib or load()
    for a in (x, conv_state, weight):
        assert a.dtype == np.uint16 and a.flags["C_CONTIGUOUS"]
    if indices is not None:
        indices = np.ascontiguousarray(indices, dtype=np.int32)
    if cache_seqlens is not None:
        cache_seqlens = np.ascontiguousarray(cache_seqlens, dtype=np.int32)
    out = np.empty((N, D, T), dtype=np.uint16)
    inter = np.zeros((N, T, D, L), dtype=np.uint16) if with_inter else None
    rc = lib.ccu_oracle_conv1d_update_multi(
        _ptr(x, ctypes.c_uint16), x_strides[0], x_strides[1], x_strides[2],
        _ptr(conv_state, ctypes.c_uint16), strides[0], strides[1], strides[2],
        _ptr(weight, ctypes.c_uint16), _ptr(bias, ctypes.c_uint16), ACT[act],
        _ptr(indices, ctypes.c_int32), _ptr(cache_seqlens, ctypes.c_int32), N, D, T, S, L, W,
        _ptr(out, ctypes.c_uint16), D * T, T, 1, _ptr(inter, ctypes.c_uint16))
    if rc != OK:
        raise ValueError(f"oracle refused the inputs (code {rc})")
    return (out, inter) if with_inter else out


def full_causal_conv(x_seq: np.ndarray, weight: np.ndarray, bias: Optional[np.ndarray], act: str,
                     init_state: Optional[np.ndarray], L: int, *, with_acc: bool = False,
                     lib: Optional[ctypes.CDLL] = None):
    """Brute-force causal conv over x_seq [T, D]; returns (y [T, D], final_state [D, L][, acc])."""
    lib = lib or load()
    T, D = x_seq.shape
    W = weight.shape[1]
    x_seq = np.ascontiguousarray(x_seq, dtype=np.uint16)
    y = np.empty((T, D), dtype=np.uint16)
    fin = np.empty((D, L), dtype=np.uint16)
    acc = np.empty((T, D), dtype=np.float32) if with_acc else None
    if init_state is not None:
        init_state = np.ascontiguousarray(init_state, dtype=np.uint16)
    rc = lib.ccu_oracle_full_causal_conv(
        _ptr(x_seq, ctypes.c_uint16), T, D, _ptr(np.ascontiguousarray(weight), ctypes.c_uint16),
        _ptr(bias, ctypes.c_uint16), ACT[act], W, _ptr(init_state, ctypes.c_uint16), L,
        _ptr(y, ctypes.c_uint16), _ptr(fin, ctypes.c_uint16), _ptr(acc, ctypes.c_float))
    if rc != OK:
        raise ValueError(f"oracle refused the inputs (code {rc})")
    return (y, fin, acc) if with_acc else (y, fin)


def check_indices(indices: np.ndarray, N: int, S: int, lib: Optional[ctypes.CDLL] = None) -> int:
    """OR of IDX_RANGE / IDX_DUPLICATE for a slot-index vector (0 when valid)."""
    lib = lib or load()
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    return lib.ccu_oracle_check_indices(_ptr(indices, ctypes.c_int32), N, S)


def run_workload(inp, layout: str = "compact", *, with_acc: bool = False, lib=None,
                 cache_seqlens: Optional[np.ndarray] = None):
    """Apply one update to a copy of a ``synthetic.Inputs``; returns (out, new_state[, acc]).

    ``new_state`` is returned as a logical [S, D, L] array whatever the layout.
    """
    wl = inp.wl
    S, D, L = wl.S, wl.D, wl.L
    if layout == "compact":
        state = inp.conv_state.copy()
        strides = (D * L, L, 1)
    elif layout == "channel_last":
        # np.array(copy=True): never a view, even when a size-1 axis makes the transpose
        # look contiguous (the oracle writes into this array)
        state = np.array(np.transpose(inp.conv_state, (0, 2, 1)), order="C", copy=True)
        strides = (L * D, 1, D)
    else:
        raise ValueError(layout)
    if cache_seqlens is None:
        res = conv1d_update(inp.x, wl.ld, state, strides, inp.weight, inp.bias, wl.act, inp.indices,
                            wl.N, D, S, L, wl.W, with_acc=with_acc, lib=lib)
    else:
        res = conv1d_update_circular(inp.x, wl.ld, state, strides, inp.weight, inp.bias, wl.act,
                                     inp.indices, cache_seqlens, wl.N, D, S, L, wl.W,
                                     with_acc=with_acc, lib=lib)
    if layout == "channel_last":
        state = np.array(np.transpose(state, (0, 2, 1)), order="C", copy=True)
    if with_acc:
        return res[0], state, res[1]
    return res, state
