"""Python binding of ``libccu_conv1d.so``: the depthwise causal conv1d decode update on GB300.

Argument marshalling only. Every step of the update runs in the library's CUDA
kernels; PyTorch supplies device memory and the current stream. There is no CPU
path: if the library is missing, importing the binding fails.

Two layers:

* ``ccu_conv1d_update`` and the other ``ccu_*`` functions mirror the C entry points
  of ``include/ccu_conv1d.h`` one to one (raw device pointers as ints).
* ``causal_conv1d_update(x, conv_state, weight, bias=None, activation=None, *,
  cache_seqlens=None, conv_state_indices=None)`` follows the signature of the cuDNN
  page "Causal Conv1d Decode Update" (section "Python API"): it mutates
  ``conv_state`` in place and returns a newly allocated BF16 ``[N, D]`` tensor.
  Declines are typed: ``NotImplementedError`` for valid but unserved requests,
  ``ValueError`` for contract violations (cuDNN page "Composing multi-kernel
  blocks", section "The shape of a block").
"""

from __future__ import annotations

import ctypes
import os

from . import _build

LIB_PATH = _build.LIB_PATH

CCU_OK = 0
CCU_ERR_INVALID_ARGUMENT = 1
CCU_ERR_NOT_IMPLEMENTED = 2
CCU_ERR_CUDA = 3

CCU_ACT_IDENTITY = 0
CCU_ACT_SILU = 1

ROUTES = {"auto": 0, "scalar": 1, "vector": 2, "staged": 3, "bulk": 4}
CCU_DEVERR_RANGE = 1
CCU_DEVERR_DUPLICATE = 2
CCU_DEVERR_TIMEOUT = 4

_ACTIVATIONS = {None: CCU_ACT_IDENTITY, "identity": CCU_ACT_IDENTITY,
                "silu": CCU_ACT_SILU, "swish": CCU_ACT_SILU}


class CudaError(RuntimeError):
    """A CUDA launch failed inside the library."""


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"` "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    upd = [vp, i64, vp, i64, i64, i64, vp, vp, ctypes.c_int, vp, vp, i64, i64, i64, i64, i64, vp]
    lib.ccu_conv1d_update.argtypes = upd + [vp]
    lib.ccu_conv1d_update_checked.argtypes = upd + [vp, vp]
    lib.ccu_conv1d_update_ex.argtypes = upd + [vp, i32, vp]
    lib.ccu_conv1d_update_checked_ex.argtypes = upd + [vp, vp, i32, vp]
    lib.ccu_conv1d_slot_scratch_bytes.argtypes = [i64]
    lib.ccu_conv1d_slot_scratch_bytes.restype = i64
    lib.ccu_conv1d_select_route.argtypes = upd + [i32, ctypes.POINTER(i32)]
    lib.ccu_conv1d_update_multi.argtypes = [vp, i64, i64, i64, vp, i64, i64, i64, vp, vp, ctypes.c_int,
                                            vp, vp, i64, i64, i64, i64, i64, i64, vp, i64, i64, i64,
                                            vp, vp, i32, vp]
    lib.ccu_conv1d_update_multi.restype = ctypes.c_int
    lib.ccu_causal_conv1d_fwd.argtypes = [vp, i64, i64, i64, vp, vp, ctypes.c_int, vp, i64, i64, i64,
                                          i64, i64, i64, i64, i64, vp, i64, i64, i64, vp, i64, i64, i64,
                                          i32, vp]
    lib.ccu_causal_conv1d_fwd.restype = ctypes.c_int
    for f in ("ccu_conv1d_update", "ccu_conv1d_update_checked", "ccu_conv1d_update_ex",
              "ccu_conv1d_update_checked_ex", "ccu_conv1d_select_route", "ccu_conv1d_check_indices"):
        getattr(lib, f).restype = ctypes.c_int
    lib.ccu_conv1d_check_indices.argtypes = [vp, i64, i64, vp, vp, vp]
    lib.ccu_conv1d_check_indices_noalloc.argtypes = [vp, i64, i64, vp, vp]
    lib.ccu_conv1d_check_indices_noalloc.restype = ctypes.c_int
    lib.ccu_conv1d_check_indices_scratch_bytes.argtypes = [i64]
    lib.ccu_conv1d_check_indices_scratch_bytes.restype = i64
    lib.ccu_status_string.argtypes = [ctypes.c_int]
    lib.ccu_status_string.restype = ctypes.c_char_p
    lib.ccu_route_name.argtypes = [i32]
    lib.ccu_route_name.restype = ctypes.c_char_p
    lib.ccu_conv1d_last_error.argtypes = []
    lib.ccu_conv1d_last_error.restype = ctypes.c_char_p
    lib.ccu_conv1d_take_device_error.argtypes = [ctypes.POINTER(i32)]
    lib.ccu_conv1d_take_device_error.restype = ctypes.c_int
    lib.ccu_conv1d_abi_version.argtypes = []
    lib.ccu_conv1d_abi_version.restype = i32
    return lib


lib = _load()


# ------------------------------------------------------------------ raw C entry points

def ccu_conv1d_update(x, ld, conv_state, stride_s, stride_d, stride_l, weight, bias, act, indices,
                      cache_seqlens, N, D, S, L, W, out, stream) -> int:
    return lib.ccu_conv1d_update(x, ld, conv_state, stride_s, stride_d, stride_l, weight, bias, act,
                                 indices, cache_seqlens, N, D, S, L, W, out, stream)


def ccu_conv1d_update_checked(x, ld, conv_state, stride_s, stride_d, stride_l, weight, bias, act,
                              indices, cache_seqlens, N, D, S, L, W, out, status_dev, stream) -> int:
    return lib.ccu_conv1d_update_checked(x, ld, conv_state, stride_s, stride_d, stride_l, weight,
                                         bias, act, indices, cache_seqlens, N, D, S, L, W, out,
                                         status_dev, stream)


def ccu_conv1d_update_ex(x, ld, conv_state, stride_s, stride_d, stride_l, weight, bias, act, indices,
                         cache_seqlens, N, D, S, L, W, out, status_dev, route, stream) -> int:
    return lib.ccu_conv1d_update_ex(x, ld, conv_state, stride_s, stride_d, stride_l, weight, bias,
                                    act, indices, cache_seqlens, N, D, S, L, W, out, status_dev,
                                    route, stream)


def ccu_conv1d_update_checked_ex(x, ld, conv_state, stride_s, stride_d, stride_l, weight, bias, act,
                                 indices, cache_seqlens, N, D, S, L, W, out, status_dev, slot_scratch,
                                 route, stream) -> int:
    return lib.ccu_conv1d_update_checked_ex(x, ld, conv_state, stride_s, stride_d, stride_l, weight,
                                            bias, act, indices, cache_seqlens, N, D, S, L, W, out,
                                            status_dev, slot_scratch, route, stream)


def ccu_conv1d_slot_scratch_bytes(S) -> int:
    return lib.ccu_conv1d_slot_scratch_bytes(S)


def ccu_conv1d_update_multi(x, x_stride_n, x_stride_d, x_stride_t, conv_state, stride_s, stride_d,
                            stride_l, weight, bias, act, indices, cache_seqlens, N, D, T, S, L, W, out,
                            out_stride_n, out_stride_d, out_stride_t, intermediate_states, status_dev,
                            route, stream) -> int:
    return lib.ccu_conv1d_update_multi(x, x_stride_n, x_stride_d, x_stride_t, conv_state, stride_s,
                                       stride_d, stride_l, weight, bias, act, indices, cache_seqlens,
                                       N, D, T, S, L, W, out, out_stride_n, out_stride_d, out_stride_t,
                                       intermediate_states, status_dev, route, stream)


def ccu_causal_conv1d_fwd(x, x_stride_b, x_stride_d, x_stride_t, weight, bias, act, initial_states,
                          init_stride_b, init_stride_d, init_stride_l, B, D, T, L, W, out, out_stride_b,
                          out_stride_d, out_stride_t, final_states, final_stride_b, final_stride_d,
                          final_stride_l, route, stream) -> int:
    return lib.ccu_causal_conv1d_fwd(x, x_stride_b, x_stride_d, x_stride_t, weight, bias, act,
                                     initial_states, init_stride_b, init_stride_d, init_stride_l, B, D,
                                     T, L, W, out, out_stride_b, out_stride_d, out_stride_t,
                                     final_states, final_stride_b, final_stride_d, final_stride_l,
                                     route, stream)


def ccu_conv1d_select_route(x, ld, conv_state, stride_s, stride_d, stride_l, weight, bias, act,
                            indices, cache_seqlens, N, D, S, L, W, out, route):
    """Returns (status, chosen_route)."""
    chosen = ctypes.c_int32(-1)
    st = lib.ccu_conv1d_select_route(x, ld, conv_state, stride_s, stride_d, stride_l, weight, bias,
                                     act, indices, cache_seqlens, N, D, S, L, W, out, route,
                                     ctypes.byref(chosen))
    return st, chosen.value


def ccu_conv1d_check_indices(indices, N, S, bitmap_scratch, status_dev, stream) -> int:
    return lib.ccu_conv1d_check_indices(indices, N, S, bitmap_scratch, status_dev, stream)


def ccu_conv1d_check_indices_noalloc(indices, N, S, status_dev, stream) -> int:
    """The index check with the library's built-in bitmap (no scratch from the caller).

    For callers that cannot allocate device memory. S is limited to
    CCU_CHECK_INDICES_NOALLOC_MAX_SLOTS; calls that overlap on the GPU race on the shared
    bitmap. The first call on a device sets up the bitmap's address.
    """
    return lib.ccu_conv1d_check_indices_noalloc(indices, N, S, status_dev, stream)


CCU_CHECK_INDICES_NOALLOC_MAX_SLOTS = 1 << 20


def ccu_conv1d_check_indices_scratch_bytes(S) -> int:
    return lib.ccu_conv1d_check_indices_scratch_bytes(S)


def ccu_status_string(status) -> str:
    return lib.ccu_status_string(status).decode()


def ccu_route_name(route) -> str:
    return lib.ccu_route_name(route).decode()


def ccu_conv1d_last_error() -> str:
    return lib.ccu_conv1d_last_error().decode()


def ccu_conv1d_take_device_error():
    """Returns (status, bits); synchronizes the current device."""
    bits = ctypes.c_int32(0)
    st = lib.ccu_conv1d_take_device_error(ctypes.byref(bits))
    return st, bits.value


def ccu_conv1d_abi_version() -> int:
    return lib.ccu_conv1d_abi_version()


def raise_for_status(status: int) -> None:
    """Map a ccu_status_t to the page's typed declines."""
    if status == CCU_OK:
        return
    msg = f"{ccu_status_string(status)}: {ccu_conv1d_last_error()}"
    if status == CCU_ERR_NOT_IMPLEMENTED:
        raise NotImplementedError(msg)
    if status == CCU_ERR_INVALID_ARGUMENT:
        raise ValueError(msg)
    raise CudaError(msg)


# ------------------------------------------------------------------ torch-level op

def _ptr(t):
    return None if t is None else t.data_ptr()


def _check_tensor(name, t, dtype, torch):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.requires_grad:
        raise ValueError(f"{name} requires grad: the update is inference-only (autograd unsupported)")


def _same_device(ref, named, ref_name="x"):
    """Every tensor of a call on the device of ``ref`` (the kernels get raw pointers)."""
    for name, t in named:
        if t is not None and t.device != ref.device:
            raise ValueError(f"{name} is on {t.device} but {ref_name} is on {ref.device}: "
                             "all tensors of a call must be on one device")


def causal_conv1d_update(x, conv_state, weight, bias=None, activation=None, *, cache_seqlens=None,
                         conv_state_indices=None, out=None, route: str = "auto", status=None,
                         intermediate_states=None, slot_scratch=None):
    """One decode step: mutate ``conv_state`` in place and return the BF16 output ``[N, D]``.

    Follows the cuDNN page "Causal Conv1d Decode Update" ("Python API" and "Semantic
    tensor contract"): ``x`` BF16 ``[N, D]`` with strides ``(ld, 1)``; ``conv_state`` BF16
    ``[S, D, L]``, compact or channel-last ``(L*D, 1, D)``; ``weight`` BF16 ``[D, W]``
    (the page's width 4; widths 2 and 3 run on every kernel, other widths with L >= 1 on the
    scalar kernel);
    ``bias`` BF16 ``[D]`` or None; ``activation`` None/"identity" or "silu"/"swish";
    ``conv_state_indices`` int32 ``[N]`` (``-1`` = padding row) or None; ``cache_seqlens``
    None (linear state) or int32 ``[N]``: the state is then a ring buffer whose oldest entry
    is at ``cache_seqlens[n] % L`` and only that entry is overwritten (use the channel-last
    layout for a ring: it then moves only the window and one entry, the compact layout moves
    the whole slab). ``out`` (optional, preallocated ``[N, D]`` BF16), ``route`` (kernel
    family), ``status`` (int32 device word: turns on the device range check) and
    ``slot_scratch`` (int32 ``[S]`` device tensor, with ``status``: also detects repeated
    slots in the same launch, see ccu_conv1d_update_checked_ex) are extensions of this
    binding. Runs on the current CUDA stream.

    A 3-D ``x`` ``[N, D, T]`` (any strides) is the multi-token update: T tokens per row,
    output ``[N, D, T]`` laid out like ``x``; ``intermediate_states`` (optional BF16
    ``[N, T, D, L]`` contiguous) receives the state after every token.
    """
    import torch

    if activation not in _ACTIVATIONS:
        raise ValueError(f"activation must be one of None, 'identity', 'silu', 'swish'; got {activation!r}")
    _check_tensor("x", x, torch.bfloat16, torch)
    if x.dim() == 3:
        if slot_scratch is not None:
            raise ValueError("slot_scratch serves the single-token update")
        return _update_multi(x, conv_state, weight, bias, activation, cache_seqlens,
                             conv_state_indices, out, route, status, intermediate_states, torch)
    if x.dim() != 2:
        raise ValueError(f"x must be 2D [N, D] or 3D [N, D, T], got {x.dim()}D")
    if intermediate_states is not None:
        raise ValueError("intermediate_states needs a multi-token x [N, D, T]")
    if x.stride(1) != 1:
        raise ValueError("x must have unit stride along D")
    _check_tensor("conv_state", conv_state, torch.bfloat16, torch)
    if conv_state.dim() != 3:
        raise ValueError("conv_state must be 3D [S, D, L]")
    _check_tensor("weight", weight, torch.bfloat16, torch)
    if weight.dim() != 2 or not weight.is_contiguous():
        raise ValueError("weight must be a contiguous 2D [D, W] tensor")
    N, D = x.shape
    S, Ds, L = conv_state.shape
    Dw, W = weight.shape
    if Ds != D or Dw != D:
        raise ValueError(f"channel counts differ: x {D}, conv_state {Ds}, weight {Dw}")
    if bias is not None:
        _check_tensor("bias", bias, torch.bfloat16, torch)
        if bias.shape != (D,) or not bias.is_contiguous():
            raise ValueError("bias must be a contiguous [D] tensor")
    if conv_state_indices is not None:
        _check_tensor("conv_state_indices", conv_state_indices, torch.int32, torch)
        if conv_state_indices.shape != (N,) or not conv_state_indices.is_contiguous():
            raise ValueError("conv_state_indices must be a contiguous int32 [N] tensor")
    if cache_seqlens is not None:
        _check_tensor("cache_seqlens", cache_seqlens, torch.int32, torch)
        if cache_seqlens.shape != (N,) or not cache_seqlens.is_contiguous():
            raise ValueError("cache_seqlens must be a contiguous int32 [N] tensor")
    if out is None:
        out = torch.empty((N, D), dtype=torch.bfloat16, device=x.device)
    else:
        _check_tensor("out", out, torch.bfloat16, torch)
        if out.shape != (N, D) or not out.is_contiguous():
            raise ValueError("out must be a contiguous [N, D] tensor")
    if route not in ROUTES:
        raise ValueError(f"route must be one of {sorted(ROUTES)}")
    if status is not None:
        _check_tensor("status", status, torch.int32, torch)
    if slot_scratch is not None:
        if status is None:
            raise ValueError("slot_scratch needs a status word")
        _check_tensor("slot_scratch", slot_scratch, torch.int32, torch)
        if slot_scratch.numel() < S or not slot_scratch.is_contiguous():
            raise ValueError("slot_scratch must be a contiguous int32 tensor of at least S elements")
    _same_device(x, (("conv_state", conv_state), ("weight", weight), ("bias", bias),
                     ("conv_state_indices", conv_state_indices), ("cache_seqlens", cache_seqlens),
                     ("out", out), ("status", status), ("slot_scratch", slot_scratch)))
    ld = x.stride(0) if N > 1 else D  # a single row's stride is never used
    ss, sd, sl = conv_state.stride()
    with torch.cuda.device(x.device):  # the library launches on the current device
        stream = torch.cuda.current_stream(x.device).cuda_stream
        if slot_scratch is not None:
            st = lib.ccu_conv1d_update_checked_ex(
                _ptr(x), ld, _ptr(conv_state), ss, sd, sl, _ptr(weight), _ptr(bias),
                _ACTIVATIONS[activation], _ptr(conv_state_indices), _ptr(cache_seqlens), N, D, S, L, W,
                _ptr(out), _ptr(status), _ptr(slot_scratch), ROUTES[route], stream)
        else:
            st = lib.ccu_conv1d_update_ex(
                _ptr(x), ld, _ptr(conv_state), ss, sd, sl, _ptr(weight), _ptr(bias),
                _ACTIVATIONS[activation], _ptr(conv_state_indices), _ptr(cache_seqlens), N, D, S, L, W,
                _ptr(out), _ptr(status), ROUTES[route], stream)
    raise_for_status(st)
    return out


def _update_multi(x, conv_state, weight, bias, activation, cache_seqlens, conv_state_indices, out,
                  route, status, intermediate_states, torch):
    if activation not in _ACTIVATIONS:
        raise ValueError(f"activation must be one of None, 'identity', 'silu', 'swish'; got {activation!r}")
    for name, t in (("conv_state", conv_state), ("weight", weight)):
        _check_tensor(name, t, torch.bfloat16, torch)
    if conv_state.dim() != 3:
        raise ValueError("conv_state must be 3D [S, D, L]")
    if weight.dim() != 2 or not weight.is_contiguous():
        raise ValueError("weight must be a contiguous 2D [D, W] tensor")
    N, D, T = x.shape
    S, Ds, L = conv_state.shape
    Dw, W = weight.shape
    if Ds != D or Dw != D:
        raise ValueError(f"channel counts differ: x {D}, conv_state {Ds}, weight {Dw}")
    if bias is not None:
        _check_tensor("bias", bias, torch.bfloat16, torch)
        if bias.shape != (D,) or not bias.is_contiguous():
            raise ValueError("bias must be a contiguous [D] tensor")
    for name, t in (("conv_state_indices", conv_state_indices), ("cache_seqlens", cache_seqlens)):
        if t is not None:
            _check_tensor(name, t, torch.int32, torch)
            if t.shape != (N,) or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous int32 [N] tensor")
    if out is None:
        out = torch.empty_like(x)  # same strides as a dense x
    else:
        _check_tensor("out", out, torch.bfloat16, torch)
        if out.shape != (N, D, T):
            raise ValueError("out must be [N, D, T]")
    if intermediate_states is not None:
        _check_tensor("intermediate_states", intermediate_states, torch.bfloat16, torch)
        if intermediate_states.shape != (N, T, D, L) or not intermediate_states.is_contiguous():
            raise ValueError("intermediate_states must be a contiguous [N, T, D, L] tensor")
    if status is not None:
        _check_tensor("status", status, torch.int32, torch)
    if route not in ROUTES:
        raise ValueError(f"route must be one of {sorted(ROUTES)}")
    _same_device(x, (("conv_state", conv_state), ("weight", weight), ("bias", bias),
                     ("conv_state_indices", conv_state_indices), ("cache_seqlens", cache_seqlens),
                     ("out", out), ("intermediate_states", intermediate_states), ("status", status)))
    with torch.cuda.device(x.device):  # the library launches on the current device
        stream = torch.cuda.current_stream(x.device).cuda_stream
        st = lib.ccu_conv1d_update_multi(
            _ptr(x), *x.stride(), _ptr(conv_state), *conv_state.stride(), _ptr(weight), _ptr(bias),
            _ACTIVATIONS[activation], _ptr(conv_state_indices), _ptr(cache_seqlens), N, D, T, S, L, W,
            _ptr(out), *out.stride(), _ptr(intermediate_states), _ptr(status), ROUTES[route], stream)
    raise_for_status(st)
    return out


def causal_conv1d_fwd(x, weight, bias=None, activation=None, *, initial_states=None,
                      return_final_states=False, final_states_out=None, final_state_len=None, out=None,
                      route: str = "auto"):
    """Full-sequence prefill: causal depthwise convolution of ``x`` [B, D, T] (any strides).

    Returns ``out`` [B, D, T] (laid out like ``x``) and, when ``return_final_states`` or
    ``final_states_out`` is given, the final state [B, D, L]: the last L inputs, by default
    L = max(W - 1, 1) in the channel-last layout (strides (L*D, 1, D)) that the decode update
    accepts without a copy. ``initial_states`` [B, D, L] (any strides) holds the inputs
    before the sequence (zeros when None).
    """
    import torch

    _check_tensor("x", x, torch.bfloat16, torch)
    if x.dim() != 3:
        raise ValueError("x must be 3D [B, D, T]")
    _check_tensor("weight", weight, torch.bfloat16, torch)
    if weight.dim() != 2 or not weight.is_contiguous():
        raise ValueError("weight must be a contiguous 2D [D, W] tensor")
    if activation not in _ACTIVATIONS:
        raise ValueError(f"activation must be one of None, 'identity', 'silu', 'swish'; got {activation!r}")
    B, D, T = x.shape
    Dw, W = weight.shape
    if Dw != D:
        raise ValueError(f"channel counts differ: x {D}, weight {Dw}")
    if bias is not None:
        _check_tensor("bias", bias, torch.bfloat16, torch)
        if bias.shape != (D,) or not bias.is_contiguous():
            raise ValueError("bias must be a contiguous [D] tensor")
    # the shortest state the width allows (a width-1 filter still keeps one entry)
    L = final_state_len if final_state_len is not None else max(W - 1, 1)
    if initial_states is not None:
        _check_tensor("initial_states", initial_states, torch.bfloat16, torch)
        if initial_states.dim() != 3 or initial_states.shape[:2] != (B, D):
            raise ValueError("initial_states must be [B, D, L]")
        L = initial_states.shape[2] if final_state_len is None else L
        if initial_states.shape[2] != L:
            raise ValueError("initial_states and the final state must have the same length L")
    fin = final_states_out
    if fin is None and return_final_states:
        fin = torch.empty((B, L, D), dtype=torch.bfloat16, device=x.device).permute(0, 2, 1)
    if fin is not None:
        _check_tensor("final_states_out", fin, torch.bfloat16, torch)
        if fin.shape != (B, D, L):
            raise ValueError("final states must be [B, D, L]")
    if out is None:
        out = torch.empty_like(x)
    else:
        _check_tensor("out", out, torch.bfloat16, torch)
        if out.shape != (B, D, T):
            raise ValueError("out must be [B, D, T]")
    if route not in ROUTES:
        raise ValueError(f"route must be one of {sorted(ROUTES)}")
    _same_device(x, (("weight", weight), ("bias", bias), ("initial_states", initial_states),
                     ("final_states_out", fin), ("out", out)))
    ist = initial_states.stride() if initial_states is not None else (0, 0, 0)
    fst = fin.stride() if fin is not None else (0, 0, 0)
    with torch.cuda.device(x.device):  # the library launches on the current device
        stream = torch.cuda.current_stream(x.device).cuda_stream
        st = lib.ccu_causal_conv1d_fwd(
            _ptr(x), *x.stride(), _ptr(weight), _ptr(bias), _ACTIVATIONS[activation],
            _ptr(initial_states), *ist, B, D, T, L, W, _ptr(out), *out.stride(), _ptr(fin), *fst,
            ROUTES[route], stream)
    raise_for_status(st)
    return (out, fin) if fin is not None else out


def check_indices(conv_state_indices, S: int, status=None, scratch=None):
    """Validate slot indices on the device (range and uniqueness) without trapping.

    Returns the int32 status word tensor (device); 0 means valid. Allocates the status
    word and the bitmap scratch with torch when not given.
    """
    import torch

    _check_tensor("conv_state_indices", conv_state_indices, torch.int32, torch)
    dev = conv_state_indices.device
    if status is None:
        status = torch.zeros((1,), dtype=torch.int32, device=dev)
    nbytes = ccu_conv1d_check_indices_scratch_bytes(S)
    if scratch is None:
        scratch = torch.empty((max(nbytes // 4, 1),), dtype=torch.int32, device=dev)
    _same_device(conv_state_indices, (("status", status), ("scratch", scratch)), "conv_state_indices")
    with torch.cuda.device(dev):  # the library launches on the current device
        stream = torch.cuda.current_stream(dev).cuda_stream
        st = lib.ccu_conv1d_check_indices(_ptr(conv_state_indices), conv_state_indices.numel(), S,
                                          _ptr(scratch), _ptr(status), stream)
    raise_for_status(st)
    return status
