"""Helpers for the GPU parity tests: device buffers with canary guard bands, one update
through the C-ABI, comparison against the oracle."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import synthetic
from oracle_pins import bf16_ulp_distance

GUARD = 4096  # bytes of 0xA5 canary before and after every guarded buffer
CANARY = 0xA5


class Guarded:
    """A device buffer of `nbytes` surrounded by canary bytes."""

    def __init__(self, nbytes: int, dev):
        self.nbytes = nbytes
        self.raw = torch.full((GUARD + max(nbytes, 16) + GUARD,), CANARY, dtype=torch.uint8, device=dev)

    def view(self, dtype, shape):
        n = int(np.prod(shape)) if len(shape) else 1
        itemsize = torch.empty((), dtype=dtype).element_size()
        return self.raw[GUARD:GUARD + n * itemsize].view(dtype).view(shape)

    def guards_intact(self) -> bool:
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + max(self.nbytes, 16):]
        return bool(torch.all(head == CANARY)) and bool(torch.all(tail == CANARY))


def to_dev_u16(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


def from_dev_u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def guarded_u16(a: np.ndarray, dev):
    g = Guarded(a.nbytes, dev)
    t = g.view(torch.int16, a.shape)
    t.copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.int16)))
    return g, t.view(torch.bfloat16)


def run_gpu(inp: synthetic.Inputs, layout="compact", route="auto", checked=False, dev="cuda:0",
            stream=None, guards=True, cache_seqlens=None, slot_scratch=None):
    """One update on the GPU through the torch binding (which calls the C-ABI).

    Returns (out, logical state [S, D, L], status or None, guards_ok).
    """
    import depthwise_causal_conv1d_gb300 as ccu

    wl = inp.wl
    S, D, L, N = wl.S, wl.D, wl.L, wl.N
    state_mem = inp.conv_state if layout == "compact" else synthetic.to_channel_last(inp.conv_state)
    gx, x = guarded_u16(inp.x, dev)
    x = x[:, :D] if wl.ld != D else x
    gs, st = guarded_u16(state_mem, dev)
    if layout == "channel_last":
        st = st.permute(0, 2, 1)  # logical [S, D, L] with strides (L*D, 1, D)
    w = to_dev_u16(inp.weight, dev)
    b = to_dev_u16(inp.bias, dev) if inp.bias is not None else None
    idx = torch.from_numpy(inp.indices).to(dev) if inp.indices is not None else None
    seq = torch.from_numpy(np.ascontiguousarray(cache_seqlens, np.int32)).to(dev) if cache_seqlens is not None else None
    go = Guarded(N * D * 2, dev)
    out = go.view(torch.bfloat16, (N, D))
    status = torch.zeros((1,), dtype=torch.int32, device=dev) if checked else None

    ctx = torch.cuda.stream(stream) if stream is not None else torch.cuda.stream(torch.cuda.current_stream())
    with ctx:
        ccu.causal_conv1d_update(x, st, w, b, wl.act, conv_state_indices=idx, cache_seqlens=seq,
                                 out=out, route=route, status=status, slot_scratch=slot_scratch)
    torch.cuda.synchronize()
    got_out = from_dev_u16(out)
    mem = from_dev_u16(gs.view(torch.int16, state_mem.shape))
    got_state = mem if layout == "compact" else synthetic.from_channel_last(mem)
    ok = (gx.guards_intact() and gs.guards_intact() and go.guards_intact()) if guards else True
    st_val = int(status.item()) if checked else None
    return got_out, got_state, st_val, ok


def assert_parity(inp, got_out, got_state, want_out, want_state, what=""):
    """State bit-exact; output within one BF16 ulp (identity: exact, +0 == -0)."""
    assert got_state.shape == want_state.shape
    if not np.array_equal(got_state, want_state):
        bad = np.argwhere(got_state != want_state)
        raise AssertionError(f"{what}: state differs at {len(bad)} places, first {bad[:3].tolist()}")
    dist = bf16_ulp_distance(got_out, want_out)
    limit = 0 if inp.wl.act == "identity" else 1
    if dist.max(initial=0) > limit:
        bad = np.argwhere(dist > limit)
        n, d = bad[0]
        raise AssertionError(f"{what}: output off by {dist.max()} ulp at {len(bad)} places, first "
                             f"(n={n}, d={d}) got {got_out[n, d]:#06x} want {want_out[n, d]:#06x}")


def oracle_ref(inp, layout="compact", cache_seqlens=None):
    return oracle.run_workload(inp, layout, cache_seqlens=cache_seqlens)


def ring_seqlens(rng, inp):
    """Seeded cache_seqlens for a workload: 0, small, multiples of L and large values;
    padding rows get -1 (never read for them)."""
    N, L = inp.wl.N, inp.wl.L
    seq = rng.integers(0, 10 * L + 7, size=N).astype(np.int32)
    seq[::5] = 0
    seq[1::7] = 2_000_000_000  # large counts: only the value mod L matters
    if inp.indices is not None:
        seq[inp.indices == -1] = -1
    return seq
