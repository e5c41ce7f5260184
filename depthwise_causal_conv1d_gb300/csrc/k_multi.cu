// Multi-token update: T tokens per row in one call, x[N, D, T].
//
// The T tokens are appended to the history in order: output t is computed from the width-4
// window ending at token t, and the new state is the last L entries of the history (with
// cache_seqlens, token t is written over ring position (q + t) mod L). Optionally the state
// after every token is written to intermediate_states [N, T, D, L] (compact, in the
// state's own entry order), so a speculative decoder can roll back to any token.
//
// The cuDNN page "Causal Conv1d Decode Update" names this extension without defining it
// ("Semantic tensor contract": a future multi-token form may admit x[N, D, Tstep] without
// changing the state or weight meanings; "Current native implementation": multi-token
// updates and speculative intermediate-state returns are declined today).
#include "ccu_internal.cuh"

namespace ccu {

int device_sm_count();

namespace {

// One thread per (row, channel), any x / out strides, any L: the correctness anchor.
template <int ACT>
__global__ void __launch_bounds__(256) k_multi_scalar(UpdateParams p, MultiParams m) {
  grid_dependency_boundary();
  const int64_t total = p.N * p.D;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = i / p.D;
    const int64_t d = i - n * p.D;
    const RowSlot r = resolve_row<0, false>(p, n);
    if (r.s < 0) {
      for (int64_t t = 0; t < m.T; ++t) p.out[n * m.son + d * m.sod + t * m.sot] = 0;
      continue;
    }
    uint16_t *st = p.state + r.s * p.ss + d * p.sd;
    const int64_t L = p.L;
    const bool ring = p.seqlens != nullptr;
    const int64_t q = ring ? r.q : 0;
    const uint16_t *xp = p.x + n * m.sxn + d * m.sxd;
    const int64_t W = p.W;
    const uint16_t *w = p.w + d * W;
    // Entry k of the time-ordered history (k < L: state entry k, oldest first; else token
    // k - L), read before any of this channel's state is overwritten.
    auto hist = [&](int64_t k) -> uint16_t {
      if (k < L) return st[(ring ? (q + k) % L : k) * p.sl];
      return xp[(k - L) * m.sxt];
    };
    // the W-1 window entries before the first token (newest last), in hw[3-(W-1) .. 2]
    uint16_t hw[3] = {0, 0, 0};
    for (int64_t k = 0; k < W - 1; ++k) hw[3 - (W - 1) + k] = hist(L - (W - 1) + k);
    for (int64_t t = 0; t < m.T; ++t) {
      const uint16_t xv = xp[t * m.sxt];
      float acc = 0.0f;
      for (int64_t k = 0; k < W - 1; ++k)
        acc = __fmaf_rn(bf16_bits(hw[3 - (W - 1) + k]), bf16_bits(w[k]), acc);
      acc = __fmaf_rn(bf16_bits(xv), bf16_bits(w[W - 1]), acc);
      if (p.bias != nullptr) acc = acc + bf16_bits(p.bias[d]);
      p.out[n * m.son + d * m.sod + t * m.sot] = round_bf16(activate<ACT>(acc));
      hw[0] = hw[1];
      hw[1] = hw[2];
      hw[2] = xv;
      if (m.inter != nullptr) {
        // the state after token t in its own order: history[t+1 .. t+L]; a ring holds the
        // entry of age (l - (q + t + 1)) mod L at position l
        uint16_t *it = m.inter + ((n * m.T + t) * p.D + d) * L;
        for (int64_t l = 0; l < L; ++l) {
          int64_t age = l;
          if (ring) {
            age = (l - (q + t + 1)) % L;
            if (age < 0) age += L;
          }
          it[l] = hist(t + 1 + age);
        }
      }
    }
    // The new state: the last L history entries. Linear: entry i takes history[T + i],
    // ascending, so each entry is read before it is overwritten. Ring: the tokens land at
    // (q + t) mod L in order; only the last L writes survive.
    if (ring) {
      for (int64_t t = (m.T > L ? m.T - L : 0); t < m.T; ++t) st[((q + t) % L) * p.sl] = xp[t * m.sxt];
    } else {
      for (int64_t l = 0; l < L; ++l) st[l * p.sl] = hist(m.T + l);
    }
  }
}

// Compact-order position of (channel c, entry l) in 4*L words, and the static transposes
// between the channel-last planes and that order.
template <int L>
__device__ __forceinline__ void planes_to_compact(const uint32_t (&pl)[4 * L], uint32_t (&cw)[4 * L]) {
#pragma unroll
  for (int i = 0; i < 4 * L; ++i) {
    const int e0 = 2 * i, e1 = 2 * i + 1;  // compact positions c*L + l
    const uint32_t v0 = get16(pl, (e0 % L) * 8 + e0 / L);
    const uint32_t v1 = get16(pl, (e1 % L) * 8 + e1 / L);
    cw[i] = v0 | (v1 << 16);
  }
}

template <int L>
__device__ __forceinline__ void compact_to_planes(const uint32_t (&cw)[4 * L], uint32_t (&pl)[4 * L]) {
#pragma unroll
  for (int i = 0; i < 4 * L; ++i) {
    const int e0 = 2 * i, e1 = 2 * i + 1;  // plane positions l*8 + c
    const uint32_t v0 = get16(cw, (e0 % 8) * L + e0 / 8);
    const uint32_t v1 = get16(cw, (e1 % 8) * L + e1 / 8);
    pl[i] = v0 | (v1 << 16);
  }
}

// 8 channels per thread, x and out channel-contiguous (16-byte vectors per token), state in
// registers in compact order for the whole row, L and layout compile-time. A thread issues
// two rows' loads (state and first four tokens) before computing either: bound by load
// latency with one row in flight, the multi-token workload went from 92.4 to 85.9 us (and
// the T = 1 shape from 217 to 180 us) at the same two CTAs per SM, which the 128-register
// cap keeps (without the cap the kernel takes 170 registers, one CTA per SM, and loses).
// The SiLU runs on channel pairs (the arithmetic is not hidden here: 86.0 -> 84.1 us), at
// 72 spilled bytes.
template <int L, int W, int ACT, int LAYOUT, bool RING, int ROWS>
__device__ __forceinline__ void multi_vector_body(const UpdateParams &p, const MultiParams &m) {
  const int64_t groups = p.D >> 3;
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= groups) return;
  const int64_t c0 = g << 3;
  uint32_t wv[16];
  load_weights_packed<W>(p.w, c0, wv);
  const bool has_bias = p.bias != nullptr;
  uint32_t bv[4] = {0u, 0u, 0u, 0u};
  if (has_bias) {
    const uint4 t = ld_keep(p.bias + c0);
    bv[0] = t.x; bv[1] = t.y; bv[2] = t.z; bv[3] = t.w;
  }

  struct MRow {
    RowSlot slot;
    int64_t n;
    uint32_t ow[4 * L];
    uint4 xg[4];
  };
  auto load_row = [&](int64_t n, MRow &r) {
    r.n = n;
    r.slot = resolve_row<L, false>(p, n);
    if (r.slot.s < 0) return;
    if constexpr (LAYOUT == (int)Layout::Compact) {
      const uint16_t *sp = p.state + r.slot.s * (p.D * L) + c0 * L;
#pragma unroll
      for (int k = 0; k < L; ++k) {
        const uint4 u = ld_stream(sp + 8 * k);
        r.ow[4 * k] = u.x; r.ow[4 * k + 1] = u.y; r.ow[4 * k + 2] = u.z; r.ow[4 * k + 3] = u.w;
      }
    } else {
      const uint16_t *sp = p.state + r.slot.s * (L * p.D) + c0;
      uint32_t pl[4 * L];
#pragma unroll
      for (int l = 0; l < L; ++l) {
        const uint4 u = ld_stream(sp + (int64_t)l * p.D);
        pl[4 * l] = u.x; pl[4 * l + 1] = u.y; pl[4 * l + 2] = u.z; pl[4 * l + 3] = u.w;
      }
      planes_to_compact<L>(pl, r.ow);
    }
    const uint16_t *xrow = p.x + n * m.sxn + c0;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (k < m.T) r.xg[k] = ld_stream(xrow + k * m.sxt);
  };
  auto process_row = [&](MRow &r) {
    const int64_t n = r.n;
    if (r.slot.s < 0) {
      for (int64_t t = 0; t < m.T; ++t)
        st_stream(p.out + n * m.son + t * m.sot + c0, make_uint4(0u, 0u, 0u, 0u));
      return;
    }
    const uint16_t *xrow = p.x + n * m.sxn + c0;
    uint16_t *orow = p.out + n * m.son + c0;
    constexpr int kGroup = 4;
    for (int64_t t0 = 0; t0 < m.T; t0 += kGroup) {
      if (t0 > 0) {
#pragma unroll
        for (int k = 0; k < kGroup; ++k)
          if (t0 + k < m.T) r.xg[k] = ld_stream(xrow + (t0 + k) * m.sxt);
      }
#pragma unroll
      for (int k = 0; k < kGroup; ++k) {
        const int64_t t = t0 + k;
        if (t >= m.T) break;
        const uint32_t xw[4] = {r.xg[k].x, r.xg[k].y, r.xg[k].z, r.xg[k].w};
        uint32_t nw[4 * L];
        uint4 outv;
        if constexpr (RING) {
          outv = update8_compact_ring<L, W, ACT, true>(xw, r.ow, wv, bv, has_bias,
                                                        (int)((r.slot.q + t) % L), nw);
        } else {
          outv = update8_compact<L, W, ACT, true>(xw, r.ow, wv, bv, has_bias, nw);
        }
        st_stream(orow + t * m.sot, outv);
#pragma unroll
        for (int i = 0; i < 4 * L; ++i) r.ow[i] = nw[i];
        if (m.inter != nullptr) {
          uint16_t *it = m.inter + ((n * m.T + t) * p.D + c0) * L;
#pragma unroll
          for (int q = 0; q < L; ++q)
            st_stream(it + 8 * q, make_uint4(r.ow[4 * q], r.ow[4 * q + 1], r.ow[4 * q + 2], r.ow[4 * q + 3]));
        }
      }
    }
    if constexpr (LAYOUT == (int)Layout::Compact) {
      uint16_t *sp = p.state + r.slot.s * (p.D * L) + c0 * L;
#pragma unroll
      for (int k = 0; k < L; ++k)
        st_stream(sp + 8 * k, make_uint4(r.ow[4 * k], r.ow[4 * k + 1], r.ow[4 * k + 2], r.ow[4 * k + 3]));
    } else {
      uint16_t *sp = p.state + r.slot.s * (L * p.D) + c0;
      uint32_t pl[4 * L];
      compact_to_planes<L>(r.ow, pl);
#pragma unroll
      for (int l = 0; l < L; ++l)
        st_stream(sp + (int64_t)l * p.D, make_uint4(pl[4 * l], pl[4 * l + 1], pl[4 * l + 2], pl[4 * l + 3]));
    }
  };
  // Two rows' loads (state and the first four tokens) in flight before either is computed.
  if constexpr (ROWS == 2) {
    for (int64_t n = blockIdx.y; n < p.N; n += 2 * (int64_t)gridDim.y) {
      const int64_t n2 = n + gridDim.y;
      MRow a, b;
      load_row(n, a);
      if (n2 < p.N) load_row(n2, b);
      process_row(a);
      if (n2 < p.N) process_row(b);
    }
  } else {
    for (int64_t n = blockIdx.y; n < p.N; n += gridDim.y) {
      MRow a;
      load_row(n, a);
      process_row(a);
    }
  }
}

// Up to L = 6: two rows in flight under a 128-register cap (two CTAs per SM).
template <int L, int W, int ACT, int LAYOUT, bool RING>
__global__ void __launch_bounds__(256, 2) k_multi_vector(UpdateParams p, MultiParams m) {
  grid_dependency_boundary();
  multi_vector_body<L, W, ACT, LAYOUT, RING, 2>(p, m);
}

// L = 7 and 8: one row in flight and the compiler's register budget (the two-row form
// spills 300-600 bytes there under the cap; N=1024, D=16384, T=4: L = 7 148.3 against
// 192.8 us, L = 8 144.7 against 206.9 us).
template <int L, int W, int ACT, int LAYOUT, bool RING>
__global__ void __launch_bounds__(256) k_multi_vector_long(UpdateParams p, MultiParams m) {
  grid_dependency_boundary();
  multi_vector_body<L, W, ACT, LAYOUT, RING, 1>(p, m);
}

template <int L, int W, int ACT, int LAYOUT, bool RING>
cudaError_t launch_vec_one(const UpdateParams &p, const MultiParams &m, dim3 grid, dim3 block,
                           cudaStream_t stream) {
  if constexpr (L >= 7) {
    return launch_overlapped(k_multi_vector_long<L, W, ACT, LAYOUT, RING>, grid, block, 0, stream, p, m);
  } else {
    return launch_overlapped(k_multi_vector<L, W, ACT, LAYOUT, RING>, grid, block, 0, stream, p, m);
  }
}

template <int L, int W, int ACT>
cudaError_t launch_vec_L(const UpdateParams &p, const MultiParams &m, dim3 grid, dim3 block,
                         cudaStream_t stream) {
  const bool ring = p.seqlens != nullptr;
  constexpr int kC = (int)Layout::Compact, kCL = (int)Layout::ChannelLast;
  if (p.layout == kC) {
    return ring ? launch_vec_one<L, W, ACT, kC, true>(p, m, grid, block, stream)
                : launch_vec_one<L, W, ACT, kC, false>(p, m, grid, block, stream);
  }
  return ring ? launch_vec_one<L, W, ACT, kCL, true>(p, m, grid, block, stream)
              : launch_vec_one<L, W, ACT, kCL, false>(p, m, grid, block, stream);
}

// Width 4 with L = 3..8; widths 2 and 3 with L = W - 1..4 (the short states they are used
// with; longer states run on the scalar kernel).
template <int ACT>
cudaError_t launch_vec_A(const UpdateParams &p, const MultiParams &m, dim3 grid, dim3 block,
                         cudaStream_t stream) {
  switch (p.W * 16 + p.L) {
    case 4 * 16 + 3: return launch_vec_L<3, 4, ACT>(p, m, grid, block, stream);
    case 4 * 16 + 4: return launch_vec_L<4, 4, ACT>(p, m, grid, block, stream);
    case 4 * 16 + 5: return launch_vec_L<5, 4, ACT>(p, m, grid, block, stream);
    case 4 * 16 + 6: return launch_vec_L<6, 4, ACT>(p, m, grid, block, stream);
    case 4 * 16 + 7: return launch_vec_L<7, 4, ACT>(p, m, grid, block, stream);
    case 4 * 16 + 8: return launch_vec_L<8, 4, ACT>(p, m, grid, block, stream);
    case 3 * 16 + 2: return launch_vec_L<2, 3, ACT>(p, m, grid, block, stream);
    case 3 * 16 + 3: return launch_vec_L<3, 3, ACT>(p, m, grid, block, stream);
    case 3 * 16 + 4: return launch_vec_L<4, 3, ACT>(p, m, grid, block, stream);
    case 2 * 16 + 1: return launch_vec_L<1, 2, ACT>(p, m, grid, block, stream);
    case 2 * 16 + 2: return launch_vec_L<2, 2, ACT>(p, m, grid, block, stream);
    case 2 * 16 + 3: return launch_vec_L<3, 2, ACT>(p, m, grid, block, stream);
    case 2 * 16 + 4: return launch_vec_L<4, 2, ACT>(p, m, grid, block, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_multi_scalar(const UpdateParams &p, const MultiParams &m, int act,
                                cudaStream_t stream) {
  const int threads = 256;
  int64_t blocks = (p.N * p.D + threads - 1) / threads;
  const int64_t cap = (int64_t)device_sm_count() * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const dim3 grid((unsigned)blocks), block(threads);
  return act == 1 ? launch_overlapped(k_multi_scalar<1>, grid, block, 0, stream, p, m)
                  : launch_overlapped(k_multi_scalar<0>, grid, block, 0, stream, p, m);
}

cudaError_t launch_multi_vector(const UpdateParams &p, const MultiParams &m, int act,
                                cudaStream_t stream) {
  const int64_t groups = p.D / 8;
  int threads = 256;
  if (groups < threads) threads = (int)((groups + 31) / 32 * 32);
  const int64_t gx = (groups + threads - 1) / threads;
  // one row per CTA row-step: each row already carries T tokens of work
  int64_t gy = (int64_t)device_sm_count() * 8 / gx;
  if (gy < 1) gy = 1;
  if (gy > p.N) gy = p.N;
  if (gy > 65535) gy = 65535;
  const dim3 grid((unsigned)gx, (unsigned)gy), block(threads);
  return act == 1 ? launch_vec_A<1>(p, m, grid, block, stream) : launch_vec_A<0>(p, m, grid, block, stream);
}

}  // namespace ccu
