// Multi-token update: T tokens per row in one call, x[N, D, T]. The vector kernel family
// (instantiated in k_multi.cu for width 4 and k_multi_narrow.cu for widths 2 and 3).
//
// The T tokens are appended to the history in order: output t is computed from the width-W
// window ending at token t, and the new state is the last L entries of the history (with
// cache_seqlens, token t is written over ring position (q + t) mod L). Optionally the state
// after every token is written to intermediate_states [N, T, D, L] (compact, in the
// state's own entry order), so a speculative decoder can roll back to any token.
//
// The cuDNN page "Causal Conv1d Decode Update" names this extension without defining it
// ("Semantic tensor contract": a future multi-token form may admit x[N, D, Tstep] without
// changing the state or weight meanings; "Current native implementation": multi-token
// updates and speculative intermediate-state returns are declined today).
#pragma once

#include "ccu_internal.cuh"

namespace ccu {

int device_sm_count();

namespace {

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
// registers in compact order for the whole row, L and layout compile-time. ROWS = 2: a thread
// issues two rows' loads (state and first four tokens) before computing either (on the
// compact L = 3 workload that took 92.4 to 85.9 us against the one-row loop of the time, at
// the same two CTAs per SM, which the 128-register cap keeps; the choice per state is in
// multi_two_rows). The SiLU runs on channel pairs (the arithmetic is not hidden here: 86.0
// -> 84.1 us).
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

// Two rows in flight under a 128-register cap (two CTAs per SM).
template <int L, int W, int ACT, int LAYOUT, bool RING>
__global__ void __launch_bounds__(256, 2) k_multi_vector(UpdateParams p, MultiParams m) {
  grid_dependency_boundary();
  multi_vector_body<L, W, ACT, LAYOUT, RING, 2>(p, m);
}

// One row in flight (the two-row form spills 300-600 bytes at L = 7, 8 under its cap). With
// no occupancy hint the compiler keeps it within 128 registers, two CTAs per SM, except at
// L = 7, where it took up to 166 and one CTA per SM; that instance is held to two CTAs
// (36 to 72 spilled bytes; N=1024, D=16384, T=4: compact L = 7 121.5 against 145.6 us,
// channel-last 119.7 against 141.0). A hint of one CTA per SM lets the compiler take 162 to
// 200 registers at L = 4, 5, 6, 8 instead, and those ran 15 to 30 % slower. One channel per
// lane, as the single-token update runs
// L = 8, lost here (each lane stepping 8 channels' states through the tokens, four tokens'
// inputs loaded ahead): L = 8 took 165.7 against 144.2 us and L = 4 138.8 against 90.2 us
// (T = 8, L = 8: 262.9 against 187.3 us); only T = 1 was faster (99.7 against 131.3 us), and
// a single token goes through the update itself.
template <int L, int W, int ACT, int LAYOUT, bool RING>
__global__ void __launch_bounds__(256) k_multi_vector_one_row(UpdateParams p, MultiParams m) {
  grid_dependency_boundary();
  multi_vector_body<L, W, ACT, LAYOUT, RING, 1>(p, m);
}

template <int L, int W, int ACT, int LAYOUT, bool RING>
__global__ void __launch_bounds__(256, 2) k_multi_vector_one_row_2cta(UpdateParams p, MultiParams m) {
  grid_dependency_boundary();
  multi_vector_body<L, W, ACT, LAYOUT, RING, 1>(p, m);
}

// The two-row form is kept where it measured ahead or level: the compact linear state up to
// L = 3 and the compact ring at L = 4. Everywhere else one row in flight wins. N=1024,
// D=16384, T=4, SiLU, us, one row (at its best grid) / two rows: compact L = 3 79.5 / 79.6,
// L = 4 87.6 / 88.8, L = 5 96.0 / 110.6, L = 6 107.2 / 115.6, L = 7 121.5 / 192.8; compact
// ring L = 3 89.2 / 99.4, L = 4 110.0 / 108.3, L = 5 123.8 / 126.0, L = 6 117.9 / 141.1;
// channel-last L = 3 80.5 / 88.4, L = 4 87.2 / 97.9, L = 5 95.0 / 114.5, L = 6 103.6 / 132.5;
// channel-last ring L = 3 90.4 / 105.0, L = 4 103.2 / 108.8, L = 5 106.9 / 138.1, L = 6
// 125.4 / 162.3.
template <int L, int LAYOUT, bool RING>
__host__ __device__ constexpr bool multi_two_rows() {
  return LAYOUT == (int)Layout::Compact && (RING ? L == 4 : L <= 3);
}

template <int L, int W, int ACT, int LAYOUT, bool RING>
cudaError_t launch_vec_one(const UpdateParams &p, const MultiParams &m, dim3 grid, dim3 block,
                           cudaStream_t stream) {
  if constexpr (multi_two_rows<L, LAYOUT, RING>()) {
    return launch_overlapped(k_multi_vector<L, W, ACT, LAYOUT, RING>, grid, block, 0, stream, p, m);
  } else if constexpr (L == 7) {
    return launch_overlapped(k_multi_vector_one_row_2cta<L, W, ACT, LAYOUT, RING>, grid, block, 0, stream, p, m);
  } else {
    return launch_overlapped(k_multi_vector_one_row<L, W, ACT, LAYOUT, RING>, grid, block, 0, stream, p, m);
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

}  // namespace

}  // namespace ccu
