// Vector kernels: each thread owns 8 consecutive channels of one row at a time and moves
// x, weight, bias, state and out as 16-byte vectors. L (W-1..8), the width W (2..4), the
// state layout, linear or ring state and the activation are compile-time, so the history
// lives in registers and the shift is a fixed permutation of 16-bit lanes.
//
// Update definition: cuDNN page "Causal Conv1d Decode Update", introduction (update
// block); layouts from its "Semantic tensor contract" (compact state, and the
// channel-last (L*D, 1, D) state a full-sequence prefill hands over).
#include "ccu_internal.cuh"

namespace ccu {

int device_sm_count();

namespace {

// W: filter width (2..4). RING: conv_state is a ring buffer indexed by cache_seqlens.
// The body of the two kernels below.
template <int L, int W, int ACT, int LAYOUT, bool RING>
__device__ __forceinline__ void update_vector(const UpdateParams &p) {
  const int64_t groups = p.D >> 3;  // 8-channel groups per row (D % 8 == 0)
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= groups) return;
  const int64_t c0 = g << 3;

  // weight[c0 .. c0+7, 0..W-1] in W 16-byte vectors, kept packed (two per word) and
  // widened at use; bias likewise. Both are reused for every row.
  uint32_t wv[16];
  load_weights_packed<W>(p.w, c0, wv);
  const bool has_bias = p.bias != nullptr;
  uint32_t bv[4] = {0u, 0u, 0u, 0u};
  if (has_bias) {
    const uint4 t = ld_keep(p.bias + c0);
    bv[0] = t.x; bv[1] = t.y; bv[2] = t.z; bv[3] = t.w;
  }

  // A thread walks R rows two at a time: the loads of both rows (slot, x and state) are
  // issued before either is computed and stored, so two rows' loads are in flight per
  // thread whatever the compiler's schedule (left to itself, the schedule of the compact
  // single-row loop varied between builds from 168 to 303 us on the large batch). Slots
  // are unique within a call, so one row's stores never touch the other row's state.
  constexpr bool kPlanes = (LAYOUT == (int)Layout::ChannelLast);
  // State words held per row: compact 4L; channel-last linear 4L (plane 0 unused when
  // L > 3); channel-last ring: the three window planes.
  constexpr int kWords = (kPlanes && RING) ? 4 * (W - 1) : 4 * L;
  struct Row {
    RowSlot slot;
    uint32_t xw[4];
    uint32_t ow[kWords];
  };

  auto load_row = [&](int64_t n, Row &r) {
    r.slot = resolve_row<L>(p, n);
    if (r.slot.s < 0) return;
    const uint4 t = ld_stream(p.x + n * p.ld + c0);
    r.xw[0] = t.x; r.xw[1] = t.y; r.xw[2] = t.z; r.xw[3] = t.w;
    if constexpr (!kPlanes) {
      const uint16_t *sp = p.state + r.slot.s * (p.D * L) + c0 * L;
#pragma unroll
      for (int k = 0; k < L; ++k) {
        const uint4 u = ld_stream(sp + 8 * k);
        r.ow[4 * k] = u.x; r.ow[4 * k + 1] = u.y; r.ow[4 * k + 2] = u.z; r.ow[4 * k + 3] = u.w;
      }
    } else if constexpr (RING) {
      const uint16_t *sp = p.state + r.slot.s * (L * p.D) + c0;
#pragma unroll
      for (int k = 0; k < W - 1; ++k) {
        const uint4 u = ld_stream(sp + (int64_t)((r.slot.q + L - (W - 1) + k) % L) * p.D);
        r.ow[4 * k] = u.x; r.ow[4 * k + 1] = u.y; r.ow[4 * k + 2] = u.z; r.ow[4 * k + 3] = u.w;
      }
    } else {
      // Plane 0 is read only when L == W - 1: it is then inside the window; otherwise it
      // is outside the window and is overwritten by plane 1.
      const uint16_t *sp = p.state + r.slot.s * (L * p.D) + c0;
      constexpr int first = (L == W - 1) ? 0 : 1;
#pragma unroll
      for (int l = 0; l < L; ++l) {
        if (l < first) {
          r.ow[4 * l] = r.ow[4 * l + 1] = r.ow[4 * l + 2] = r.ow[4 * l + 3] = 0u;
          continue;
        }
        const uint4 u = ld_stream(sp + (int64_t)l * p.D);
        r.ow[4 * l] = u.x; r.ow[4 * l + 1] = u.y; r.ow[4 * l + 2] = u.z; r.ow[4 * l + 3] = u.w;
      }
    }
  };

  auto store_row = [&](int64_t n, const Row &r) {
    uint16_t *outp = p.out + n * p.D + c0;
    if (r.slot.s < 0) {  // padding row: zero output, state untouched
      st_stream(outp, make_uint4(0u, 0u, 0u, 0u));
      return;
    }
    uint4 outv;
    if constexpr (!kPlanes) {
      uint32_t nw[4 * L];
      if constexpr (RING) {
        outv = update8_compact_ring<L, W, ACT>(r.xw, r.ow, wv, bv, has_bias, r.slot.q, nw);
      } else {
        outv = update8_compact<L, W, ACT>(r.xw, r.ow, wv, bv, has_bias, nw);
      }
      uint16_t *sp = p.state + r.slot.s * (p.D * L) + c0 * L;
#pragma unroll
      for (int k = 0; k < L; ++k)
        st_stream(sp + 8 * k, make_uint4(nw[4 * k], nw[4 * k + 1], nw[4 * k + 2], nw[4 * k + 3]));
    } else {
      uint16_t *sp = p.state + r.slot.s * (L * p.D) + c0;
      // window planes: the ring's W-1, or the linear state's last W-1
      constexpr int wp0 = RING ? 0 : L - (W - 1);
      uint32_t h[3][8], xs[8];
#pragma unroll
      for (int k = 0; k < W - 1; ++k)
        unpack8(make_uint4(r.ow[4 * (wp0 + k)], r.ow[4 * (wp0 + k) + 1], r.ow[4 * (wp0 + k) + 2],
                           r.ow[4 * (wp0 + k) + 3]),
                h[k]);
      unpack8(make_uint4(r.xw[0], r.xw[1], r.xw[2], r.xw[3]), xs);
      outv = outputs8_window<W, ACT>(h, xs, wv, bv, has_bias);
      if constexpr (RING) {
        st_stream(sp + (int64_t)r.slot.q * p.D, make_uint4(r.xw[0], r.xw[1], r.xw[2], r.xw[3]));
      } else {
        // plane l takes old plane l+1; the newest plane takes x
#pragma unroll
        for (int l = 0; l + 1 < L; ++l)
          st_stream(sp + (int64_t)l * p.D, make_uint4(r.ow[4 * (l + 1)], r.ow[4 * (l + 1) + 1],
                                                      r.ow[4 * (l + 1) + 2], r.ow[4 * (l + 1) + 3]));
        st_stream(sp + (int64_t)(L - 1) * p.D, make_uint4(r.xw[0], r.xw[1], r.xw[2], r.xw[3]));
      }
    }
    st_stream(outp, outv);
  };

  const int64_t R = p.rows_per_cta;
  for (int64_t r0 = (int64_t)blockIdx.y * R; r0 < p.N; r0 += (int64_t)gridDim.y * R) {
    const int64_t r1 = r0 + R < p.N ? r0 + R : p.N;
    if constexpr (kPlanes && RING) {
      // The channel-last ring update holds 16 registers of loaded data per row and was
      // bound by load latency with two rows in flight: four rows in flight took the large
      // batch from 142.5 to 125.2 us (the other forms measured slower this way).
      for (int64_t n = r0; n < r1; n += 4) {
        Row rw[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (n + k < r1) load_row(n + k, rw[k]);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (n + k < r1) store_row(n + k, rw[k]);
      }
    } else {
      for (int64_t n = r0; n < r1; n += 2) {
        Row a, b;
        load_row(n, a);
        if (n + 1 < r1) load_row(n + 1, b);
        store_row(n, a);
        if (n + 1 < r1) store_row(n + 1, b);
      }
    }
  }
}

// Register budget left to the compiler (two CTAs per SM at the register counts it picks).
template <int L, int W, int ACT, int LAYOUT, bool RING>
__global__ void __launch_bounds__(256) k_update_vector(UpdateParams p) {
  grid_dependency_boundary();
  update_vector<L, W, ACT, LAYOUT, RING>(p);
}

// Width 3 at three CTAs per SM (at most 85 registers a thread): measured on the large batch at
// L = 2, 118.6 us against 130.7 us with the compiler's budget; the other widths measured
// slower with that cap.
template <int L, int ACT, int LAYOUT, bool RING>
__global__ void __launch_bounds__(256, 3) k_update_vector_w3(UpdateParams p) {
  grid_dependency_boundary();
  update_vector<L, 3, ACT, LAYOUT, RING>(p);
}

template <int L, int W, int ACT, int LAYOUT, bool RING>
cudaError_t launch_one(const UpdateParams &p, dim3 grid, dim3 block, cudaStream_t stream) {
  if constexpr (W == 3) {
    return launch_overlapped(k_update_vector_w3<L, ACT, LAYOUT, RING>, grid, block, 0, stream, p);
  } else {
    return launch_overlapped(k_update_vector<L, W, ACT, LAYOUT, RING>, grid, block, 0, stream, p);
  }
}

template <int L, int W, int ACT>
cudaError_t launch_LW(const UpdateParams &p, dim3 grid, dim3 block, cudaStream_t stream) {
  const bool ring = p.seqlens != nullptr;
  if (p.layout == (int)Layout::Compact) {
    return ring ? launch_one<L, W, ACT, (int)Layout::Compact, true>(p, grid, block, stream)
                : launch_one<L, W, ACT, (int)Layout::Compact, false>(p, grid, block, stream);
  }
  return ring ? launch_one<L, W, ACT, (int)Layout::ChannelLast, true>(p, grid, block, stream)
              : launch_one<L, W, ACT, (int)Layout::ChannelLast, false>(p, grid, block, stream);
}

// L from W - 1 (the shortest state the contract allows) up to kVectorMaxL.
template <int W, int ACT>
cudaError_t launch_W(const UpdateParams &p, dim3 grid, dim3 block, cudaStream_t stream) {
  switch (p.L) {
    case 1: if constexpr (W - 1 <= 1) return launch_LW<1, W, ACT>(p, grid, block, stream); break;
    case 2: if constexpr (W - 1 <= 2) return launch_LW<2, W, ACT>(p, grid, block, stream); break;
    case 3: return launch_LW<3, W, ACT>(p, grid, block, stream);
    case 4: return launch_LW<4, W, ACT>(p, grid, block, stream);
    case 5: return launch_LW<5, W, ACT>(p, grid, block, stream);
    case 6: return launch_LW<6, W, ACT>(p, grid, block, stream);
    case 7: return launch_LW<7, W, ACT>(p, grid, block, stream);
    case 8: return launch_LW<8, W, ACT>(p, grid, block, stream);
    default: break;
  }
  return cudaErrorInvalidValue;
}

template <int ACT>
cudaError_t launch_act(const UpdateParams &p, dim3 grid, dim3 block, cudaStream_t stream) {
  switch (p.W) {
    case 2: return launch_W<2, ACT>(p, grid, block, stream);
    case 3: return launch_W<3, ACT>(p, grid, block, stream);
    case 4: return launch_W<4, ACT>(p, grid, block, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_vector(const UpdateParams &p_in, int act, cudaStream_t stream) {
  UpdateParams p = p_in;
  const int64_t groups = p.D / 8;
  int threads = 256;
  if (groups < threads) threads = (int)((groups + 31) / 32 * 32);
  const int64_t gx = (groups + threads - 1) / threads;
  // Rows per CTA: enough CTAs for several waves on every SM, a few rows each so the
  // weights loaded into registers are reused and a thread has a pair of rows in flight.
  // At least 4 rows once that still leaves a full wave of CTAs (two per SM): measured at
  // D = 16384, 1024 rows took 63.6 us at one row per CTA and 47.2 us at four; 4096 rows
  // take 164.4 us at six (the computed R), 170.0 at four and 242.4 at one.
  const int64_t sms = device_sm_count();
  const int64_t target_ctas = sms * 32;
  int64_t R = (p.N * gx) / target_ctas;
  R = R > 8 ? 8 : R;
  if (R < 4) R = p.N * gx >= 4 * 2 * sms ? 4 : 1;
  // The channel-last ring form walks its rows four at a time: whole groups of four.
  if (p.layout == (int)Layout::ChannelLast && p.seqlens != nullptr) R = R < 4 ? 4 : (R + 3) / 4 * 4;
  int64_t gy = (p.N + R - 1) / R;
  if (gy > 65535) gy = 65535;  // the row loop strides over the rest
  p.rows_per_cta = (int)R;
  const dim3 grid((unsigned)gx, (unsigned)gy);
  const dim3 block(threads);
  return act == 1 ? launch_act<1>(p, grid, block, stream) : launch_act<0>(p, grid, block, stream);
}

}  // namespace ccu
