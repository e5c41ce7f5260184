// Update kernel for the compact linear state at L = 1, 2, 4 and 8 (widths 2..4), one channel
// per lane at a time.
//
// At these L one channel's state is 2L bytes, a naturally aligned element (at L = 8 exactly
// 16 bytes), so the compact slab of a slot is an array of one element per channel. The vector kernels give a lane 8
// consecutive channels, i.e. 128 contiguous bytes of state: a warp's 16-byte load then
// touches 32 different 128-byte lines, so each load or store instruction costs 32 L1
// wavefronts, and at L = 8 that request rate, not DRAM, set the time (N=4096, D=16384: 526
// us, 0.64 of the copy rate). Here lane i of a warp takes channels cb + 32 j + i (j = 0..7)
// of the warp's 256-channel block: a warp reads and writes 64 L contiguous bytes of state per
// instruction (4 wavefronts at L = 8), and x, out, weight and bias are read and written as
// coalesced 2- to 8-byte elements. Any D and any padded ld are served (no 16-byte alignment of x rows
// is needed).
//
// Update definition: cuDNN page "Causal Conv1d Decode Update", introduction (update
// block); compact state layout from its "Semantic tensor contract".
#include "ccu_internal.cuh"

namespace ccu {

int device_sm_count();

namespace {

constexpr int kLThreads = 256;            // 8 warps
constexpr int kLanesJ = 8;                // channels per lane per row
constexpr int64_t kWarpCh = 32 * kLanesJ; // channels per warp
constexpr int64_t kCtaCh = 8 * kWarpCh;   // channels per CTA

// Taps of channel c (W of them, zero-padded to 4) packed two per word, and its bias.
template <int W>
__device__ __forceinline__ void channel_weights(const UpdateParams &p, int64_t c, uint32_t (&w)[2], uint32_t &b) {
  if constexpr (W == 4) {
    const uint2 t = __ldg(reinterpret_cast<const uint2 *>(p.w + c * 4));
    w[0] = t.x;
    w[1] = t.y;
  } else if constexpr (W == 2) {
    w[0] = __ldg(reinterpret_cast<const uint32_t *>(p.w + c * 2));
    w[1] = 0u;
  } else {
    const uint16_t *wp = p.w + c * 3;
    w[0] = (uint32_t)__ldg(wp) | ((uint32_t)__ldg(wp + 1) << 16);
    w[1] = (uint32_t)__ldg(wp + 2);
  }
  b = p.bias != nullptr ? (uint32_t)__ldg(p.bias + c) : 0u;
}

// A channel's state at L = 1, 2, 4, 8: 2L bytes, one naturally aligned element.
template <int L> struct Chunk;
template <> struct Chunk<1> { using T = uint16_t; };
template <> struct Chunk<2> { using T = uint32_t; };
template <> struct Chunk<4> { using T = uint2; };
template <> struct Chunk<8> { using T = uint4; };

template <int L>
__device__ __forceinline__ void chunk_words(const typename Chunk<L>::T &c, uint32_t (&w)[4]) {
  if constexpr (L == 1) { w[0] = c; }
  else if constexpr (L == 2) { w[0] = c; }
  else if constexpr (L == 4) { w[0] = c.x; w[1] = c.y; }
  else { w[0] = c.x; w[1] = c.y; w[2] = c.z; w[3] = c.w; }
}

// The shifted state: entries 1 .. L-1, then x.
template <int L>
__device__ __forceinline__ typename Chunk<L>::T shifted(const uint32_t (&s)[4], uint32_t x) {
  if constexpr (L == 1) {
    return (uint16_t)x;
  } else if constexpr (L == 2) {
    return (s[0] >> 16) | (x << 16);
  } else if constexpr (L == 4) {
    return make_uint2(__funnelshift_r(s[0], s[1], 16), (s[1] >> 16) | (x << 16));
  } else {
    return make_uint4(__funnelshift_r(s[0], s[1], 16), __funnelshift_r(s[1], s[2], 16),
                      __funnelshift_r(s[2], s[3], 16), (s[3] >> 16) | (x << 16));
  }
}

// One channel: state s (L entries, oldest first) and input x; returns the BF16 output and
// writes the shifted state to ns. Tap j of width W multiplies history entry L + 1 - W + j of
// the L + 1 (entry L is x), summed in ascending j with FP32 fused multiply-adds (each BF16 x
// BF16 product is exact), then the bias.
template <int L, int W, int ACT>
__device__ __forceinline__ uint32_t one_channel(const typename Chunk<L>::T s, uint32_t x, const uint32_t (&w)[2],
                                                uint32_t b, bool has_bias, typename Chunk<L>::T &ns) {
  uint32_t sw[4] = {0u, 0u, 0u, 0u};
  chunk_words<L>(s, sw);
  float acc = 0.0f;
#pragma unroll
  for (int j = 0; j < W; ++j) {
    const int e = L + 1 - W + j;  // history entry
    const uint32_t h = e == L ? x : get16(sw, e);
    acc = __fmaf_rn(bf16_bits(h), bf16_bits(get16(w, j)), acc);
  }
  if (has_bias) acc = acc + bf16_bits(b);
  ns = shifted<L>(sw, x);
  return round_bf16(activate<ACT>(acc));
}

template <int L, int W, int ACT, bool DEDUP>
__global__ void __launch_bounds__(kLThreads, 3) k_update_lanes(UpdateParams p) {
  grid_dependency_boundary();
  using C = typename Chunk<L>::T;
  const int lane = threadIdx.x & 31;
  const int64_t cb = (int64_t)blockIdx.x * kCtaCh + (int64_t)(threadIdx.x >> 5) * kWarpCh;
  if (cb >= p.D) return;  // the whole warp
  const bool has_bias = p.bias != nullptr;
  // Each lane's weights and bias, kept in shared memory rather than registers (24 registers
  // a thread spilled at the three-CTA budget). A lane reads back only what it wrote, so no
  // barrier is needed; consecutive lanes hold consecutive entries (conflict-free).
  __shared__ uint2 ws[8][kLanesJ][32];
  __shared__ uint32_t bs[8][kLanesJ][32];
  const int wp = threadIdx.x >> 5;
#pragma unroll
  for (int j = 0; j < kLanesJ; ++j) {
    const int64_t c = cb + 32 * j + lane;
    uint32_t w[2] = {0u, 0u}, b = 0u;
    if (c < p.D) channel_weights<W>(p, c, w, b);
    ws[wp][j][lane] = make_uint2(w[0], w[1]);
    bs[wp][j][lane] = b;
  }
  const int64_t R = p.rows_per_cta;
  for (int64_t r0 = (int64_t)blockIdx.y * R; r0 < p.N; r0 += (int64_t)gridDim.y * R) {
    const int64_t r1 = r0 + R < p.N ? r0 + R : p.N;
    for (int64_t n = r0; n < r1; ++n) {
      RowSlot slot = resolve_row<L, false>(p, n);  // one row per warp: the same for every lane
      uint16_t *orow = p.out + n * p.D;
      C st[kLanesJ];
      uint32_t xv[kLanesJ];
      if (slot.s >= 0) {
        const uint16_t *xrow = p.x + n * p.ld;
        const C *srow = reinterpret_cast<const C *>(p.state + slot.s * (p.D * L));
#pragma unroll
        for (int j = 0; j < kLanesJ; ++j) {
          const int64_t c = cb + 32 * j + lane;
          if (c < p.D) {
            xv[j] = __ldcs(xrow + c);
            st[j] = __ldcs(srow + c);
          }
        }
        if constexpr (DEDUP) {
          // the claim after the row's loads: lane 0 for the warp (all 32 lanes are live)
          if (p.owner != nullptr) {
            int own = 1;
            if (lane == 0) {
              own = claim_slot(p.owner, slot.s, n) ? 1 : 0;
              if (!own) atomicOr(p.status, 2);  // CCU_DEVERR_DUPLICATE
            }
            if (!__shfl_sync(0xffffffffu, own, 0)) slot.s = -1;
          }
        }
      }
      if (slot.s < 0) {  // padding row: zero output, state untouched
#pragma unroll
        for (int j = 0; j < kLanesJ; ++j) {
          const int64_t c = cb + 32 * j + lane;
          if (c < p.D) __stcs(orow + c, (uint16_t)0);
        }
        continue;
      }
      C *srow = reinterpret_cast<C *>(p.state + slot.s * (p.D * L));
#pragma unroll
      for (int j = 0; j < kLanesJ; ++j) {
        const int64_t c = cb + 32 * j + lane;
        if (c < p.D) {
          C ns;
          const uint2 wj = ws[wp][j][lane];
          const uint32_t w[2] = {wj.x, wj.y};
          const uint32_t y = one_channel<L, W, ACT>(st[j], xv[j], w, bs[wp][j][lane], has_bias, ns);
          __stcs(srow + c, ns);
          __stcs(orow + c, (uint16_t)y);
        }
      }
    }
  }
}

template <int L, int W, bool DEDUP>
cudaError_t launch_lwd(const UpdateParams &p_in, int act, cudaStream_t stream) {
  UpdateParams p = p_in;
  const int64_t gx = (p.D + kCtaCh - 1) / kCtaCh;
  // Rows per CTA as in the lean vector kernel: one per CTA while the batch does not fill the
  // GPU, three beyond (the weights a CTA loads serve a few rows; CTAs stay short-lived).
  const int64_t sms = device_sm_count();
  const int64_t R = p.N * gx >= 8 * sms ? 3 : 1;
  int64_t gy = (p.N + R - 1) / R;
  if (gy > 65535) gy = 65535;
  p.rows_per_cta = (int)R;
  const dim3 grid((unsigned)gx, (unsigned)gy), block(kLThreads);
  return act == 1 ? launch_overlapped(k_update_lanes<L, W, 1, DEDUP>, grid, block, 0, stream, p)
                  : launch_overlapped(k_update_lanes<L, W, 0, DEDUP>, grid, block, 0, stream, p);
}

template <int L, int W>
cudaError_t launch_lw(const UpdateParams &p, int act, cudaStream_t stream) {
  return p.owner != nullptr ? launch_lwd<L, W, true>(p, act, stream) : launch_lwd<L, W, false>(p, act, stream);
}

}  // namespace

bool lanes_serve(const UpdateParams &p) {
  return p.layout == (int)Layout::Compact && p.seqlens == nullptr && p.W >= 2 && p.W <= kW &&
         p.L >= p.W - 1 && (p.L == 1 || p.L == 2 || p.L == 4 || p.L == 8);
}

// The compact linear state at L = 1, 2, 4, 8 (L >= W - 1), widths 2..4 (anything else:
// cudaErrorInvalidValue).
cudaError_t launch_lanes(const UpdateParams &p, int act, cudaStream_t stream) {
  if (!lanes_serve(p)) return cudaErrorInvalidValue;
  switch (p.W * 16 + p.L) {
    case 2 * 16 + 1: return launch_lw<1, 2>(p, act, stream);
    case 2 * 16 + 2: return launch_lw<2, 2>(p, act, stream);
    case 2 * 16 + 4: return launch_lw<4, 2>(p, act, stream);
    case 2 * 16 + 8: return launch_lw<8, 2>(p, act, stream);
    case 3 * 16 + 2: return launch_lw<2, 3>(p, act, stream);
    case 3 * 16 + 4: return launch_lw<4, 3>(p, act, stream);
    case 3 * 16 + 8: return launch_lw<8, 3>(p, act, stream);
    case 4 * 16 + 4: return launch_lw<4, 4>(p, act, stream);
    case 4 * 16 + 8: return launch_lw<8, 4>(p, act, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ccu
