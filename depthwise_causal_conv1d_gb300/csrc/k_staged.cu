// Staged kernels for any state length L (W-1..256) and width W (2..4) with 8-channel groups
// (D % 8 == 0); linear or ring-buffer state.
//
// Compact layout: a CTA owns a tile of C channels of one row at a time. The tile's state
// slab (C*L contiguous BF16) and its x values are copied into shared memory with
// coalesced 16-byte loads; outputs are computed from shared memory; the new slab is
// written back with coalesced 16-byte stores. Seen as one flat array, the compact
// update is new[e] = (e % L == L-1) ? x[e / L] : old[e + 1], so every 16-byte output
// chunk is a one-element shift of the staged slab with x spliced in.
//
// Channel-last layout (L*D, 1, D): every plane is contiguous over channels, so the shift
// is plane l <- plane l+1 and plane L-1 <- x, done with 16-byte vectors per thread.
//
// Update definition: cuDNN page "Causal Conv1d Decode Update", introduction (update
// block) and "Semantic tensor contract" (conv_state [S, D, L] with L >= W - 1).
#include <atomic>

#include "ccu_internal.cuh"

namespace ccu {

int device_sm_count();
int current_device();

namespace {

constexpr int kMaxDevices = 64;

// weight[c0 .. c0+7, 0..W-1] (W 16-byte vectors) widened to floats wf[c][j], and the bias.
__device__ __forceinline__ void load_weights8(const UpdateParams &p, int64_t c0, float (&wf)[8][kW],
                                              float (&bf)[8]) {
  const int W = (int)p.W;
  const uint16_t *wp = p.w + c0 * W;
  for (int k = 0; k < W; ++k) {
    const uint4 t = ld_keep(wp + 8 * k);
    const uint32_t v[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = 8 * k + 2 * i;  // flat c*W + j of the low half
      wf[e / W][e % W] = bf16_lo(v[i]);
      wf[(e + 1) / W][(e + 1) % W] = bf16_hi(v[i]);
    }
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) bf[c] = 0.0f;
  if (p.bias != nullptr) {
    const uint4 t = ld_keep(p.bias + c0);
    const uint32_t v[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      bf[2 * i] = bf16_lo(v[i]);
      bf[2 * i + 1] = bf16_hi(v[i]);
    }
  }
}

// Outputs of 8 channels from the W-1 window entries h[k][c] (k < W-1) and x.
template <int ACT>
__device__ __forceinline__ uint4 outputs8(const uint32_t (&h)[3][8], const uint32_t (&xs)[8],
                                          const float (&wf)[8][kW], const float (&bf)[8],
                                          bool has_bias, int W) {
  float y[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    float acc = 0.0f;
    for (int k = 0; k < W - 1; ++k) acc = __fmaf_rn(bf16_bits(h[k][c]), wf[c][k], acc);
    acc = __fmaf_rn(bf16_bits(xs[c]), wf[c][W - 1], acc);
    if (has_bias) acc = acc + bf[c];
    y[c] = activate<ACT>(acc);
  }
  return make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                    pack_bf16x2(y[6], y[7]));
}

// Compact layout. Dynamic shared memory: 8*T*L BF16 for the slab, then 8*T BF16 for x.
template <int ACT>
__global__ void __launch_bounds__(256) k_update_staged_compact(UpdateParams p) {
  grid_dependency_boundary();
  extern __shared__ uint4 smem[];
  const int T = blockDim.x;
  const int tid = threadIdx.x;
  const int64_t L = p.L;
  const int64_t c_base = (int64_t)blockIdx.x * 8 * T;
  const int64_t rem = p.D - c_base;
  const int64_t C = rem < 8 * T ? rem : 8 * T;  // channels in this tile, multiple of 8
  uint16_t *s_state = reinterpret_cast<uint16_t *>(smem);
  uint16_t *s_x = s_state + (int64_t)8 * T * L;
  const int64_t nvec = C * L / 8;  // 16-byte chunks of the slab
  const bool mine = (int64_t)8 * tid < C;
  const bool has_bias = p.bias != nullptr;

  float wf[8][kW], bf[8];
  if (mine) load_weights8(p, c_base + 8 * tid, wf, bf);

  const bool ring = p.seqlens != nullptr;
  for (int64_t n = blockIdx.y; n < p.N; n += gridDim.y) {
    const RowSlot row = resolve_row(p, n);  // same for the whole CTA
    const int64_t s = row.s;
    const int64_t q = row.q;                // ring position of the oldest entry
    uint16_t *outp = p.out + n * p.D + c_base + 8 * tid;
    if (s < 0) {
      if (mine) st_stream(outp, make_uint4(0u, 0u, 0u, 0u));
      continue;
    }
    uint16_t *slab = p.state + s * (p.D * L) + c_base * L;
    for (int64_t v = tid; v < nvec; v += T)
      reinterpret_cast<uint4 *>(s_state)[v] = ld_stream(slab + 8 * v);
    if (mine)
      reinterpret_cast<uint4 *>(s_x)[tid] = ld_stream(p.x + n * p.ld + c_base + 8 * tid);
    __syncthreads();

    if (mine) {
      uint32_t h[3][8], xs[8];
      const int W = (int)p.W;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int64_t base = (int64_t)(8 * tid + c) * L;
        // the window: the last W-1 state entries (the ring read from q: q+L-W+1 .. q+L-1)
        for (int k = 0; k < W - 1; ++k)
          h[k][c] = s_state[base + (q + L - (W - 1) + k) % L];
        xs[c] = s_x[8 * tid + c];
      }
      st_stream(outp, outputs8<ACT>(h, xs, wf, bf, has_bias, W));
    }

    for (int64_t v = tid; v < nvec; v += T) {
      const int64_t e0 = 8 * v;
      int64_t c = e0 / L;
      int64_t l = e0 - c * L;
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t val;
        if (ring) {  // ring: only the oldest entry q of each channel takes x
          val = (l == q) ? (uint32_t)s_x[c] : (uint32_t)s_state[e0 + i];
          if (++l == L) {
            l = 0;
            ++c;
          }
        } else if (l == L - 1) {
          val = s_x[c];
          l = 0;
          ++c;
        } else {
          val = s_state[e0 + i + 1];
          ++l;
        }
        if (i & 1) {
          w[i >> 1] |= val << 16;
        } else {
          w[i >> 1] = val;
        }
      }
      st_stream(slab + e0, make_uint4(w[0], w[1], w[2], w[3]));
    }
    __syncthreads();  // the next row reuses the buffers
  }
}

// Channel-last layout, any L: planes move down by one, four at a time so several loads are
// in flight before their stores.
template <int ACT>
__global__ void __launch_bounds__(256) k_update_staged_chlast(UpdateParams p) {
  grid_dependency_boundary();
  const int64_t groups = p.D >> 3;
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= groups) return;
  const int64_t c0 = g << 3;
  const int64_t L = p.L;
  const bool has_bias = p.bias != nullptr;
  float wf[8][kW], bf[8];
  load_weights8(p, c0, wf, bf);

  for (int64_t n = blockIdx.y; n < p.N; n += gridDim.y) {
    const RowSlot row = resolve_row(p, n);
    const int64_t s = row.s;
    uint16_t *outp = p.out + n * p.D + c0;
    if (s < 0) {
      st_stream(outp, make_uint4(0u, 0u, 0u, 0u));
      continue;
    }
    const uint4 xv = ld_stream(p.x + n * p.ld + c0);
    uint16_t *sp = p.state + s * (L * p.D) + c0;
    const int W = (int)p.W;
    uint32_t h[3][8], xs[8];
    unpack8(xv, xs);
    if (p.seqlens != nullptr) {
      // Ring in planes: read the W-1 window planes, write x over the oldest plane.
      const int64_t q = row.q;
      for (int k = 0; k < W - 1; ++k) unpack8(ld_stream(sp + ((q + L - (W - 1) + k) % L) * p.D), h[k]);
      st_stream(sp + q * p.D, xv);
      st_stream(outp, outputs8<ACT>(h, xs, wf, bf, has_bias, W));
      continue;
    }
    // Linear: plane l <- plane l+1, four planes in flight; the window planes L-W+1 .. L-1 are
    // kept as they pass (plane 0 is read only when L == W - 1: it is then in the window).
    if (L == W - 1) unpack8(ld_stream(sp), h[0]);
    for (int64_t l = 1; l < L; l += 4) {
      uint4 t[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (l + k < L) t[k] = ld_stream(sp + (l + k) * p.D);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (l + k < L) {
          st_stream(sp + (l + k - 1) * p.D, t[k]);
          const int64_t wi = (l + k) - (L - (W - 1));
          if (wi >= 0 && wi < W - 1) unpack8(t[k], h[wi]);
        }
      }
    }
    st_stream(sp + (L - 1) * p.D, xv);
    st_stream(outp, outputs8<ACT>(h, xs, wf, bf, has_bias, W));
  }
}

std::atomic<bool> g_smem_opt_in[kMaxDevices][2];

template <int ACT>
cudaError_t launch_compact(const UpdateParams &p, cudaStream_t stream) {
  // Tile width: the largest power-of-two thread count (<= 256) whose slab fits 64 KB, so
  // several CTAs share an SM; long states fall back to narrower tiles (and up to 227 KB).
  int T = 256;
  while (T > 32 && (size_t)16 * T * (p.L + 1) > 64 * 1024) T /= 2;
  const size_t smem = (size_t)16 * T * (p.L + 1);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  if (smem > 48 * 1024) {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!g_smem_opt_in[dev][ACT].load(std::memory_order_acquire)) {
      cudaError_t e = cudaFuncSetAttribute(k_update_staged_compact<ACT>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           227 * 1024);
      if (e != cudaSuccess) return e;
      g_smem_opt_in[dev][ACT].store(true, std::memory_order_release);
    }
  }
  const int64_t gx = (p.D + 8 * T - 1) / (8 * T);
  int64_t gy = (int64_t)device_sm_count() * 8 / gx;
  if (gy < 1) gy = 1;
  if (gy > p.N) gy = p.N;
  if (gy > 65535) gy = 65535;
  return launch_overlapped(k_update_staged_compact<ACT>, dim3((unsigned)gx, (unsigned)gy), dim3(T), smem,
                           stream, p);
}

template <int ACT>
cudaError_t launch_chlast(const UpdateParams &p, cudaStream_t stream) {
  const int64_t groups = p.D / 8;
  int T = 256;
  if (groups < T) T = (int)((groups + 31) / 32 * 32);
  const int64_t gx = (groups + T - 1) / T;
  int64_t gy = (int64_t)device_sm_count() * 8 / gx;
  if (gy < 1) gy = 1;
  if (gy > p.N) gy = p.N;
  if (gy > 65535) gy = 65535;
  return launch_overlapped(k_update_staged_chlast<ACT>, dim3((unsigned)gx, (unsigned)gy), dim3(T), 0,
                           stream, p);
}

}  // namespace

cudaError_t launch_staged(const UpdateParams &p, int act, cudaStream_t stream) {
  if (p.layout == (int)Layout::Compact)
    return act == 1 ? launch_compact<1>(p, stream) : launch_compact<0>(p, stream);
  return act == 1 ? launch_chlast<1>(p, stream) : launch_chlast<0>(p, stream);
}

}  // namespace ccu
