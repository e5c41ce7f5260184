// Internal declarations shared by the C-ABI host code and the kernels.
//
// The operation is the decode update of the cuDNN page "Causal Conv1d Decode Update"
// (introduction, update block); the argument contract is documented in ccu_conv1d.h.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ccu {

// Filter width served by the kernels ("Current native implementation": width four).
constexpr int kW = 4;

enum class Layout : int { Compact = 0, ChannelLast = 1 };

// Everything a kernel needs, by value (fits the kernel parameter space easily).
struct UpdateParams {
  const uint16_t *x;      // [N, ld] BF16 bits
  int64_t ld;
  uint16_t *state;        // logical [S, D, L] BF16 bits, compact or channel-last
  const uint16_t *w;      // [D, 4]
  const uint16_t *bias;   // [D] or nullptr
  const int32_t *idx;     // [N] or nullptr
  uint16_t *out;          // [N, D]
  int32_t *status;        // nullptr: unchecked; else device error word (range check on)
  int64_t N, D, S, L;
  int64_t ss, sd, sl;     // element strides of the state (used by the scalar kernel)
  int layout;             // Layout
  int rows_per_cta;       // rows each CTA walks (vector kernels)
};

// Launch description chosen on the host.
struct LaunchShape {
  dim3 grid;
  dim3 block;
  size_t smem;
};

// ---------------------------------------------------------------------------------------
// Device helpers. BF16 values travel as raw 16-bit patterns packed two per 32-bit word
// (the lower address in the low half, as memory is little-endian).

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_bits(uint32_t h) { return __uint_as_float(h << 16); }

// Round two floats to BF16 (nearest-even) and pack: lo -> low half, hi -> high half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint16_t round_bf16(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t *>(&b);
}

// The activation, a compile-time choice: identity kernels carry no SiLU code.
// SiLU is a * sigmoid(a). With e = exp(-|a|) in (0, 1], sigmoid(a) = 1 / (1 + e) for
// a >= 0 and e / (1 + e) for a < 0, so a * sigmoid(a) = (a >= 0 ? a : a * e) / (1 + e):
// no overflow for any finite a (a / (1 + exp(-a)) overflows to -0 below a ~ -88.7, where
// the true value is still a representable float). The exponential and the division use
// the hardware approximations (__expf, __fdividef with a denominator in [1, 2]): a few
// float ulps of error, far below the half BF16 ulp (2^15 float ulps) the result keeps, so
// the rounded output stays within one BF16 ulp of the exact value. The accurate library
// versions made this path issue-bound on the large batch.
template <int ACT>
__device__ __forceinline__ float activate(float a) {
  if constexpr (ACT == 1) {
    const float e = __expf(-fabsf(a));
    const float num = a >= 0.0f ? a : a * e;
    return __fdividef(num, 1.0f + e);
  } else {
    return a;
  }
}

// Streaming (evict-first) 16-byte global accesses for data touched once per call.
__device__ __forceinline__ uint4 ld_stream(const uint16_t *p) {
  return __ldcs(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ void st_stream(uint16_t *p, uint4 v) {
  __stcs(reinterpret_cast<uint4 *>(p), v);
}
// Read-only, cached: weights and bias are re-read by every row.
__device__ __forceinline__ uint4 ld_keep(const uint16_t *p) {
  return __ldg(reinterpret_cast<const uint4 *>(p));
}

// Slot of row n, or -1 for "no state access" (a padding row, or in checked mode a slot
// out of range, which also raises CCU_DEVERR_RANGE in *status).
__device__ __forceinline__ int64_t resolve_slot(const UpdateParams &p, int64_t n) {
  if (p.idx == nullptr) return n;
  int64_t s = __ldg(p.idx + n);
  if (p.status != nullptr && (s < -1 || s >= p.S)) {
    atomicOr(p.status, 1);  // CCU_DEVERR_RANGE
    return -1;
  }
  return s;
}

__device__ __forceinline__ uint32_t get16(const uint32_t *w, int pos) {
  return (w[pos >> 1] >> ((pos & 1) * 16)) & 0xffffu;
}

// The update of 8 consecutive channels whose compact state [8][L] sits in 4*L words `ow`
// (two BF16 per word, flat position c*L + l) and whose inputs sit in 4 words `xw`:
//   out[c]      = act(sum_j h_c[L-3+j] * w[c][j] + bias[c]),  h_c = (state[c][0..L-1], x[c])
//   new state   = state[c][1..L-1] followed by x[c]   (written to `nw`, same packing)
// `wv` holds weight[8][4] (16 words), `bv` bias[8] (4 words). Returns the packed outputs.
template <int L, int ACT>
__device__ __forceinline__ uint4 update8_compact(const uint32_t (&xw)[4], const uint32_t (&ow)[4 * L],
                                                 const uint32_t (&wv)[16], const uint32_t (&bv)[4],
                                                 bool has_bias, uint32_t (&nw)[4 * L]) {
  float y[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    float acc = 0.0f;
#pragma unroll
    for (int j = 0; j < kW; ++j) {
      const int hidx = L - (kW - 1) + j;  // index into the L + 1 history entries
      const uint32_t h = (hidx == L) ? get16(xw, c) : get16(ow, c * L + hidx);
      acc = __fmaf_rn(bf16_bits(h), bf16_bits(get16(wv, c * kW + j)), acc);
    }
    if (has_bias) acc = acc + bf16_bits(get16(bv, c));
    y[c] = activate<ACT>(acc);
  }
#pragma unroll
  for (int i = 0; i < 4 * L; ++i) {
    const int e0 = 2 * i, e1 = 2 * i + 1;  // flat positions c*L + l
    const uint32_t v0 = (e0 % L == L - 1) ? get16(xw, e0 / L) : get16(ow, e0 + 1);
    const uint32_t v1 = (e1 % L == L - 1) ? get16(xw, e1 / L) : get16(ow, e1 + 1);
    nw[i] = v0 | (v1 << 16);
  }
  return make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                    pack_bf16x2(y[6], y[7]));
}

// ---------------------------------------------------------------------------------------
// Kernel launchers (one per family). Each returns the cudaError_t of its launch.

cudaError_t launch_scalar(const UpdateParams &p, int act, cudaStream_t stream);
cudaError_t launch_vector(const UpdateParams &p, int act, cudaStream_t stream);
cudaError_t launch_staged(const UpdateParams &p, int act, cudaStream_t stream);
cudaError_t launch_bulk(const UpdateParams &p, int act, cudaStream_t stream);
// Sets the calling thread's message returned by ccu_conv1d_last_error.
void record_error(const char *msg);
// Reads and clears the device error word that kernels without a status word report into.
cudaError_t take_async_error(int32_t *bits);
cudaError_t launch_check_indices(const int32_t *idx, int64_t N, int64_t S, uint32_t *bitmap,
                                 int32_t *status, cudaStream_t stream);

// CCU_DEVERR_TIMEOUT: a bounded wait inside a kernel gave up.
constexpr int32_t kDevErrTimeout = 4;
// Largest L the register-resident vector and bulk kernels are compiled for.
constexpr int64_t kVectorMaxL = 8;
// Largest L the shared-memory staged kernel accepts.
constexpr int64_t kStagedMaxL = 256;

}  // namespace ccu
