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
template <int ACT>
__device__ __forceinline__ float activate(float a) {
  if constexpr (ACT == 1) {
    return a / (1.0f + expf(-a));  // SiLU: a * sigmoid(a)
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

// ---------------------------------------------------------------------------------------
// Kernel launchers (one per family). Each returns the cudaError_t of its launch.

cudaError_t launch_scalar(const UpdateParams &p, int act, cudaStream_t stream);
cudaError_t launch_vector(const UpdateParams &p, int act, cudaStream_t stream);
cudaError_t launch_staged(const UpdateParams &p, int act, cudaStream_t stream);
cudaError_t launch_bulk(const UpdateParams &p, int act, cudaStream_t stream);
cudaError_t launch_check_indices(const int32_t *idx, int64_t N, int64_t S, uint32_t *bitmap,
                                 int32_t *status, cudaStream_t stream);

// Largest L the register-resident vector and bulk kernels are compiled for.
constexpr int64_t kVectorMaxL = 8;
// Largest L the shared-memory staged kernel accepts.
constexpr int64_t kStagedMaxL = 256;

}  // namespace ccu
