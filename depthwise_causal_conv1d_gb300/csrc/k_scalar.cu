// Scalar kernels: the correctness anchor of the update (any D, any ld, any width W >= 1
// and L >= max(W - 1, 1), both state layouts through explicit strides) and the index
// checker.
//
// Update definition: cuDNN page "Causal Conv1d Decode Update", introduction (update
// block) and the conv_state_indices paragraph.
#include "ccu_internal.cuh"

namespace ccu {

int device_sm_count();

namespace {

// One thread per (row, channel), grid-stride. Each thread reads the W-1 newest state
// entries and x, computes the output, then shifts its own channel's state in place.
template <int ACT>
__global__ void __launch_bounds__(256) k_update_scalar(UpdateParams p) {
  grid_dependency_boundary();
  const int64_t total = p.N * p.D;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = i / p.D;
    const int64_t d = i - n * p.D;
    const RowSlot r = resolve_row(p, n);
    if (r.s < 0) {
      p.out[n * p.D + d] = 0;  // padding row: +0, no state access
      continue;
    }
    uint16_t *st = p.state + r.s * p.ss + d * p.sd;
    const int64_t L = p.L;
    const uint16_t xv = p.x[n * p.ld + d];
    // history = [st[0], ..., st[L-1], x] (linear), or the ring read from its oldest entry
    // q followed by x; the width-W window is the last W entries of the history.
    const int64_t q = p.seqlens != nullptr ? r.q : 0;
    const int64_t W = p.W;
    const uint16_t *w = p.w + d * W;
    float acc = 0.0f;
    for (int64_t k = 0; k < W - 1; ++k) {
      const uint16_t h = st[((q + L - (W - 1) + k) % L) * p.sl];
      acc = __fmaf_rn(bf16_bits(h), bf16_bits(w[k]), acc);
    }
    acc = __fmaf_rn(bf16_bits(xv), bf16_bits(w[W - 1]), acc);
    if (p.bias != nullptr) acc = acc + bf16_bits(p.bias[d]);
    p.out[n * p.D + d] = round_bf16(activate<ACT>(acc));
    if (p.seqlens != nullptr) {
      st[q * p.sl] = xv;  // ring: the new input replaces the oldest entry
    } else {
      // conv_state[s, d, :] = history[1:], ascending so each entry is read before overwritten
      for (int64_t l = 0; l + 1 < L; ++l) st[l * p.sl] = st[(l + 1) * p.sl];
      st[(L - 1) * p.sl] = xv;
    }
  }
}

// Marks each non-padding slot in a bitmap; a slot seen twice, or out of range, raises a
// bit in *status. No trap, no wait.
__global__ void __launch_bounds__(256) k_check_indices(const int32_t *idx, int64_t N, int64_t S,
                                                       uint32_t *bitmap, int32_t *status) {
  grid_dependency_boundary();
  for (int64_t n = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; n < N;
       n += (int64_t)gridDim.x * blockDim.x) {
    const int64_t s = idx[n];
    if (s == -1) continue;
    if (s < -1 || s >= S) {
      atomicOr(status, 1);  // CCU_DEVERR_RANGE
      continue;
    }
    const uint32_t bit = 1u << (s & 31);
    const uint32_t old = atomicOr(bitmap + (s >> 5), bit);
    if (old & bit) atomicOr(status, 2);  // CCU_DEVERR_DUPLICATE
  }
}

// Zeroes n 32-bit words (the duplicate check's slot scratch). A kernel rather than a
// memset so that it joins the programmatic overlap of consecutive launches: it waits, at its
// boundary, for the previous kernel on the stream (which may still read the scratch), and
// the update launched after it waits for it in the same way.
__global__ void __launch_bounds__(256) k_clear_words(int32_t *w, int64_t n) {
  grid_dependency_boundary();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    w[i] = 0;
}

int64_t grid_for(int64_t work, int threads) {
  const int64_t blocks = (work + threads - 1) / threads;
  const int64_t cap = (int64_t)device_sm_count() * 16;
  return blocks < cap ? (blocks > 0 ? blocks : 1) : cap;
}

}  // namespace

cudaError_t launch_scalar(const UpdateParams &p, int act, cudaStream_t stream) {
  const int threads = 256;
  const dim3 grid((unsigned)grid_for(p.N * p.D, threads));
  return act == 1 ? launch_overlapped(k_update_scalar<1>, grid, dim3(threads), 0, stream, p)
                  : launch_overlapped(k_update_scalar<0>, grid, dim3(threads), 0, stream, p);
}

cudaError_t launch_clear_words(int32_t *w, int64_t n, cudaStream_t stream) {
  const int threads = 256;
  const dim3 grid((unsigned)grid_for(n, threads));
  return launch_overlapped(k_clear_words, grid, dim3(threads), 0, stream, w, n);
}

cudaError_t launch_check_indices(const int32_t *idx, int64_t N, int64_t S, uint32_t *bitmap,
                                 int32_t *status, cudaStream_t stream) {
  const int threads = 256;
  const dim3 grid((unsigned)grid_for(N, threads));
  return launch_overlapped(k_check_indices, grid, dim3(threads), 0, stream, idx, N, S, bitmap, status);
}

}  // namespace ccu
