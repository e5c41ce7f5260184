// Bulk-copy kernel for the channel-last state layout (L*D, 1, D), L = 3..8, D % 8 == 0.
//
// In this layout every plane l of a slot is contiguous over channels, so a warp's slice
// (row n, 512 consecutive channels) of each plane is one contiguous 1 KB run. Per slice,
// lane 0 brings x and the planes the update reads into one stage of the warp's two-stage
// ring with cp.async.bulk (completing on the stage's mbarrier), the lanes compute the
// outputs from shared memory, and lane 0 writes back with bulk stores:
//   linear state: plane l <- old plane l+1 for l < L-1 and plane L-1 <- x, stored
//     straight from the staged planes (the shift costs no arithmetic); plane 0 is read
//     only when L == 3, where it is inside the width-4 window;
//   ring-buffer state (cache_seqlens): only the three window planes (q+L-3 .. q+L-1 mod
//     L) are read and only plane q (the oldest) is written, with x.
// Like the compact bulk kernel, every warp is an independent pipeline and every mbarrier
// wait is bounded (CCU_DEVERR_TIMEOUT on expiry, then a bounded wait for the warp's own
// copies before it returns).
//
// Update definition: cuDNN page "Causal Conv1d Decode Update", introduction (update
// block); the channel-last layout is the one its "Semantic tensor contract" accepts from a
// full-sequence prefill.
#include <atomic>

#include "ccu_bulk.cuh"

namespace ccu {

int device_sm_count();
int current_device();

namespace {

using namespace bulk;

__device__ int32_t g_planes_error = 0;  // CCU_DEVERR_* bits raised with no status word
__device__ int32_t g_planes_error_taken = 0;  // the value the last exchange read

// Reads and clears the error word in one atomic step (a kernel that raises a bit
// meanwhile leaves it for the next exchange).
__global__ void k_exchange_planes_error() {
  grid_dependency_boundary();
  g_planes_error_taken = atomicExch(&g_planes_error, 0);
}

constexpr int kG = 2;                 // 8-channel groups per lane: slices of 512 channels
constexpr int64_t kSlice = 256 * kG;  // channels per slice
constexpr int64_t kPlane = 2 * kSlice;  // bytes of one plane's slice

// Stage layout (kPlane-byte buffers): [x][plane buffers ...][out].
template <int L, bool RING>
__host__ __device__ constexpr int plane_buffers() {
  return RING ? kW - 1 : (L == kW - 1 ? L : L - 1);
}

// Refill schedule as in the compact bulk kernel: ahead == 0 refills the stage of slice k - 1
// after slice k is stored (P slices loaded before the loop); 1 <= ahead <= stages - 1 issues
// slice k + ahead at the top of iteration k, before the wait on slice k.
template <int L, int ACT, bool RING>
__global__ void __launch_bounds__(kThreads) k_update_bulk_planes(UpdateParams p, int stages, int ahead,
                                                                 int64_t stage_bytes) {
  grid_dependency_boundary();
  constexpr int NB = plane_buffers<L, RING>();
  // First plane held in buffer 0 for the linear state (0 when L == 3, else 1).
  constexpr int first = (L == kW - 1) ? 0 : 1;
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = stages, A = ahead;
  unsigned char *wbase = smem + (int64_t)warp * (kBarrierBytes + P * stage_bytes);
  uint64_t *bars = reinterpret_cast<uint64_t *>(wbase);
  unsigned char *bufs = wbase + kBarrierBytes;

  const int64_t slices = (p.D + kSlice - 1) / kSlice;
  const int64_t items = p.N * slices;
  const int64_t first_item = (int64_t)blockIdx.x * kWarps + warp;
  const int64_t stride = (int64_t)gridDim.x * kWarps;
  const int64_t mine = items > first_item ? (items - first_item + stride - 1) / stride : 0;
  const int64_t plane_stride = p.D;  // elements between planes of a slot

  if (lane == 0) {
    for (int k = 0; k < P; ++k) mbar_init(&bars[k], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // Plane held in buffer b for a slice whose ring position is q.
  auto plane_of = [&](int b, int q) -> int64_t {
    if constexpr (RING) {
      return (q + L - (kW - 1) + b) % L;
    } else {
      return first + b;
    }
  };

  auto issue = [&](int64_t k) {
    const Slice sl = slice_of<kG, L, false>(p, first_item + k * stride, slices, true);
    uint64_t *bar = &bars[k % P];
    unsigned char *buf = bufs + (k % P) * stage_bytes;
    if (sl.s < 0) {
      mbar_arrive(bar);
      return;
    }
    const uint32_t bytes = (uint32_t)(sl.cn * 2);
    mbar_arrive_expect_tx(bar, bytes * (1 + NB));
    bulk_load(buf, p.x + sl.n * p.ld + sl.c_base, bytes, bar);
    const uint16_t *slot = p.state + sl.s * (L * p.D) + sl.c_base;
#pragma unroll
    for (int b = 0; b < NB; ++b)
      bulk_load(buf + (1 + b) * kPlane, slot + plane_of(b, sl.q) * plane_stride, bytes, bar);
    claim_after_issue(p, sl);
  };

  const int64_t pre = A > 0 ? A : P;
  const int64_t prologue = mine < pre ? mine : pre;
  if (lane == 0)
    for (int64_t k = 0; k < prologue; ++k) issue(k);

  const bool has_bias = p.bias != nullptr;
  uint32_t wv[kG][16], bv[kG][4];
  int64_t w_base = -1;
  bool failed = false;
  int64_t k = 0;

  for (; k < mine; ++k) {
    const int st = (int)(k % P);
    const uint32_t parity = (uint32_t)((k / P) & 1);
    if (A > 0 && lane == 0 && k + A < mine) {
      // Stage (k + A) % P last held slice k + A - P, stored P - A - 1 groups before the newest.
      bulk_wait_read_n(P - A - 1);
      issue(k + A);
    }
    const Slice sl = slice_of<kG, L>(p, first_item + k * stride, slices, false);
    unsigned char *buf = bufs + st * stage_bytes;

    if (sl.c_base != w_base) {
#pragma unroll
      for (int g = 0; g < kG; ++g) {
        const int64_t c = sl.c_base + 8 * (lane + 32 * g);
        if (8 * (lane + 32 * g) < sl.cn) {
          const uint16_t *wp = p.w + c * kW;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 t = ld_keep(wp + 8 * q);
            wv[g][4 * q] = t.x; wv[g][4 * q + 1] = t.y; wv[g][4 * q + 2] = t.z; wv[g][4 * q + 3] = t.w;
          }
          if (has_bias) {
            const uint4 t = ld_keep(p.bias + c);
            bv[g][0] = t.x; bv[g][1] = t.y; bv[g][2] = t.z; bv[g][3] = t.w;
          } else {
            bv[g][0] = bv[g][1] = bv[g][2] = bv[g][3] = 0u;
          }
        }
      }
      w_base = sl.c_base;
    }

    const bool ok = mbar_wait(&bars[st], parity);
    if (!__all_sync(kFull, ok)) {
      failed = true;
      break;
    }

    unsigned char *out_buf = buf + (1 + NB) * kPlane;
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      const int q8 = lane + 32 * g;
      if (8 * q8 >= sl.cn) continue;
      if (sl.s < 0) {
        st_stream(p.out + sl.n * p.D + sl.c_base + 8 * q8, make_uint4(0u, 0u, 0u, 0u));
        continue;
      }
      // Window buffers: the ring's three window planes, or the linear state's last three.
      constexpr int wb0 = RING ? 0 : NB - (kW - 1);
      uint32_t h[3][8], xs[8];
#pragma unroll
      for (int j = 0; j < kW - 1; ++j)
        unpack8(reinterpret_cast<const uint4 *>(buf + (1 + wb0 + j) * kPlane)[q8], h[j]);
      unpack8(reinterpret_cast<const uint4 *>(buf)[q8], xs);
      reinterpret_cast<uint4 *>(out_buf)[q8] = outputs8_window<kW, ACT>(h, xs, wv[g], bv[g], has_bias);
    }
    fence_proxy_async();
    __syncwarp();

    if (lane == 0) {
      if (sl.s >= 0) {
        const uint32_t bytes = (uint32_t)(sl.cn * 2);
        uint16_t *slot = p.state + sl.s * (L * p.D) + sl.c_base;
        bulk_store(p.out + sl.n * p.D + sl.c_base, out_buf, bytes);
        if constexpr (RING) {
          bulk_store(slot + (int64_t)sl.q * plane_stride, buf, bytes);  // x over the oldest plane
        } else {
          // plane l <- old plane l+1 (held in buffer l+1-first), plane L-1 <- x
#pragma unroll
          for (int l = 0; l + 1 < L; ++l)
            bulk_store(slot + (int64_t)l * plane_stride, buf + (1 + (l + 1 - first)) * kPlane, bytes);
          bulk_store(slot + (int64_t)(L - 1) * plane_stride, buf, bytes);
        }
      }
      bulk_commit();
      if (A == 0 && k >= 1 && k - 1 + P < mine) {
        bulk_wait_read<1>();
        issue(k - 1 + P);
      }
    }
    __syncwarp();
  }

  if (failed && lane == 0) {
    atomicOr(p.status != nullptr ? p.status : &g_planes_error, kDevErrTimeout);
    // slices k .. issued - 1 were issued and not consumed
    const int64_t last = A > 0 ? k + A + 1 : (k > 0 ? k - 1 : 0) + P;
    const int64_t issued = last < mine ? last : mine;
    for (int64_t q = k; q < issued; ++q) mbar_wait(&bars[q % P], (uint32_t)((q / P) & 1));
  }
  if (lane == 0) bulk_wait_all();
}

constexpr int kMaxDevices = 64;
std::atomic<bool> g_opted_in[kMaxDevices][kVectorMaxL + 1][2][2];

template <int L, int ACT, bool RING>
cudaError_t launch_LAR(const UpdateParams &p, cudaStream_t stream) {
  constexpr int NB = plane_buffers<L, RING>();
  const int64_t sb = (2 + NB) * kPlane;  // x, the plane buffers, out
  // Refill after compute for the linear state (large batch: 163.0 against 167.7 us issuing
  // ahead); the ring state measured the same either way (143.2 / 142.9 us).
  const int P = 2, A = RING ? 1 : 0;
  const size_t smem = (size_t)kWarps * (kBarrierBytes + (size_t)P * sb);
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!g_opted_in[dev][L][ACT][RING].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(k_update_bulk_planes<L, ACT, RING>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    g_opted_in[dev][L][ACT][RING].store(true, std::memory_order_release);
  }
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm, k_update_bulk_planes<L, ACT, RING>, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int64_t slices = (p.D + kSlice - 1) / kSlice;
  const int64_t items = p.N * slices;
  int64_t warps = (int64_t)device_sm_count() * per_sm * kWarps;
  if (warps >= slices) warps = warps / slices * slices;
  if (warps > items) warps = items;
  int64_t grid = (warps + kWarps - 1) / kWarps;
  if (grid < 1) grid = 1;
  return launch_overlapped(k_update_bulk_planes<L, ACT, RING>, dim3((unsigned)grid), dim3(kThreads), smem,
                           stream, p, P, A, sb);
}

template <int L, int ACT>
cudaError_t launch_LA(const UpdateParams &p, cudaStream_t stream) {
  return p.seqlens != nullptr ? launch_LAR<L, ACT, true>(p, stream) : launch_LAR<L, ACT, false>(p, stream);
}

template <int ACT>
cudaError_t launch_A(const UpdateParams &p, cudaStream_t stream) {
  switch (p.L) {
    case 3: return launch_LA<3, ACT>(p, stream);
    case 4: return launch_LA<4, ACT>(p, stream);
    case 5: return launch_LA<5, ACT>(p, stream);
    case 6: return launch_LA<6, ACT>(p, stream);
    case 7: return launch_LA<7, ACT>(p, stream);
    case 8: return launch_LA<8, ACT>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t take_planes_error(int32_t *bits) {
  // read and clear in one atomic step on the device (the legacy default stream orders
  // the copy after the exchange)
  cudaError_t e = launch_overlapped(k_exchange_planes_error, dim3(1), dim3(1), 0, (cudaStream_t)0);
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(bits, g_planes_error_taken, sizeof(int32_t));
  return e;
}

cudaError_t launch_bulk_planes(const UpdateParams &p, int act, cudaStream_t stream) {
  if (p.layout != (int)Layout::ChannelLast || p.W != kW) return cudaErrorInvalidValue;
  return act == 1 ? launch_A<1>(p, stream) : launch_A<0>(p, stream);
}

}  // namespace ccu
