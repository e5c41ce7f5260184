// Bulk-copy kernel for large batches (compact state layout, D % 8 == 0, linear or
// ring-buffer state; width 4 with L = 3..8, widths 2 and 3 with L = W-1..4; the channel-last
// layout has its own bulk kernel in k_bulk_planes.cu, width 4).
//
// Every warp is an independent pipeline. Its work items are slices (row n, 256*G
// consecutive channels); lane 0 moves whole slices between global and shared memory with
// the bulk-copy engine (cp.async.bulk): the x slice (512*G bytes) and the slot's state
// slab (512*G*L bytes, contiguous in the compact layout) land in one stage of the warp's
// own ring of P stages and complete on that stage's mbarrier. The 32 lanes then update 8
// channels per group in shared memory (the new state in place over the old, the output
// over x), and lane 0 writes the output slice and the state slab back with bulk stores.
// Loads run P-1 slices ahead. No barrier spans more than one warp, so warps drift freely
// and one warp's arithmetic overlaps other warps' copies.
//
// Every mbarrier wait has an iteration limit: on expiry the warp records
// CCU_DEVERR_TIMEOUT, waits (again bounded) for its own copies in flight and returns.
//
// Update definition: cuDNN page "Causal Conv1d Decode Update", introduction (update
// block) and the conv_state_indices paragraph; compact state layout from its "Semantic
// tensor contract".
#include <atomic>
#include <mutex>

#include "ccu_bulk.cuh"

namespace ccu {

int device_sm_count();
int current_device();

__device__ int32_t g_async_error = 0;  // CCU_DEVERR_* bits raised by a kernel with no status word
__device__ int32_t g_async_error_taken = 0;  // the value the last exchange read

// Reads and clears the error word in one atomic step (a kernel that raises a bit
// meanwhile leaves it for the next exchange).
__global__ void k_exchange_async_error() {
  grid_dependency_boundary();
  g_async_error_taken = atomicExch(&g_async_error, 0);
}

namespace {

using namespace bulk;

// Shared memory per warp: kBarrierBytes of mbarriers, then P stages of stage_bytes.
// RING: conv_state is a ring buffer indexed by cache_seqlens (entry q replaced by x).
// Two refill schedules, chosen by `ahead`:
//   ahead == 0: the stage of slice k - 1 is refilled (with slice k - 1 + P) after slice k has
//     been computed and stored; P slices are loaded before the loop.
//   1 <= ahead <= P - 1: slice k + ahead is issued at the top of iteration k, before the wait
//     on slice k, so a load is in flight while the warp waits and while it computes; ahead
//     slices are loaded before the loop.
template <int L, int W, int ACT, int G, bool RING>
__global__ void __launch_bounds__(kThreads) k_update_bulk(UpdateParams p, int stages, int ahead,
                                                          int64_t stage_bytes) {
  grid_dependency_boundary();
  constexpr int64_t kSlice = 256 * G;
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = stages, A = ahead;
  unsigned char *wbase = smem + (int64_t)warp * (kBarrierBytes + P * stage_bytes);
  uint64_t *bars = reinterpret_cast<uint64_t *>(wbase);
  unsigned char *bufs = wbase + kBarrierBytes;

  const int64_t slices = (p.D + kSlice - 1) / kSlice;
  const int64_t items = p.N * slices;
  const int64_t first = (int64_t)blockIdx.x * kWarps + warp;
  const int64_t stride = (int64_t)gridDim.x * kWarps;
  const int64_t mine = items > first ? (items - first + stride - 1) / stride : 0;

  if (lane == 0) {
    for (int k = 0; k < P; ++k) mbar_init(&bars[k], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // Lane 0: put this warp's k-th slice into stage k % P.
  auto issue = [&](int64_t k) {
    const Slice sl = slice_of<G, L, false>(p, first + k * stride, slices, true);
    uint64_t *bar = &bars[k % P];
    unsigned char *buf = bufs + (k % P) * stage_bytes;
    if (sl.s < 0) {
      mbar_arrive(bar);  // padding row: nothing to load
    } else {
      const uint32_t bx = (uint32_t)(sl.cn * 2), bs = (uint32_t)(sl.cn * L * 2);
      mbar_arrive_expect_tx(bar, bx + bs);
      bulk_load(buf, p.x + sl.n * p.ld + sl.c_base, bx, bar);
      bulk_load(buf + 2 * kSlice, p.state + sl.s * (p.D * L) + sl.c_base * L, bs, bar);
      claim_after_issue(p, sl);
    }
  };

  const int64_t pre = A > 0 ? A : P;
  const int64_t prologue = mine < pre ? mine : pre;
  if (lane == 0)
    for (int64_t k = 0; k < prologue; ++k) issue(k);

  const bool has_bias = p.bias != nullptr;
  uint32_t wv[G][16], bv[G][4];
  int64_t w_base = -1;
  bool failed = false;
  int64_t k = 0;

  for (; k < mine; ++k) {
    const int st = (int)(k % P);
    const uint32_t parity = (uint32_t)((k / P) & 1);
    if (A > 0 && lane == 0 && k + A < mine) {
      // Stage (k + A) % P last held slice k + A - P, whose stores were committed in iteration
      // k + A - P: P - A - 1 groups before the newest. Wait until they have read it.
      bulk_wait_read_n(P - A - 1);
      issue(k + A);
    }
    const Slice sl = slice_of<G, L>(p, first + k * stride, slices, false);
    unsigned char *buf = bufs + st * stage_bytes;

    if (sl.c_base != w_base) {  // weights of this slice, kept while it repeats
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const int64_t c = sl.c_base + 8 * (lane + 32 * g);
        if (8 * (lane + 32 * g) < sl.cn) {
          load_weights_packed<W>(p.w, c, wv[g]);
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

    // Every lane waits (bounded); the verdict is made warp-uniform.
    const bool ok = mbar_wait(&bars[st], parity);
    if (!__all_sync(kFull, ok)) {
      failed = true;
      break;
    }

#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int q8 = lane + 32 * g;  // 8-channel group within the slice
      if (8 * q8 >= sl.cn) continue;
      if (sl.s < 0) {
        st_stream(p.out + sl.n * p.D + sl.c_base + 8 * q8, make_uint4(0u, 0u, 0u, 0u));
        continue;
      }
      uint4 *sx = reinterpret_cast<uint4 *>(buf) + q8;
      uint4 *ss = reinterpret_cast<uint4 *>(buf + 2 * kSlice) + q8 * L;
      const uint4 xv = *sx;
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
      uint32_t ow[4 * L], nw[4 * L];
#pragma unroll
      for (int q = 0; q < L; ++q) {
        const uint4 t = ss[q];
        ow[4 * q] = t.x; ow[4 * q + 1] = t.y; ow[4 * q + 2] = t.z; ow[4 * q + 3] = t.w;
      }
      uint4 outv;
      if constexpr (RING) {
        outv = update8_compact_ring<L, W, ACT>(xw, ow, wv[g], bv[g], has_bias, sl.q, nw);
      } else {
        outv = update8_compact<L, W, ACT>(xw, ow, wv[g], bv[g], has_bias, nw);
      }
#pragma unroll
      for (int q = 0; q < L; ++q) ss[q] = make_uint4(nw[4 * q], nw[4 * q + 1], nw[4 * q + 2], nw[4 * q + 3]);
      *sx = outv;
    }
    fence_proxy_async();
    __syncwarp();

    if (lane == 0) {
      if (sl.s >= 0) {
        bulk_store(p.out + sl.n * p.D + sl.c_base, buf, (uint32_t)(sl.cn * 2));
        bulk_store(p.state + sl.s * (p.D * L) + sl.c_base * L, buf + 2 * kSlice,
                   (uint32_t)(sl.cn * L * 2));
      }
      bulk_commit();  // one group per iteration, empty for a padding slice
      // Refill the previous stage once its stores have read their shared memory.
      if (A == 0 && k >= 1 && k - 1 + P < mine) {
        bulk_wait_read<1>();
        issue(k - 1 + P);
      }
    }
    __syncwarp();
  }

  if (failed && lane == 0) {
    // Record the error, then let this warp's own loads land before shared memory goes away:
    // slices k .. issued - 1 were issued and not consumed (ahead == 0: the P slices of the
    // prologue and one refill per iteration from k = 1 on, so up to slice max(k, 1) + P - 2).
    atomicOr(p.status != nullptr ? p.status : &g_async_error, kDevErrTimeout);
    const int64_t last = A > 0 ? k + A + 1 : (k > 0 ? k - 1 : 0) + P;
    const int64_t issued = last < mine ? last : mine;
    for (int64_t q = k; q < issued; ++q) mbar_wait(&bars[q % P], (uint32_t)((q / P) & 1));
  }
  if (lane == 0) bulk_wait_all();  // stores complete before the warp retires
}

constexpr int kMaxDevices = 64;
std::atomic<bool> g_opted_in[kMaxDevices][kVectorMaxL + 1][kW + 1][2][2];

constexpr int kGroups = 2;  // 8-channel groups per lane: slices of 512 channels

int64_t stage_bytes_for(int64_t L) {
  const int64_t b = (int64_t)256 * kGroups * 2 * (L + 1);
  return (b + 127) / 128 * 128;
}

// Stage bytes a warp may hold (see launch_LAR).
constexpr int64_t kWarpStageBudget = 8 * 1024;

template <int L, int W, int ACT, bool RING>
cudaError_t launch_LAR(const UpdateParams &p, cudaStream_t stream) {
  const int64_t sb = stage_bytes_for(L);
  // About 8 KB of stages per warp (two 4 KB stages at L = 3), 66 KB a CTA; the registers
  // (99 a thread at L = 3) keep 2 CTAs of 8 warps resident per SM. Measured on the large
  // batch: slices of 512 channels with two stages beat 256-channel slices with four (larger
  // bulk copies); one CTA per SM was slower.
  int P = (int)(kWarpStageBudget / sb);
  P = P < 2 ? 2 : (P > kMaxStages ? kMaxStages : P);
  // Refill schedule, measured at N=4096, D=16384 (us, refilled after compute / issued one
  // ahead): linear L = 3 160.2 / 168.8 (and 169.7 with two ahead at three stages), L = 4
  // 199.6 / 213.7, L = 5 247.3 / 248.1, L = 6 289.2 / 288.2, L = 7 309.3 / 325.8, L = 8
  // 656.7 / 570.4; the ring state at L = 3 166.9 / 161.5. At L = 8 a lane's state is 128
  // bytes, so the lanes of a quarter-warp read and write the same shared-memory banks.
  const int A = (RING || L == 8) ? 1 : 0;
  const size_t smem = (size_t)kWarps * (kBarrierBytes + (size_t)P * sb);
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!g_opted_in[dev][L][W][ACT][RING].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(k_update_bulk<L, W, ACT, kGroups, RING>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    g_opted_in[dev][L][W][ACT][RING].store(true, std::memory_order_release);
  }
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm, k_update_bulk<L, W, ACT, kGroups, RING>, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int64_t slices = (p.D + 256 * kGroups - 1) / (256 * kGroups);
  const int64_t items = p.N * slices;
  int64_t warps = (int64_t)device_sm_count() * per_sm * kWarps;
  // A warp count that is a multiple of the slice count keeps every warp on one slice, so
  // its weights stay in registers.
  if (warps >= slices) warps = warps / slices * slices;
  if (warps > items) warps = items;
  int64_t grid = (warps + kWarps - 1) / kWarps;
  if (grid < 1) grid = 1;
  return launch_overlapped(k_update_bulk<L, W, ACT, kGroups, RING>, dim3((unsigned)grid), dim3(kThreads),
                           smem, stream, p, P, A, sb);
}

template <int L, int W, int ACT>
cudaError_t launch_LWA(const UpdateParams &p, cudaStream_t stream) {
  return p.seqlens != nullptr ? launch_LAR<L, W, ACT, true>(p, stream)
                              : launch_LAR<L, W, ACT, false>(p, stream);
}

template <int ACT>
cudaError_t launch_A(const UpdateParams &p, cudaStream_t stream) {
  switch (p.W * 16 + p.L) {
    case 4 * 16 + 3: return launch_LWA<3, 4, ACT>(p, stream);
    case 4 * 16 + 4: return launch_LWA<4, 4, ACT>(p, stream);
    case 4 * 16 + 5: return launch_LWA<5, 4, ACT>(p, stream);
    case 4 * 16 + 6: return launch_LWA<6, 4, ACT>(p, stream);
    case 4 * 16 + 7: return launch_LWA<7, 4, ACT>(p, stream);
    case 4 * 16 + 8: return launch_LWA<8, 4, ACT>(p, stream);
    case 3 * 16 + 2: return launch_LWA<2, 3, ACT>(p, stream);
    case 3 * 16 + 3: return launch_LWA<3, 3, ACT>(p, stream);
    case 3 * 16 + 4: return launch_LWA<4, 3, ACT>(p, stream);
    case 2 * 16 + 1: return launch_LWA<1, 2, ACT>(p, stream);
    case 2 * 16 + 2: return launch_LWA<2, 2, ACT>(p, stream);
    case 2 * 16 + 3: return launch_LWA<3, 2, ACT>(p, stream);
    case 2 * 16 + 4: return launch_LWA<4, 2, ACT>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t take_async_error(int32_t *bits) {
  // One caller at a time, after every kernel issued so far has finished. Each word is read
  // and cleared by one atomic exchange on the device, so a bit raised by a kernel that runs
  // meanwhile (on a stream that does not synchronize with the legacy default stream) is
  // kept for the next call rather than lost between a read and a clear.
  static std::mutex serial;
  std::lock_guard<std::mutex> lock(serial);
  int32_t mine = 0, planes = 0, prefill = 0, multi = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) {
    e = launch_overlapped(k_exchange_async_error, dim3(1), dim3(1), 0, (cudaStream_t)0);
  }
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&mine, g_async_error_taken, sizeof(int32_t));
  if (e == cudaSuccess) e = take_planes_error(&planes);
  if (e == cudaSuccess) e = take_prefill_error(&prefill);
  if (e == cudaSuccess) e = take_multi_bulk_error(&multi);
  if (e == cudaSuccess) *bits = mine | planes | prefill | multi;
  return e;
}

cudaError_t launch_bulk(const UpdateParams &p, int act, cudaStream_t stream) {
  if (p.layout == (int)Layout::ChannelLast) return launch_bulk_planes(p, act, stream);
  return act == 1 ? launch_A<1>(p, stream) : launch_A<0>(p, stream);
}

}  // namespace ccu
