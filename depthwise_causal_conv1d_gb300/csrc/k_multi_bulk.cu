// Bulk-copy kernel for the multi-token update: x[N, T, D] and out in device memory with
// channel-contiguous token rows, the compact state layout (linear or ring), width 4,
// L = 3..8, T = 1..kMultiBulkMaxT, no intermediate states.
//
// The decode bulk kernel (k_bulk.cu) with T tokens per slice: every warp is an independent
// pipeline over slices (row n, 256 consecutive channels). Lane 0 brings the slice's T token
// rows of x (512 bytes each) and the slot's state slab (512 * L bytes, contiguous in the
// compact layout) into one stage of the warp's ring with cp.async.bulk, completing on the
// stage's mbarrier. Each lane then steps its 8 channels' state through the T tokens in
// registers, writing token t's outputs over token t's x row and the final state over the
// slab, and lane 0 writes the T output rows and the slab back with bulk stores. The bytes a
// warp keeps in flight (a whole stage per slice, several slices deep) cost no registers, which
// is what bounds the vector kernel's rate here.
//
// Every mbarrier wait has an iteration limit: on expiry the warp records
// CCU_DEVERR_TIMEOUT, waits (again bounded) for its own copies in flight and returns.
//
// The multi-token reading: the T tokens are appended to the history in order; output t is
// the update of the cuDNN page "Causal Conv1d Decode Update" (introduction, update block)
// applied after t earlier tokens; the new state is the last L history entries ("Semantic
// tensor contract": a future form may admit x[N, D, Tstep]).
#include <atomic>

#include "ccu_bulk.cuh"

namespace ccu {

int device_sm_count();
int current_device();

__device__ int32_t g_multi_bulk_error = 0;  // CCU_DEVERR_* bits raised with no status word
__device__ int32_t g_multi_bulk_error_taken = 0;  // the value the last exchange read

// Reads and clears the error word in one atomic step (a kernel that raises a bit
// meanwhile leaves it for the next exchange).
__global__ void k_exchange_multi_bulk_error() {
  grid_dependency_boundary();
  g_multi_bulk_error_taken = atomicExch(&g_multi_bulk_error, 0);
}

namespace {

using namespace bulk;

constexpr int64_t kMRow = 512;  // bytes of one token row of a 256-channel slice

// P stages per warp of stage_bytes each: T token rows at t * 512, then the state slab.
template <int L, int W, int ACT, bool RING>
__global__ void __launch_bounds__(kThreads) k_multi_bulk(UpdateParams p, MultiParams m, int stages,
                                                         int64_t stage_bytes) {
  grid_dependency_boundary();
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = stages;
  const int T = (int)m.T;
  unsigned char *wbase = smem + (int64_t)warp * (kBarrierBytes + P * stage_bytes);
  uint64_t *bars = reinterpret_cast<uint64_t *>(wbase);
  unsigned char *bufs = wbase + kBarrierBytes;

  const int64_t slices = (p.D + 255) / 256;
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
    const Slice sl = slice_of<1, L, false>(p, first + k * stride, slices, true);
    uint64_t *bar = &bars[k % P];
    unsigned char *buf = bufs + (k % P) * stage_bytes;
    if (sl.s < 0) {
      mbar_arrive(bar);  // padding row: nothing to load
    } else {
      const uint32_t bx = (uint32_t)(sl.cn * 2), bs = (uint32_t)(sl.cn * L * 2);
      mbar_arrive_expect_tx(bar, bx * (uint32_t)T + bs);
      const uint16_t *xr = p.x + sl.n * m.sxn + sl.c_base;
      for (int t = 0; t < T; ++t) bulk_load(buf + t * kMRow, xr + t * m.sxt, bx, bar);
      bulk_load(buf + T * kMRow, p.state + sl.s * (p.D * L) + sl.c_base * L, bs, bar);
    }
  };

  const int64_t prologue = mine < P ? mine : P;
  if (lane == 0)
    for (int64_t k = 0; k < prologue; ++k) issue(k);

  const bool has_bias = p.bias != nullptr;
  uint32_t wv[16], bv[4];
  int64_t w_base = -1;
  bool failed = false;
  int64_t k = 0;

  for (; k < mine; ++k) {
    const int st = (int)(k % P);
    const uint32_t parity = (uint32_t)((k / P) & 1);
    const Slice sl = slice_of<1, L, false>(p, first + k * stride, slices, false);
    unsigned char *buf = bufs + st * stage_bytes;
    const bool active = 8 * lane < sl.cn;
    const int64_t c = sl.c_base + 8 * lane;

    if (sl.c_base != w_base) {  // weights of this slice, kept while it repeats
      if (active) {
        load_weights_packed<W>(p.w, c, wv);
        if (has_bias) {
          const uint4 t = ld_keep(p.bias + c);
          bv[0] = t.x; bv[1] = t.y; bv[2] = t.z; bv[3] = t.w;
        } else {
          bv[0] = bv[1] = bv[2] = bv[3] = 0u;
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

    if (active) {
      if (sl.s < 0) {
        for (int t = 0; t < T; ++t)
          st_stream(p.out + sl.n * m.son + t * m.sot + c, make_uint4(0u, 0u, 0u, 0u));
      } else {
        uint4 *ss = reinterpret_cast<uint4 *>(buf + T * kMRow) + lane * L;
        uint32_t ow[4 * L];
#pragma unroll
        for (int q = 0; q < L; ++q) {
          const uint4 t = ss[q];
          ow[4 * q] = t.x; ow[4 * q + 1] = t.y; ow[4 * q + 2] = t.z; ow[4 * q + 3] = t.w;
        }
        for (int t = 0; t < T; ++t) {
          uint4 *sx = reinterpret_cast<uint4 *>(buf + t * kMRow) + lane;
          const uint4 xv = *sx;
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
          uint32_t nw[4 * L];
          if constexpr (RING) {
            *sx = update8_compact_ring<L, W, ACT, true>(xw, ow, wv, bv, has_bias, (sl.q + t) % L, nw);
          } else {
            *sx = update8_compact<L, W, ACT, true>(xw, ow, wv, bv, has_bias, nw);
          }
#pragma unroll
          for (int i = 0; i < 4 * L; ++i) ow[i] = nw[i];
        }
#pragma unroll
        for (int q = 0; q < L; ++q) ss[q] = make_uint4(ow[4 * q], ow[4 * q + 1], ow[4 * q + 2], ow[4 * q + 3]);
      }
    }
    fence_proxy_async();
    __syncwarp();

    if (lane == 0) {
      if (sl.s >= 0) {
        const uint32_t bx = (uint32_t)(sl.cn * 2);
        uint16_t *orow = p.out + sl.n * m.son + sl.c_base;
        for (int t = 0; t < T; ++t) bulk_store(orow + t * m.sot, buf + t * kMRow, bx);
        bulk_store(p.state + sl.s * (p.D * L) + sl.c_base * L, buf + T * kMRow, (uint32_t)(sl.cn * L * 2));
      }
      bulk_commit();  // one group per iteration, empty for a padding slice
      // Refill the previous stage once its stores have read their shared memory.
      if (k >= 1 && k - 1 + P < mine) {
        bulk_wait_read<1>();
        issue(k - 1 + P);
      }
    }
    __syncwarp();
  }

  if (failed && lane == 0) {
    // Record the error, then let this warp's own loads land before shared memory goes away:
    // the P slices of the prologue and one refill per iteration from k = 1 on were issued,
    // so slices k .. max(k, 1) + P - 2 are in flight.
    atomicOr(p.status != nullptr ? p.status : &g_multi_bulk_error, kDevErrTimeout);
    const int64_t last = (k > 0 ? k - 1 : 0) + P;
    const int64_t issued = last < mine ? last : mine;
    for (int64_t q = k; q < issued; ++q) mbar_wait(&bars[q % P], (uint32_t)((q / P) & 1));
  }
  if (lane == 0) bulk_wait_all();  // stores complete before the warp retires
}

constexpr int kMaxDevices = 64;
std::atomic<bool> g_opted_in[kMaxDevices][kVectorMaxL + 1][2][2];

// Stage bytes a warp may hold: two stages of T + L rows at T = 4, L = 3 (7 KB), a CTA of 8
// warps then needing 57 KB. Larger budgets (more stages, fewer CTAs per SM) lost: N=1024,
// D=16384, T=4, us, 8 / 12 / 16 KB: ring L = 4 99.3 / 112.1 / 177.2, ring L = 5 106.9 / 107.3 /
// 121.8, L = 3 95.7 / 105.7 / 107.7.
constexpr int64_t kWarpStageBudget = 8 * 1024;

// Stage bytes, stages and shared memory per CTA for T tokens at state length L.
struct MbSizes {
  int64_t sb;
  int P;
  size_t smem;
};
MbSizes mb_sizes(int64_t T, int64_t L) {
  MbSizes z;
  z.sb = ((T + L) * kMRow + 127) / 128 * 128;
  int P = (int)(kWarpStageBudget / z.sb);
  z.P = P < 2 ? 2 : (P > kMaxStages ? kMaxStages : P);
  z.smem = (size_t)kWarps * (kBarrierBytes + (size_t)z.P * z.sb);
  return z;
}

template <int L, int ACT, bool RING>
cudaError_t launch_mb(const UpdateParams &p, const MultiParams &m, cudaStream_t stream) {
  const MbSizes z = mb_sizes(m.T, L);
  const int64_t sb = z.sb;
  const int P = z.P;
  const size_t smem = z.smem;
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!g_opted_in[dev][L][ACT][RING].load(std::memory_order_acquire)) {
    // The shared memory of a launch depends on T: opt in once for the largest T served.
    size_t most = 0;
    for (int64_t t = 1; t <= kMultiBulkMaxT; ++t) {
      const size_t b = mb_sizes(t, L).smem;
      most = b > most ? b : most;
    }
    cudaError_t e = cudaFuncSetAttribute(k_multi_bulk<L, kW, ACT, RING>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most);
    if (e != cudaSuccess) return e;
    g_opted_in[dev][L][ACT][RING].store(true, std::memory_order_release);
  }
  int per_sm = 0;
  cudaError_t e =
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_multi_bulk<L, kW, ACT, RING>, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int64_t slices = (p.D + 255) / 256;
  const int64_t items = p.N * slices;
  int64_t warps = (int64_t)device_sm_count() * per_sm * kWarps;
  // A warp count that is a multiple of the slice count keeps every warp on one slice, so
  // its weights stay in registers.
  if (warps >= slices) warps = warps / slices * slices;
  if (warps > items) warps = items;
  int64_t grid = (warps + kWarps - 1) / kWarps;
  if (grid < 1) grid = 1;
  return launch_overlapped(k_multi_bulk<L, kW, ACT, RING>, dim3((unsigned)grid), dim3(kThreads), smem, stream,
                           p, m, P, sb);
}

template <int L, int ACT>
cudaError_t launch_mb_l(const UpdateParams &p, const MultiParams &m, cudaStream_t stream) {
  return p.seqlens != nullptr ? launch_mb<L, ACT, true>(p, m, stream) : launch_mb<L, ACT, false>(p, m, stream);
}

template <int ACT>
cudaError_t launch_mb_a(const UpdateParams &p, const MultiParams &m, cudaStream_t stream) {
  switch (p.L) {
    case 3: return launch_mb_l<3, ACT>(p, m, stream);
    case 4: return launch_mb_l<4, ACT>(p, m, stream);
    case 5: return launch_mb_l<5, ACT>(p, m, stream);
    case 6: return launch_mb_l<6, ACT>(p, m, stream);
    case 7: return launch_mb_l<7, ACT>(p, m, stream);
    case 8: return launch_mb_l<8, ACT>(p, m, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_multi_bulk(const UpdateParams &p, const MultiParams &m, int act, cudaStream_t stream) {
  if (p.W != kW || p.layout != (int)Layout::Compact || m.T < 1 || m.T > kMultiBulkMaxT || m.inter != nullptr)
    return cudaErrorInvalidValue;
  return act == 1 ? launch_mb_a<1>(p, m, stream) : launch_mb_a<0>(p, m, stream);
}

cudaError_t take_multi_bulk_error(int32_t *bits) {
  // read and clear in one atomic step on the device (the legacy default stream orders the
  // copy after the exchange)
  cudaError_t e = launch_overlapped(k_exchange_multi_bulk_error, dim3(1), dim3(1), 0, (cudaStream_t)0);
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(bits, g_multi_bulk_error_taken, sizeof(int32_t));
  return e;
}

}  // namespace ccu
