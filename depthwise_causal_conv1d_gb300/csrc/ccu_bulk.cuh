// Building blocks of the bulk-copy kernels (k_bulk.cu: compact state; k_bulk_planes.cu:
// channel-last state): inline PTX for mbarriers and cp.async.bulk, and the work split of a
// warp into slices (row n, 256*G consecutive channels).
#pragma once

#include "ccu_internal.cuh"

namespace ccu {
namespace bulk {

constexpr int kThreads = 256;              // 8 warps per CTA
constexpr int kWarps = kThreads / 32;
constexpr int kMaxStages = 8;
constexpr int kBarrierBytes = 64;           // a warp's P mbarriers, padded
constexpr uint32_t kMaxSpins = 1u << 22;    // try_wait rounds before a wait is declared failed
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < kMaxSpins; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// global -> shared bulk copy; completes `bytes` of transaction count on `bar`.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// shared -> global bulk copy, tracked by bulk async-groups.
__device__ __forceinline__ void bulk_store(void *dst, const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_addr(src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// All but the newest N committed store groups have finished reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// bulk_wait_read<N> for a run-time N in [0, kMaxStages - 2].
__device__ __forceinline__ void bulk_wait_read_n(int n) {
  switch (n) {
    case 0: bulk_wait_read<0>(); break;
    case 1: bulk_wait_read<1>(); break;
    case 2: bulk_wait_read<2>(); break;
    case 3: bulk_wait_read<3>(); break;
    case 4: bulk_wait_read<4>(); break;
    case 5: bulk_wait_read<5>(); break;
    default: bulk_wait_read<6>(); break;
  }
}

__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Generic-proxy writes to shared memory become visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One work item of a warp.
struct Slice {
  int64_t n, c_base, cn, s;
  int q;  // ring position of the oldest entry (ring-buffer state only)
};

// LC: L known at compile time. The cache_seqlens load is issued together with the index
// load, as in resolve_row. DEDUP = false leaves out the duplicate check (the producer lane
// makes it after issuing the slice's copies, see claim_after_issue).
template <int G, int LC, bool DEDUP = true>
__device__ __forceinline__ Slice slice_of(const UpdateParams &p, int64_t t, int64_t slices, bool report) {
  constexpr int64_t kSlice = 256 * G;
  Slice sl;
  sl.n = t / slices;
  sl.c_base = (t - sl.n * slices) * kSlice;
  const int64_t rem = p.D - sl.c_base;
  sl.cn = rem < kSlice ? rem : kSlice;
  const int32_t v = p.seqlens != nullptr ? __ldg(p.seqlens + sl.n) : 0;
  if (p.idx == nullptr) {
    sl.s = sl.n;
  } else {
    sl.s = __ldg(p.idx + sl.n);
    if (p.status != nullptr && (sl.s < -1 || sl.s >= p.S)) {
      if (report) atomicOr(p.status, 1);  // CCU_DEVERR_RANGE
      sl.s = -1;
    }
    // Duplicate check (every slice of the row gets the same answer; see claim_slot).
    if constexpr (DEDUP) {
      if (p.owner != nullptr && sl.s >= 0 && !claim_slot(p.owner, sl.s, sl.n)) {
        if (report) atomicOr(p.status, 2);  // CCU_DEVERR_DUPLICATE
        sl.s = -1;
      }
    }
  }
  sl.q = 0;
  if (sl.s >= 0 && p.seqlens != nullptr) {
    if (v < 0 && p.status != nullptr) {
      if (report) atomicOr(p.status, 1);  // CCU_DEVERR_RANGE
      sl.s = -1;
    } else {
      const int m = v % LC;
      sl.q = m < 0 ? m + LC : m;
    }
  }
  return sl;
}

// The producer lane's duplicate check, after it has issued the slice's copies: raises
// CCU_DEVERR_DUPLICATE if another row owns the slot. The lanes that compute the slice call
// slice_of with the check and get the same answer, so they drop the staged data.
__device__ __forceinline__ void claim_after_issue(const UpdateParams &p, const Slice &sl) {
  if (p.owner != nullptr && sl.s >= 0 && !claim_slot(p.owner, sl.s, sl.n)) atomicOr(p.status, 2);
}

}  // namespace bulk
}  // namespace ccu
