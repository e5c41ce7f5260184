// C-ABI entry points: argument checks (typed declines), kernel-family selection, launch.
//
// The contract checked here is the one of the cuDNN page "Causal Conv1d Decode Update":
// "Semantic tensor contract" (shapes, ld rule, L >= W - 1, the two state layouts) and
// "Current native implementation" (16-byte pointer alignment for BF16 tensors, 4 bytes
// for indices). Widths other than 4 (any W >= 1 with L >= 1) and the multi-token,
// ring-buffer and prefill forms, which the page names but does not serve, are served here
// too. The declines follow the
// cuDNN page "Composing multi-kernel blocks", section "The shape of a block": a contract
// violation is CCU_ERR_INVALID_ARGUMENT, a valid but unserved request
// CCU_ERR_NOT_IMPLEMENTED, and nothing is launched or changed in either case.
#include <atomic>
#include <cstdarg>
#include <cstdio>

#include "ccu_conv1d.h"
#include "ccu_internal.cuh"

namespace ccu {

int device_sm_count();

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
thread_local char g_last_error[512];

ccu_status_t fail(ccu_status_t st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return st;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// a * b <= limit for non-negative a, b, without overflow.
bool mul_le(int64_t a, int64_t b, int64_t limit) { return a == 0 || b <= limit / a; }

struct Args {
  const void *x;
  int64_t ld;
  const void *state;
  int64_t ss, sd, sl;
  const void *w;
  const void *bias;
  int act;
  const int32_t *idx;
  const int32_t *cache_seqlens;
  int64_t N, D, S, L, W;
  const void *out;
  const int32_t *status;
  int32_t *owner = nullptr;  // slot-owner scratch [S]: the duplicate check (checked mode only)
};

// Every check of the contract. On CCU_OK, *noop says whether there is nothing to launch
// and *layout which state layout the strides describe.
ccu_status_t validate(const Args &a, bool *noop, Layout *layout) {
  g_last_error[0] = '\0';
  if (a.act != CCU_ACT_IDENTITY && a.act != CCU_ACT_SILU)
    return fail(CCU_ERR_INVALID_ARGUMENT, "act must be CCU_ACT_IDENTITY or CCU_ACT_SILU, got %d",
                a.act);
  if (a.N < 0 || a.D < 0 || a.S < 0)
    return fail(CCU_ERR_INVALID_ARGUMENT, "N, D and S must be >= 0");
  if (a.W < 1) return fail(CCU_ERR_INVALID_ARGUMENT, "W must be >= 1, got %lld", (long long)a.W);
  if (a.L < a.W - 1)
    return fail(CCU_ERR_INVALID_ARGUMENT, "L must be >= W - 1 (L=%lld, W=%lld)", (long long)a.L,
                (long long)a.W);
  if (a.L < 1) return fail(CCU_ERR_NOT_IMPLEMENTED, "an empty state (L = 0) is not served");
  if (!mul_le(a.D, a.W, INT64_MAX / 4))
    return fail(CCU_ERR_INVALID_ARGUMENT, "tensor sizes overflow 64-bit indexing");
  if (a.status != nullptr && !aligned(a.status, 4))
    return fail(CCU_ERR_INVALID_ARGUMENT, "status word must be 4-byte aligned");
  if (a.owner != nullptr) {
    if (a.status == nullptr)
      return fail(CCU_ERR_INVALID_ARGUMENT, "the duplicate check needs a status word");
    if (!aligned(a.owner, 4))
      return fail(CCU_ERR_INVALID_ARGUMENT, "slot_scratch must be 4-byte aligned");
    if (a.N >= INT32_MAX)
      return fail(CCU_ERR_NOT_IMPLEMENTED, "the duplicate check serves N < 2^31 - 1 rows");
  }
  if (a.N == 0 || a.D == 0) {
    *noop = true;  // nothing to read or write, whatever the strides
    return CCU_OK;
  }
  *noop = false;
  if (a.ld < a.D)
    return fail(CCU_ERR_INVALID_ARGUMENT, "ld must be >= D (ld=%lld, D=%lld)", (long long)a.ld,
                (long long)a.D);
  if (a.ld > a.D && a.ld % 8 != 0)
    return fail(CCU_ERR_INVALID_ARGUMENT,
                "a padded row stride ld > D must be a multiple of 8, got ld=%lld", (long long)a.ld);
  if (a.x == nullptr || a.w == nullptr || a.out == nullptr || (a.state == nullptr && a.S > 0))
    return fail(CCU_ERR_INVALID_ARGUMENT, "x, conv_state, weight and out must not be NULL");
  if (!aligned(a.x, 16) || !aligned(a.state, 16) || !aligned(a.w, 16) || !aligned(a.out, 16) ||
      (a.bias != nullptr && !aligned(a.bias, 16)))
    return fail(CCU_ERR_INVALID_ARGUMENT, "BF16 tensors must be 16-byte aligned");
  if (a.idx != nullptr && !aligned(a.idx, 4))
    return fail(CCU_ERR_INVALID_ARGUMENT, "conv_state_indices must be 4-byte aligned");
  if (a.cache_seqlens != nullptr && !aligned(a.cache_seqlens, 4))
    return fail(CCU_ERR_INVALID_ARGUMENT, "cache_seqlens must be 4-byte aligned");
  if (a.idx == nullptr && a.S < a.N)
    return fail(CCU_ERR_INVALID_ARGUMENT,
                "without conv_state_indices row n uses slot n, so S must be >= N (S=%lld, N=%lld)",
                (long long)a.S, (long long)a.N);
  const int64_t lim = INT64_MAX / 4;
  if (!mul_le(a.N, a.ld, lim) || !mul_le(a.D, a.L, lim) || !mul_le(a.S, a.D * a.L, lim))
    return fail(CCU_ERR_INVALID_ARGUMENT, "tensor sizes overflow 64-bit indexing");
  if (a.ss == a.D * a.L && a.sd == a.L && a.sl == 1) {
    *layout = Layout::Compact;
  } else if (a.ss == a.L * a.D && a.sd == 1 && a.sl == a.D) {
    *layout = Layout::ChannelLast;
  } else {
    return fail(CCU_ERR_NOT_IMPLEMENTED,
                "conv_state strides (%lld, %lld, %lld) are neither compact (D*L, L, 1) nor "
                "channel-last (L*D, 1, D)",
                (long long)a.ss, (long long)a.sd, (long long)a.sl);
  }
  return CCU_OK;
}

// The bulk family is compiled for width 4 with L <= 8 (both layouts) and, in the compact
// layout, for widths 2 and 3 with L <= 4 (the short states those widths are used with).
constexpr int64_t kBulkNarrowMaxL = 4;

bool route_serves(int route, const Args &a, Layout layout) {
  // The 8-channel kernels are compiled for widths 2 to 4; every other width runs on the
  // scalar kernel.
  const bool vec8 = (a.D % 8 == 0) && (a.ld % 8 == 0) && a.W >= 2 && a.W <= kW;
  switch (route) {
    case CCU_ROUTE_SCALAR: return true;
    case CCU_ROUTE_VECTOR: return vec8 && a.L <= kVectorMaxL;
    case CCU_ROUTE_STAGED: return vec8 && a.L <= kStagedMaxL;
    case CCU_ROUTE_BULK:
      if (!vec8) return false;
      if (a.W == kW) return a.L <= kVectorMaxL;
      return layout == Layout::Compact && a.L <= kBulkNarrowMaxL;
    default: return false;
  }
}

// Below this many (row, channel) elements a call is launch-bound and the plain vector
// kernel's shorter start-up wins; above it the bulk-copy pipeline keeps more bytes in flight
// (compact state, cold L2, D = 16384: tied at 64 rows, 12.3 vs 14.8 us at 128 rows, 24.6 vs
// 27.5 us at 512).
constexpr int64_t kBulkMinElements = 1 << 20;
constexpr int64_t kWindowOnlyW3VectorElements = int64_t(3) << 24;

ccu_status_t choose(int requested, const Args &a, Layout layout, int *chosen) {
  if (requested < 0 || requested >= CCU_ROUTE_COUNT)
    return fail(CCU_ERR_INVALID_ARGUMENT, "unknown route %d", requested);
  if (requested == CCU_ROUTE_AUTO) {
    // The bulk kernel serves the linear compact state from 2^20 elements where it measured
    // ahead of the vector kernel (D = 16384, us, bulk / vector):
    //  - L = 7 (N = 4096, back to back: 310.2 / 362.9), and L = 4 at widths 2 and 3 (width 3:
    //    199.9 / 203.2); width 4 at L = 4 takes the vector route's one-channel-per-lane kernel
    //    (cold, N = 1024: 56.8 / 53.5; back to back at N = 4096 199.0 / 200.6);
    //  - width 3 with L = 2 (a state of just the window) below 3 * 2^24 elements (back to
    //    back, 1024 rows: 36.8 / 41.0; 4096 rows: 119.0 / 116.5).
    // Everything else takes the vector kernel: L = 3, 5, 6 at every size (cold, on rotating
    // copies: N = 64 6.6 / 6.0, N = 256 15.7 / 13.9, N = 512 25.9 / 23.4, N = 768 37.2 / 33.2,
    // N = 256 at D = 8192 10.0 / 9.2; back to back the two are within 8 % from 2^20 to 2^23
    // elements and the vector kernel leads beyond: N = 4096 160.1 / 155.5; L = 5 and 6:
    // 247.3 / 237.8 and 289.2 / 286.7); L = 8 (570.4 / 337.1, where the vector route takes
    // one channel per lane; a lane's 128-byte state makes the bulk kernel's shared-memory
    // accesses bank-conflicted); L = 1, which moves 8 bytes
    // per element, too little per 512-channel slice (W = 2: 100.8 / 80.7); the ring state
    // (compact, N = 4096: 161.5 / 158.6; N = 1024: 45.3 / 43.7) and the channel-last state
    // (linear: N = 4096, 162.3 plane-bulk / 154.3; ring: the vector kernel leads from 128 rows).
    const int64_t elements = a.N * a.D;
    const bool ring = a.cache_seqlens != nullptr;
    const bool window_only_w3 = a.W == 3 && a.L == 2 && elements >= kWindowOnlyW3VectorElements;
    const bool vector_leads = a.L == 3 || a.L == 5 || a.L == 6 || (a.L == 4 && a.W == kW);
    const bool bulk_size = layout == Layout::Compact && !ring && elements >= kBulkMinElements && a.L >= 2 &&
                           a.L != 8 && !window_only_w3 && !vector_leads;
    if (bulk_size && route_serves(CCU_ROUTE_BULK, a, layout)) {
      *chosen = CCU_ROUTE_BULK;
    } else if (route_serves(CCU_ROUTE_VECTOR, a, layout)) {
      *chosen = CCU_ROUTE_VECTOR;
    } else if (route_serves(CCU_ROUTE_STAGED, a, layout)) {
      *chosen = CCU_ROUTE_STAGED;
    } else {
      *chosen = CCU_ROUTE_SCALAR;
    }
    return CCU_OK;
  }
  if (!route_serves(requested, a, layout))
    return fail(CCU_ERR_NOT_IMPLEMENTED, "route '%s' does not serve these arguments",
                ccu_route_name(requested));
  *chosen = requested;
  return CCU_OK;
}

// True when p is host memory (pinned or pageable) rather than device or managed memory.
bool is_host_memory(const void *p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeUnregistered;
}

ccu_status_t run(const Args &a, int route, cudaStream_t stream) {
  bool noop = false;
  Layout layout = Layout::Compact;
  ccu_status_t st = validate(a, &noop, &layout);
  if (st != CCU_OK || noop) return st;
  int chosen = CCU_ROUTE_AUTO;
  st = choose(route, a, layout, &chosen);
  if (st != CCU_OK) return st;
  // The bulk kernel's copies run between device memory and shared memory. x and out may
  // also be host memory the device can address (for example pinned with cudaHostAlloc):
  // the vector kernel reads and writes those with ordinary loads and stores.
  if (chosen == CCU_ROUTE_BULK && (is_host_memory(a.x) || is_host_memory(a.out))) {
    if (route == CCU_ROUTE_BULK)
      return fail(CCU_ERR_NOT_IMPLEMENTED,
                  "route 'bulk' needs x and out in device memory; x or out is host memory");
    chosen = CCU_ROUTE_VECTOR;  // serves every call the bulk family serves
  }

  UpdateParams p;
  p.x = static_cast<const uint16_t *>(a.x);
  p.ld = a.ld;
  p.state = static_cast<uint16_t *>(const_cast<void *>(a.state));
  p.w = static_cast<const uint16_t *>(a.w);
  p.bias = static_cast<const uint16_t *>(a.bias);
  p.idx = a.idx;
  p.seqlens = a.cache_seqlens;
  p.out = static_cast<uint16_t *>(const_cast<void *>(a.out));
  p.status = const_cast<int32_t *>(a.status);
  // Without indices row n uses slot n: no two rows can share a slot.
  p.owner = a.idx != nullptr ? a.owner : nullptr;
  p.N = a.N;
  p.D = a.D;
  p.S = a.S;
  p.L = a.L;
  p.W = a.W;
  p.ss = a.ss;
  p.sd = a.sd;
  p.sl = a.sl;
  p.layout = (int)layout;
  p.rows_per_cta = 1;

  cudaError_t e = cudaSuccess;
  if (p.owner != nullptr && a.S > 0) e = launch_clear_words(p.owner, a.S, stream);
  if (e != cudaSuccess)
    return fail(CCU_ERR_CUDA, "clearing slot_scratch failed: %s", cudaGetErrorString(e));
  e = cudaErrorInvalidValue;
  switch (chosen) {
    case CCU_ROUTE_SCALAR: e = launch_scalar(p, a.act, stream); break;
    case CCU_ROUTE_VECTOR: e = launch_vector(p, a.act, stream); break;
    case CCU_ROUTE_STAGED: e = launch_staged(p, a.act, stream); break;
    case CCU_ROUTE_BULK: e = launch_bulk(p, a.act, stream); break;
    default: break;
  }
  if (e != cudaSuccess)
    return fail(CCU_ERR_CUDA, "launch of the %s kernel failed: %s", ccu_route_name(chosen),
                cudaGetErrorString(e));
  return CCU_OK;
}

// ---------------------------------------------------------------- multi-token update

struct MultiArgs {
  Args a;  // x, state, weight, bias, act, indices, seqlens, N, D, S, L, W, out, status
  int64_t T, sxn, sxd, sxt, son, sod, sot;
  const void *inter;
};

ccu_status_t validate_multi(const MultiArgs &m, bool *noop, Layout *layout) {
  const Args &a = m.a;
  g_last_error[0] = '\0';
  if (a.act != CCU_ACT_IDENTITY && a.act != CCU_ACT_SILU)
    return fail(CCU_ERR_INVALID_ARGUMENT, "act must be CCU_ACT_IDENTITY or CCU_ACT_SILU, got %d",
                a.act);
  if (a.N < 0 || a.D < 0 || a.S < 0 || m.T < 0)
    return fail(CCU_ERR_INVALID_ARGUMENT, "N, D, T and S must be >= 0");
  if (a.W < 1) return fail(CCU_ERR_INVALID_ARGUMENT, "W must be >= 1, got %lld", (long long)a.W);
  if (a.L < a.W - 1)
    return fail(CCU_ERR_INVALID_ARGUMENT, "L must be >= W - 1 (L=%lld, W=%lld)", (long long)a.L,
                (long long)a.W);
  if (a.L < 1) return fail(CCU_ERR_NOT_IMPLEMENTED, "an empty state (L = 0) is not served");
  if (!mul_le(a.D, a.W, INT64_MAX / 4))
    return fail(CCU_ERR_INVALID_ARGUMENT, "tensor sizes overflow 64-bit indexing");
  if (a.status != nullptr && !aligned(a.status, 4))
    return fail(CCU_ERR_INVALID_ARGUMENT, "status word must be 4-byte aligned");
  if (a.N == 0 || a.D == 0 || m.T == 0) {
    *noop = true;
    return CCU_OK;
  }
  *noop = false;
  if (m.sxn < 0 || m.sxd < 0 || m.sxt < 0 || m.son < 0 || m.sod < 0 || m.sot < 0)
    return fail(CCU_ERR_INVALID_ARGUMENT, "x and out strides must be >= 0");
  if (a.x == nullptr || a.w == nullptr || a.out == nullptr || (a.state == nullptr && a.S > 0))
    return fail(CCU_ERR_INVALID_ARGUMENT, "x, conv_state, weight and out must not be NULL");
  if (!aligned(a.x, 16) || !aligned(a.state, 16) || !aligned(a.w, 16) || !aligned(a.out, 16) ||
      (a.bias != nullptr && !aligned(a.bias, 16)) || (m.inter != nullptr && !aligned(m.inter, 16)))
    return fail(CCU_ERR_INVALID_ARGUMENT, "BF16 tensors must be 16-byte aligned");
  if (a.idx != nullptr && !aligned(a.idx, 4))
    return fail(CCU_ERR_INVALID_ARGUMENT, "conv_state_indices must be 4-byte aligned");
  if (a.cache_seqlens != nullptr && !aligned(a.cache_seqlens, 4))
    return fail(CCU_ERR_INVALID_ARGUMENT, "cache_seqlens must be 4-byte aligned");
  if (a.idx == nullptr && a.S < a.N)
    return fail(CCU_ERR_INVALID_ARGUMENT,
                "without conv_state_indices row n uses slot n, so S must be >= N (S=%lld, N=%lld)",
                (long long)a.S, (long long)a.N);
  const int64_t lim = INT64_MAX / 4;
  if (!mul_le(a.D, a.L, lim) || !mul_le(a.S, a.D * a.L, lim) || !mul_le(a.N, m.T, lim) ||
      !mul_le(a.N * m.T, a.D * a.L, lim))
    return fail(CCU_ERR_INVALID_ARGUMENT, "tensor sizes overflow 64-bit indexing");
  if (a.ss == a.D * a.L && a.sd == a.L && a.sl == 1) {
    *layout = Layout::Compact;
  } else if (a.ss == a.L * a.D && a.sd == 1 && a.sl == a.D) {
    *layout = Layout::ChannelLast;
  } else {
    return fail(CCU_ERR_NOT_IMPLEMENTED,
                "conv_state strides (%lld, %lld, %lld) are neither compact (D*L, L, 1) nor "
                "channel-last (L*D, 1, D)",
                (long long)a.ss, (long long)a.sd, (long long)a.sl);
  }
  return CCU_OK;
}

// The vector multi-token kernel moves 8 channels of one token as one 16-byte vector.
constexpr int64_t kMultiNarrowMaxL = 4;

bool multi_vector_serves(const MultiArgs &m) {
  const Args &a = m.a;
  // width 4 up to L = 8; widths 2 and 3 up to L = 4; other widths on the scalar kernel
  const bool served_l = a.W == kW ? a.L <= kVectorMaxL : a.L <= kMultiNarrowMaxL;
  return a.W >= 2 && a.W <= kW && a.D % 8 == 0 && served_l && m.sxd == 1 && m.sod == 1 &&
         m.sxn % 8 == 0 && m.sxt % 8 == 0 && m.son % 8 == 0 && m.sot % 8 == 0;
}

// The bulk-copy multi-token kernel: width 4, the compact state at L = 3..8, T <= 8 tokens,
// no intermediate states, the vector kernel's stride conditions, and x and out in device
// memory (checked last: it queries the pointers).
bool multi_bulk_serves(const MultiArgs &m, Layout layout) {
  const Args &a = m.a;
  return a.W == kW && a.L >= 3 && a.L <= kVectorMaxL && layout == Layout::Compact && m.T >= 1 &&
         m.T <= kMultiBulkMaxT && m.inter == nullptr && multi_vector_serves(m) && !is_host_memory(a.x) &&
         !is_host_memory(a.out);
}

ccu_status_t run_multi(const MultiArgs &m, int route, cudaStream_t stream) {
  bool noop = false;
  Layout layout = Layout::Compact;
  ccu_status_t st = validate_multi(m, &noop, &layout);
  if (st != CCU_OK || noop) return st;
  int chosen;
  if (route == CCU_ROUTE_AUTO) {
    // The bulk-copy kernel where it measured ahead of the vector kernel: the compact ring
    // state at L = 4, 5 and 7 (N=1024, D=16384, T=4, us, bulk / vector: 98.9 / 109.4, 107.0 /
    // 123.4, 131.2 / 158.8). Elsewhere the vector kernel leads (compact linear L = 3 95.2 /
    // 81.0, L = 5 112.5 / 97.1, L = 8 185.7 / 145.2; ring L = 3 97.3 / 89.6, L = 6 128.2 /
    // 119.3, L = 8 184.8 / 170.5; T = 1, 2, 8 and N = 256, 4096 at L = 3 likewise).
    const bool bulk_leads = m.a.cache_seqlens != nullptr && (m.a.L == 4 || m.a.L == 5 || m.a.L == 7);
    if (bulk_leads && layout == Layout::Compact && multi_bulk_serves(m, layout)) {
      chosen = CCU_ROUTE_BULK;
    } else {
      chosen = multi_vector_serves(m) ? CCU_ROUTE_VECTOR : CCU_ROUTE_SCALAR;
    }
  } else if (route == CCU_ROUTE_SCALAR || (route == CCU_ROUTE_VECTOR && multi_vector_serves(m)) ||
             (route == CCU_ROUTE_BULK && multi_bulk_serves(m, layout))) {
    chosen = route;
  } else if (route >= 0 && route < CCU_ROUTE_COUNT) {
    return fail(CCU_ERR_NOT_IMPLEMENTED, "route '%s' does not serve these multi-token arguments",
                ccu_route_name(route));
  } else {
    return fail(CCU_ERR_INVALID_ARGUMENT, "unknown route %d", route);
  }
  const Args &a = m.a;
  UpdateParams p = {};
  p.x = static_cast<const uint16_t *>(a.x);
  p.ld = 0;
  p.state = static_cast<uint16_t *>(const_cast<void *>(a.state));
  p.w = static_cast<const uint16_t *>(a.w);
  p.bias = static_cast<const uint16_t *>(a.bias);
  p.idx = a.idx;
  p.seqlens = a.cache_seqlens;
  p.out = static_cast<uint16_t *>(const_cast<void *>(a.out));
  p.status = const_cast<int32_t *>(a.status);
  p.N = a.N;
  p.D = a.D;
  p.S = a.S;
  p.L = a.L;
  p.W = a.W;
  p.ss = a.ss;
  p.sd = a.sd;
  p.sl = a.sl;
  p.layout = (int)layout;
  p.rows_per_cta = 1;
  MultiParams mp;
  mp.T = m.T;
  mp.sxn = m.sxn;
  mp.sxd = m.sxd;
  mp.sxt = m.sxt;
  mp.son = m.son;
  mp.sod = m.sod;
  mp.sot = m.sot;
  mp.inter = static_cast<uint16_t *>(const_cast<void *>(m.inter));
  cudaError_t e = chosen == CCU_ROUTE_BULK     ? launch_multi_bulk(p, mp, a.act, stream)
                  : chosen == CCU_ROUTE_VECTOR ? launch_multi_vector(p, mp, a.act, stream)
                                               : launch_multi_scalar(p, mp, a.act, stream);
  if (e != cudaSuccess)
    return fail(CCU_ERR_CUDA, "launch of the multi-token %s kernel failed: %s",
                ccu_route_name(chosen), cudaGetErrorString(e));
  return CCU_OK;
}

// ---------------------------------------------------------------- full-sequence prefill

struct PrefillArgs {
  const void *x, *w, *bias, *init, *out, *fin;
  int act;
  int64_t sxb, sxd, sxt, sib, sid, sil, sob, sod, sot, sfb, sfd, sfl;
  int64_t B, D, T, L, W;
};

// Prefill sizes (B*D*T) from which AUTO takes the bulk-copy kernel.
constexpr int64_t kPrefillBulkMinElements = int64_t(1) << 20;

// Tokens per thread: enough (batch row, channel group, chunk) items to fill the GPU several
// times over, and at least 32 tokens so the 3-token halo stays a small overhead.
int64_t prefill_chunk(int64_t B, int64_t lanes, int64_t T) {
  const int64_t want = (int64_t)device_sm_count() * 2048 * 2;  // thread items to aim for
  int64_t chunks = want / (B * lanes > 0 ? B * lanes : 1);
  if (chunks < 1) chunks = 1;
  int64_t chunk = (T + chunks - 1) / chunks;
  chunk = (chunk + 3) / 4 * 4;
  if (chunk < 32) chunk = 32;
  return chunk;
}

ccu_status_t run_prefill(const PrefillArgs &a, int route, cudaStream_t stream) {
  g_last_error[0] = '\0';
  if (a.act != CCU_ACT_IDENTITY && a.act != CCU_ACT_SILU)
    return fail(CCU_ERR_INVALID_ARGUMENT, "act must be CCU_ACT_IDENTITY or CCU_ACT_SILU, got %d",
                a.act);
  if (a.B < 0 || a.D < 0 || a.T < 0) return fail(CCU_ERR_INVALID_ARGUMENT, "B, D and T must be >= 0");
  if (a.W < 1) return fail(CCU_ERR_INVALID_ARGUMENT, "W must be >= 1, got %lld", (long long)a.W);
  if (a.L < a.W - 1)
    return fail(CCU_ERR_INVALID_ARGUMENT, "L must be >= W - 1 (L=%lld, W=%lld)", (long long)a.L,
                (long long)a.W);
  if (a.L < 1) return fail(CCU_ERR_NOT_IMPLEMENTED, "an empty state (L = 0) is not served");
  if (!mul_le(a.D, a.W, INT64_MAX / 4))
    return fail(CCU_ERR_INVALID_ARGUMENT, "tensor sizes overflow 64-bit indexing");
  if (a.B == 0 || a.D == 0 || a.T == 0) return CCU_OK;
  const int64_t strides[] = {a.sxb, a.sxd, a.sxt, a.sib, a.sid, a.sil, a.sob, a.sod, a.sot,
                             a.sfb, a.sfd, a.sfl};
  for (int64_t v : strides)
    if (v < 0) return fail(CCU_ERR_INVALID_ARGUMENT, "strides must be >= 0");
  if (a.x == nullptr || a.w == nullptr || a.out == nullptr)
    return fail(CCU_ERR_INVALID_ARGUMENT, "x, weight and out must not be NULL");
  if (!aligned(a.x, 16) || !aligned(a.w, 16) || !aligned(a.out, 16) ||
      (a.bias != nullptr && !aligned(a.bias, 16)) || (a.init != nullptr && !aligned(a.init, 16)) ||
      (a.fin != nullptr && !aligned(a.fin, 16)))
    return fail(CCU_ERR_INVALID_ARGUMENT, "BF16 tensors must be 16-byte aligned");
  if (a.fin != nullptr && a.fin == a.init)
    return fail(CCU_ERR_INVALID_ARGUMENT,
                "final_states must not be the initial_states buffer (write the new state elsewhere)");
  const int64_t lim = INT64_MAX / 4;
  if (!mul_le(a.B, a.D, lim) || !mul_le(a.B * a.D, a.T, lim) || !mul_le(a.B * a.D, a.L, lim))
    return fail(CCU_ERR_INVALID_ARGUMENT, "tensor sizes overflow 64-bit indexing");

  // The vector and bulk kernels serve widths 2 to 4; other widths run on the scalar kernel.
  const bool vec_ok = a.W >= 2 && a.W <= kW && a.D % 8 == 0 && a.sxd == 1 && a.sod == 1 && a.sxb % 8 == 0 &&
                      a.sxt % 8 == 0 && a.sob % 8 == 0 && a.sot % 8 == 0 && a.B <= 65535;
  PrefillParams f;
  f.B = a.B;
  f.T = a.T;
  f.sxb = a.sxb; f.sxd = a.sxd; f.sxt = a.sxt;
  f.sob = a.sob; f.sod = a.sod; f.sot = a.sot;
  f.init = static_cast<const uint16_t *>(a.init);
  f.sib = a.sib; f.sid = a.sid; f.sil = a.sil;
  f.fin = static_cast<uint16_t *>(const_cast<void *>(a.fin));
  f.sfb = a.sfb; f.sfd = a.sfd; f.sfl = a.sfl;
  // The bulk kernel's copies run between device memory and shared memory (as for the
  // update, host-resident x or out go to the vector kernel). The pointer query runs only
  // when the bulk kernel is in question.
  auto on_device = [&]() { return !is_host_memory(a.x) && !is_host_memory(a.out); };
  bool vector, bulk = false;
  if (route == CCU_ROUTE_AUTO) {
    vector = vec_ok;
    bulk = vec_ok && a.B * a.D * a.T >= kPrefillBulkMinElements && on_device();
  } else if (route == CCU_ROUTE_SCALAR) {
    vector = false;
  } else if (route == CCU_ROUTE_VECTOR && vec_ok) {
    vector = true;
  } else if (route == CCU_ROUTE_BULK && vec_ok && on_device()) {
    vector = bulk = true;
  } else if (route >= 0 && route < CCU_ROUTE_COUNT) {
    return fail(CCU_ERR_NOT_IMPLEMENTED, "route '%s' does not serve these prefill arguments",
                ccu_route_name(route));
  } else {
    return fail(CCU_ERR_INVALID_ARGUMENT, "unknown route %d", route);
  }
  f.chunk = prefill_chunk(a.B, vector ? a.D / 8 : a.D, a.T);
  if (vector && (a.T + f.chunk - 1) / f.chunk > 65535) vector = false;
  UpdateParams p = {};
  p.x = static_cast<const uint16_t *>(a.x);
  p.w = static_cast<const uint16_t *>(a.w);
  p.bias = static_cast<const uint16_t *>(a.bias);
  p.out = static_cast<uint16_t *>(const_cast<void *>(a.out));
  p.D = a.D;
  p.L = a.L;
  p.W = a.W;
  cudaError_t e = bulk ? launch_prefill_bulk(p, f, a.act, stream)
                       : launch_prefill(p, f, a.act, vector, stream);
  if (e != cudaSuccess)
    return fail(CCU_ERR_CUDA, "launch of the prefill kernel failed: %s", cudaGetErrorString(e));
  return CCU_OK;
}

}  // namespace

void record_error(const char *msg) { snprintf(g_last_error, sizeof g_last_error, "%s", msg); }

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

int device_sm_count() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return 1;
  int v = g_sm_count[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
    return 1;
  g_sm_count[dev].store(v, std::memory_order_relaxed);
  return v;
}

}  // namespace ccu

using ccu::Args;

extern "C" {

ccu_status_t ccu_conv1d_update_ex(const void *x, int64_t ld, void *conv_state, int64_t stride_s,
                                  int64_t stride_d, int64_t stride_l, const void *weight,
                                  const void *bias, ccu_act_t act, const int32_t *indices,
                                  const int32_t *cache_seqlens, int64_t N, int64_t D, int64_t S,
                                  int64_t L, int64_t W, void *out, int32_t *status_dev,
                                  int32_t route, ccu_stream_t stream) {
  const Args a{x,    ld,      conv_state, stride_s,      stride_d, stride_l, weight, bias,
               (int)act, indices, cache_seqlens, N, D, S, L, W, out, status_dev};
  return ccu::run(a, route, reinterpret_cast<cudaStream_t>(stream));
}

ccu_status_t ccu_conv1d_update(const void *x, int64_t ld, void *conv_state, int64_t stride_s,
                               int64_t stride_d, int64_t stride_l, const void *weight,
                               const void *bias, ccu_act_t act, const int32_t *indices,
                               const int32_t *cache_seqlens, int64_t N, int64_t D, int64_t S,
                               int64_t L, int64_t W, void *out, ccu_stream_t stream) {
  return ccu_conv1d_update_ex(x, ld, conv_state, stride_s, stride_d, stride_l, weight, bias, act,
                              indices, cache_seqlens, N, D, S, L, W, out, nullptr,
                              CCU_ROUTE_AUTO, stream);
}

ccu_status_t ccu_conv1d_update_checked(const void *x, int64_t ld, void *conv_state,
                                       int64_t stride_s, int64_t stride_d, int64_t stride_l,
                                       const void *weight, const void *bias, ccu_act_t act,
                                       const int32_t *indices, const int32_t *cache_seqlens,
                                       int64_t N, int64_t D, int64_t S, int64_t L, int64_t W,
                                       void *out, int32_t *status_dev, ccu_stream_t stream) {
  if (status_dev == nullptr)
    return ccu::fail(CCU_ERR_INVALID_ARGUMENT, "status_dev must not be NULL");
  return ccu_conv1d_update_ex(x, ld, conv_state, stride_s, stride_d, stride_l, weight, bias, act,
                              indices, cache_seqlens, N, D, S, L, W, out, status_dev,
                              CCU_ROUTE_AUTO, stream);
}

ccu_status_t ccu_conv1d_update_checked_ex(const void *x, int64_t ld, void *conv_state,
                                          int64_t stride_s, int64_t stride_d, int64_t stride_l,
                                          const void *weight, const void *bias, ccu_act_t act,
                                          const int32_t *indices, const int32_t *cache_seqlens,
                                          int64_t N, int64_t D, int64_t S, int64_t L, int64_t W,
                                          void *out, int32_t *status_dev, int32_t *slot_scratch,
                                          int32_t route, ccu_stream_t stream) {
  if (status_dev == nullptr)
    return ccu::fail(CCU_ERR_INVALID_ARGUMENT, "status_dev must not be NULL");
  if (slot_scratch == nullptr && indices != nullptr && N > 0 && D > 0 && S > 0)
    return ccu::fail(CCU_ERR_INVALID_ARGUMENT, "slot_scratch must not be NULL");
  Args a{x,    ld,      conv_state, stride_s,      stride_d, stride_l, weight, bias,
         (int)act, indices, cache_seqlens, N, D, S, L, W, out, status_dev};
  a.owner = slot_scratch;
  return ccu::run(a, route, reinterpret_cast<cudaStream_t>(stream));
}

int64_t ccu_conv1d_slot_scratch_bytes(int64_t S) { return S > 0 ? S * (int64_t)sizeof(int32_t) : 0; }

ccu_status_t ccu_conv1d_select_route(const void *x, int64_t ld, const void *conv_state,
                                     int64_t stride_s, int64_t stride_d, int64_t stride_l,
                                     const void *weight, const void *bias, ccu_act_t act,
                                     const int32_t *indices, const int32_t *cache_seqlens,
                                     int64_t N, int64_t D, int64_t S, int64_t L, int64_t W,
                                     const void *out, int32_t route, int32_t *chosen_route) {
  if (chosen_route == nullptr)
    return ccu::fail(CCU_ERR_INVALID_ARGUMENT, "chosen_route must not be NULL");
  const Args a{x,    ld,      conv_state, stride_s,      stride_d, stride_l, weight, bias,
               (int)act, indices, cache_seqlens, N, D, S, L, W, out, nullptr};
  bool noop = false;
  ccu::Layout layout = ccu::Layout::Compact;
  ccu_status_t st = ccu::validate(a, &noop, &layout);
  if (st != CCU_OK) return st;
  if (noop) {
    *chosen_route = CCU_ROUTE_AUTO;
    return CCU_OK;
  }
  int chosen = CCU_ROUTE_AUTO;
  st = ccu::choose(route, a, layout, &chosen);
  if (st == CCU_OK) *chosen_route = chosen;
  return st;
}

ccu_status_t ccu_conv1d_update_multi(const void *x, int64_t x_stride_n, int64_t x_stride_d,
                                     int64_t x_stride_t, void *conv_state, int64_t stride_s,
                                     int64_t stride_d, int64_t stride_l, const void *weight,
                                     const void *bias, ccu_act_t act, const int32_t *indices,
                                     const int32_t *cache_seqlens, int64_t N, int64_t D, int64_t T,
                                     int64_t S, int64_t L, int64_t W, void *out,
                                     int64_t out_stride_n, int64_t out_stride_d,
                                     int64_t out_stride_t, void *intermediate_states,
                                     int32_t *status_dev, int32_t route, ccu_stream_t stream) {
  ccu::MultiArgs m;
  m.a = Args{x,    0,       conv_state,    stride_s, stride_d, stride_l, weight, bias, (int)act,
             indices, cache_seqlens, N, D, S, L, W, out, status_dev};
  m.T = T;
  m.sxn = x_stride_n;
  m.sxd = x_stride_d;
  m.sxt = x_stride_t;
  m.son = out_stride_n;
  m.sod = out_stride_d;
  m.sot = out_stride_t;
  m.inter = intermediate_states;
  return ccu::run_multi(m, route, reinterpret_cast<cudaStream_t>(stream));
}

ccu_status_t ccu_causal_conv1d_fwd(const void *x, int64_t x_stride_b, int64_t x_stride_d,
                                   int64_t x_stride_t, const void *weight, const void *bias,
                                   ccu_act_t act, const void *initial_states, int64_t init_stride_b,
                                   int64_t init_stride_d, int64_t init_stride_l, int64_t B, int64_t D,
                                   int64_t T, int64_t L, int64_t W, void *out, int64_t out_stride_b,
                                   int64_t out_stride_d, int64_t out_stride_t, void *final_states,
                                   int64_t final_stride_b, int64_t final_stride_d,
                                   int64_t final_stride_l, int32_t route, ccu_stream_t stream) {
  ccu::PrefillArgs a;
  a.x = x; a.w = weight; a.bias = bias; a.init = initial_states; a.out = out; a.fin = final_states;
  a.act = (int)act;
  a.sxb = x_stride_b; a.sxd = x_stride_d; a.sxt = x_stride_t;
  a.sib = init_stride_b; a.sid = init_stride_d; a.sil = init_stride_l;
  a.sob = out_stride_b; a.sod = out_stride_d; a.sot = out_stride_t;
  a.sfb = final_stride_b; a.sfd = final_stride_d; a.sfl = final_stride_l;
  a.B = B; a.D = D; a.T = T; a.L = L; a.W = W;
  return ccu::run_prefill(a, route, reinterpret_cast<cudaStream_t>(stream));
}

int64_t ccu_conv1d_check_indices_scratch_bytes(int64_t S) {
  if (S <= 0) return 0;
  return ((S + 31) / 32) * 4;
}

ccu_status_t ccu_conv1d_check_indices(const int32_t *indices, int64_t N, int64_t S,
                                      uint32_t *bitmap_scratch, int32_t *status_dev,
                                      ccu_stream_t stream) {
  ccu::g_last_error[0] = '\0';
  if (N < 0 || S < 0) return ccu::fail(CCU_ERR_INVALID_ARGUMENT, "N and S must be >= 0");
  if (N == 0) return CCU_OK;
  if (indices == nullptr || status_dev == nullptr || (S > 0 && bitmap_scratch == nullptr))
    return ccu::fail(CCU_ERR_INVALID_ARGUMENT, "indices, bitmap_scratch and status_dev must not be NULL");
  if (!ccu::aligned(indices, 4) || !ccu::aligned(status_dev, 4) ||
      !ccu::aligned(bitmap_scratch, 4))
    return ccu::fail(CCU_ERR_INVALID_ARGUMENT, "indices, bitmap_scratch and status_dev must be 4-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  const int64_t bytes = ccu_conv1d_check_indices_scratch_bytes(S);
  if (bytes > 0) e = cudaMemsetAsync(bitmap_scratch, 0, (size_t)bytes, s);
  if (e == cudaSuccess) e = ccu::launch_check_indices(indices, N, S, bitmap_scratch, status_dev, s);
  if (e != cudaSuccess)
    return ccu::fail(CCU_ERR_CUDA, "index check failed to launch: %s", cudaGetErrorString(e));
  return CCU_OK;
}

const char *ccu_status_string(ccu_status_t status) {
  switch (status) {
    case CCU_OK: return "ok";
    case CCU_ERR_INVALID_ARGUMENT: return "invalid argument (contract violation)";
    case CCU_ERR_NOT_IMPLEMENTED: return "not implemented (valid but not served)";
    case CCU_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

const char *ccu_route_name(int32_t route) {
  switch (route) {
    case CCU_ROUTE_AUTO: return "auto";
    case CCU_ROUTE_SCALAR: return "scalar";
    case CCU_ROUTE_VECTOR: return "vector";
    case CCU_ROUTE_STAGED: return "staged";
    case CCU_ROUTE_BULK: return "bulk";
    default: return "unknown";
  }
}

ccu_status_t ccu_conv1d_take_device_error(int32_t *bits) {
  ccu::g_last_error[0] = '\0';
  if (bits == nullptr) return ccu::fail(CCU_ERR_INVALID_ARGUMENT, "bits must not be NULL");
  cudaError_t e = ccu::take_async_error(bits);
  if (e != cudaSuccess)
    return ccu::fail(CCU_ERR_CUDA, "reading the device error word failed: %s", cudaGetErrorString(e));
  return CCU_OK;
}

const char *ccu_conv1d_last_error(void) { return ccu::g_last_error; }

int32_t ccu_conv1d_abi_version(void) { return CCU_CONV1D_ABI_VERSION; }

}  // extern "C"
