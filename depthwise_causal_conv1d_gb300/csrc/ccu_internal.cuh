// Internal declarations shared by the C-ABI host code and the kernels.
//
// The operation is the decode update of the cuDNN page "Causal Conv1d Decode Update"
// (introduction, update block); the argument contract is documented in ccu_conv1d.h.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ccu {

// The widest filter served (the page's native width, "Current native implementation");
// widths 2 and 3 are served too. Kernels tuned for the large batch are width four only.
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
  const int32_t *seqlens; // [N] cache_seqlens (ring-buffer state) or nullptr (linear state)
  uint16_t *out;          // [N, D]
  int32_t *status;        // nullptr: unchecked; else device error word (range check on)
  int32_t *owner;         // nullptr, or [S] slot owners (checked mode: duplicate check on)
  int64_t N, D, S, L, W;  // W: filter width (2, 3 or 4)
  int64_t ss, sd, sl;     // element strides of the state (used by the scalar kernel)
  int layout;             // Layout
  int rows_per_cta;       // rows each CTA walks (vector kernels)
};

// The extra arguments of the multi-token update (x[N, D, T] and out[N, D, T] by element
// strides; intermediate_states [N, T, D, L] compact, or nullptr).
struct MultiParams {
  int64_t T;
  int64_t sxn, sxd, sxt;
  int64_t son, sod, sot;
  uint16_t *inter;
};

// The arguments of the full-sequence prefill beyond UpdateParams (x, w, bias, out, D, L):
// x / out [B, D, T] and the optional initial / final states [B, D, L] by element strides.
struct PrefillParams {
  int64_t B, T, chunk;  // chunk: tokens per thread
  int64_t sxb, sxd, sxt;
  int64_t sob, sod, sot;
  const uint16_t *init;  // nullptr: the inputs before the sequence are zero
  int64_t sib, sid, sil;
  uint16_t *fin;         // nullptr: no final state
  int64_t sfb, sfd, sfl;
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

// PTX approximations (documented in the PTX ISA: ex2.approx has a relative error of about
// 2^-22 over the normal range, rcp.approx about one float ulp), flushing subnormals.
__device__ __forceinline__ float ex2_approx_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx_ftz(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The activation, a compile-time choice: identity kernels carry no SiLU code.
// SiLU is a * sigmoid(a) with sigmoid(a) = 1 / (1 + exp(-a)). In float, exp(-a) overflows
// below a ~ -88.7, where a * sigmoid(a) is still a representable float (a version that
// returned -0 there failed the extreme-value parity test). So the exponential is taken
// scaled down by 2^32,
//   v = 2^(-a log2 e - 32) = exp(-a) 2^-32           finite down to a ~ -110.9,
//   sigmoid(a) = 2^-32 / (v + 2^-32) = rcp(v + 2^-32) * 2^-32,
// with ex2.approx and rcp.approx. For a > ~65, v flushes to zero and sigmoid is exactly 1, so
// nothing overflows for any finite a. Below a ~ -87.3 the final multiply makes sigmoid a
// float subnormal, with an absolute error under 1e-45, far below the ~9e-41 BF16 subnormal
// step that a * sigmoid(a) is rounded to; below a ~ -103 it is 0, and a * sigmoid(a) rounds
// to -0 in BF16 anyway. Elsewhere the error is a few float ulps, far below the half BF16 ulp
// (2^15 float ulps) the result keeps, so the rounded output stays within one BF16 ulp of
// the exact value. Six operations (four a channel in the paired form below): the kernels
// that move 4 bytes per element are issue-bound on the SiLU.
template <int ACT>
__device__ __forceinline__ float activate(float a) {
  if constexpr (ACT == 1) {
    const float v = ex2_approx_ftz(fmaf(a, -1.4426950408889634f, -32.0f));
    return a * (rcp_approx_ftz(v + 0x1p-32f) * 0x1p-32f);
  } else {
    return a;
  }
}

// The same SiLU on a pair of channels: the multiplies and adds go through the paired FP32
// instructions (two IEEE operations each, rounded exactly as the scalar ones), so the result
// equals activate<ACT> on each half bit for bit.
template <int ACT>
__device__ __forceinline__ float2 activate2(float2 a) {
  if constexpr (ACT == 1) {
    const float2 t = __ffma2_rn(a, make_float2(-1.4426950408889634f, -1.4426950408889634f),
                                make_float2(-32.0f, -32.0f));
    const float2 d = __fadd2_rn(make_float2(ex2_approx_ftz(t.x), ex2_approx_ftz(t.y)),
                                make_float2(0x1p-32f, 0x1p-32f));
    const float2 sig = __fmul2_rn(make_float2(rcp_approx_ftz(d.x), rcp_approx_ftz(d.y)),
                                  make_float2(0x1p-32f, 0x1p-32f));
    return __fmul2_rn(a, sig);
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

// ---------------------------------------------------------------------------------------
// Programmatic dependent launch. Every kernel of the library is launched by
// launch_overlapped, with programmatic stream serialization: the hardware may schedule its
// CTAs while the previous kernel on the stream is still finishing. The first statement of
// every kernel is grid_dependency_boundary(): griddepcontrol.wait holds the CTA until all
// prior grids on the stream have completed and their memory is visible, so no global
// access overlaps earlier work and the stream order is the same as for a plain launch;
// griddepcontrol.launch_dependents then lets the next kernel's CTAs be scheduled as soon
// as every CTA of this grid has started (so they can never hold resources this grid still
// needs). What overlaps is the launch and CTA start-up of the next call: on the large-batch
// decode, 162.9 -> 160.5 us per call back to back, and 13.8 -> 11.3 us at 256 rows.
__device__ __forceinline__ void grid_dependency_boundary() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Duplicate check: row n claims slot s in owner[] (zeroed before the launch), which then
// holds n + 1 for good. Every thread, CTA and slice working on row n may call this; all of
// them get the same answer: true if row n owns the slot (it claimed it first), false if
// another row did. The owner word is read from L2 first, so only the first claims of a slot
// are atomic operations.
__device__ __forceinline__ bool claim_slot(int32_t *owner, int64_t s, int64_t n) {
  const int32_t me = (int32_t)(n + 1);
  int32_t v = __ldcg(owner + s);
  if (v == 0) {
    v = atomicCAS(owner + s, 0, me);
    if (v == 0) return true;
  }
  return v == me;
}

// Slot of row n, or -1 for "no state access" (a padding row; in checked mode also a slot
// out of range, which raises CCU_DEVERR_RANGE in *status, and with the duplicate check a
// slot another row has claimed, which raises CCU_DEVERR_DUPLICATE). DEDUP = false leaves
// the duplicate check out of the code (kernels whose entry points never turn it on: the
// multi-token update, whose two-row form spilled 164 instead of 72 bytes with it).
template <bool DEDUP = true>
__device__ __forceinline__ int64_t resolve_slot(const UpdateParams &p, int64_t n) {
  if (p.idx == nullptr) return n;
  int64_t s = __ldg(p.idx + n);
  if (p.status != nullptr && (s < -1 || s >= p.S)) {
    atomicOr(p.status, 1);  // CCU_DEVERR_RANGE
    return -1;
  }
  if constexpr (DEDUP) {
    if (p.owner != nullptr && s >= 0 && !claim_slot(p.owner, s, n)) {
      atomicOr(p.status, 2);  // CCU_DEVERR_DUPLICATE
      return -1;
    }
  }
  return s;
}

__device__ __forceinline__ uint32_t get16(const uint32_t *w, int pos) {
  return (w[pos >> 1] >> ((pos & 1) * 16)) & 0xffffu;
}

// The SiLU (or identity) of 8 channel sums on channel pairs (activate2, bit-identical to
// the scalar form in fewer instructions), packed to BF16. For kernels whose arithmetic is
// not hidden behind memory traffic: the multi-token update took 84.2 against 86.0 us on its
// N=1024, D=16384, T=4 workload with it, and 1-2 % less on every shape measured.
template <int ACT>
__device__ __forceinline__ uint4 activate_pairs8(const float (&a)[8]) {
  uint32_t y[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = activate2<ACT>(make_float2(a[2 * i], a[2 * i + 1]));
    y[i] = pack_bf16x2(v.x, v.y);
  }
  return make_uint4(y[0], y[1], y[2], y[3]);
}

// The update of 8 consecutive channels whose compact state [8][L] sits in 4*L words `ow`
// (two BF16 per word, flat position c*L + l) and whose inputs sit in 4 words `xw`:
//   out[c]      = act(sum_{j<W} h_c[L+1-W+j] * w[c][j] + bias[c]),  h_c = (state[c][0..L-1], x[c])
//   new state   = state[c][1..L-1] followed by x[c]   (written to `nw`, same packing)
// `wv` holds weight[8][W] (4*W of its 16 words), `bv` bias[8] (4 words). Returns the
// packed outputs. PAIRED: the activation through activate_pairs8.
template <int L, int W, int ACT, bool PAIRED = false>
__device__ __forceinline__ uint4 update8_compact(const uint32_t (&xw)[4], const uint32_t (&ow)[4 * L],
                                                 const uint32_t (&wv)[16], const uint32_t (&bv)[4],
                                                 bool has_bias, uint32_t (&nw)[4 * L]) {
  float y[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    float acc = 0.0f;
#pragma unroll
    for (int j = 0; j < W; ++j) {
      const int hidx = L - (W - 1) + j;  // index into the L + 1 history entries
      const uint32_t h = (hidx == L) ? get16(xw, c) : get16(ow, c * L + hidx);
      acc = __fmaf_rn(bf16_bits(h), bf16_bits(get16(wv, c * W + j)), acc);
    }
    if (has_bias) acc = acc + bf16_bits(get16(bv, c));
    y[c] = PAIRED ? acc : activate<ACT>(acc);
  }
#pragma unroll
  for (int i = 0; i < 4 * L; ++i) {
    const int e0 = 2 * i, e1 = 2 * i + 1;  // flat positions c*L + l
    const uint32_t v0 = (e0 % L == L - 1) ? get16(xw, e0 / L) : get16(ow, e0 + 1);
    const uint32_t v1 = (e1 % L == L - 1) ? get16(xw, e1 / L) : get16(ow, e1 + 1);
    nw[i] = v0 | (v1 << 16);
  }
  if constexpr (PAIRED) return activate_pairs8<ACT>(y);
  return make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                    pack_bf16x2(y[6], y[7]));
}

// Slot of row n and, for a ring-buffer state, the ring position of its oldest entry:
// q = cache_seqlens[n] mod L (taken non-negative, so every access stays inside the slot
// whatever the value). In checked mode a negative cache_seqlens of a non-padding row
// raises CCU_DEVERR_RANGE and the row is treated as padding.
struct RowSlot {
  int64_t s;
  int q;
};

// The cache_seqlens load is issued together with the index load (every row has an entry,
// and it does not depend on the slot), so a ring row waits for one round of loads before
// its state address is known, not two. LC: L known at compile time (0: use p.L).
template <int LC = 0, bool DEDUP = true>
__device__ __forceinline__ RowSlot resolve_row(const UpdateParams &p, int64_t n) {
  RowSlot r;
  const int32_t v = p.seqlens != nullptr ? __ldg(p.seqlens + n) : 0;
  r.s = resolve_slot<DEDUP>(p, n);
  r.q = 0;
  if (r.s >= 0 && p.seqlens != nullptr) {
    if (v < 0 && p.status != nullptr) {
      atomicOr(p.status, 1);  // CCU_DEVERR_RANGE
      r.s = -1;
    } else if constexpr (LC > 0) {
      const int m = v % LC;
      r.q = m < 0 ? m + LC : m;
    } else {
      const int64_t m = (int64_t)v % p.L;
      r.q = (int)(m < 0 ? m + p.L : m);
    }
  }
  return r;
}

// The duplicate check of a row whose slot resolved without it (resolve_row<LC, false>),
// made after the row's loads have been issued so that its latency overlaps theirs: if
// another row owns the slot, the row becomes a padding row (the loaded values are dropped:
// output +0, no state written; the reads stayed inside the range-checked slot).
__device__ __forceinline__ void drop_if_duplicate(const UpdateParams &p, int64_t n, RowSlot &r) {
  if (p.owner != nullptr && r.s >= 0 && !claim_slot(p.owner, r.s, n)) {
    atomicOr(p.status, 2);  // CCU_DEVERR_DUPLICATE
    r.s = -1;
  }
}

// The lanes of the calling thread's warp whose 8-channel group g is below `groups` (the
// others exit early in the vector kernels).
__device__ __forceinline__ unsigned live_lanes(int64_t groups) {
  const int64_t first = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31);
  const int64_t live = groups - first;
  return live >= 32 ? 0xffffffffu : ((1u << live) - 1u);
}

// drop_if_duplicate for the vector kernels, whose warps work on one row at a time and whose
// lanes past the last 8-channel group (p.D / 8) have exited: lane 0 claims the slot for the
// whole warp and passes the answer to the live lanes (lane 0 is always one of them), so a
// row costs one claim per warp rather than one per thread (at N=4096, D=16384 per-thread
// claims made the checked update 45 % slower).
__device__ __forceinline__ void drop_if_duplicate_warp(const UpdateParams &p, int64_t n, RowSlot &r) {
  if (p.owner == nullptr || r.s < 0) return;  // the same for every lane: one row per warp
  const unsigned live = live_lanes(p.D >> 3);
  int own = 1;
  if ((threadIdx.x & 31) == 0) {
    own = claim_slot(p.owner, r.s, n) ? 1 : 0;
    if (!own) atomicOr(p.status, 2);  // CCU_DEVERR_DUPLICATE
  }
  if (!__shfl_sync(live, own, 0)) r.s = -1;
}

// The ring-buffer form of update8_compact for a ring position Q known at compile time:
// the 8 channels' rings sit in `ow` (flat position c*L + l) and Q is the ring position of
// the oldest entry. The history, oldest first, is ring[Q], ring[Q+1], ..., ring[Q+L-1]
// (mod L) followed by x, so the width-W window is ring[(Q+L-(W-1)+k) % L] for
// k = 0..W-2, then x. The new rings in `nw` equal the old ones with entry Q replaced by x.
template <int L, int W, int ACT, int Q, bool PAIRED = false>
__device__ __forceinline__ uint4 update8_ring_q(const uint32_t (&xw)[4], const uint32_t (&ow)[4 * L],
                                                const uint32_t (&wv)[16], const uint32_t (&bv)[4],
                                                bool has_bias, uint32_t (&nw)[4 * L]) {
  float y[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    float acc = 0.0f;
#pragma unroll
    for (int k = 0; k < W - 1; ++k) {
      const uint32_t h = get16(ow, c * L + (Q + L - (W - 1) + k) % L);
      acc = __fmaf_rn(bf16_bits(h), bf16_bits(get16(wv, c * W + k)), acc);
    }
    acc = __fmaf_rn(bf16_bits(get16(xw, c)), bf16_bits(get16(wv, c * W + W - 1)), acc);
    if (has_bias) acc = acc + bf16_bits(get16(bv, c));
    y[c] = PAIRED ? acc : activate<ACT>(acc);
  }
#pragma unroll
  for (int i = 0; i < 4 * L; ++i) {
    const int e0 = 2 * i, e1 = 2 * i + 1;
    const uint32_t v0 = (e0 % L == Q) ? get16(xw, e0 / L) : get16(ow, e0);
    const uint32_t v1 = (e1 % L == Q) ? get16(xw, e1 / L) : get16(ow, e1);
    nw[i] = v0 | (v1 << 16);
  }
  if constexpr (PAIRED) return activate_pairs8<ACT>(y);
  return make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                    pack_bf16x2(y[6], y[7]));
}

// Runtime ring position q in [0, L): one branch to the matching compile-time form (q is
// the same for every lane of a row, so the branch does not diverge within a row).
template <int L, int W, int ACT, bool PAIRED = false>
__device__ __forceinline__ uint4 update8_compact_ring(const uint32_t (&xw)[4], const uint32_t (&ow)[4 * L],
                                                      const uint32_t (&wv)[16], const uint32_t (&bv)[4],
                                                      bool has_bias, int q, uint32_t (&nw)[4 * L]) {
  switch (q) {
    case 0: return update8_ring_q<L, W, ACT, 0, PAIRED>(xw, ow, wv, bv, has_bias, nw);
    case 1: return update8_ring_q<L, W, ACT, 1 % L, PAIRED>(xw, ow, wv, bv, has_bias, nw);
    case 2: return update8_ring_q<L, W, ACT, 2 % L, PAIRED>(xw, ow, wv, bv, has_bias, nw);
    case 3: return update8_ring_q<L, W, ACT, 3 % L, PAIRED>(xw, ow, wv, bv, has_bias, nw);
    case 4: return update8_ring_q<L, W, ACT, 4 % L, PAIRED>(xw, ow, wv, bv, has_bias, nw);
    case 5: return update8_ring_q<L, W, ACT, 5 % L, PAIRED>(xw, ow, wv, bv, has_bias, nw);
    case 6: return update8_ring_q<L, W, ACT, 6 % L, PAIRED>(xw, ow, wv, bv, has_bias, nw);
    default: return update8_ring_q<L, W, ACT, 7 % L, PAIRED>(xw, ow, wv, bv, has_bias, nw);
  }
}

// Outputs of 8 channels from the W-1 window entries before x (h[k][c], k < W-1) and x
// (xs[c]); weight[8][W] packed in wv.
template <int W, int ACT>
__device__ __forceinline__ uint4 outputs8_window(const uint32_t (&h)[3][8], const uint32_t (&xs)[8],
                                                 const uint32_t (&wv)[16], const uint32_t (&bv)[4],
                                                 bool has_bias) {
  float y[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    float acc = 0.0f;
#pragma unroll
    for (int k = 0; k < W - 1; ++k)
      acc = __fmaf_rn(bf16_bits(h[k][c]), bf16_bits(get16(wv, c * W + k)), acc);
    acc = __fmaf_rn(bf16_bits(xs[c]), bf16_bits(get16(wv, c * W + W - 1)), acc);
    if (has_bias) acc = acc + bf16_bits(get16(bv, c));
    y[c] = activate<ACT>(acc);
  }
  return make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                    pack_bf16x2(y[6], y[7]));
}

// Load weight[c0 .. c0+7, 0..W-1]: 8*W BF16 = W 16-byte vectors, packed two per word.
template <int W>
__device__ __forceinline__ void load_weights_packed(const uint16_t *w, int64_t c0, uint32_t (&wv)[16]) {
  const uint16_t *wp = w + c0 * W;
#pragma unroll
  for (int k = 0; k < W; ++k) {
    const uint4 t = __ldg(reinterpret_cast<const uint4 *>(wp + 8 * k));
    wv[4 * k] = t.x; wv[4 * k + 1] = t.y; wv[4 * k + 2] = t.z; wv[4 * k + 3] = t.w;
  }
#pragma unroll
  for (int k = W; k < 4; ++k) wv[4 * k] = wv[4 * k + 1] = wv[4 * k + 2] = wv[4 * k + 3] = 0u;
}

// Unpack a 16-byte vector of 8 BF16 into 8 raw 16-bit values.
__device__ __forceinline__ void unpack8(const uint4 v, uint32_t (&e)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    e[2 * i] = w[i] & 0xffffu;
    e[2 * i + 1] = w[i] >> 16;
  }
}

// ---------------------------------------------------------------------------------------
// Width-4 arithmetic on channel pairs (the prefill and the multi-token update): 8 channels
// as 4 float pairs, the window sums and the SiLU through the paired FP32 instructions.

// Widen 8 packed BF16 to 4 float pairs (channels 2i, 2i+1).
__device__ __forceinline__ void widen8(const uint4 v, float2 (&f)[4]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) f[i] = make_float2(bf16_lo(w[i]), bf16_hi(w[i]));
}

// The width-W weights of channels c0..c0+7 as float pairs: wf[j][i] = weight[c0 + 2i (+1), j]
// for j < W (taps j >= W are zero and unused).
template <int W = kW>
__device__ __forceinline__ void load_weights_f(const uint16_t *w, int64_t c0, float2 (&wf)[kW][4]) {
  if constexpr (W == kW) {
    const uint16_t *wp = w + c0 * kW;
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // 16 bytes = channels 2k, 2k+1, all four taps each
      const uint4 t = ld_keep(wp + 8 * k);
      wf[0][k] = make_float2(bf16_lo(t.x), bf16_lo(t.z));
      wf[1][k] = make_float2(bf16_hi(t.x), bf16_hi(t.z));
      wf[2][k] = make_float2(bf16_lo(t.y), bf16_lo(t.w));
      wf[3][k] = make_float2(bf16_hi(t.y), bf16_hi(t.w));
    }
  } else {
    uint32_t wv[16];
    load_weights_packed<W>(w, c0, wv);
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int j = 0; j < kW; ++j)
        wf[j][k] = j < W ? make_float2(bf16_bits(get16(wv, (2 * k) * W + j)), bf16_bits(get16(wv, (2 * k + 1) * W + j)))
                         : make_float2(0.0f, 0.0f);
  }
}

// Outputs of 8 channels (4 pairs) for one token from the window a, b, c (oldest first) and
// the token's inputs x. The accumulation order is the update's: width 4 ((0 + a*w0) + b*w1)
// + c*w2 + x*w3, width 3 (0 + b*w0) + c*w1 + x*w2, width 2 (0 + c*w0) + x*w1, then the bias
// (each product of two BF16 values is exact in FP32); the paired FP32 instructions round each
// half exactly as the scalar ones.
template <int ACT, int W = kW>
__device__ __forceinline__ uint4 outputs8f(const float2 (&wf)[kW][4], const float2 (&bf)[4],
                                           bool has_bias, const float2 (&a)[4], const float2 (&b)[4],
                                           const float2 (&c)[4], const float2 (&x)[4]) {
  uint32_t y[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 acc;
    if constexpr (W == 4) {
      acc = __ffma2_rn(a[i], wf[0][i], make_float2(0.0f, 0.0f));
      acc = __ffma2_rn(b[i], wf[1][i], acc);
      acc = __ffma2_rn(c[i], wf[2][i], acc);
      acc = __ffma2_rn(x[i], wf[3][i], acc);
    } else if constexpr (W == 3) {
      acc = __ffma2_rn(b[i], wf[0][i], make_float2(0.0f, 0.0f));
      acc = __ffma2_rn(c[i], wf[1][i], acc);
      acc = __ffma2_rn(x[i], wf[2][i], acc);
    } else {
      acc = __ffma2_rn(c[i], wf[0][i], make_float2(0.0f, 0.0f));
      acc = __ffma2_rn(x[i], wf[1][i], acc);
    }
    if (has_bias) acc = __fadd2_rn(acc, bf[i]);
    const float2 v = activate2<ACT>(acc);
    y[i] = pack_bf16x2(v.x, v.y);
  }
  return make_uint4(y[0], y[1], y[2], y[3]);
}

// The window slides by one token: (h0, h1, h2) <- (h1, h2, x).
__device__ __forceinline__ void slide(float2 (&h0)[4], float2 (&h1)[4], float2 (&h2)[4],
                                      const float2 (&x)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h0[i] = h1[i];
    h1[i] = h2[i];
    h2[i] = x[i];
  }
}

// ---------------------------------------------------------------------------------------
// Kernel launchers (one per family). Each returns the cudaError_t of its launch.

cudaError_t launch_scalar(const UpdateParams &p, int act, cudaStream_t stream);
cudaError_t launch_vector(const UpdateParams &p, int act, cudaStream_t stream);
cudaError_t launch_staged(const UpdateParams &p, int act, cudaStream_t stream);
cudaError_t launch_bulk(const UpdateParams &p, int act, cudaStream_t stream);
cudaError_t launch_bulk_planes(const UpdateParams &p, int act, cudaStream_t stream);
cudaError_t take_planes_error(int32_t *bits);
// Sets the calling thread's message returned by ccu_conv1d_last_error.
void record_error(const char *msg);
// Reads and clears the device error word that kernels without a status word report into.
cudaError_t take_async_error(int32_t *bits);
cudaError_t launch_multi_scalar(const UpdateParams &p, const MultiParams &m, int act,
                                cudaStream_t stream);
cudaError_t launch_multi_vector(const UpdateParams &p, const MultiParams &m, int act,
                                cudaStream_t stream);
cudaError_t launch_prefill(const UpdateParams &p, const PrefillParams &f, int act, bool vector,
                           cudaStream_t stream);
// Bulk-copy prefill (width 4, channel-contiguous x and out); sets the run length itself.
cudaError_t launch_prefill_bulk(const UpdateParams &p, const PrefillParams &f, int act,
                                cudaStream_t stream);
cudaError_t take_prefill_error(int32_t *bits);
// Bulk-copy multi-token update (compact state, width 4, L = 3..8, T <= kMultiBulkMaxT, no
// intermediate states, x and out in device memory with channel-contiguous token rows).
cudaError_t launch_multi_bulk(const UpdateParams &p, const MultiParams &m, int act, cudaStream_t stream);
cudaError_t take_multi_bulk_error(int32_t *bits);
// Zeroes n words on the stream as a kernel in the overlapped launch sequence (k_scalar.cu).
cudaError_t launch_clear_words(int32_t *w, int64_t n, cudaStream_t stream);
cudaError_t launch_check_indices(const int32_t *idx, int64_t N, int64_t S, uint32_t *bitmap,
                                 int32_t *status, cudaStream_t stream);

// CCU_DEVERR_TIMEOUT: a bounded wait inside a kernel gave up.
constexpr int32_t kDevErrTimeout = 4;
// Largest L the register-resident vector and bulk kernels are compiled for.
constexpr int64_t kVectorMaxL = 8;
// Most tokens per row the bulk-copy multi-token kernel takes.
constexpr int64_t kMultiBulkMaxT = 8;
// Largest L the shared-memory staged kernel accepts.
constexpr int64_t kStagedMaxL = 256;

}  // namespace ccu
