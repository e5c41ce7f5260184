// The vector kernel family (instantiated in k_vector.cu and k_vector_checked.cu): each
// thread owns 8 consecutive channels of one row at a time and moves x, state and out as
// 16-byte vectors. L (W-1..8), the width W (2..4), the state layout,
// linear or ring state and the activation are compile-time, so the history lives in
// registers and the shift is a fixed permutation of 16-bit lanes.
//
// What sets this kernel's speed is the number of bytes in flight per SM, and that grows
// with the warps an SM can hold, so a thread keeps as little as it can in registers: its
// row's x and state. The weights and bias of its 8 channels sit in shared memory, written
// once per CTA, one 16-byte vector per channel pair, laid out [pair][thread] so that a
// warp's reads are conflict-free; they are read pair by pair while the outputs are formed.
// At L = 3 that is 48 registers a thread and five CTAs of 8 warps per SM. Measured on the
// large batch (N=4096, D=16384, L=3, SiLU): 155.9 us, against 162.4 us with the weights in
// registers (110 registers, two CTAs per SM) and 160.3 us for the bulk-copy kernel; at
// N=1024, 41.9 us against 45.3 us for both.
//
// Update definition: cuDNN page "Causal Conv1d Decode Update", introduction (update
// block); layouts from its "Semantic tensor contract" (compact state, and the
// channel-last (L*D, 1, D) state a full-sequence prefill hands over).
#pragma once

#include <type_traits>

#include "ccu_internal.cuh"

namespace ccu {

int device_sm_count();
cudaError_t launch_lanes(const UpdateParams &p, int act, cudaStream_t stream);

namespace {

constexpr int kThreads = 256;

// The weights and bias of a CTA's channels: for thread t (channels c0 .. c0+7), w[k][t]
// holds the taps of channels c0+2k (words 0, 1) and c0+2k+1 (words 2, 3), tap j in half j
// of word j/2 of its channel (taps j >= W are zero), and b[k][t] their bias (low, high).
struct PairTables {
  uint4 w[4][kThreads];
  uint32_t b[4][kThreads];
};

// The pair vectors of channels c0 .. c0+7 (the layout of PairTables) and their bias words.
template <int W>
__device__ __forceinline__ void pair_weights(const UpdateParams &p, int64_t c0, uint4 (&wp)[4], uint32_t (&bp)[4]) {
  if constexpr (W == kW) {  // weight[D, 4]: 16 bytes are exactly two channels' taps
#pragma unroll
    for (int k = 0; k < 4; ++k) wp[k] = ld_keep(p.w + c0 * kW + 8 * k);
  } else {
    uint32_t wv[16];
    load_weights_packed<W>(p.w, c0, wv);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t q[4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = 2 * k + h;
        uint32_t tap[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) tap[j] = j < W ? get16(wv, c * W + j) : 0u;
        q[2 * h] = tap[0] | (tap[1] << 16);
        q[2 * h + 1] = tap[2] | (tap[3] << 16);
      }
      wp[k] = make_uint4(q[0], q[1], q[2], q[3]);
    }
  }
  const uint4 b = p.bias != nullptr ? ld_keep(p.bias + c0) : make_uint4(0u, 0u, 0u, 0u);
  bp[0] = b.x;
  bp[1] = b.y;
  bp[2] = b.z;
  bp[3] = b.w;
}

// The outputs of the 8 channels: hist(c, j) is the history entry tap j of channel c
// multiplies (entry L + 1 - W + j of the L + 1 entries; hist(c, W - 1) is x); wsrc(k) and
// bsrc(k) give pair k's weight vector and bias word. The products are summed in ascending
// j with FP32 fused multiply-adds (each BF16 x BF16 product is exact in FP32), then the
// bias, then the activation, rounded to BF16 and packed.
template <int W, int ACT, typename Hist, typename WSrc, typename BSrc>
__device__ __forceinline__ uint4 outputs8(Hist hist, WSrc wsrc, BSrc bsrc, bool has_bias) {
  uint32_t y[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint4 wk = wsrc(k);
    const uint32_t wa[4] = {wk.x, wk.y, wk.z, wk.w};
    const uint32_t bk = has_bias ? bsrc(k) : 0u;
    float v[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = 2 * k + h;
      float acc = 0.0f;
#pragma unroll
      for (int j = 0; j < W; ++j)
        acc = __fmaf_rn(bf16_bits(hist(c, j)), bf16_bits(get16(wa, 4 * h + j)), acc);
      if (has_bias) acc = acc + bf16_bits((bk >> (16 * h)) & 0xffffu);
      v[h] = activate<ACT>(acc);
    }
    y[k] = pack_bf16x2(v[0], v[1]);
  }
  return make_uint4(y[0], y[1], y[2], y[3]);
}

// Words of state a thread holds per row: compact 4L (8 channels x L entries); channel-last
// linear 4L (plane l in words 4l .. 4l+3; plane 0 only when it is in the window);
// channel-last ring: the W - 1 window planes.
template <int L, int W, int LAYOUT, bool RING>
__host__ __device__ constexpr int state_words() {
  return (LAYOUT == (int)Layout::ChannelLast && RING) ? 4 * (W - 1) : 4 * L;
}

// How an instance runs: rif rows' loads issued per thread before the first of them is
// computed; minb resident CTAs per SM the register budget is set for (__launch_bounds__;
// 1 leaves the budget to the compiler); wreg: update_vector_regs (weights and bias held in
// registers for all of a CTA's rows) instead of the lean form.
struct VecCfg {
  int rif, minb;
  bool wreg;
};

// The lean form (one row in flight, weights in shared memory) at an occupancy set by the
// registers it needs: about 32 of addresses and temporaries plus the row's x and state, and
// 16 more for the compact ring form, whose branch over the ring position keeps more values
// live (at the plain budget it spilled 8 to 16 bytes).
template <int L, int W, int LAYOUT, bool RING>
__host__ __device__ constexpr int lean_min_ctas() {
  constexpr int need =
      32 + 4 + state_words<L, W, LAYOUT, RING>() + ((RING && LAYOUT == (int)Layout::Compact) ? 16 : 0);
  return need <= 48 ? 5 : (need <= 64 ? 4 : (need <= 80 ? 3 : 2));
}

// Measured at N=4096, D=16384 (us, lean form / weights in registers with two rows in
// flight): compact L = 3 155.6 / 162.4, compact ring L = 3 160.5 / 165.0, channel-last L = 3
// 154.3 / 157.3, channel-last ring 125.9 / 125.2 (N=1024: 32.2 / 34.6), W = 3 at L = 3
// 154.2 / 165.4, L = 5 237.8 / 242.1; but L = 4 211.1 / 201.0, W = 2 at L = 1 88.9 / 80.4
// and W = 3 at L = 2 117.5 / 116.5. The
// second form runs at four CTAs per SM for L = 1 (64 registers), three for L = 2 (85; at
// W = 3, L = 2: 118.6 us against 130.7 us with the compiler's budget) and two at L = 4. The
// compact linear state at L = 8 runs on neither (see launch_LW).
template <int L, int W, int LAYOUT, bool RING>
__host__ __device__ constexpr VecCfg vec_cfg() {
  constexpr bool compact_linear = LAYOUT == (int)Layout::Compact && !RING;
  constexpr bool keep_regs = compact_linear && (L == 4 || (L == W - 1 && W < 4));
  if constexpr (keep_regs) return VecCfg{2, L == 1 ? 4 : (L == 2 ? 3 : 2), true};
  return VecCfg{1, lean_min_ctas<L, W, LAYOUT, RING>(), false};
}

// The lean form: weights and bias from the CTA's shared-memory tables. TWO_ROWS: two rows'
// loads in flight per thread (the small-batch form, see launch_one).
template <int L, int W, int ACT, int LAYOUT, bool RING, bool DEDUP, bool TWO_ROWS>
__device__ __forceinline__ void update_vector(const UpdateParams &p, PairTables &tab) {
  constexpr VecCfg cfg = vec_cfg<L, W, LAYOUT, RING>();
  const int t = threadIdx.x;
  const int64_t groups = p.D >> 3;  // 8-channel groups per row (D % 8 == 0)
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + t;
  const int64_t c0 = g << 3;
  const bool has_bias = p.bias != nullptr;
  if (g < groups) {
    uint4 wr[4];
    uint32_t br[4];
    pair_weights<W>(p, c0, wr, br);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      tab.w[k][t] = wr[k];
      tab.b[k][t] = br[k];
    }
  }
  __syncthreads();
  if (g >= groups) return;
  auto wsrc = [&](int k) -> uint4 { return tab.w[k][t]; };
  auto bsrc = [&](int k) -> uint32_t { return tab.b[k][t]; };

  constexpr bool kPlanes = (LAYOUT == (int)Layout::ChannelLast);
  constexpr int kWords = state_words<L, W, LAYOUT, RING>();
  struct Row {
    RowSlot slot;
    uint32_t xw[4];
    uint32_t ow[kWords];
  };

  auto load_row = [&](int64_t n, Row &r) {
    r.slot = resolve_row<L, false>(p, n);  // the duplicate check follows the loads
    if (r.slot.s < 0) return;
    const uint4 xv = ld_stream(p.x + n * p.ld + c0);
    r.xw[0] = xv.x; r.xw[1] = xv.y; r.xw[2] = xv.z; r.xw[3] = xv.w;
    if constexpr (!kPlanes) {
      const uint16_t *sp = p.state + r.slot.s * (p.D * L) + c0 * L;
#pragma unroll
      for (int k = 0; k < L; ++k) {
        const uint4 u = ld_stream(sp + 8 * k);
        r.ow[4 * k] = u.x; r.ow[4 * k + 1] = u.y; r.ow[4 * k + 2] = u.z; r.ow[4 * k + 3] = u.w;
      }
    } else if constexpr (RING) {
      const uint16_t *sp = p.state + r.slot.s * (L * p.D) + c0;
#pragma unroll
      for (int k = 0; k < W - 1; ++k) {
        const uint4 u = ld_stream(sp + (int64_t)((r.slot.q + L - (W - 1) + k) % L) * p.D);
        r.ow[4 * k] = u.x; r.ow[4 * k + 1] = u.y; r.ow[4 * k + 2] = u.z; r.ow[4 * k + 3] = u.w;
      }
    } else {
      // Plane 0 is read only when L == W - 1: it is then inside the window; otherwise it
      // is outside the window and is overwritten by plane 1.
      const uint16_t *sp = p.state + r.slot.s * (L * p.D) + c0;
      constexpr int first = (L == W - 1) ? 0 : 1;
#pragma unroll
      for (int l = 0; l < L; ++l) {
        if (l < first) {
          r.ow[4 * l] = r.ow[4 * l + 1] = r.ow[4 * l + 2] = r.ow[4 * l + 3] = 0u;
          continue;
        }
        const uint4 u = ld_stream(sp + (int64_t)l * p.D);
        r.ow[4 * l] = u.x; r.ow[4 * l + 1] = u.y; r.ow[4 * l + 2] = u.z; r.ow[4 * l + 3] = u.w;
      }
    }
    if constexpr (DEDUP) drop_if_duplicate_warp(p, n, r.slot);
  };

  auto store_row = [&](int64_t n, const Row &r) {
    uint16_t *outp = p.out + n * p.D + c0;
    if (r.slot.s < 0) {  // padding row: zero output, state untouched
      st_stream(outp, make_uint4(0u, 0u, 0u, 0u));
      return;
    }
    const uint32_t(&xw)[4] = r.xw;
    const uint32_t(&ow)[kWords] = r.ow;
    uint4 outv;
    if constexpr (!kPlanes) {
      uint16_t *sp = p.state + r.slot.s * (p.D * L) + c0 * L;
      // new compact state at flat position e = c*L + l: entry l+1 of channel c, or x[c] for
      // the newest entry (linear); entry l, or x[c] at the ring position q (ring)
      auto store_state = [&](auto newest_at, auto take_from) {
        uint32_t nw[4 * L];
#pragma unroll
        for (int i = 0; i < 4 * L; ++i) {
          const int e0 = 2 * i, e1 = 2 * i + 1;
          const uint32_t v0 = newest_at(e0) ? get16(xw, e0 / L) : get16(ow, take_from(e0));
          const uint32_t v1 = newest_at(e1) ? get16(xw, e1 / L) : get16(ow, take_from(e1));
          nw[i] = v0 | (v1 << 16);
        }
#pragma unroll
        for (int k = 0; k < L; ++k)
          st_stream(sp + 8 * k, make_uint4(nw[4 * k], nw[4 * k + 1], nw[4 * k + 2], nw[4 * k + 3]));
      };
      if constexpr (RING) {
        // one branch to a compile-time ring position (q is the same for the whole row)
        auto ring_q = [&](auto qc) {
          constexpr int Q = decltype(qc)::value;
          outv = outputs8<W, ACT>(
              [&](int c, int j) {
                return j == W - 1 ? get16(xw, c) : get16(ow, c * L + (Q + L - (W - 1) + j) % L);
              },
              wsrc, bsrc, has_bias);
          store_state([](int e) { return e % L == Q; }, [](int e) { return e; });
        };
        switch (r.slot.q) {
          case 0: ring_q(std::integral_constant<int, 0>()); break;
          case 1: ring_q(std::integral_constant<int, 1 % L>()); break;
          case 2: ring_q(std::integral_constant<int, 2 % L>()); break;
          case 3: ring_q(std::integral_constant<int, 3 % L>()); break;
          case 4: ring_q(std::integral_constant<int, 4 % L>()); break;
          case 5: ring_q(std::integral_constant<int, 5 % L>()); break;
          case 6: ring_q(std::integral_constant<int, 6 % L>()); break;
          default: ring_q(std::integral_constant<int, 7 % L>()); break;
        }
      } else {
        outv = outputs8<W, ACT>(
            [&](int c, int j) { return j == W - 1 ? get16(xw, c) : get16(ow, c * L + L - (W - 1) + j); }, wsrc,
            bsrc, has_bias);
        store_state([](int e) { return e % L == L - 1; }, [](int e) { return e + 1; });
      }
    } else {
      uint16_t *sp = p.state + r.slot.s * (L * p.D) + c0;
      // window planes: the ring's W-1 (held in order), or the linear state's last W-1
      constexpr int wp0 = RING ? 0 : L - (W - 1);
      outv = outputs8<W, ACT>(
          [&](int c, int j) { return j == W - 1 ? get16(xw, c) : get16(ow, 8 * (wp0 + j) + c); }, wsrc, bsrc,
          has_bias);
      if constexpr (RING) {
        st_stream(sp + (int64_t)r.slot.q * p.D, make_uint4(xw[0], xw[1], xw[2], xw[3]));
      } else {
        // plane l takes old plane l+1; the newest plane takes x
#pragma unroll
        for (int l = 0; l + 1 < L; ++l)
          st_stream(sp + (int64_t)l * p.D,
                    make_uint4(ow[4 * (l + 1)], ow[4 * (l + 1) + 1], ow[4 * (l + 1) + 2], ow[4 * (l + 1) + 3]));
        st_stream(sp + (int64_t)(L - 1) * p.D, make_uint4(xw[0], xw[1], xw[2], xw[3]));
      }
    }
    st_stream(outp, outv);
  };

  // A CTA walks R consecutive rows (rows_per_cta), rif rows' loads in flight per thread.
  // Slots are unique within a call, so one row's stores never touch another row's state.
  constexpr int RIF = TWO_ROWS ? 2 : cfg.rif;
  const int64_t R = p.rows_per_cta;
  for (int64_t r0 = (int64_t)blockIdx.y * R; r0 < p.N; r0 += (int64_t)gridDim.y * R) {
    const int64_t r1 = r0 + R < p.N ? r0 + R : p.N;
    for (int64_t n = r0; n < r1; n += RIF) {
      Row rw[RIF];
#pragma unroll
      for (int k = 0; k < RIF; ++k)
        if (n + k < r1) load_row(n + k, rw[k]);
#pragma unroll
      for (int k = 0; k < RIF; ++k)
        if (n + k < r1) store_row(n + k, rw[k]);
    }
  }
}

// The form with the weights and bias in registers (compact linear state only): a thread
// loads its channels' weights once and walks the CTA's rows two at a time, issuing both
// rows' loads (slot, x and state) before computing either (left to the compiler, the
// schedule of a single-row loop varied between builds from 168 to 303 us on the large
// batch at L = 3).
template <int L, int W, int ACT, bool DEDUP>
__device__ __forceinline__ void update_vector_regs(const UpdateParams &p) {
  const int64_t groups = p.D >> 3;
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= groups) return;
  const int64_t c0 = g << 3;
  uint32_t wv[16];  // weight[c0 .. c0+7, 0..W-1], packed two per word, widened at use
  load_weights_packed<W>(p.w, c0, wv);
  const bool has_bias = p.bias != nullptr;
  uint32_t bv[4] = {0u, 0u, 0u, 0u};
  if (has_bias) {
    const uint4 t = ld_keep(p.bias + c0);
    bv[0] = t.x; bv[1] = t.y; bv[2] = t.z; bv[3] = t.w;
  }
  struct Row {
    RowSlot slot;
    uint32_t xw[4];
    uint32_t ow[4 * L];
  };
  auto load_row = [&](int64_t n, Row &r) {
    r.slot = resolve_row<L, false>(p, n);  // the duplicate check follows the loads
    if (r.slot.s < 0) return;
    const uint4 t = ld_stream(p.x + n * p.ld + c0);
    r.xw[0] = t.x; r.xw[1] = t.y; r.xw[2] = t.z; r.xw[3] = t.w;
    const uint16_t *sp = p.state + r.slot.s * (p.D * L) + c0 * L;
#pragma unroll
    for (int k = 0; k < L; ++k) {
      const uint4 u = ld_stream(sp + 8 * k);
      r.ow[4 * k] = u.x; r.ow[4 * k + 1] = u.y; r.ow[4 * k + 2] = u.z; r.ow[4 * k + 3] = u.w;
    }
    if constexpr (DEDUP) drop_if_duplicate_warp(p, n, r.slot);
  };
  auto store_row = [&](int64_t n, const Row &r) {
    uint16_t *outp = p.out + n * p.D + c0;
    if (r.slot.s < 0) {  // padding row: zero output, state untouched
      st_stream(outp, make_uint4(0u, 0u, 0u, 0u));
      return;
    }
    uint32_t nw[4 * L];
    const uint4 outv = update8_compact<L, W, ACT>(r.xw, r.ow, wv, bv, has_bias, nw);
    uint16_t *sp = p.state + r.slot.s * (p.D * L) + c0 * L;
#pragma unroll
    for (int k = 0; k < L; ++k)
      st_stream(sp + 8 * k, make_uint4(nw[4 * k], nw[4 * k + 1], nw[4 * k + 2], nw[4 * k + 3]));
    st_stream(outp, outv);
  };
  const int64_t R = p.rows_per_cta;
  for (int64_t r0 = (int64_t)blockIdx.y * R; r0 < p.N; r0 += (int64_t)gridDim.y * R) {
    const int64_t r1 = r0 + R < p.N ? r0 + R : p.N;
    for (int64_t n = r0; n < r1; n += 2) {
      Row a, b;
      load_row(n, a);
      if (n + 1 < r1) load_row(n + 1, b);
      store_row(n, a);
      if (n + 1 < r1) store_row(n + 1, b);
    }
  }
}

// The duplicate check's warp-wide claim needs a few more registers: its instances are
// budgeted for one resident CTA fewer (at the lean form's budget they spilled up to 56 bytes).
// The two-rows-in-flight lean form holds a second row's x and state: four CTAs per SM.
template <int L, int W, bool DEDUP, int LAYOUT, bool RING, bool TWO_ROWS>
__host__ __device__ constexpr int kernel_min_ctas() {
  constexpr int m = TWO_ROWS ? 4 : vec_cfg<L, W, LAYOUT, RING>().minb;
  return (DEDUP && m > 1) ? m - 1 : m;
}

template <int L, int W, int ACT, int LAYOUT, bool RING, bool DEDUP, bool TWO_ROWS>
__global__ void __launch_bounds__(kThreads, kernel_min_ctas<L, W, DEDUP, LAYOUT, RING, TWO_ROWS>())
    k_update_vector(UpdateParams p) {
  grid_dependency_boundary();
  if constexpr (vec_cfg<L, W, LAYOUT, RING>().wreg) {
    update_vector_regs<L, W, ACT, DEDUP>(p);
  } else {
    __shared__ PairTables tab;
    update_vector<L, W, ACT, LAYOUT, RING, DEDUP, TWO_ROWS>(p, tab);
  }
}

// The small-batch two-row form is built for the compact linear state at L = 3, width 4 (at
// widths 2 and 3 it measured 2 % slower: N=256, D=8192 cold 8.18 / 8.30 against 7.98 / 8.11
// us).
template <int L, int W, int LAYOUT, bool RING>
__host__ __device__ constexpr bool two_row_form() {
  return L == 3 && W == 4 && LAYOUT == (int)Layout::Compact && !RING && !vec_cfg<L, W, LAYOUT, RING>().wreg;
}

// Rows per CTA once the batch fills the GPU. Lean form: enough that the weights a CTA
// writes into shared memory serve a few rows, few enough that CTAs stay short-lived (N=4096,
// D=16384: 155.9 us at 2.7 rows per CTA, 156.1 at 5.4, 161.0 at 10.8 and 182.6 with one
// long-lived CTA per slot; N=1024: 41.9 us at 2.7 rows, 44.8 at 1.3); the compact ring
// state takes four (158.6 against 160.4 us at three). The form with weights in registers
// keeps about 32 CTAs per SM and 4 to 8 rows each (its weights are loaded once per CTA).
template <int L, int W, int ACT, int LAYOUT, bool RING, bool DEDUP>
cudaError_t launch_one(UpdateParams p, int64_t gx, int threads, cudaStream_t stream) {
  constexpr VecCfg cfg = vec_cfg<L, W, LAYOUT, RING>();
  const int64_t sms = device_sm_count();
  const int64_t work = p.N * gx;  // (row, channel block) pairs
  int64_t R = 1;
  if constexpr (cfg.wreg) {
    R = work / (sms * 32);
    R = R > 8 ? 8 : R;
    if (R < 4) R = work >= 4 * 2 * sms ? 4 : 1;
  } else {
    // Small batches take one row per CTA: every (row, channel block) is a CTA of its own.
    // From six to eight (row, channel block) pairs per SM, the compact linear L = 3 state
    // takes two rows per CTA, both in flight, at four CTAs per SM: one wave instead of a
    // wave and a ragged second at five one-row CTAs per SM (cold, us, two rows / one row: N=256,
    // D=8192 8.51 / 9.21; N=300, D=8192 9.01 / 10.14; N=128, D=16384 8.55 / 9.09; but N=192,
    // D=8192, where one-row CTAs fit one wave, 8.16 / 7.32).
    constexpr int64_t kRows = (RING && LAYOUT == (int)Layout::Compact) ? 4 : 3;
    R = work >= 8 * sms ? kRows : 1;
    if constexpr (two_row_form<L, W, LAYOUT, RING>()) {
      if (R == 1 && work >= 6 * sms) {
        int64_t gy = (p.N + 1) / 2;
        if (gy > 65535) gy = 65535;
        p.rows_per_cta = 2;
        return launch_overlapped(k_update_vector<L, W, ACT, LAYOUT, RING, DEDUP, true>,
                                 dim3((unsigned)gx, (unsigned)gy), dim3(threads), 0, stream, p);
      }
    }
  }
  // The channel-last ring state (a row is 12 bytes an element, few registers) runs two rows
  // in flight at four CTAs per SM once the batch fills the GPU, four rows per CTA (six from
  // 16 x 8 pairs per SM). us, two rows (4 rows per CTA / 6) against one: N=4096 123.5 / 121.8
  // against 125.7 (cold 124.0 / 121.8 against 126.0), N=2048 64.2 / 64.2 against 65.5, N=1024
  // 31.4 / 31.4 against 32.1 (cold 34.9 / 35.8 against 35.4), N=512 17.3 / 18.6 against 17.6.
  // The channel-last linear state lost with it (156.3 against 154.3 us at N=4096).
  if constexpr (LAYOUT == (int)Layout::ChannelLast && RING && !cfg.wreg) {
    if (R > 1) {
      R = work >= 16 * 8 * sms ? 6 : 4;
      int64_t gy = (p.N + R - 1) / R;
      if (gy > 65535) gy = 65535;
      p.rows_per_cta = (int)R;
      return launch_overlapped(k_update_vector<L, W, ACT, LAYOUT, RING, DEDUP, true>,
                               dim3((unsigned)gx, (unsigned)gy), dim3(threads), 0, stream, p);
    }
  }
  int64_t gy = (p.N + R - 1) / R;
  if (gy > 65535) gy = 65535;  // the row loop strides over the rest
  p.rows_per_cta = (int)R;
  return launch_overlapped(k_update_vector<L, W, ACT, LAYOUT, RING, DEDUP, false>,
                           dim3((unsigned)gx, (unsigned)gy), dim3(threads), 0, stream, p);
}

// The linear compact states that run one channel per lane (k_lanes.cu) instead: L = 8
// (N=4096, D=16384: 337.1 us, 1.007 of the copy rate, against 527.2 us on this family, where
// each 16-byte access of a lane's 128-byte state costs its own L1 wavefront; N=64, D=6144
// cold 5.0 against 7.1 us) and width 4 at L = 4 (cold, N=1024: 53.5 against 56.1 us, and
// 56.8 on the bulk kernel; N=256, D=8192: 10.1 against 11.4 and 12.6; back to back at
// N=4096 200.6 against 202.9 and 199.0). Widths 3 at L = 4 (212.7 against 203.2 us), and
// L = 1 and 2, whose 2- and 4-byte states make many small accesses (W = 2, L = 1: 115.4
// against 80.6 us), stay here.
template <int L, int W>
__host__ __device__ constexpr bool lanes_form() {
  return L == 8 || (L == 4 && W == 4);
}

template <int L, int W, int ACT, bool DEDUP>
cudaError_t launch_LW(const UpdateParams &p, int64_t gx, int threads, cudaStream_t stream) {
  const bool ring = p.seqlens != nullptr;
  constexpr int kC = (int)Layout::Compact, kCL = (int)Layout::ChannelLast;
  if (p.layout == kC) {
    if constexpr (lanes_form<L, W>()) {
      return ring ? launch_one<L, W, ACT, kC, true, DEDUP>(p, gx, threads, stream) : launch_lanes(p, ACT, stream);
    } else {
      return ring ? launch_one<L, W, ACT, kC, true, DEDUP>(p, gx, threads, stream)
                  : launch_one<L, W, ACT, kC, false, DEDUP>(p, gx, threads, stream);
    }
  }
  return ring ? launch_one<L, W, ACT, kCL, true, DEDUP>(p, gx, threads, stream)
              : launch_one<L, W, ACT, kCL, false, DEDUP>(p, gx, threads, stream);
}

// L from W - 1 (the shortest state the contract allows) up to kVectorMaxL.
template <int W, int ACT, bool DEDUP>
cudaError_t launch_W(const UpdateParams &p, int64_t gx, int threads, cudaStream_t stream) {
  switch (p.L) {
    case 1: if constexpr (W - 1 <= 1) return launch_LW<1, W, ACT, DEDUP>(p, gx, threads, stream); break;
    case 2: if constexpr (W - 1 <= 2) return launch_LW<2, W, ACT, DEDUP>(p, gx, threads, stream); break;
    case 3: return launch_LW<3, W, ACT, DEDUP>(p, gx, threads, stream);
    case 4: return launch_LW<4, W, ACT, DEDUP>(p, gx, threads, stream);
    case 5: return launch_LW<5, W, ACT, DEDUP>(p, gx, threads, stream);
    case 6: return launch_LW<6, W, ACT, DEDUP>(p, gx, threads, stream);
    case 7: return launch_LW<7, W, ACT, DEDUP>(p, gx, threads, stream);
    case 8: return launch_LW<8, W, ACT, DEDUP>(p, gx, threads, stream);
    default: break;
  }
  return cudaErrorInvalidValue;
}

template <int ACT, bool DEDUP>
cudaError_t launch_act(const UpdateParams &p, int64_t gx, int threads, cudaStream_t stream) {
  switch (p.W) {
    case 2: return launch_W<2, ACT, DEDUP>(p, gx, threads, stream);
    case 3: return launch_W<3, ACT, DEDUP>(p, gx, threads, stream);
    case 4: return launch_W<4, ACT, DEDUP>(p, gx, threads, stream);
    default: return cudaErrorInvalidValue;
  }
}


// The vector family's launcher: DEDUP instances carry the duplicate check of
// ccu_conv1d_update_checked_ex (their own translation unit); the others have none of its
// code, which at the lean form's 48-register budget would cost spills.
template <bool DEDUP>
cudaError_t launch_vector_impl(const UpdateParams &p, int act, cudaStream_t stream) {
  const int64_t groups = p.D / 8;
  int threads = kThreads;
  if (groups < threads) threads = (int)((groups + 31) / 32 * 32);
  const int64_t gx = (groups + threads - 1) / threads;
  return act == 1 ? launch_act<1, DEDUP>(p, gx, threads, stream) : launch_act<0, DEDUP>(p, gx, threads, stream);
}

}  // namespace

}  // namespace ccu
