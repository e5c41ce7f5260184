// Full-sequence prefill: the causal depthwise convolution over T tokens per batch row,
// and the final state that the decode update continues from.
//
//   y[b, d, t] = act( sum_{j=0}^{W-1} w[d, j] * xx(b, d, t - (W-1) + j) + bias[d] )
//   xx(b, d, t) = x[b, d, t] for t >= 0; initial_states[b, d, L + t] for t < 0 (zero
//                 when no initial state is given)
//   final_states[b, d, l] = xx(b, d, T - L + l), l = 0..L-1
//
// This is the operation the cuDNN page "Causal Conv1d Decode Update" points to for
// prefill (introduction: use causal_conv1d for full-sequence prefill; its width-four
// final state can be passed directly to the decode update) and whose L = 3 final state in
// the channel-last stride (3*D, 1, D) the update accepts without a copy ("Semantic tensor
// contract"). The page does not define that operation; the convolution above is the
// update's definition applied to every token of a sequence.
//
// Work split: a thread owns 8 channels (vector and bulk kernels) or 1 channel (scalar
// kernel) of one batch row and a chunk of consecutive tokens; it reads the W-1 inputs before
// its chunk (the halo) and then slides the window through the chunk.
#include <atomic>

#include "ccu_bulk.cuh"

namespace ccu {

int device_sm_count();
int current_device();

namespace {

// Input xx(b, d, t) for any t >= -L (scalar access, any strides).
__device__ __forceinline__ uint32_t input_at(const UpdateParams &p, const PrefillParams &f, int64_t b,
                                             int64_t d, int64_t t) {
  if (t >= 0) return p.x[b * f.sxb + d * f.sxd + t * f.sxt];
  if (f.init == nullptr) return 0u;
  return f.init[b * f.sib + d * f.sid + (p.L + t) * f.sil];
}

// The final state of channel d: the last L inputs, in the layout the strides describe.
__device__ __forceinline__ void write_final(const UpdateParams &p, const PrefillParams &f, int64_t b,
                                            int64_t d) {
  for (int64_t l = 0; l < p.L; ++l)
    f.fin[b * f.sfb + d * f.sfd + l * f.sfl] = (uint16_t)input_at(p, f, b, d, f.T - p.L + l);
}

// One thread per (batch row, channel, token chunk); any strides and widths.
template <int ACT>
__global__ void __launch_bounds__(256) k_prefill_scalar(UpdateParams p, PrefillParams f) {
  grid_dependency_boundary();
  const int64_t chunks = (f.T + f.chunk - 1) / f.chunk;
  const int64_t total = f.B * p.D * chunks;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t d = i % p.D;
    const int64_t rest = i / p.D;
    const int64_t k = rest % chunks;
    const int64_t b = rest / chunks;
    const int64_t t0 = k * f.chunk;
    const int64_t t1 = t0 + f.chunk < f.T ? t0 + f.chunk : f.T;
    const int64_t W = p.W;
    const uint16_t *w = p.w + d * W;
    // the W-1 inputs before the chunk (newest last) in hw[3-(W-1) .. 2] (widths up to 4; a
    // wider window is read input by input)
    uint32_t hw[3] = {0u, 0u, 0u};
    if (W <= kW)
      for (int64_t k = 0; k < W - 1; ++k) hw[3 - (W - 1) + k] = input_at(p, f, b, d, t0 - (W - 1) + k);
    for (int64_t t = t0; t < t1; ++t) {
      const uint32_t xv = p.x[b * f.sxb + d * f.sxd + t * f.sxt];
      float acc = 0.0f;
      if (W <= kW) {
        for (int64_t k = 0; k < W - 1; ++k)
          acc = __fmaf_rn(bf16_bits(hw[3 - (W - 1) + k]), bf16_bits(w[k]), acc);
      } else {
        for (int64_t k = 0; k < W - 1; ++k)
          acc = __fmaf_rn(bf16_bits(input_at(p, f, b, d, t - (W - 1) + k)), bf16_bits(w[k]), acc);
      }
      acc = __fmaf_rn(bf16_bits(xv), bf16_bits(w[W - 1]), acc);
      if (p.bias != nullptr) acc = acc + bf16_bits(p.bias[d]);
      p.out[b * f.sob + d * f.sod + t * f.sot] = round_bf16(activate<ACT>(acc));
      hw[0] = hw[1];
      hw[1] = hw[2];
      hw[2] = xv;
    }
    if (f.fin != nullptr && t1 == f.T) write_final(p, f, b, d);
  }
}

// The window before token t0 for channels c0..c0+7: inputs t0-3, t0-2, t0-1 (from x, or the
// initial state / zeros before the sequence). Width W reads only the last W - 1 of them (an
// earlier one can lie before the initial state, which holds L >= W - 1 entries); the others
// are set to zero and never used.
template <int W>
__device__ __forceinline__ void load_halo(const UpdateParams &p, const PrefillParams &f, int64_t b,
                                          int64_t c0, int64_t t0, float2 (&h0)[4], float2 (&h1)[4],
                                          float2 (&h2)[4]) {
  const uint16_t *xb = p.x + b * f.sxb + c0;
  float2 *hs[3] = {h0, h1, h2};
#pragma unroll
  for (int k = 0; k < kW - 1; ++k) {
    const int64_t t = t0 - (kW - 1) + k;
    if (k < kW - W) {
#pragma unroll
      for (int i = 0; i < 4; ++i) hs[k][i] = make_float2(0.0f, 0.0f);
      continue;
    }
    if (t >= 0) {
      float2 tmp[4];
      widen8(ld_keep(xb + t * f.sxt), tmp);
#pragma unroll
      for (int i = 0; i < 4; ++i) hs[k][i] = tmp[i];
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        hs[k][i] = make_float2(bf16_bits(input_at(p, f, b, c0 + 2 * i, t)),
                               bf16_bits(input_at(p, f, b, c0 + 2 * i + 1, t)));
    }
  }
}

// Scalar-float forms of the paired helpers in ccu_internal.cuh, for the vector kernel (paired FP32 arithmetic
// made it spill at 128 registers).

// Widen 8 packed BF16 to floats.
__device__ __forceinline__ void widen8s(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16_lo(w[i]);
    f[2 * i + 1] = bf16_hi(w[i]);
  }
}

// The width-W weights of channels c0..c0+7 as floats: wf[j][c] = weight[c0 + c, j], j < W.
template <int W>
__device__ __forceinline__ void load_weights_s(const UpdateParams &p, int64_t c0, float (&wf)[kW][8]) {
  uint32_t wv[16];
  load_weights_packed<W>(p.w, c0, wv);
#pragma unroll
  for (int c = 0; c < 8; ++c)
#pragma unroll
    for (int j = 0; j < kW; ++j) wf[j][c] = j < W ? bf16_bits(get16(wv, c * W + j)) : 0.0f;
}

// Outputs of 8 channels for one token from the window a, b, c (oldest first) and the token's
// inputs x. The accumulation order is the update's: for width 4 ((0 + a*w0) + b*w1) + c*w2 +
// x*w3, for width 3 (0 + b*w0) + c*w1 + x*w2, for width 2 (0 + c*w0) + x*w1, then the bias
// (each product of two BF16 values is exact in FP32).
template <int ACT, int W>
__device__ __forceinline__ uint4 outputs8s(const float (&wf)[kW][8], const float (&bf)[8],
                                           bool has_bias, const float (&a)[8], const float (&b)[8],
                                           const float (&c)[8], const float (&x)[8]) {
  float y[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float acc;
    if constexpr (W == 4) {
      acc = __fmaf_rn(a[i], wf[0][i], 0.0f);
      acc = __fmaf_rn(b[i], wf[1][i], acc);
      acc = __fmaf_rn(c[i], wf[2][i], acc);
      acc = __fmaf_rn(x[i], wf[3][i], acc);
    } else if constexpr (W == 3) {
      acc = __fmaf_rn(b[i], wf[0][i], 0.0f);
      acc = __fmaf_rn(c[i], wf[1][i], acc);
      acc = __fmaf_rn(x[i], wf[2][i], acc);
    } else {
      acc = __fmaf_rn(c[i], wf[0][i], 0.0f);
      acc = __fmaf_rn(x[i], wf[1][i], acc);
    }
    if (has_bias) acc = acc + bf[i];
    y[i] = activate<ACT>(acc);
  }
  return make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                    pack_bf16x2(y[6], y[7]));
}

// The window before token t0 for channels c0..c0+7: inputs t0-3, t0-2, t0-1 (from x, or the
// initial state / zeros before the sequence).
template <int W>
__device__ __forceinline__ void load_halo_s(const UpdateParams &p, const PrefillParams &f, int64_t b,
                                          int64_t c0, int64_t t0, float (&h0)[8], float (&h1)[8],
                                          float (&h2)[8]) {
  const uint16_t *xb = p.x + b * f.sxb + c0;
  float *hs[3] = {h0, h1, h2};
#pragma unroll
  for (int k = 0; k < kW - 1; ++k) {
    const int64_t t = t0 - (kW - 1) + k;
    if (k < kW - W) {  // outside a width-W window (see load_halo)
#pragma unroll
      for (int c = 0; c < 8; ++c) hs[k][c] = 0.0f;
      continue;
    }
    if (t >= 0) {
      float tmp[8];
      widen8s(ld_keep(xb + t * f.sxt), tmp);
#pragma unroll
      for (int c = 0; c < 8; ++c) hs[k][c] = tmp[c];
    } else {
#pragma unroll
      for (int c = 0; c < 8; ++c) hs[k][c] = bf16_bits(input_at(p, f, b, c0 + c, t));
    }
  }
}

// 8 channels per thread, width W (2..4); x and out channel-contiguous (one 16-byte vector per
// token). The prefill moves 4 bytes per element, a quarter of the decode update's 16, so its
// arithmetic is kept lean: weights and bias are widened to floats once, the width-4 window
// is kept as floats, and tokens go four at a time so the window slides by register
// renaming; the next four tokens' loads are issued before the current four are computed
// (measured on B=8, T=4096, D=4096 with SiLU: 298 us for the first version, 159 us with
// float windows, 105 us with the loads one group ahead).
template <int ACT, int W>
__global__ void __launch_bounds__(256) k_prefill_vector(UpdateParams p, PrefillParams f) {
  grid_dependency_boundary();
  const int64_t groups = p.D >> 3;
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= groups) return;
  const int64_t c0 = g << 3;
  const int64_t b = blockIdx.z;
  const int64_t t0 = (int64_t)blockIdx.y * f.chunk;
  if (t0 >= f.T) return;
  const int64_t t1 = t0 + f.chunk < f.T ? t0 + f.chunk : f.T;

  float wf[kW][8];  // wf[j][c] = weight[c0 + c, j]
  load_weights_s<W>(p, c0, wf);
  const bool has_bias = p.bias != nullptr;
  float bf[8];
  if (has_bias) {
    widen8s(ld_keep(p.bias + c0), bf);
  }

  // The window before the chunk: inputs t0-3, t0-2, t0-1 (from x, or the initial state).
  float h0[8], h1[8], h2[8];
  load_halo_s<W>(p, f, b, c0, t0, h0, h1, h2);
  const uint16_t *xb = p.x + b * f.sxb + c0;

  auto outputs = [&](const float (&a)[8], const float (&bb)[8], const float (&cc)[8],
                     const float (&xx)[8]) -> uint4 {
    return outputs8s<ACT, W>(wf, bf, has_bias, a, bb, cc, xx);
  };

  uint16_t *ob = p.out + b * f.sob + c0;
  int64_t t = t0;
  uint4 nx[4];
  if (t + 4 <= t1) {
#pragma unroll
    for (int k = 0; k < 4; ++k) nx[k] = ld_stream(xb + (t + k) * f.sxt);
  }
  for (; t + 4 <= t1; t += 4) {
    uint4 cx[4] = {nx[0], nx[1], nx[2], nx[3]};
    if (t + 8 <= t1) {
#pragma unroll
      for (int k = 0; k < 4; ++k) nx[k] = ld_stream(xb + (t + 4 + k) * f.sxt);
    }
    float x0[8], x1[8], x2[8], x3[8];
    widen8s(cx[0], x0);
    widen8s(cx[1], x1);
    widen8s(cx[2], x2);
    widen8s(cx[3], x3);
    st_stream(ob + t * f.sot, outputs(h0, h1, h2, x0));
    st_stream(ob + (t + 1) * f.sot, outputs(h1, h2, x0, x1));
    st_stream(ob + (t + 2) * f.sot, outputs(h2, x0, x1, x2));
    st_stream(ob + (t + 3) * f.sot, outputs(x0, x1, x2, x3));
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      h0[c] = x1[c];
      h1[c] = x2[c];
      h2[c] = x3[c];
    }
  }
  for (; t < t1; ++t) {  // the chunk's last 0..3 tokens
    float x0[8];
    widen8s(ld_stream(xb + t * f.sxt), x0);
    st_stream(ob + t * f.sot, outputs(h0, h1, h2, x0));
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      h0[c] = h1[c];
      h1[c] = h2[c];
      h2[c] = x0[c];
    }
  }
  if (f.fin != nullptr && t1 == f.T) {
#pragma unroll
    for (int c = 0; c < 8; ++c) write_final(p, f, b, c0 + c);
  }
}

// ------------------------------------------------------------------ bulk-copy prefill
//
// Width W (2..4), channel-contiguous x and out. The vector kernel above keeps its next four tokens
// in registers, and at 128 registers a thread only 16 warps fit on an SM: too few bytes in
// flight for HBM. Here x travels through shared memory instead. Each warp is a pipeline over
// a run of consecutive tokens of one sequence and 256 channels (8 per lane): lane 0 brings
// kTG tokens at a time (one 512-byte cp.async.bulk per token) into a kP-stage ring that
// completes on per-stage mbarriers, the lanes slide their float windows through the stage
// from shared memory and store the outputs as 16-byte streaming stores, and the stage is
// refilled kP groups ahead. The warps share the groups evenly (see Run below); a warp's runs
// are long, so the 3-token halo and the weights are read rarely. At 4 bytes per element the
// SiLU prefill is bound by instruction issue rather than by HBM, so the arithmetic runs on
// channel pairs with the paired FP32 instructions (half the multiply-add instructions,
// identical rounding). Every mbarrier wait is bounded: on expiry the warp raises
// CCU_DEVERR_TIMEOUT, waits (bounded) for its own copies and returns.

__device__ int32_t g_prefill_error = 0;  // CCU_DEVERR_* bits raised by the bulk prefill
__device__ int32_t g_prefill_error_taken = 0;  // the value the last exchange read

// Reads and clears the error word in one atomic step (a kernel that raises a bit
// meanwhile leaves it for the next exchange).
__global__ void k_exchange_prefill_error() {
  grid_dependency_boundary();
  g_prefill_error_taken = atomicExch(&g_prefill_error, 0);
}

constexpr int kPThreads = 384;                 // 12 warps per CTA, up to 170 registers each
constexpr int kPWarps = kPThreads / 32;
constexpr int64_t kRunCh = 256;                // channels per warp (8 per lane)
constexpr int64_t kRowBytes = 2 * kRunCh;      // one token of a run
constexpr int kTG = 8;                         // tokens per stage
constexpr int kP = 3;                          // stages per warp
constexpr int64_t kStageBytes = kTG * kRowBytes;
constexpr int64_t kHeadBytes = 128;  // per warp: kP mbarriers, then the producer cursor
constexpr int64_t kWarpBytes = kHeadBytes + kP * kStageBytes;

// The work is the flattened space of groups (pair, g): pair = b * slices + s is a batch row
// and a 256-channel slice, g = 0 .. ceil(T / kTG) - 1 its kTG-token groups. Each warp takes
// one contiguous span of it, the same length to one group, so the warps finish together
// whatever B, D and T are. A span crosses pair boundaries where it must: the stretch of a
// span inside one pair is a run, over which the window slides without a restart.
struct Run {
  int64_t b, c_base, cn, t0, t1;  // batch row, channels c_base .. c_base+cn-1, tokens t0 .. t1-1
  int64_t next;                   // the group where the span's next run starts
};

// The run that starts at group q of a span ending at group q_end.
__device__ __forceinline__ Run run_at(const UpdateParams &p, const PrefillParams &f, int64_t q,
                                      int64_t q_end, int64_t slices, int64_t groups) {
  Run r;
  const int64_t pair = q / groups;
  const int64_t pair_end = (pair + 1) * groups;
  r.next = q_end < pair_end ? q_end : pair_end;
  r.b = pair / slices;
  r.c_base = (pair - r.b * slices) * kRunCh;
  const int64_t rem = p.D - r.c_base;
  r.cn = rem < kRunCh ? rem : kRunCh;
  r.t0 = (q - pair * groups) * kTG;
  const int64_t t1 = (r.next - pair * groups) * kTG;
  r.t1 = t1 < f.T ? t1 : f.T;
  return r;
}

// Lane 0's producer cursor: the next group's first x row, the tokens of its run from there,
// the row bytes, the group where the next run starts, the stage of the next load and the
// loads issued but not yet consumed. It lives in shared memory, out of the registers the
// lanes need for their windows and weights.
struct Cursor {
  const uint16_t *src;
  int64_t left, next;
  uint32_t bytes;
  int st, inflight;
};
static_assert(kP * 8 + 8 + sizeof(Cursor) <= kHeadBytes, "warp header too small");

template <int ACT, int W>
__global__ void __launch_bounds__(kPThreads, 1) k_prefill_bulk(UpdateParams p, PrefillParams f) {
  grid_dependency_boundary();
  using namespace bulk;
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char *wbase = smem + (int64_t)warp * kWarpBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(wbase);
  Cursor *cur = reinterpret_cast<Cursor *>(wbase + 8 * ((kP + 1) & ~1));
  unsigned char *bufs = wbase + kHeadBytes;

  // This warp's span [q0, q1) of the B * slices * groups groups.
  const int64_t slices = (p.D + kRunCh - 1) / kRunCh;
  const int64_t groups = (f.T + kTG - 1) / kTG;
  const int64_t total = f.B * slices * groups;
  const int64_t nw = (int64_t)gridDim.x * kPWarps;
  const int64_t w = (int64_t)blockIdx.x * kPWarps + warp;
  const int64_t share = total / nw, extra = total % nw;
  const int64_t q0 = w * share + (w < extra ? w : extra);
  const int64_t q1 = q0 + share + (w < extra ? 1 : 0);
  if (q0 >= q1) return;

  // Lane 0: point the cursor at the run that starts at group q.
  auto start_run = [&](Cursor &c, int64_t q) {
    const Run r = run_at(p, f, q, q1, slices, groups);
    c.src = p.x + r.b * f.sxb + r.t0 * f.sxt + r.c_base;
    c.left = r.t1 - r.t0;
    c.bytes = (uint32_t)(r.cn * 2);
    c.next = r.next;
  };
  // Lane 0: load the cursor's group (up to kTG tokens) into its stage and advance.
  auto issue_next = [&]() {
    Cursor c = *cur;
    if (c.left == 0) return;  // the span is all issued
    const int nt = c.left < kTG ? (int)c.left : kTG;
    uint64_t *bar = &bars[c.st];
    unsigned char *buf = bufs + c.st * kStageBytes;
    mbar_arrive_expect_tx(bar, c.bytes * (uint32_t)nt);
    for (int k = 0; k < nt; ++k) bulk_load(buf + k * kRowBytes, c.src + k * f.sxt, c.bytes, bar);
    ++c.inflight;
    if (++c.st == kP) c.st = 0;
    c.left -= nt;
    c.src += nt * f.sxt;
    if (c.left == 0 && c.next < q1) start_run(c, c.next);
    *cur = c;
  };
  if (lane == 0) {
    for (int k = 0; k < kP; ++k) mbar_init(&bars[k], 1);
    fence_mbar_init();
    Cursor c;
    start_run(c, q0);
    c.st = 0;
    c.inflight = 0;
    *cur = c;
    for (int k = 0; k < kP; ++k) issue_next();
  }
  __syncwarp();

  const bool has_bias = p.bias != nullptr;
  float2 wf[kW][4], bf[4], h0[4], h1[4], h2[4];
  int64_t w_base = -1;
  int st = 0;
  uint32_t phase = 0;
  bool failed = false;
  for (int64_t q = q0; q < q1 && !failed;) {
    // A new run: weights (when the channels change) and the halo.
    const Run r = run_at(p, f, q, q1, slices, groups);
    q = r.next;
    const bool active = 8 * lane < r.cn;
    const int64_t c0 = r.c_base + 8 * lane;
    if (active) {
      if (r.c_base != w_base) {
        load_weights_f<W>(p.w, c0, wf);
        if (has_bias) widen8(ld_keep(p.bias + c0), bf);
      }
      load_halo<W>(p, f, r.b, c0, r.t0, h0, h1, h2);
    }
    w_base = r.c_base;
    const bool ends = f.fin != nullptr && r.t1 == f.T;
    const int64_t b = r.b;
    uint16_t *ob = p.out + b * f.sob + r.t0 * f.sot + c0;
    for (int64_t left = r.t1 - r.t0; left > 0; left -= kTG) {
      const bool ok = mbar_wait(&bars[st], phase);
      if (!__all_sync(kFull, ok)) {
        failed = true;
        break;
      }
      if (active) {
        const uint4 *row = reinterpret_cast<const uint4 *>(bufs + st * kStageBytes) + lane;
        if (left >= kTG) {
#pragma unroll
          for (int k = 0; k < kTG; ++k) {  // unrolled: the window slides by register renaming
            float2 xk[4];
            widen8(row[k * (kRowBytes / 16)], xk);
            st_stream(ob + k * f.sot, outputs8f<ACT, W>(wf, bf, has_bias, h0, h1, h2, xk));
            slide(h0, h1, h2, xk);
          }
        } else {
          for (int k = 0; k < (int)left; ++k) {
            float2 xk[4];
            widen8(row[k * (kRowBytes / 16)], xk);
            st_stream(ob + k * f.sot, outputs8f<ACT, W>(wf, bf, has_bias, h0, h1, h2, xk));
            slide(h0, h1, h2, xk);
          }
        }
        if (ends && left <= kTG) {
#pragma unroll
          for (int c = 0; c < 8; ++c) write_final(p, f, b, c0 + c);
        }
      }
      ob += kTG * f.sot;
      // Every lane has read the stage; order those reads before the refill's async writes.
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        --cur->inflight;
        issue_next();
      }
      if (++st == kP) {
        st = 0;
        phase ^= 1u;
      }
    }
  }

  if (failed && lane == 0) {
    atomicOr(&g_prefill_error, kDevErrTimeout);
    for (int q = cur->inflight; q > 0; --q) {  // the warp's loads still in flight
      mbar_wait(&bars[st], phase);
      if (++st == kP) {
        st = 0;
        phase ^= 1u;
      }
    }
  }
}

constexpr int kMaxDevices = 64;
std::atomic<bool> g_bulk_opted_in[kMaxDevices][2][kW + 1];

template <int ACT, int W>
cudaError_t launch_prefill_bulk_aw(const UpdateParams &p, PrefillParams f, cudaStream_t stream) {
  const size_t smem = (size_t)kPWarps * kWarpBytes;
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!g_bulk_opted_in[dev][ACT][W].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(k_prefill_bulk<ACT, W>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    g_bulk_opted_in[dev][ACT][W].store(true, std::memory_order_release);
  }
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_prefill_bulk<ACT, W>,
                                                                kPThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int64_t ctas = (int64_t)device_sm_count() * per_sm;
  // One CTA per SM (fewer when there are fewer groups than warps to share them).
  const int64_t groups = f.B * ((p.D + kRunCh - 1) / kRunCh) * ((f.T + kTG - 1) / kTG);
  int64_t grid = (groups + kPWarps - 1) / kPWarps;
  if (grid > ctas) grid = ctas;
  return launch_overlapped(k_prefill_bulk<ACT, W>, dim3((unsigned)grid), dim3(kPThreads), smem, stream, p, f);
}

template <int ACT>
cudaError_t launch_prefill_bulk_act(const UpdateParams &p, const PrefillParams &f, cudaStream_t stream) {
  switch (p.W) {
    case 2: return launch_prefill_bulk_aw<ACT, 2>(p, f, stream);
    case 3: return launch_prefill_bulk_aw<ACT, 3>(p, f, stream);
    case 4: return launch_prefill_bulk_aw<ACT, 4>(p, f, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int ACT>
cudaError_t launch_prefill_vector_act(const UpdateParams &p, const PrefillParams &f, dim3 grid, int threads,
                                      cudaStream_t stream) {
  switch (p.W) {
    case 2: return launch_overlapped(k_prefill_vector<ACT, 2>, grid, dim3(threads), 0, stream, p, f);
    case 3: return launch_overlapped(k_prefill_vector<ACT, 3>, grid, dim3(threads), 0, stream, p, f);
    case 4: return launch_overlapped(k_prefill_vector<ACT, 4>, grid, dim3(threads), 0, stream, p, f);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_prefill(const UpdateParams &p, const PrefillParams &f, int act, bool vector,
                           cudaStream_t stream) {
  if (vector) {
    const int64_t groups = p.D / 8;
    int threads = 256;
    if (groups < threads) threads = (int)((groups + 31) / 32 * 32);
    const int64_t gx = (groups + threads - 1) / threads;
    const int64_t gy = (f.T + f.chunk - 1) / f.chunk;
    if (gy > 65535 || f.B > 65535) return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)gx, (unsigned)gy, (unsigned)f.B);
    return act == 1 ? launch_prefill_vector_act<1>(p, f, grid, threads, stream)
                    : launch_prefill_vector_act<0>(p, f, grid, threads, stream);
  } else {
    const int threads = 256;
    const int64_t chunks = (f.T + f.chunk - 1) / f.chunk;
    int64_t blocks = (f.B * p.D * chunks + threads - 1) / threads;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const dim3 grid((unsigned)blocks), block(threads);
    return act == 1 ? launch_overlapped(k_prefill_scalar<1>, grid, block, 0, stream, p, f)
                    : launch_overlapped(k_prefill_scalar<0>, grid, block, 0, stream, p, f);
  }
}

cudaError_t launch_prefill_bulk(const UpdateParams &p, const PrefillParams &f, int act,
                                cudaStream_t stream) {
  return act == 1 ? launch_prefill_bulk_act<1>(p, f, stream) : launch_prefill_bulk_act<0>(p, f, stream);
}

cudaError_t take_prefill_error(int32_t *bits) {
  // read and clear in one atomic step on the device (the legacy default stream orders
  // the copy after the exchange)
  cudaError_t e = launch_overlapped(k_exchange_prefill_error, dim3(1), dim3(1), 0, (cudaStream_t)0);
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(bits, g_prefill_error_taken, sizeof(int32_t));
  return e;
}

}  // namespace ccu
