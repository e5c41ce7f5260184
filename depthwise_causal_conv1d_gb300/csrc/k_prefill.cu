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
// Work split: a thread owns 8 channels (vector kernel) or 1 channel (scalar kernel) of one
// batch row and a chunk of consecutive tokens; it reads the 3 inputs before its chunk
// (the halo) and then slides the width-4 window through the chunk.
#include "ccu_internal.cuh"

namespace ccu {

int device_sm_count();

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

// One thread per (batch row, channel, token chunk); any strides.
template <int ACT>
__global__ void __launch_bounds__(256) k_prefill_scalar(UpdateParams p, PrefillParams f) {
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
    // the W-1 inputs before the chunk (newest last) in hw[3-(W-1) .. 2]
    uint32_t hw[3] = {0u, 0u, 0u};
    for (int64_t k = 0; k < W - 1; ++k) hw[3 - (W - 1) + k] = input_at(p, f, b, d, t0 - (W - 1) + k);
    for (int64_t t = t0; t < t1; ++t) {
      const uint32_t xv = p.x[b * f.sxb + d * f.sxd + t * f.sxt];
      float acc = 0.0f;
      for (int64_t k = 0; k < W - 1; ++k)
        acc = __fmaf_rn(bf16_bits(hw[3 - (W - 1) + k]), bf16_bits(w[k]), acc);
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

// Widen 8 packed BF16 to floats.
__device__ __forceinline__ void widen8(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16_lo(w[i]);
    f[2 * i + 1] = bf16_hi(w[i]);
  }
}

// 8 channels per thread, width 4; x and out channel-contiguous (one 16-byte vector per
// token). The prefill moves 4 bytes per element, a quarter of the decode update's 16, so its
// arithmetic is kept lean: weights and bias are widened to floats once, the width-4 window
// is kept as floats, and tokens go four at a time so the window slides by register
// renaming; the next four tokens' loads are issued before the current four are computed
// (measured on B=8, T=4096, D=4096 with SiLU: 298 us for the first version, 159 us with
// float windows, 105 us with the loads one group ahead). The accumulation order is the
// update's: ((0 + h0*w0) + h1*w1) + h2*w2 + x*w3, then the bias (each product of two
// BF16 values is exact in FP32).
template <int ACT>
__global__ void __launch_bounds__(256) k_prefill_vector(UpdateParams p, PrefillParams f) {
  const int64_t groups = p.D >> 3;
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= groups) return;
  const int64_t c0 = g << 3;
  const int64_t b = blockIdx.z;
  const int64_t t0 = (int64_t)blockIdx.y * f.chunk;
  if (t0 >= f.T) return;
  const int64_t t1 = t0 + f.chunk < f.T ? t0 + f.chunk : f.T;

  float wf[kW][8];  // wf[j][c] = weight[c0 + c, j]
  {
    const uint16_t *wp = p.w + c0 * kW;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 t = ld_keep(wp + 8 * k);
      const uint32_t v[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int e = 8 * k + 2 * i;  // flat c*4 + j of the low half
        wf[e % kW][e / kW] = bf16_lo(v[i]);
        wf[(e + 1) % kW][(e + 1) / kW] = bf16_hi(v[i]);
      }
    }
  }
  const bool has_bias = p.bias != nullptr;
  float bf[8];
  if (has_bias) {
    widen8(ld_keep(p.bias + c0), bf);
  }

  // The window before the chunk: inputs t0-3, t0-2, t0-1 (from x, or the initial state).
  float h0[8], h1[8], h2[8];
  const uint16_t *xb = p.x + b * f.sxb + c0;
  {
    float *hs[3] = {h0, h1, h2};
#pragma unroll
    for (int k = 0; k < kW - 1; ++k) {
      const int64_t t = t0 - (kW - 1) + k;
      if (t >= 0) {
        float tmp[8];
        widen8(ld_keep(xb + t * f.sxt), tmp);
#pragma unroll
        for (int c = 0; c < 8; ++c) hs[k][c] = tmp[c];
      } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) hs[k][c] = bf16_bits(input_at(p, f, b, c0 + c, t));
      }
    }
  }

  auto outputs = [&](const float (&a)[8], const float (&bb)[8], const float (&cc)[8],
                     const float (&xx)[8]) -> uint4 {
    float y[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float acc = __fmaf_rn(a[c], wf[0][c], 0.0f);
      acc = __fmaf_rn(bb[c], wf[1][c], acc);
      acc = __fmaf_rn(cc[c], wf[2][c], acc);
      acc = __fmaf_rn(xx[c], wf[3][c], acc);
      if (has_bias) acc = acc + bf[c];
      y[c] = activate<ACT>(acc);
    }
    return make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                      pack_bf16x2(y[6], y[7]));
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
    widen8(cx[0], x0);
    widen8(cx[1], x1);
    widen8(cx[2], x2);
    widen8(cx[3], x3);
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
    widen8(ld_stream(xb + t * f.sxt), x0);
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
    if (act == 1) {
      k_prefill_vector<1><<<grid, threads, 0, stream>>>(p, f);
    } else {
      k_prefill_vector<0><<<grid, threads, 0, stream>>>(p, f);
    }
  } else {
    const int threads = 256;
    const int64_t chunks = (f.T + f.chunk - 1) / f.chunk;
    int64_t blocks = (f.B * p.D * chunks + threads - 1) / threads;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (act == 1) {
      k_prefill_scalar<1><<<(unsigned)blocks, threads, 0, stream>>>(p, f);
    } else {
      k_prefill_scalar<0><<<(unsigned)blocks, threads, 0, stream>>>(p, f);
    }
  }
  return cudaGetLastError();
}

}  // namespace ccu
