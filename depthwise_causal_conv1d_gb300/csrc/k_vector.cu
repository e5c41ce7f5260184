// Vector kernels: each thread owns 8 consecutive channels of one row at a time and moves
// x, weight, bias, state and out as 16-byte vectors. L (3..8), the state layout and the
// activation are compile-time, so the history lives in registers and the shift is a
// fixed permutation of 16-bit lanes.
//
// Update definition: cuDNN page "Causal Conv1d Decode Update", introduction (update
// block); layouts from its "Semantic tensor contract" (compact state, and the
// channel-last (L*D, 1, D) state a full-sequence prefill hands over).
#include "ccu_internal.cuh"

namespace ccu {

int device_sm_count();

namespace {

// Position of state element (channel c of the thread's 8, entry l) inside the thread's
// registers: 4*L words, two BF16 per word.
//   compact      [8 channels][L]: flat c*L + l
//   channel-last [L planes][8 channels]: plane l is one 16-byte vector
template <int L, int LAYOUT>
__device__ __forceinline__ constexpr int elem_pos(int c, int l) {
  return LAYOUT == (int)Layout::Compact ? c * L + l : l * 8 + c;
}

template <int L, int ACT, int LAYOUT>
__global__ void __launch_bounds__(256) k_update_vector(UpdateParams p) {
  const int64_t groups = p.D >> 3;  // 8-channel groups per row (D % 8 == 0)
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= groups) return;
  const int64_t c0 = g << 3;

  // weight[c0 .. c0+7, 0..3]: 32 BF16 in four 16-byte vectors, kept packed (two per
  // word) and widened at use; bias likewise. Both are reused for every row.
  uint32_t wv[16];
  {
    const uint16_t *wp = p.w + c0 * kW;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 t = ld_keep(wp + 8 * k);
      wv[4 * k] = t.x; wv[4 * k + 1] = t.y; wv[4 * k + 2] = t.z; wv[4 * k + 3] = t.w;
    }
  }
  const bool has_bias = p.bias != nullptr;
  uint32_t bv[4] = {0u, 0u, 0u, 0u};
  if (has_bias) {
    const uint4 t = ld_keep(p.bias + c0);
    bv[0] = t.x; bv[1] = t.y; bv[2] = t.z; bv[3] = t.w;
  }

  const int64_t R = p.rows_per_cta;
  for (int64_t r0 = (int64_t)blockIdx.y * R; r0 < p.N; r0 += (int64_t)gridDim.y * R) {
    const int64_t r1 = r0 + R < p.N ? r0 + R : p.N;
    for (int64_t n = r0; n < r1; ++n) {
      const int64_t s = resolve_slot(p, n);
      uint16_t *outp = p.out + n * p.D + c0;
      if (s < 0) {  // padding row: zero output, state untouched
        st_stream(outp, make_uint4(0u, 0u, 0u, 0u));
        continue;
      }

      uint32_t xw[4];
      {
        const uint4 t = ld_stream(p.x + n * p.ld + c0);
        xw[0] = t.x; xw[1] = t.y; xw[2] = t.z; xw[3] = t.w;
      }

      // Old state of the 8 channels. Channel-last with L > 3 never reads plane 0: it
      // is outside the width-4 window and is overwritten by plane 1.
      uint32_t ow[4 * L];
      uint16_t *sp;
      if constexpr (LAYOUT == (int)Layout::Compact) {
        sp = p.state + s * (p.D * L) + c0 * L;
#pragma unroll
        for (int k = 0; k < L; ++k) {
          const uint4 t = ld_stream(sp + 8 * k);
          ow[4 * k] = t.x; ow[4 * k + 1] = t.y; ow[4 * k + 2] = t.z; ow[4 * k + 3] = t.w;
        }
      } else {
        sp = p.state + s * (L * p.D) + c0;
        constexpr int first = (L == kW - 1) ? 0 : 1;
#pragma unroll
        for (int l = 0; l < L; ++l) {
          if (l < first) {
            ow[4 * l] = ow[4 * l + 1] = ow[4 * l + 2] = ow[4 * l + 3] = 0u;
            continue;
          }
          const uint4 t = ld_stream(sp + (int64_t)l * p.D);
          ow[4 * l] = t.x; ow[4 * l + 1] = t.y; ow[4 * l + 2] = t.z; ow[4 * l + 3] = t.w;
        }
      }

      uint32_t nw[4 * L];
      uint4 outv;
      if constexpr (LAYOUT == (int)Layout::Compact) {
        outv = update8_compact<L, ACT>(xw, ow, wv, bv, has_bias, nw);
#pragma unroll
        for (int k = 0; k < L; ++k)
          st_stream(sp + 8 * k, make_uint4(nw[4 * k], nw[4 * k + 1], nw[4 * k + 2], nw[4 * k + 3]));
      } else {
        // acc = sum_j history[L-3+j] * w[j] (j = 0..3, history[L] = x), then bias.
        float y[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          float acc = 0.0f;
#pragma unroll
          for (int j = 0; j < kW; ++j) {
            const int hidx = L - (kW - 1) + j;
            const uint32_t h = (hidx == L) ? get16(xw, c) : get16(ow, elem_pos<L, LAYOUT>(c, hidx));
            acc = __fmaf_rn(bf16_bits(h), bf16_bits(get16(wv, c * kW + j)), acc);
          }
          if (has_bias) acc = acc + bf16_bits(get16(bv, c));
          y[c] = activate<ACT>(acc);
        }
        outv = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                          pack_bf16x2(y[6], y[7]));
        // New state: plane l takes old plane l+1; the newest plane takes x.
#pragma unroll
        for (int l = 0; l + 1 < L; ++l)
#pragma unroll
          for (int i = 0; i < 4; ++i) nw[4 * l + i] = ow[4 * (l + 1) + i];
#pragma unroll
        for (int i = 0; i < 4; ++i) nw[4 * (L - 1) + i] = xw[i];
#pragma unroll
        for (int l = 0; l < L; ++l)
          st_stream(sp + (int64_t)l * p.D,
                    make_uint4(nw[4 * l], nw[4 * l + 1], nw[4 * l + 2], nw[4 * l + 3]));
      }
      st_stream(outp, outv);
    }
  }
}

template <int L, int ACT>
cudaError_t launch_L(const UpdateParams &p, dim3 grid, dim3 block, cudaStream_t stream) {
  if (p.layout == (int)Layout::Compact) {
    k_update_vector<L, ACT, (int)Layout::Compact><<<grid, block, 0, stream>>>(p);
  } else {
    k_update_vector<L, ACT, (int)Layout::ChannelLast><<<grid, block, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

template <int ACT>
cudaError_t launch_act(const UpdateParams &p, dim3 grid, dim3 block, cudaStream_t stream) {
  switch (p.L) {
    case 3: return launch_L<3, ACT>(p, grid, block, stream);
    case 4: return launch_L<4, ACT>(p, grid, block, stream);
    case 5: return launch_L<5, ACT>(p, grid, block, stream);
    case 6: return launch_L<6, ACT>(p, grid, block, stream);
    case 7: return launch_L<7, ACT>(p, grid, block, stream);
    case 8: return launch_L<8, ACT>(p, grid, block, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_vector(const UpdateParams &p_in, int act, cudaStream_t stream) {
  UpdateParams p = p_in;
  const int64_t groups = p.D / 8;
  int threads = 256;
  if (groups < threads) threads = (int)((groups + 31) / 32 * 32);
  const int64_t gx = (groups + threads - 1) / threads;
  // Rows per CTA: enough CTAs for several waves on every SM, a few rows each so the
  // weights loaded into registers are reused.
  const int64_t target_ctas = (int64_t)device_sm_count() * 32;
  int64_t R = (p.N * gx) / target_ctas;
  R = R < 1 ? 1 : (R > 8 ? 8 : R);
  int64_t gy = (p.N + R - 1) / R;
  if (gy > 65535) gy = 65535;  // the row loop strides over the rest
  p.rows_per_cta = (int)R;
  const dim3 grid((unsigned)gx, (unsigned)gy);
  const dim3 block(threads);
  return act == 1 ? launch_act<1>(p, grid, block, stream) : launch_act<0>(p, grid, block, stream);
}

}  // namespace ccu
