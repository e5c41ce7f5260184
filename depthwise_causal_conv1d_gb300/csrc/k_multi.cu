// Multi-token update: T tokens per row in one call, x[N, D, T].
//
// The T tokens are appended to the history in order: output t is computed from the width-W
// window ending at token t, and the new state is the last L entries of the history (with
// cache_seqlens, token t is written over ring position (q + t) mod L). Optionally the state
// after every token is written to intermediate_states [N, T, D, L] (compact, in the
// state's own entry order), so a speculative decoder can roll back to any token.
//
// The cuDNN page "Causal Conv1d Decode Update" names this extension without defining it
// ("Semantic tensor contract": a future multi-token form may admit x[N, D, Tstep] without
// changing the state or weight meanings; "Current native implementation": multi-token
// updates and speculative intermediate-state returns are declined today).
#include "ccu_multi.cuh"

namespace ccu {

// Widths 2 and 3 (k_multi_narrow.cu).
cudaError_t launch_multi_vector_narrow(const UpdateParams &p, const MultiParams &m, int act, dim3 grid,
                                       dim3 block, cudaStream_t stream);

namespace {

// One thread per (row, channel), any x / out strides, any L and W: the correctness anchor.
template <int ACT>
__global__ void __launch_bounds__(256) k_multi_scalar(UpdateParams p, MultiParams m) {
  grid_dependency_boundary();
  const int64_t total = p.N * p.D;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = i / p.D;
    const int64_t d = i - n * p.D;
    const RowSlot r = resolve_row<0, false>(p, n);
    if (r.s < 0) {
      for (int64_t t = 0; t < m.T; ++t) p.out[n * m.son + d * m.sod + t * m.sot] = 0;
      continue;
    }
    uint16_t *st = p.state + r.s * p.ss + d * p.sd;
    const int64_t L = p.L;
    const bool ring = p.seqlens != nullptr;
    const int64_t q = ring ? r.q : 0;
    const uint16_t *xp = p.x + n * m.sxn + d * m.sxd;
    const int64_t W = p.W;
    const uint16_t *w = p.w + d * W;
    // Entry k of the time-ordered history (k < L: state entry k, oldest first; else token
    // k - L), read before any of this channel's state is overwritten.
    auto hist = [&](int64_t k) -> uint16_t {
      if (k < L) return st[(ring ? (q + k) % L : k) * p.sl];
      return xp[(k - L) * m.sxt];
    };
    // the W-1 window entries before the first token (newest last), in hw[3-(W-1) .. 2]
    // (widths up to 4; a wider window is read from the history tap by tap)
    uint16_t hw[3] = {0, 0, 0};
    if (W <= kW)
      for (int64_t k = 0; k < W - 1; ++k) hw[3 - (W - 1) + k] = hist(L - (W - 1) + k);
    for (int64_t t = 0; t < m.T; ++t) {
      const uint16_t xv = xp[t * m.sxt];
      float acc = 0.0f;
      if (W <= kW) {
        for (int64_t k = 0; k < W - 1; ++k)
          acc = __fmaf_rn(bf16_bits(hw[3 - (W - 1) + k]), bf16_bits(w[k]), acc);
      } else {
        // token t is history entry L + t; its window is entries L + t - (W-1) .. L + t
        for (int64_t k = 0; k < W - 1; ++k)
          acc = __fmaf_rn(bf16_bits(hist(L + t - (W - 1) + k)), bf16_bits(w[k]), acc);
      }
      acc = __fmaf_rn(bf16_bits(xv), bf16_bits(w[W - 1]), acc);
      if (p.bias != nullptr) acc = acc + bf16_bits(p.bias[d]);
      p.out[n * m.son + d * m.sod + t * m.sot] = round_bf16(activate<ACT>(acc));
      hw[0] = hw[1];
      hw[1] = hw[2];
      hw[2] = xv;
      if (m.inter != nullptr) {
        // the state after token t in its own order: history[t+1 .. t+L]; a ring holds the
        // entry of age (l - (q + t + 1)) mod L at position l
        uint16_t *it = m.inter + ((n * m.T + t) * p.D + d) * L;
        for (int64_t l = 0; l < L; ++l) {
          int64_t age = l;
          if (ring) {
            age = (l - (q + t + 1)) % L;
            if (age < 0) age += L;
          }
          it[l] = hist(t + 1 + age);
        }
      }
    }
    // The new state: the last L history entries. Linear: entry i takes history[T + i],
    // ascending, so each entry is read before it is overwritten. Ring: the tokens land at
    // (q + t) mod L in order; only the last L writes survive.
    if (ring) {
      for (int64_t t = (m.T > L ? m.T - L : 0); t < m.T; ++t) st[((q + t) % L) * p.sl] = xp[t * m.sxt];
    } else {
      for (int64_t l = 0; l < L; ++l) st[l * p.sl] = hist(m.T + l);
    }
  }
}

// Width 4 with L = 3..8 (widths 2 and 3 in k_multi_narrow.cu).
template <int ACT>
cudaError_t launch_vec_A(const UpdateParams &p, const MultiParams &m, dim3 grid, dim3 block,
                         cudaStream_t stream) {
  switch (p.L) {
    case 3: return launch_vec_L<3, 4, ACT>(p, m, grid, block, stream);
    case 4: return launch_vec_L<4, 4, ACT>(p, m, grid, block, stream);
    case 5: return launch_vec_L<5, 4, ACT>(p, m, grid, block, stream);
    case 6: return launch_vec_L<6, 4, ACT>(p, m, grid, block, stream);
    case 7: return launch_vec_L<7, 4, ACT>(p, m, grid, block, stream);
    case 8: return launch_vec_L<8, 4, ACT>(p, m, grid, block, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_multi_scalar(const UpdateParams &p, const MultiParams &m, int act,
                                cudaStream_t stream) {
  const int threads = 256;
  int64_t blocks = (p.N * p.D + threads - 1) / threads;
  const int64_t cap = (int64_t)device_sm_count() * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const dim3 grid((unsigned)blocks), block(threads);
  return act == 1 ? launch_overlapped(k_multi_scalar<1>, grid, block, 0, stream, p, m)
                  : launch_overlapped(k_multi_scalar<0>, grid, block, 0, stream, p, m);
}

// CTAs per SM the grid is sized for: one wave (two per SM, each CTA walking its rows) or
// four waves (eight per SM), whichever measured faster. N=1024, D=16384, T=4, us, one wave /
// four waves, one row in flight: ring states (compact L = 3 90.1 / 89.2, L = 5 135.8 / 123.8,
// L = 6 119.3 / 117.9, L = 7 176.0 / 160.5, L = 8 172.4 / 165.5; channel-last L = 3 91.1 /
// 90.4, L = 4 105.7 / 103.2, L = 5 111.4 / 106.9, L = 6 133.3 / 125.4, L = 7 132.8 / 128.3)
// and the linear state at L = 6 (compact 109.9 / 107.2, channel-last 105.2 / 103.6) and at
// L = 8 in the channel-last layout (123.3 / 120.3) take four waves; the other linear states
// one (compact L = 4 87.6 / 89.1, L = 5 96.0 / 97.8, L = 7 144.7 / 152.7, L = 8 142.0 / 144.2;
// channel-last L = 3 80.5 / 81.0, L = 7 140.3 / 143.2; the two-row form at compact L = 3
// 77.8 / 81.4, T = 1 45.8 / 48.7, T = 8 136.2 / 138.1, N=256 20.2 / 22.1, N=128 11.4 / 13.6,
// and at the compact ring L = 4). A form that kept each thread's next rows in flight in
// shared memory (cp.async, three rows ahead, one wave) measured 83.3 at L = 3, 100.4 at
// L = 4 and 183.9 at L = 8.
static int multi_grid_ctas_per_sm(const UpdateParams &p) {
  const bool ring = p.seqlens != nullptr;
  const bool compact = p.layout == (int)Layout::Compact;
  if (ring) return (compact && p.L == 4) ? 2 : 8;  // the compact ring at L = 4 runs two rows
  const bool four_waves = p.L == 6 || (p.L == 8 && !compact);
  return four_waves ? 8 : 2;
}

cudaError_t launch_multi_vector(const UpdateParams &p, const MultiParams &m, int act,
                                cudaStream_t stream) {
  const int64_t groups = p.D / 8;
  int threads = 256;
  if (groups < threads) threads = (int)((groups + 31) / 32 * 32);
  const int64_t gx = (groups + threads - 1) / threads;
  int64_t gy = (int64_t)device_sm_count() * multi_grid_ctas_per_sm(p) / gx;
  if (gy < 1) gy = 1;
  if (gy > p.N) gy = p.N;
  if (gy > 65535) gy = 65535;
  const dim3 grid((unsigned)gx, (unsigned)gy), block(threads);
  if (p.W != kW) return launch_multi_vector_narrow(p, m, act, grid, block, stream);
  return act == 1 ? launch_vec_A<1>(p, m, grid, block, stream) : launch_vec_A<0>(p, m, grid, block, stream);
}

}  // namespace ccu
