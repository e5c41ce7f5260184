/*
 * CPU oracle for the depthwise causal conv1d decode update.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg; never by the product path. It shares no code,
 * header, table or helper with the CUDA library.
 *
 * It is the plain definition written out, one (row, channel) at a time, from
 * the cuDNN page "Causal Conv1d Decode Update":
 *   - introduction, update block: history = concat(conv_state[s, d, :], x[n, d]);
 *     conv_state[s, d, :] = history[-L:]; acc = sum_j history[-W + j] * weight[d, j]
 *     + bias[d]; output = activation(acc);
 *   - the paragraph after it: bias is zero when omitted; identity returns acc;
 *     "silu"/"swish" are the same SiLU;
 *   - the conv_state_indices paragraph: s = n without indices, else indices[n];
 *     -1 is a padding row (zero output, no state change); other slots in range
 *     and unique;
 *   - "Semantic tensor contract": x [N, D] with row stride ld, weight [D, W],
 *     conv_state [S, D, L] with L >= W - 1, output [N, D].
 *
 * Readings where the page is silent:
 *   - the accumulator is FP32, summed over j = 0..W-1 in ascending order, each
 *     term a float product of the two widened BF16 values, bias added last and
 *     skipped (not +0) when omitted;
 *   - SiLU is a / (1 + exp(-a)), evaluated in double from the FP32 accumulator and
 *     rounded to float;
 *   - the output is the float result rounded to BF16, nearest-even;
 *   - a padding row's output is +0;
 *   - the circular-buffer state the page reserves cache_seqlens for (its section on the
 *     keyword says only that a future version may use it so): the slot is a ring of L
 *     entries, p = cache_seqlens[n] mod L indexes its oldest entry, the history is the
 *     ring read from p onward followed by x, and the step overwrites only that oldest
 *     entry with x. Read this way, a ring read from p is exactly the linear state;
 *   - the multi-token update x[N, D, T] the page says may come later: the T tokens are
 *     appended to the history in order, output t is computed from the window ending at
 *     token t, and the new state is the last L entries (T single steps in one call).
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared (no fast-math, no FMA contraction).
 */
#include "ccu_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

float ccu_oracle_bf16_to_f32(uint16_t bits) {
  /* BF16 is the upper half of an IEEE-754 binary32. */
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

uint16_t ccu_oracle_f32_to_bf16(float value) {
  uint32_t u;
  memcpy(&u, &value, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) {
    /* NaN: keep the sign and the top payload bits, force it quiet. */
    return (uint16_t)((u >> 16) | 0x0040u);
  }
  uint32_t upper = u >> 16;      /* truncated result */
  uint32_t lower = u & 0xffffu;  /* the discarded half */
  if (lower > 0x8000u) {
    upper += 1;                  /* above the halfway point: round up in magnitude */
  } else if (lower == 0x8000u) {
    upper += (upper & 1u);       /* exactly halfway: round to the even neighbour */
  }
  /* A carry out of the mantissa bumps the exponent, which is the correct
   * rounded value (and gives infinity past the largest finite BF16). */
  return (uint16_t)upper;
}

float ccu_oracle_silu(float acc) {
  double a = (double)acc;
  double y = a / (1.0 + exp(-a));
  return (float)y;
}

static float activation(float acc, int act) {
  return act == CCU_ORACLE_ACT_SILU ? ccu_oracle_silu(acc) : acc;
}

int ccu_oracle_check_indices(const int32_t *indices, int64_t N, int64_t S) {
  int flags = 0;
  if (indices == NULL || N <= 0) return 0;
  unsigned char *seen = (unsigned char *)calloc((size_t)(S > 0 ? S : 1), 1);
  if (seen == NULL) return CCU_ORACLE_NO_MEMORY;
  for (int64_t n = 0; n < N; ++n) {
    int64_t s = indices[n];
    if (s == -1) continue;
    if (s < -1 || s >= S) {
      flags |= CCU_ORACLE_IDX_RANGE;
      continue;
    }
    if (seen[s]) flags |= CCU_ORACLE_IDX_DUPLICATE;
    seen[s] = 1;
  }
  free(seen);
  return flags;
}

int ccu_oracle_conv1d_update(const uint16_t *x, int64_t ld, uint16_t *conv_state,
                             int64_t stride_s, int64_t stride_d, int64_t stride_l,
                             const uint16_t *weight, const uint16_t *bias, int act,
                             const int32_t *indices, int64_t N, int64_t D, int64_t S,
                             int64_t L, int64_t W, uint16_t *out, float *acc_out) {
  if (N < 0 || D < 0 || S < 0 || W < 1 || L < W - 1 || ld < D) return CCU_ORACLE_BAD_ARGS;
  if (act != CCU_ORACLE_ACT_IDENTITY && act != CCU_ORACLE_ACT_SILU) return CCU_ORACLE_BAD_ARGS;
  if (N == 0 || D == 0) return CCU_ORACLE_OK;
  if (x == NULL || conv_state == NULL || weight == NULL || out == NULL) return CCU_ORACLE_BAD_ARGS;
  if (indices == NULL && S < N) return CCU_ORACLE_BAD_ARGS;
  if (indices != NULL) {
    int flags = ccu_oracle_check_indices(indices, N, S);
    if (flags < 0) return flags;
    if (flags != 0) return CCU_ORACLE_BAD_INDICES;
  }

  /* history holds the L state entries followed by the new input: L + 1 values. */
  uint16_t *history = (uint16_t *)malloc((size_t)(L + 1) * sizeof(uint16_t));
  if (history == NULL) return CCU_ORACLE_NO_MEMORY;

  for (int64_t n = 0; n < N; ++n) {
    int64_t s = indices ? (int64_t)indices[n] : n;
    if (s == -1) {
      for (int64_t d = 0; d < D; ++d) {
        out[n * D + d] = 0x0000u; /* +0.0 */
        if (acc_out) acc_out[n * D + d] = 0.0f;
      }
      continue; /* padding row: conv_state is not read or written */
    }
    for (int64_t d = 0; d < D; ++d) {
      uint16_t *st = conv_state + s * stride_s + d * stride_d;

      /* history = concat(conv_state[s, d, :], x[n, d]) */
      for (int64_t l = 0; l < L; ++l) history[l] = st[l * stride_l];
      history[L] = x[n * ld + d];

      /* acc = sum_j history[-W + j] * weight[d, j] + bias[d]; history[-W + j] is
       * history[(L + 1) - W + j] counted from the front. */
      float acc = 0.0f;
      for (int64_t j = 0; j < W; ++j) {
        float h = ccu_oracle_bf16_to_f32(history[(L + 1) - W + j]);
        float w = ccu_oracle_bf16_to_f32(weight[d * W + j]);
        float term = h * w;
        acc = acc + term;
      }
      if (bias != NULL) acc = acc + ccu_oracle_bf16_to_f32(bias[d]);

      out[n * D + d] = ccu_oracle_f32_to_bf16(activation(acc, act));
      if (acc_out) acc_out[n * D + d] = acc;

      /* conv_state[s, d, :] = history[-L:], i.e. history[1..L]: raw bit copies */
      for (int64_t l = 0; l < L; ++l) st[l * stride_l] = history[l + 1];
    }
  }
  free(history);
  return CCU_ORACLE_OK;
}

int ccu_oracle_conv1d_update_circular(const uint16_t *x, int64_t ld, uint16_t *conv_state,
                                      int64_t stride_s, int64_t stride_d, int64_t stride_l,
                                      const uint16_t *weight, const uint16_t *bias, int act,
                                      const int32_t *indices, const int32_t *cache_seqlens,
                                      int64_t N, int64_t D, int64_t S, int64_t L, int64_t W,
                                      uint16_t *out, float *acc_out) {
  if (N < 0 || D < 0 || S < 0 || W < 1 || L < W - 1 || L < 1 || ld < D) return CCU_ORACLE_BAD_ARGS;
  if (act != CCU_ORACLE_ACT_IDENTITY && act != CCU_ORACLE_ACT_SILU) return CCU_ORACLE_BAD_ARGS;
  if (N == 0 || D == 0) return CCU_ORACLE_OK;
  if (x == NULL || conv_state == NULL || weight == NULL || out == NULL || cache_seqlens == NULL)
    return CCU_ORACLE_BAD_ARGS;
  if (indices == NULL && S < N) return CCU_ORACLE_BAD_ARGS;
  if (indices != NULL) {
    int flags = ccu_oracle_check_indices(indices, N, S);
    if (flags < 0) return flags;
    if (flags != 0) return CCU_ORACLE_BAD_INDICES;
  }
  for (int64_t n = 0; n < N; ++n) {
    int64_t s = indices ? (int64_t)indices[n] : n;
    if (s != -1 && cache_seqlens[n] < 0) return CCU_ORACLE_BAD_ARGS;
  }

  uint16_t *history = (uint16_t *)malloc((size_t)(L + 1) * sizeof(uint16_t));
  if (history == NULL) return CCU_ORACLE_NO_MEMORY;

  for (int64_t n = 0; n < N; ++n) {
    int64_t s = indices ? (int64_t)indices[n] : n;
    if (s == -1) {
      for (int64_t d = 0; d < D; ++d) {
        out[n * D + d] = 0x0000u;
        if (acc_out) acc_out[n * D + d] = 0.0f;
      }
      continue;
    }
    const int64_t p = (int64_t)cache_seqlens[n] % L; /* position of the oldest entry */
    for (int64_t d = 0; d < D; ++d) {
      uint16_t *ring = conv_state + s * stride_s + d * stride_d;

      /* history, oldest first: the ring read from position p, then x */
      for (int64_t i = 0; i < L; ++i) history[i] = ring[((p + i) % L) * stride_l];
      history[L] = x[n * ld + d];

      float acc = 0.0f;
      for (int64_t j = 0; j < W; ++j) {
        float h = ccu_oracle_bf16_to_f32(history[(L + 1) - W + j]);
        float w = ccu_oracle_bf16_to_f32(weight[d * W + j]);
        float term = h * w;
        acc = acc + term;
      }
      if (bias != NULL) acc = acc + ccu_oracle_bf16_to_f32(bias[d]);

      out[n * D + d] = ccu_oracle_f32_to_bf16(activation(acc, act));
      if (acc_out) acc_out[n * D + d] = acc;

      /* the new input replaces the oldest entry; the others stay where they are */
      ring[p * stride_l] = history[L];
    }
  }
  free(history);
  return CCU_ORACLE_OK;
}

int ccu_oracle_conv1d_update_multi(const uint16_t *x, int64_t sxn, int64_t sxd, int64_t sxt,
                                   uint16_t *conv_state, int64_t stride_s, int64_t stride_d,
                                   int64_t stride_l, const uint16_t *weight, const uint16_t *bias,
                                   int act, const int32_t *indices, const int32_t *cache_seqlens,
                                   int64_t N, int64_t D, int64_t T, int64_t S, int64_t L, int64_t W,
                                   uint16_t *out, int64_t son, int64_t sod, int64_t sot,
                                   uint16_t *inter) {
  if (N < 0 || D < 0 || T < 0 || S < 0 || W < 1 || L < W - 1 || L < 1) return CCU_ORACLE_BAD_ARGS;
  if (act != CCU_ORACLE_ACT_IDENTITY && act != CCU_ORACLE_ACT_SILU) return CCU_ORACLE_BAD_ARGS;
  if (N == 0 || D == 0 || T == 0) return CCU_ORACLE_OK;
  if (x == NULL || conv_state == NULL || weight == NULL || out == NULL) return CCU_ORACLE_BAD_ARGS;
  if (indices == NULL && S < N) return CCU_ORACLE_BAD_ARGS;
  if (indices != NULL) {
    int flags = ccu_oracle_check_indices(indices, N, S);
    if (flags < 0) return flags;
    if (flags != 0) return CCU_ORACLE_BAD_INDICES;
  }
  if (cache_seqlens != NULL) {
    for (int64_t n = 0; n < N; ++n) {
      int64_t s = indices ? (int64_t)indices[n] : n;
      if (s != -1 && cache_seqlens[n] < 0) return CCU_ORACLE_BAD_ARGS;
    }
  }

  /* the state entries in time order (oldest first), then the T tokens */
  uint16_t *history = (uint16_t *)malloc((size_t)(L + T) * sizeof(uint16_t));
  if (history == NULL) return CCU_ORACLE_NO_MEMORY;

  for (int64_t n = 0; n < N; ++n) {
    int64_t s = indices ? (int64_t)indices[n] : n;
    if (s == -1) {
      for (int64_t d = 0; d < D; ++d)
        for (int64_t t = 0; t < T; ++t) out[n * son + d * sod + t * sot] = 0x0000u;
      continue;
    }
    const int64_t q = cache_seqlens ? (int64_t)cache_seqlens[n] % L : 0;
    for (int64_t d = 0; d < D; ++d) {
      uint16_t *st = conv_state + s * stride_s + d * stride_d;
      for (int64_t i = 0; i < L; ++i) {
        /* linear state: entry i; ring: the ring read from its oldest entry q */
        int64_t pos = cache_seqlens ? (q + i) % L : i;
        history[i] = st[pos * stride_l];
      }
      for (int64_t t = 0; t < T; ++t) history[L + t] = x[n * sxn + d * sxd + t * sxt];

      for (int64_t t = 0; t < T; ++t) {
        /* token t is history[L + t]; its window is history[L + t + 1 - W .. L + t] */
        float acc = 0.0f;
        for (int64_t j = 0; j < W; ++j) {
          float h = ccu_oracle_bf16_to_f32(history[L + t + 1 - W + j]);
          float w = ccu_oracle_bf16_to_f32(weight[d * W + j]);
          float term = h * w;
          acc = acc + term;
        }
        if (bias != NULL) acc = acc + ccu_oracle_bf16_to_f32(bias[d]);
        out[n * son + d * sod + t * sot] = ccu_oracle_f32_to_bf16(activation(acc, act));

        if (inter != NULL) {
          /* the state after token t, in the state's own order */
          uint16_t *it = inter + ((n * T + t) * D + d) * L;
          for (int64_t l = 0; l < L; ++l) {
            if (cache_seqlens) {
              /* ring after t+1 writes: position (q + k) mod L holds token k for the last
               * writes, so read the time-ordered history back into ring positions */
              int64_t age = (l - (q + t + 1)) % L; /* 0 = oldest entry after token t */
              if (age < 0) age += L;
              it[l] = history[t + 1 + age];
            } else {
              it[l] = history[t + 1 + l];
            }
          }
        }
      }

      /* the new state: the last L history entries, in the state's own order */
      for (int64_t i = 0; i < L; ++i) {
        if (cache_seqlens) {
          int64_t pos = (q + T + i) % L; /* after T writes the oldest entry sits at q + T */
          st[pos * stride_l] = history[T + i];
        } else {
          st[i * stride_l] = history[T + i];
        }
      }
    }
  }
  free(history);
  return CCU_ORACLE_OK;
}

int ccu_oracle_full_causal_conv(const uint16_t *x_seq, int64_t T, int64_t D,
                                const uint16_t *weight, const uint16_t *bias, int act,
                                int64_t W, const uint16_t *init_state, int64_t L,
                                uint16_t *y, uint16_t *final_state, float *acc_out) {
  if (T < 0 || D < 0 || W < 1 || L < W - 1) return CCU_ORACLE_BAD_ARGS;
  if (act != CCU_ORACLE_ACT_IDENTITY && act != CCU_ORACLE_ACT_SILU) return CCU_ORACLE_BAD_ARGS;
  if (D == 0) return CCU_ORACLE_OK;
  if (weight == NULL || (T > 0 && (x_seq == NULL || y == NULL))) return CCU_ORACLE_BAD_ARGS;

  for (int64_t d = 0; d < D; ++d) {
    for (int64_t t = 0; t < T; ++t) {
      float acc = 0.0f;
      for (int64_t j = 0; j < W; ++j) {
        int64_t tau = t - (W - 1) + j; /* time of the input this tap sees */
        uint16_t v;
        if (tau >= 0) {
          v = x_seq[tau * D + d];
        } else {
          v = init_state ? init_state[d * L + (L + tau)] : 0x0000u;
        }
        float term = ccu_oracle_bf16_to_f32(v) * ccu_oracle_bf16_to_f32(weight[d * W + j]);
        acc = acc + term;
      }
      if (bias != NULL) acc = acc + ccu_oracle_bf16_to_f32(bias[d]);
      y[t * D + d] = ccu_oracle_f32_to_bf16(activation(acc, act));
      if (acc_out) acc_out[t * D + d] = acc;
    }
    if (final_state != NULL) {
      for (int64_t l = 0; l < L; ++l) {
        int64_t tau = T - L + l;
        uint16_t v;
        if (tau >= 0) {
          v = x_seq[tau * D + d];
        } else {
          v = init_state ? init_state[d * L + (L + tau)] : 0x0000u;
        }
        final_state[d * L + l] = v;
      }
    }
  }
  return CCU_ORACLE_OK;
}
