/*
 * CPU oracle for the depthwise causal conv1d decode update.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library. The product path (the CUDA library
 * and its Python binding) never calls it, links it or shares code with it.
 *
 * Source of truth: the cuDNN page "Causal Conv1d Decode Update" -- the update
 * block in its introduction (history, shift, weighted sum, activation), the
 * paragraphs on bias/activation and on conv_state_indices that follow it, and
 * the section "Semantic tensor contract".
 *
 * BF16 tensors are passed as uint16_t bit patterns. All arrays are host memory
 * owned by the caller. Single-threaded, no SIMD intrinsics, plain loops.
 */
#ifndef CCU_ORACLE_H
#define CCU_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  CCU_ORACLE_OK = 0,
  CCU_ORACLE_BAD_ARGS = -1,     /* a size, stride or pointer breaks the contract */
  CCU_ORACLE_BAD_INDICES = -2,  /* a slot index out of range or repeated */
  CCU_ORACLE_NO_MEMORY = -3
};

enum { CCU_ORACLE_ACT_IDENTITY = 0, CCU_ORACLE_ACT_SILU = 1 };

/* Flags returned by ccu_oracle_check_indices. */
enum { CCU_ORACLE_IDX_RANGE = 1, CCU_ORACLE_IDX_DUPLICATE = 2 };

/* One decode step, in place on conv_state.
 *   x          [N, ld] BF16 bits; element (n, d) at n*ld + d
 *   conv_state logical [S, D, L] BF16 bits at s*stride_s + d*stride_d + l*stride_l
 *   weight     [D, W] BF16 bits, contiguous
 *   bias       [D] BF16 bits or NULL (no bias)
 *   act        CCU_ORACLE_ACT_IDENTITY or CCU_ORACLE_ACT_SILU
 *   indices    int32 [N] or NULL (row n uses slot n); -1 marks a padding row
 *   out        [N, D] BF16 bits, contiguous
 *   acc_out    optional float [N, D]: the FP32 accumulator before activation
 *              (0 for padding rows); NULL to skip
 * Returns CCU_ORACLE_OK, or a negative code without touching anything. */
int ccu_oracle_conv1d_update(const uint16_t *x, int64_t ld, uint16_t *conv_state,
                             int64_t stride_s, int64_t stride_d, int64_t stride_l,
                             const uint16_t *weight, const uint16_t *bias, int act,
                             const int32_t *indices, int64_t N, int64_t D, int64_t S,
                             int64_t L, int64_t W, uint16_t *out, float *acc_out);

/* One decode step with conv_state[s, d, :] used as a ring of L entries (the
 * circular-buffer state the page reserves the cache_seqlens keyword for). With
 * p = cache_seqlens[n] mod L, the slot's history, oldest first, is
 * ring[p], ring[p+1], ..., ring[p+L-1] (indices mod L), followed by x[n, d]; the sum
 * takes its last W entries as in ccu_oracle_conv1d_update, and the step writes only
 * ring[p] = x[n, d] (the oldest entry). cache_seqlens [N] holds the number of inputs each
 * row's slot has already received; it must be >= 0 for non-padding rows and is not
 * modified. Other arguments as ccu_oracle_conv1d_update. */
int ccu_oracle_conv1d_update_circular(const uint16_t *x, int64_t ld, uint16_t *conv_state,
                                      int64_t stride_s, int64_t stride_d, int64_t stride_l,
                                      const uint16_t *weight, const uint16_t *bias, int act,
                                      const int32_t *indices, const int32_t *cache_seqlens,
                                      int64_t N, int64_t D, int64_t S, int64_t L, int64_t W,
                                      uint16_t *out, float *acc_out);

/* T tokens per row in one call: the multi-token form of the update, x[N, D, T].
 * history = concat(state entries, x[n, d, 0], ..., x[n, d, T-1]); output t is computed
 * from the W history entries ending at token t; the new state is the last L entries of
 * the history. With cache_seqlens (ring-buffer state), token t is written over ring
 * position (cache_seqlens[n] + t) mod L, each token seeing the ring as it stands.
 *   x        element (n, d, t) at x[n*sxn + d*sxd + t*sxt]
 *   out      element (n, d, t) at out[n*son + d*sod + t*sot]
 *   inter    NULL, or [N, T, D, L] compact: inter[((n*T + t)*D + d)*L + l] is entry l of
 *            the state (in the state's own order, linear or ring) after token t; padding
 *            rows leave their entries untouched
 * Other arguments as ccu_oracle_conv1d_update / ccu_oracle_conv1d_update_circular
 * (cache_seqlens NULL for the linear state). */
int ccu_oracle_conv1d_update_multi(const uint16_t *x, int64_t sxn, int64_t sxd, int64_t sxt,
                                   uint16_t *conv_state, int64_t stride_s, int64_t stride_d,
                                   int64_t stride_l, const uint16_t *weight, const uint16_t *bias,
                                   int act, const int32_t *indices, const int32_t *cache_seqlens,
                                   int64_t N, int64_t D, int64_t T, int64_t S, int64_t L, int64_t W,
                                   uint16_t *out, int64_t son, int64_t sod, int64_t sot,
                                   uint16_t *inter);

/* Full-sequence causal depthwise convolution over T steps, written directly
 * from the convolution sum (no state shifting):
 *   y[t, d] = act( sum_{j=0}^{W-1} w[d, j] * xx(t - (W-1) + j, d) + b[d] )
 * where xx(t, d) = x_seq[t, d] for t >= 0 and init_state[d, L + t] for t < 0
 * (zero when init_state is NULL). final_state[d, l] = xx(T - L + l, d).
 *   x_seq [T, D], y [T, D], init_state / final_state [D, L] (compact, BF16 bits)
 *   acc_out optional float [T, D]. */
int ccu_oracle_full_causal_conv(const uint16_t *x_seq, int64_t T, int64_t D,
                                const uint16_t *weight, const uint16_t *bias, int act,
                                int64_t W, const uint16_t *init_state, int64_t L,
                                uint16_t *y, uint16_t *final_state, float *acc_out);

/* Index preconditions of the decode batch: each non-padding slot in [0, S) and
 * used once; -1 may repeat. Returns an OR of CCU_ORACLE_IDX_* (0 when valid),
 * or CCU_ORACLE_NO_MEMORY. */
int ccu_oracle_check_indices(const int32_t *indices, int64_t N, int64_t S);

/* The oracle's own scalar conversions, exported so the tests can pin them. */
float ccu_oracle_bf16_to_f32(uint16_t bits);
uint16_t ccu_oracle_f32_to_bf16(float value);
float ccu_oracle_silu(float acc);

#ifdef __cplusplus
}
#endif

#endif /* CCU_ORACLE_H */
