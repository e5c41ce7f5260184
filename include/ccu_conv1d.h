/*
 * ccu_conv1d -- depthwise causal conv1d decode update for NVIDIA GB300 (sm_103a).
 *
 * The operation is the decode step of a depthwise causal convolution with a
 * mutable state cache, as defined on the cuDNN page "Causal Conv1d Decode Update"
 * (introduction, update block). For every row n and channel d with slot s:
 *
 *     history            = concat(conv_state[s, d, :], x[n, d])        (L + 1 values)
 *     conv_state[s, d, :] = history[-L:]                                 (in place)
 *     acc                = sum_{j=0}^{W-1} history[-W + j] * weight[d, j] + bias[d]
 *     out[n, d]          = activation(acc)
 *
 * s = n when indices is NULL, else s = indices[n]; s == -1 marks a padding row whose
 * output is +0 and which reads and writes no state (same page, paragraph on
 * conv_state_indices). The bias is zero when omitted; identity and SiLU are the two
 * activations and are compiled as separate kernels (paragraph after the update block).
 *
 * Numerics: BF16 storage, FP32 accumulation in ascending tap order (j = 0..W-1, each
 * term a product of the two widened BF16 values, fused multiply-add allowed because a
 * BF16 x BF16 product is exact in FP32), bias added last, SiLU as a / (1 + exp(-a)) in
 * FP32, output rounded to BF16 to nearest-even. The state update is a bit copy.
 *
 * Conventions shared by every entry point below:
 *  - All tensor pointers are device-accessible memory owned by the caller: device memory,
 *    and for x and out of the update also host memory the device can address directly
 *    (pinned with cudaHostAlloc / cudaMallocHost, or registered with cudaHostRegister's
 *    mapped flag, under unified addressing). Host-resident x or out are read and written
 *    in place by the kernel (no staging copy); a call the library would give to the bulk
 *    family then runs on the vector family, which is found with cudaPointerGetAttributes
 *    on those two pointers (launching entry points only, large calls only). The library never
 *    allocates, frees or copies between host and device, and only
 *    ccu_conv1d_take_device_error synchronizes. The update entry points only enqueue
 *    kernels on `stream`, so an update call can be captured in a CUDA graph. The first
 *    launch of a bulk-copy kernel on a device (the bulk route of the update, the
 *    multi-token update and the prefill) sets that kernel's shared-memory limit with
 *    cudaFuncSetAttribute, so make one such call before capturing it. Launch
 *    errors are reported as CCU_ERR_CUDA; errors of the asynchronous execution surface
 *    at the caller's next synchronization.
 *  - `stream` is a cudaStream_t; NULL is the legacy default stream.
 *  - Kernels are launched with programmatic stream serialization (programmatic dependent
 *    launch), and each one waits for all earlier work on `stream` to complete
 *    (griddepcontrol.wait) before it touches memory, so the order is that of a plain
 *    launch: only the launch and start-up of consecutive calls overlap. Work the caller
 *    enqueues after a call sees its results, as usual, unless the caller launches its own
 *    kernel with programmatic dependent launch: such a kernel must wait itself
 *    (griddepcontrol.wait / cudaGridDependencySynchronize) before reading them.
 *  - BF16 tensors are passed as `const void*` / `void*` to 16-bit storage.
 *  - Every argument check happens before any launch; a declined call changes nothing.
 *  - Sizes are elements, not bytes. Strides are elements.
 *  - The functions are thread-safe; ccu_conv1d_last_error() is per calling thread.
 */
#ifndef CCU_CONV1D_H
#define CCU_CONV1D_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CCU_CONV1D_ABI_VERSION 2

/* Every entry point is exported from the shared library (the rest is hidden). */
#if defined(__GNUC__)
#define CCU_API __attribute__((visibility("default")))
#else
#define CCU_API
#endif

/* Same type as cudaStream_t; declared here so this header needs no CUDA header. */
typedef struct CUstream_st *ccu_stream_t;

/* Status of a call. The two declines mirror the typed declines of the cuDNN page
 * "Composing multi-kernel blocks" (section "The shape of a block"): a contract
 * violation versus a valid request that this library does not serve. */
typedef enum ccu_status {
  CCU_OK = 0,
  CCU_ERR_INVALID_ARGUMENT = 1, /* the arguments break the tensor contract */
  CCU_ERR_NOT_IMPLEMENTED = 2,  /* valid, but not served (e.g. an empty state, L = 0) */
  CCU_ERR_CUDA = 3              /* a CUDA launch or runtime call failed */
} ccu_status_t;

/* Activation. "identity" (or none) and "silu"/"swish" on the page map to these. */
typedef enum ccu_act { CCU_ACT_IDENTITY = 0, CCU_ACT_SILU = 1 } ccu_act_t;

/* Kernel families, for ccu_conv1d_update_ex and ccu_conv1d_select_route. AUTO lets the
 * library choose; the others force one family and decline (CCU_ERR_NOT_IMPLEMENTED)
 * when it cannot serve the arguments. */
typedef enum ccu_route {
  CCU_ROUTE_AUTO = 0,
  CCU_ROUTE_SCALAR = 1, /* one thread per (row, channel); any D, ld, L, W and layout */
  CCU_ROUTE_VECTOR = 2, /* 8 channels per thread, 16-byte vectors; D % 8 == 0, W = 2..4,
                           L <= 8 (multi-token widths 2 and 3: L <= 4) */
  CCU_ROUTE_STAGED = 3, /* shared-memory staged tiles; D % 8 == 0, W = 2..4, L <= 256 */
  CCU_ROUTE_BULK = 4,   /* persistent CTAs, bulk async copies through shared memory;
                           D % 8 == 0; width 4 with L <= 8 in both layouts, widths 2
                           and 3 with L <= 4 in the compact layout (multi-token: width 4,
                           compact, 3 <= L <= 8, T <= 8; prefill: widths 2 to 4) */
  CCU_ROUTE_COUNT = 5
} ccu_route_t;

/* Bits ORed into a device status word (the caller's, or the library's own, see
 * ccu_conv1d_take_device_error). */
#define CCU_DEVERR_RANGE 1     /* a slot index < -1 or >= S */
#define CCU_DEVERR_DUPLICATE 2 /* a non-padding slot used by more than one row */
#define CCU_DEVERR_TIMEOUT 4   /* a bounded wait inside a kernel gave up; that call's
                                  results are incomplete */

/*
 * ccu_conv1d_update -- one decode step, in place on conv_state.
 *
 * Defined by the update block in the introduction of "Causal Conv1d Decode Update";
 * argument meanings follow its "Semantic tensor contract" and the served subset in
 * "Current native implementation".
 *
 *   x           BF16, logical [N, D], element (n, d) at x[n * ld + d]. 16-byte aligned.
 *   ld          row stride of x in elements: ld == D (any D), or ld > D with ld % 8 == 0.
 *               Columns D..ld-1 are never read.
 *   conv_state  BF16, logical [S, D, L], element (s, d, l) at
 *               conv_state[s * stride_s + d * stride_d + l * stride_l]; updated in place.
 *               Two layouts are served: compact (stride_s, stride_d, stride_l) =
 *               (D * L, L, 1), and channel-last (L * D, 1, D), the layout of the final
 *               state of a full-sequence prefill. 16-byte aligned.
 *   weight      BF16, contiguous [D, W]. 16-byte aligned.
 *   bias        BF16, contiguous [D], or NULL for no bias. 16-byte aligned.
 *   act         CCU_ACT_IDENTITY or CCU_ACT_SILU.
 *   indices     int32 [N] slot per row, or NULL (row n uses slot n, which needs S >= N).
 *               -1 marks a padding row. Every other value must lie in [0, S) and appear
 *               at most once: these two preconditions are NOT checked here (use
 *               ccu_conv1d_update_checked / ccu_conv1d_check_indices). A repeated slot
 *               gives an unspecified state for that slot; an out-of-range one is
 *               undefined behaviour. 4-byte aligned.
 *   cache_seqlens  NULL for the linear state above, or int32 [N] (4-byte aligned) for a
 *               ring-buffer state, the use the page reserves this keyword for (section on
 *               cache_seqlens). Then conv_state[s, d, :] is a ring of L entries whose oldest
 *               entry sits at q = cache_seqlens[n] mod L: the history is ring[q], ...,
 *               ring[q+L-1] (mod L) followed by x, the output is computed from its last W
 *               entries as above, and the call writes only ring[q] = x (one entry per
 *               channel instead of L). cache_seqlens counts the inputs the row's slot has
 *               received and is not modified; the caller advances it. Values must be >= 0
 *               for non-padding rows (checked entry: a negative value is reported as
 *               CCU_DEVERR_RANGE and the row treated as padding). Pick the channel-last
 *               layout for a ring: there a step reads the W - 1 window planes and writes one
 *               plane, so it moves 12 bytes per element at W = 4; in the compact layout the
 *               L entries of a channel share their 32-byte sectors, so the whole slab is read
 *               and written, 16 bytes per element at L = 3 (large batch: 118 against 157 us).
 *   N, D, S     rows, channels, cache slots. N == 0 or D == 0 is a no-op.
 *   L, W        state length and filter width, L >= W - 1 (W >= 1). Served: every W with
 *               L >= 1 (the page's native width is 4; it names other widths as semantically
 *               valid). Widths 2, 3 and 4 run on every kernel family; W = 1 and W > 4 run on
 *               the scalar kernel (AUTO picks it). An empty state (W = 1, L = 0) is declined
 *               with CCU_ERR_NOT_IMPLEMENTED.
 *   out         BF16, contiguous [N, D], written for every row (+0 for padding rows).
 *               16-byte aligned; must not overlap any input.
 *
 * Returns CCU_OK after enqueueing, CCU_ERR_INVALID_ARGUMENT / CCU_ERR_NOT_IMPLEMENTED
 * without enqueueing anything, or CCU_ERR_CUDA if the launch failed.
 */
CCU_API ccu_status_t ccu_conv1d_update(const void *x, int64_t ld, void *conv_state, int64_t stride_s,
                               int64_t stride_d, int64_t stride_l, const void *weight,
                               const void *bias, ccu_act_t act, const int32_t *indices,
                               const int32_t *cache_seqlens, int64_t N, int64_t D, int64_t S,
                               int64_t L, int64_t W, void *out, ccu_stream_t stream);

/*
 * ccu_conv1d_update_checked -- ccu_conv1d_update that range-checks every slot on the
 * device instead of trusting it.
 *
 * The page's kernel traps on an index below -1 or past the cache ("Current native
 * implementation", last paragraph); a trap kills the CUDA context, so this library
 * reports instead: a row whose slot is < -1 or >= S is treated as a padding row (output
 * +0, no state access) and CCU_DEVERR_RANGE is ORed into *status_dev. Duplicate slots
 * are not detected here (see ccu_conv1d_update_checked_ex, or ccu_conv1d_check_indices).
 *
 *   status_dev  device int32 word, not cleared by the call: errors accumulate until the
 *               caller resets it. 4-byte aligned, must not be NULL.
 * Other arguments and returns as ccu_conv1d_update.
 */
CCU_API ccu_status_t ccu_conv1d_update_checked(const void *x, int64_t ld, void *conv_state,
                                       int64_t stride_s, int64_t stride_d, int64_t stride_l,
                                       const void *weight, const void *bias, ccu_act_t act,
                                       const int32_t *indices, const int32_t *cache_seqlens,
                                       int64_t N, int64_t D, int64_t S, int64_t L, int64_t W,
                                       void *out, int32_t *status_dev, ccu_stream_t stream);

/*
 * ccu_conv1d_update_checked_ex -- the checked update that also detects duplicate slots, in
 * the same launch, on the kernel family `route` selects.
 *
 * The page's kernel checks the slot indices on the device and traps on values below -1, on
 * slots past the cache and on non-padding slots repeated across rows ("Current native
 * implementation", last paragraph; conv_state_indices paragraph). Here nothing traps: a row
 * whose slot is out of range raises CCU_DEVERR_RANGE and a row whose slot another row has
 * already claimed raises CCU_DEVERR_DUPLICATE, and either row is then treated as a padding
 * row (output +0, no state access). Of the rows that share a slot exactly one updates it:
 * whichever claims it first, which may differ from one call to the next; so the state of a
 * repeated slot is one of its rows' updates, not a mix of them (the page leaves the update
 * non-transactional).
 *
 *   status_dev    device int32 word as in ccu_conv1d_update_checked; must not be NULL.
 *   slot_scratch  device int32 [S] (ccu_conv1d_slot_scratch_bytes(S) bytes), 4-byte
 *                 aligned, owned by the caller. The call clears it on `stream` before the
 *                 update (so its contents on entry do not matter) and leaves in it, for each
 *                 slot, 1 + the row that updated it (0: no row). May be NULL only when
 *                 indices is NULL (row n uses slot n: no slot can repeat). Calls that
 *                 overlap on the GPU must not share it.
 *   N             at most 2^31 - 2 (CCU_ERR_NOT_IMPLEMENTED beyond).
 *   route         CCU_ROUTE_AUTO or a family, as in ccu_conv1d_update_ex.
 * Other arguments and returns as ccu_conv1d_update.
 */
CCU_API ccu_status_t ccu_conv1d_update_checked_ex(const void *x, int64_t ld, void *conv_state,
                                                  int64_t stride_s, int64_t stride_d, int64_t stride_l,
                                                  const void *weight, const void *bias, ccu_act_t act,
                                                  const int32_t *indices, const int32_t *cache_seqlens,
                                                  int64_t N, int64_t D, int64_t S, int64_t L, int64_t W,
                                                  void *out, int32_t *status_dev, int32_t *slot_scratch,
                                                  int32_t route, ccu_stream_t stream);

/* Bytes of slot_scratch ccu_conv1d_update_checked_ex needs for S slots (4 * S; 0 for
 * S <= 0). */
CCU_API int64_t ccu_conv1d_slot_scratch_bytes(int64_t S);

/*
 * ccu_conv1d_update_ex -- the update with an explicit kernel family (for tests and A/B
 * benchmarks of the families on the same inputs).
 *
 *   status_dev  NULL for the unchecked update, else as in ccu_conv1d_update_checked.
 *   route       a ccu_route_t; a forced family that cannot serve the arguments returns
 *               CCU_ERR_NOT_IMPLEMENTED without launching.
 * Other arguments and returns as ccu_conv1d_update.
 */
CCU_API ccu_status_t ccu_conv1d_update_ex(const void *x, int64_t ld, void *conv_state, int64_t stride_s,
                                  int64_t stride_d, int64_t stride_l, const void *weight,
                                  const void *bias, ccu_act_t act, const int32_t *indices,
                                  const int32_t *cache_seqlens, int64_t N, int64_t D, int64_t S,
                                  int64_t L, int64_t W, void *out, int32_t *status_dev,
                                  int32_t route, ccu_stream_t stream);

/*
 * ccu_conv1d_select_route -- run every argument check of ccu_conv1d_update_ex and report,
 * in *chosen_route, the kernel family a call with these arguments would launch when x and
 * out are device memory. Touches no memory behind the pointers and makes no CUDA call, so
 * it also works without a GPU.
 *
 *   chosen_route  host int32 out-parameter; set only when CCU_OK is returned (to
 *                 CCU_ROUTE_AUTO for a no-op call with N == 0 or D == 0).
 */
CCU_API ccu_status_t ccu_conv1d_select_route(const void *x, int64_t ld, const void *conv_state,
                                     int64_t stride_s, int64_t stride_d, int64_t stride_l,
                                     const void *weight, const void *bias, ccu_act_t act,
                                     const int32_t *indices, const int32_t *cache_seqlens,
                                     int64_t N, int64_t D, int64_t S, int64_t L, int64_t W,
                                     const void *out, int32_t route, int32_t *chosen_route);

/*
 * ccu_conv1d_update_multi -- T tokens per row in one call (multi-token update, with the
 * state after every token on request, for speculative decoding).
 *
 * The cuDNN page "Causal Conv1d Decode Update" says a future multi-token extension can
 * admit x[N, D, Tstep] without changing the meaning of the state and the weights ("Semantic
 * tensor contract"), and lists multi-token updates and speculative intermediate-state
 * returns as not yet served ("Current native implementation"). This entry point serves
 * them with that meaning: the T tokens of row n are appended to the slot's history in
 * order; output t is the activation of the width-4 window ending at token t (plus bias);
 * the new state is the last L history entries. It equals T calls of ccu_conv1d_update
 * with x[:, :, 0], ..., x[:, :, T-1] (and, with cache_seqlens, cache_seqlens + t for token
 * t: token t lands at ring position (cache_seqlens[n] + t) mod L).
 *
 *   x            BF16, element (n, d, t) at x[n*x_stride_n + d*x_stride_d + t*x_stride_t];
 *                any non-negative strides. Channel-contiguous x (x_stride_d == 1, the
 *                other two strides multiples of 8, 16-byte aligned) runs the vector kernel.
 *   out          BF16, element (n, d, t) at out[n*out_stride_n + d*out_stride_d +
 *                t*out_stride_t]; must not overlap itself or any input. Padding rows get
 *                +0 for every token.
 *   intermediate_states  NULL, or BF16 [N, T, D, L] contiguous, 16-byte aligned: entry
 *                (n, t, d, l) is entry l of the slot's state (in the state's own order,
 *                linear or ring) after token t. Padding rows' entries are not written.
 *   T            tokens per row; T == 0 is a no-op.
 *   status_dev   NULL, or a device status word as in ccu_conv1d_update_checked.
 *   route        CCU_ROUTE_AUTO, CCU_ROUTE_SCALAR, CCU_ROUTE_VECTOR or CCU_ROUTE_BULK (others
 *                decline). BULK: the bulk-copy kernel (x rows and the state slab staged through
 *                shared memory by cp.async.bulk) for width 4, the compact state at L = 3..8,
 *                T <= 8, no intermediate states, x and out in device memory with the vector
 *                kernel's stride conditions; AUTO takes it for the compact ring state at
 *                L = 4, 5 and 7, where it measured faster. Its waits are bounded: on expiry it
 *                stops and raises CCU_DEVERR_TIMEOUT (the status word, else the library's own,
 *                read with ccu_conv1d_take_device_error).
 * Other arguments (state layouts, weight, bias, act, indices, cache_seqlens, N, D, S, L, W,
 * stream) and returns as ccu_conv1d_update.
 */
CCU_API ccu_status_t ccu_conv1d_update_multi(const void *x, int64_t x_stride_n, int64_t x_stride_d,
                                             int64_t x_stride_t, void *conv_state, int64_t stride_s,
                                             int64_t stride_d, int64_t stride_l, const void *weight,
                                             const void *bias, ccu_act_t act, const int32_t *indices,
                                             const int32_t *cache_seqlens, int64_t N, int64_t D,
                                             int64_t T, int64_t S, int64_t L, int64_t W, void *out,
                                             int64_t out_stride_n, int64_t out_stride_d,
                                             int64_t out_stride_t, void *intermediate_states,
                                             int32_t *status_dev, int32_t route, ccu_stream_t stream);

/*
 * ccu_causal_conv1d_fwd -- full-sequence prefill: the causal depthwise convolution over T
 * tokens of B sequences, and the final state the decode update continues from.
 *
 * The cuDNN page "Causal Conv1d Decode Update" sends full-sequence prefill to a separate
 * causal_conv1d operation whose width-four final state the update accepts directly, the
 * L = 3 state in the channel-last stride (3*D, 1, D) without a copy (introduction;
 * "Semantic tensor contract"). The page does not define that operation; this is the
 * update's definition applied to every token of a sequence:
 *
 *   out[b, d, t]  = act( sum_{j=0}^{W-1} weight[d, j] * xx(b, d, t - (W-1) + j) + bias[d] )
 *   xx(b, d, t)   = x[b, d, t] for t >= 0, initial_states[b, d, L + t] for t < 0 (zero when
 *                   initial_states is NULL)
 *   final_states[b, d, l] = xx(b, d, T - L + l),  l = 0..L-1
 *
 * So running the decode update on final_states with the next token continues the same
 * convolution. All tensors are device memory; element (b, d, t) of x is at
 * x[b*x_stride_b + d*x_stride_d + t*x_stride_t] (any non-negative strides; channel-
 * contiguous x and out -- stride_d == 1, the other strides multiples of 8 -- run the vector
 * or the bulk-copy kernel), and likewise for out, initial_states (b, d, l) and final_states
 * (b, d, l). For the
 * hand-off layout pass final strides (L*D, 1, D). initial_states and final_states may be
 * NULL; final_states must not overlap initial_states, x or out, and out must not overlap x.
 * Any W >= 1 with L >= W - 1 and L >= 1 (L = 0 is declined with CCU_ERR_NOT_IMPLEMENTED);
 * widths 2, 3 and 4 run on every kernel, other widths on the scalar kernel (AUTO picks it;
 * the vector and bulk routes decline them). B, D or T == 0 is a
 * no-op. route: CCU_ROUTE_AUTO, CCU_ROUTE_SCALAR, CCU_ROUTE_VECTOR or CCU_ROUTE_BULK (x staged
 * through shared memory by cp.async.bulk; the vector kernel's conditions; AUTO takes it from
 * B*D*T >= 2^20). The bulk kernel bounds its waits: on expiry it stops and raises
 * CCU_DEVERR_TIMEOUT, read with ccu_conv1d_take_device_error.
 * Returns as ccu_conv1d_update.
 */
CCU_API ccu_status_t ccu_causal_conv1d_fwd(const void *x, int64_t x_stride_b, int64_t x_stride_d,
                                           int64_t x_stride_t, const void *weight, const void *bias,
                                           ccu_act_t act, const void *initial_states,
                                           int64_t init_stride_b, int64_t init_stride_d,
                                           int64_t init_stride_l, int64_t B, int64_t D, int64_t T,
                                           int64_t L, int64_t W, void *out, int64_t out_stride_b,
                                           int64_t out_stride_d, int64_t out_stride_t,
                                           void *final_states, int64_t final_stride_b,
                                           int64_t final_stride_d, int64_t final_stride_l,
                                           int32_t route, ccu_stream_t stream);

/*
 * ccu_conv1d_check_indices -- validate a slot-index vector on the device without trapping.
 *
 * Checks the two preconditions of the conv_state_indices paragraph of "Causal Conv1d
 * Decode Update": every non-padding slot in [0, S) (else CCU_DEVERR_RANGE) and used by
 * one row only (else CCU_DEVERR_DUPLICATE); any number of -1 rows is allowed.
 *
 *   indices         device int32 [N], 4-byte aligned.
 *   bitmap_scratch  device scratch of ccu_conv1d_check_indices_scratch_bytes(S) bytes,
 *                   4-byte aligned, owned by the caller; the call clears it itself
 *                   (cudaMemsetAsync on `stream`) before use and leaves it dirty.
 *   status_dev      device int32 word; error bits are ORed in, never cleared.
 * N == 0 is a no-op. Calls that share a scratch buffer must not overlap on the GPU.
 */
CCU_API ccu_status_t ccu_conv1d_check_indices(const int32_t *indices, int64_t N, int64_t S,
                                      uint32_t *bitmap_scratch, int32_t *status_dev,
                                      ccu_stream_t stream);

/*
 * ccu_conv1d_check_indices_noalloc -- ccu_conv1d_check_indices without caller scratch.
 *
 * The cuDNN pages have no counterpart to this entry point; it exists for callers that
 * cannot hand the library a scratch buffer because they cannot allocate device memory:
 * a plugin that reaches this library through a C function table without access to the
 * host application's allocator, or a serving loop whose owner forbids cudaMalloc between
 * steps because it can synchronize the whole device and stall every other stream.
 *
 * The one-bit-per-slot bitmap lives in a fixed 128 KB array compiled into the library
 * (CCU_CHECK_INDICES_NOALLOC_MAX_SLOTS slots); every GPU on which the library's device
 * code is loaded keeps that array until the process exits. The call allocates nothing
 * and calls no allocating routine: it clears the bitmap words it needs with a
 * cudaMemsetAsync on `stream`, then runs the same check kernel on `stream`.
 *
 *   indices     device int32 [N], 4-byte aligned.
 *   N, S        rows and cache slots; N == 0 is a no-op. S greater than
 *               CCU_CHECK_INDICES_NOALLOC_MAX_SLOTS is declined with
 *               CCU_ERR_NOT_IMPLEMENTED (use ccu_conv1d_check_indices with your own
 *               bitmap instead).
 *   status_dev  device int32 word; CCU_DEVERR_RANGE / CCU_DEVERR_DUPLICATE are ORed in,
 *               never cleared.
 *
 * Each call whose stream is not being captured looks up the array's device address (a
 * runtime symbol lookup, which can load the library's device code onto that device), so
 * the address stays right after a cudaDeviceReset. A call on a stream that is being
 * captured cannot do that lookup and uses the address of the last uncaptured call on the
 * same device: make the first call on a device, and the first after a reset of it, outside
 * any stream capture (otherwise the call fails with CCU_ERR_CUDA). All calls in the process
 * share the one array per device, and it keeps the previous call's contents until the
 * next call clears it: calls that overlap on the GPU (on different streams, or from
 * different threads without ordering) race on it and can report false duplicates or miss
 * real ones. Order such calls, or use ccu_conv1d_check_indices with separate buffers.
 */
#define CCU_CHECK_INDICES_NOALLOC_MAX_SLOTS (1 << 20)
CCU_API ccu_status_t ccu_conv1d_check_indices_noalloc(const int32_t *indices, int64_t N, int64_t S,
                                                      int32_t *status_dev, ccu_stream_t stream);

/* Bytes of scratch ccu_conv1d_check_indices needs for S slots (one bit per slot, rounded
 * up to whole 32-bit words); 0 for S <= 0. */
CCU_API int64_t ccu_conv1d_check_indices_scratch_bytes(int64_t S);

/*
 * ccu_conv1d_take_device_error -- read and clear the library's own device error word.
 *
 * Kernels that wait on their own asynchronous copies (the bulk family of the update and
 * of the prefill) never wait without
 * limit; if a wait gives up they OR CCU_DEVERR_TIMEOUT into the caller's status word when
 * there is one (checked entry points), and otherwise into this per-process, per-device
 * word. This call SYNCHRONIZES the current device (it waits for all work issued so far,
 * then reads and clears the word in one atomic step and copies it to the host; a bit
 * raised by a kernel issued later is kept for the next call). Calls from several host
 * threads are serialized.
 *
 *   bits  host int32 out-parameter: the CCU_DEVERR_* bits raised since the last call.
 */
CCU_API ccu_status_t ccu_conv1d_take_device_error(int32_t *bits);

/* Static English text for a status code. Never NULL. */
CCU_API const char *ccu_status_string(ccu_status_t status);

/* Static name of a kernel family ("auto", "scalar", "vector", "staged", "bulk"). */
CCU_API const char *ccu_route_name(int32_t route);

/* Message of the last failed call on the calling thread (empty string if none). The
 * pointer stays valid until the thread's next call into this library. */
CCU_API const char *ccu_conv1d_last_error(void);

/* CCU_CONV1D_ABI_VERSION of the loaded library. */
CCU_API int32_t ccu_conv1d_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CCU_CONV1D_H */
