/*
 * moonep.h -- C ABI of the GB300 (sm_103a) balanced expert-parallel hot path.
 *
 * One process, one GPU.  The R expert-parallel ranks of the method are R
 * logical partitions of this device's HBM: rank j's dispatched rows are rows
 * [j*NvS, (j+1)*NvS) of one [R*NvS, H] buffer, so a "remote" write of the
 * method is an ordinary scatter inside one allocation.
 *
 * Sources (page title, section):
 *   [API]    "MoonEP Public API Visual Guide": Notation; Buffer(...);
 *            Buffer.dispatch(...); Buffer.prefetch_weight(...);
 *            Buffer.combine(...); Buffer.reduce_grad(...);
 *            Buffer.hidden_nvsh_buffer_view; Buffer.router_weight_buffer_view;
 *            Buffer.destroy(); MoonEPCommPlan and MoonEPCommPlan.clone().
 *   [README] "MoonshotAI/MoonEP" README: items 1-3; "Weight buffer";
 *            "How to set B".
 *   [vLLM]   "vllm ... prepare_finalize.moonep": prepare() and finalize().
 *
 * Conventions shared by every entry point
 *   - Arrays are dense, row-major, and live in device memory unless stated.
 *     bf16 tensors travel as uint16_t bit patterns.
 *   - Every device pointer must be 16-byte aligned; H % 8 == 0 and, for the
 *     weight entry points, HHp % 8 == 0 (16-byte rows).  moonep_prefetch_rows
 *     takes any alignment and row size (other than 16-byte multiples on a
 *     16-byte aligned base, rows move byte by byte).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *     is stream-ordered and asynchronous: nothing synchronises with the host
 *     except moonep_get_status, moonep_ctx_destroy and moonep_plan_destroy
 *     (fixed shapes need no per-layer host synchronisation [README item 3]).
 *   - Return value: MOONEP_OK (0) or a negative MOONEP_ERR_*.  Errors found on
 *     the host (bad argument, destroyed context, CUDA launch failure) return
 *     at once and launch nothing.  Errors found by a kernel (bad expert id,
 *     histogram mismatch, too many slots, corrupted plan) are latched in the
 *     context's device status word and read with moonep_get_status; outputs of
 *     the failing call and of calls that use its plan are then unspecified but
 *     every kernel stays inside the buffers it was given.
 *   - The caller owns every tensor argument.  The library owns the context's
 *     scratch and status word, the plan's arrays and the optional zero-copy
 *     buffers behind moonep_hidden_view / moonep_weight_view.
 *   - One context plans one batch at a time: its planner scratch (counters,
 *     per-rank totals) is shared by its moonep_plan calls, so two of them
 *     must not overlap on the GPU (issue them on one stream, or order the
 *     streams); use one context per concurrent stream.  The copy entry points
 *     keep no state between calls and may overlap freely.
 *   - Kernels are launched with programmatic dependent launch: each waits
 *     for the previous kernel on its stream before touching memory, so
 *     stream order is kept as with plain launches.
 */
#ifndef MOONEP_H
#define MOONEP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOONEP_OK 0
#define MOONEP_ERR_INVALID_ARG (-1)   /* bad argument or configuration (host) */
#define MOONEP_ERR_BAD_EXPERT (-2)    /* a top-k id outside [0, E) (device) */
#define MOONEP_ERR_HIST_MISMATCH (-3) /* tokens_per_expert != recount of topk (device) */
#define MOONEP_ERR_SLOTS (-4)         /* a rank needs more than B slots (device) */
#define MOONEP_ERR_CUDA (-5)          /* a CUDA call failed (host) */
#define MOONEP_ERR_DESTROYED (-6)     /* context already destroyed (host) */
#define MOONEP_ERR_PLAN (-7)          /* plan row outside [0, R*NvS) (device) */
#define MOONEP_ERR_NOMEM (-8)         /* device allocation failed (host) */
#define MOONEP_ERR_TIMEOUT (-9)       /* a planner block gave up waiting (device) */

/* Constructor controls [API, Buffer(...)]: E % R == 0; B prefetch slots per
 * rank (B = E/R is what training needs [README, How to set B]; smaller B is
 * allowed and reported as MOONEP_ERR_SLOTS when a plan needs more);
 * token_padding = row alignment of every non-empty segment; num_sms caps the
 * SMs the copy kernels use (<= 0: the MOONEP_NUM_SMS environment variable
 * when set to a positive count, else every SM). */
typedef struct moonep_config {
  int R;             /* expert-parallel ranks (logical partitions), >= 1 */
  int E;             /* experts, multiple of R */
  int K;             /* routes per token, 1..32 */
  int S;             /* tokens per rank, >= 0 */
  int H;             /* hidden size, multiple of 8 */
  int B;             /* prefetch slots per rank, >= 0 */
  int token_padding; /* >= 1 */
  int num_sms;       /* <= 0: MOONEP_NUM_SMS, else all SMs */
} moonep_config;

typedef struct moonep_ctx moonep_ctx;

/* Plan flags */
#define MOONEP_PLAN_DUP_RECORDS 1 /* also build dup_groups / dup_loffs */

/* A communication plan [API, MoonEPCommPlan].  All pointers are device
 * arrays owned by the plan (moonep_plan_create / _clone / _destroy).
 *   dst[R, S*K]              encoded global row of every route i = s*K + k of
 *                            source rank r: g = j*NvS + w for the first route
 *                            of the token that lands on rank j, -(g+1) for a
 *                            later route of that token on the same rank
 *                            [API, Buffer.combine: positive/negative encoding]
 *   experts_to_copy[R, B]    expert held by each prefetch slot, -1 = unused
 *   cu_seqlens[R, E+B]       inclusive padded end offset of every segment,
 *                            rank-local rows, no leading 0 [API,
 *                            Buffer.dispatch; vLLM prepare: diff(cu_seqlens)]
 *   zero_fill_ranges[R,E+B,2] [start, end) padding rows of every segment
 *   remote_stats[R, 2]       {routes received from a remote home group,
 *                            prefetch slots used}
 *   dup_counts[R, 2]         {local duplicate routes, duplicate groups}
 *   dup_groups[R, NvS, 3]    (primary row, first index into dup_loffs, number
 *                            of duplicates), ascending primary row; valid
 *                            prefix dup_counts[j][1]; NULL unless the plan was
 *                            created with MOONEP_PLAN_DUP_RECORDS
 *   dup_loffs[R, NvS]        duplicate rows, grouped as dup_groups says; valid
 *                            prefix dup_counts[j][0]
 *   internal                 library-private tables (do not touch)
 * Segments of rank j: x = e for its home experts e in [j*E/R, (j+1)*E/R),
 * x = E + b for prefetch slot b; other segments are empty.  Rows
 * [cu_seqlens[j][E+B-1], NvS) of a rank (the tail) are never written. */
typedef struct moonep_comm_plan {
  int32_t *dst;
  int32_t *experts_to_copy;
  int32_t *cu_seqlens;
  int32_t *zero_fill_ranges;
  int32_t *remote_stats;
  int32_t *dup_counts;
  int32_t *dup_groups;
  int32_t *dup_loffs;
  int32_t *internal;
  int N;          /* routes per rank, S*K */
  int R, E, B, K, S;
  int NvS;        /* dispatched-row capacity per rank */
  int NvS_padded; /* row stride between ranks (== NvS) */
  int flags;
  size_t internal_bytes;
} moonep_comm_plan;

/* Sizes for a configuration: NvS = roundup(S*K + (E/R + B)*(tp-1), tp) and the
 * context's device scratch in bytes.  Any output pointer may be NULL. */
int moonep_query_sizes(const moonep_config *cfg, int *NvS, int *NvS_padded,
                       size_t *scratch_bytes);

/* Create a context on the current CUDA device [API, Buffer(...)]: validates
 * the configuration, allocates planner scratch and the status word, and, when
 * alloc_views != 0, the persistent [R*NvS, H] bf16 hidden buffer and [R*NvS]
 * fp32 weight buffer behind the zero-copy views.  *out is set on success. */
int moonep_ctx_create(const moonep_config *cfg, int alloc_views,
                      moonep_ctx **out);

/* Synchronise the device, free everything the context owns, mark it
 * destroyed [API, Buffer.destroy()].  Idempotent; NULL is accepted.  The
 * handle itself stays allocated so that later calls on it return
 * MOONEP_ERR_DESTROYED; moonep_ctx_free releases it. */
int moonep_ctx_destroy(moonep_ctx *ctx);
void moonep_ctx_free(moonep_ctx *ctx);
/* 1 once moonep_ctx_destroy has completed [API, Buffer.destroyed]. */
int moonep_ctx_destroyed(const moonep_ctx *ctx);

/* Allocate a plan's device arrays for the context's configuration.  flags:
 * MOONEP_PLAN_DUP_RECORDS. */
int moonep_plan_create(moonep_ctx *ctx, int flags, moonep_comm_plan *plan);
/* Free a plan's arrays (synchronises the device first); idempotent. */
int moonep_plan_destroy(moonep_comm_plan *plan);
/* Deep copy of every array and scalar [API, MoonEPCommPlan.clone()]: dst
 * must be a plan created for the same configuration and flags. */
int moonep_plan_clone(const moonep_comm_plan *src, moonep_comm_plan *dst, void *stream);

/* Online planner [API, Buffer.dispatch(...): the planning step that turns
 * every rank's S*K routes into the dst map; README items 1-2].
 *   topk  [R, S, K] int32 expert ids, each in [0, E)
 *   tpe   [R, E] int32 per-rank histogram, or NULL; when given it is checked
 *         against a recount of topk: a mismatch latches
 *         MOONEP_ERR_HIST_MISMATCH, and the plan is built from the recount
 * Fills every array of `plan`.  Deterministic: the same inputs give the same
 * plan, bit for bit.  Every rank receives exactly S*K routes; the experts a
 * rank prefetches come from one remote home group, at most B of them. */
int moonep_plan(moonep_ctx *ctx, const int32_t *topk, const int32_t *tpe,
                moonep_comm_plan *plan, void *stream);

/* Rank-local planner: the per-rank form of moonep_plan when each of the R
 * ranks is its own GPU [API, Buffer.dispatch(...): planning is collective,
 * every rank plans from the cross-rank statistics (MoonEPCommPlan
 * remote_stats); README, "How to set B"].  The one exchange step is an
 * all-gather of every rank's [E] tokens_per_expert into hist_all; each rank
 * then derives the same balance tables from hist_all and assigns only its own
 * routes, so no other routing data crosses between ranks.
 *   rank      source rank r of this call, 0 <= r < R
 *   topk_r    [S, K] int32 expert ids of rank r only
 *   hist_all  [R, E] int32 gathered per-rank histograms; row r is checked
 *             against a recount of topk_r (a mismatch latches
 *             MOONEP_ERR_HIST_MISMATCH; the tables stay those of hist_all,
 *             which every rank shares, and rank r's rows are unspecified)
 * Writes rank r's row of dst ([S*K] at plan->dst + r*S*K; other rows are not
 * touched), and experts_to_copy, cu_seqlens, zero_fill_ranges, remote_stats
 * and the plan's internal tables for every rank, equal to moonep_plan's.
 * dup_counts[j] is written with rank r's share: {duplicate routes of rank
 * r's tokens landing on rank j, their groups}; summed over the R calls (an
 * all-reduce across GPUs) it equals moonep_plan's.  The R calls together
 * give moonep_plan's plan, bit for bit.  Plans with MOONEP_PLAN_DUP_RECORDS,
 * and configurations whose planner tables do not fit in shared memory, are
 * refused (MOONEP_ERR_INVALID_ARG).  Rank-local calls of one context must
 * not overlap on the GPU (they share its scratch, as moonep_plan calls do). */
int moonep_plan_rank(moonep_ctx *ctx, int rank, const int32_t *topk_r,
                     const int32_t *hist_all, moonep_comm_plan *plan, void *stream);

/* Rank-local dispatch [API, Buffer.dispatch(...): tokens written straight
 * into the receiving ranks' buffers; README item 3]: rank r's tokens go to
 * their K destination rows in R rank windows, each its own allocation (on R
 * GPUs, peer pointers), and rank r zero-fills the padding rows of its own
 * window.  The R calls together give moonep_dispatch's rows.
 *   hidden_r   [S, H] bf16 rows of rank r
 *   w_r        [S, K] fp32 route weights of rank r, or NULL
 *   windows    HOST array of R device pointers: windows[j] = rank j's
 *              [NvS, H] bf16 rows (16-byte aligned)
 *   w_windows  HOST array of R device pointers to [NvS] fp32, or NULL
 *              (given exactly when w_r is)
 * Uses the plan's dst row r and its tables (moonep_plan or moonep_plan_rank). */
int moonep_dispatch_rank(moonep_ctx *ctx, const moonep_comm_plan *plan, int rank,
                         const uint16_t *hidden_r, const float *w_r,
                         uint16_t *const *windows, float *const *w_windows, void *stream);

/* Rank-local combine [API, Buffer.combine(...): the owner gathers its
 * tokens' K rows and reduces them; vLLM finalize(): an unweighted K-sum]:
 * out_r[s,:] = bf16_rne(fp32 sum over k = 0..K-1, in k order, of the row
 * |dst(r,s,k)| read from the rank window that holds it).
 *   y_windows  HOST array of R device pointers: rank j's [NvS, H] bf16 rows
 *   w_windows  HOST array of R device pointers to [NvS] fp32, or NULL
 *   out_r      [S, H] bf16 out
 *   w_out_r    [S, K] fp32 out (bit copies of the routes' weights), given
 *              exactly when w_windows is */
int moonep_combine_rank(moonep_ctx *ctx, const moonep_comm_plan *plan, int rank,
                        const uint16_t *const *y_windows, const float *const *w_windows,
                        uint16_t *out_r, float *w_out_r, void *stream);

/* Planner for callers that cannot allocate device memory.  The pages have no
 * counterpart: it exists for callers that must not call cudaMalloc, such as a
 * framework whose caching allocator owns (and accounts for) all device memory,
 * or a host path that cannot absorb cudaMalloc's implicit synchronisation.
 * It needs no context and no plan object and allocates nothing.
 *   cfg          as for moonep_ctx_create (H and num_sms are not used)
 *   topk, tpe    as for moonep_plan
 *   dst[R,S*K], experts_to_copy[R,B], cu_seqlens[R,E+B],
 *   zero_fill_ranges[R,E+B,2], remote_stats[R,2], dup_counts[R,2]
 *                caller-allocated device outputs, same contents as the
 *                fields of the same name that moonep_plan writes
 *   status       caller-allocated device int32: cleared by the call, then set
 *                to the first MOONEP_ERR_* a kernel meets (0 if none)
 * The planner's intermediate tables live in one file-scope device array of
 * 4 MiB (1 << 20 int32 words) that every GPU loading the library keeps until
 * the process exits; configurations whose tables do not fit (roughly
 * E*R*ceil(S*K/2048) + R*S*K + a few tables of E+B words) are rejected with
 * MOONEP_ERR_INVALID_ARG.  The first call on a device looks up that array's
 * device address, and the first call for each new (R, E, B) raises the
 * planner kernels' shared-memory limits, so make those calls before any
 * stream capture.  All calls share the array and a call overwrites what the last
 * one left there: calls that overlap on the GPU (on different streams, or
 * from several host threads without ordering) race and give wrong plans.
 * The plan it produces feeds no other entry point (they take a
 * moonep_comm_plan). */
int moonep_plan_noalloc(const moonep_config *cfg, const int32_t *topk,
                        const int32_t *tpe, int32_t *dst,
                        int32_t *experts_to_copy, int32_t *cu_seqlens,
                        int32_t *zero_fill_ranges, int32_t *remote_stats,
                        int32_t *dup_counts, int32_t *status, void *stream);

/* Fused-permute dispatch [API, Buffer.dispatch; README item 3].
 *   hidden      [R, S, H] bf16 source rows
 *   w_sk        [R, S, K] fp32 route weights, or NULL
 *   hidden_nvsh [R*NvS, H] bf16 out: row |dst| of every route = its token's
 *               row; padding rows zero; tail rows untouched
 *   w_nvs       [R*NvS] fp32 out, or NULL: route weight per row, 0 on padding
 *               (w_sk and w_nvs are both given or both NULL, else
 *               MOONEP_ERR_INVALID_ARG; an empty batch, R*S = 0, takes
 *               either without complaint)
 * Passing a saved plan again is the plan-reuse path (combine-backward
 * dispatch of an [R, S, H] gradient, weights NULL) [API, Buffer.dispatch:
 * a saved plan skips planning and ignores the routing inputs]. */
int moonep_dispatch(moonep_ctx *ctx, const moonep_comm_plan *plan,
                    const uint16_t *hidden, const float *w_sk,
                    uint16_t *hidden_nvsh, float *w_nvs, void *stream);

/* Combine [API, Buffer.combine; vLLM finalize: the K-sum is unweighted].
 *   y_nvsh   [R*NvS, H] bf16 expert outputs in dispatched order
 *   w_nvs    [R*NvS] fp32 or NULL
 *   out_sh   [R, S, H] bf16 out: out[r,s,:] = bf16_rne(fp32 sum over
 *            k = 0..K-1, in k order, of y[|dst(r,s,k)|,:])
 *   w_sk_out [R, S, K] fp32 out or NULL: w_nvs[|dst|] (bit copy); given
 *            together with w_nvs or not at all (any pair for an empty batch)
 * Reads only rows that dst names (never padding or tail rows). */
int moonep_combine(moonep_ctx *ctx, const moonep_comm_plan *plan,
                   const uint16_t *y_nvsh, const float *w_nvs,
                   uint16_t *out_sh, float *w_sk_out, void *stream);

/* Deduplicated dispatch [API, Buffer.dispatch: a token routed to several
 * experts on one rank is transferred once and expanded locally in an
 * epilogue].  Same arguments and results as moonep_dispatch, bit for bit,
 * in two launches: the copy writes the primary rows (dst >= 0) and every
 * route weight, then the expand epilogue copies each primary row to the
 * duplicate rows that plan->dup_groups / dup_loffs list for it.  Requires a
 * plan created with MOONEP_PLAN_DUP_RECORDS (else MOONEP_ERR_INVALID_ARG).
 * A record that points outside its rank sets MOONEP_ERR_PLAN in the status
 * word and is skipped. */
int moonep_dispatch_dedup(moonep_ctx *ctx, const moonep_comm_plan *plan,
                          const uint16_t *hidden, const float *w_sk,
                          uint16_t *hidden_nvsh, float *w_nvs, void *stream);

/* Deduplicated combine [API, Buffer.combine: duplicate rows are accumulated
 * into their primaries in fp32 before the gather].  Two launches:
 *   1. fold prologue, IN PLACE on y_nvsh: for every group of rank j,
 *      y[primary] = bf16_rne(fp32 y[primary] + y[dup_1] + ... ) in k order;
 *      the duplicate rows are left as they were;
 *   2. out[r,s,:] = bf16_rne(fp32 sum, in k order, over the token's primary
 *      routes only (dst >= 0; route 0 always is)); w_sk_out as moonep_combine.
 * The result can differ from moonep_combine by the fold's extra rounding
 * (at most 2^-7 * sum |y| per element).  Requires MOONEP_PLAN_DUP_RECORDS.
 * y_nvsh is written: a second call on the same buffer folds twice. */
int moonep_combine_dedup(moonep_ctx *ctx, const moonep_comm_plan *plan,
                         uint16_t *y_nvsh, const float *w_nvs,
                         uint16_t *out_sh, float *w_sk_out, void *stream);

/* Redundant-expert weight prefetch [API, Buffer.prefetch_weight; README,
 * Weight buffer].  W[p] (p < n_proj <= 4) is a device pointer to one
 * [E + R*B, HHp] bf16 tensor: rows [0, E) are the experts, rows E + j*B + b
 * are rank j's slots.  For every slot with experts_to_copy[j][b] = e >= 0:
 * row E + j*B + b = row e (bit copy).  Unused slots are not touched.
 * `W` itself is a host array of n_proj device pointers. */
int moonep_prefetch_weight(moonep_ctx *ctx, const moonep_comm_plan *plan,
                           int n_proj, uint16_t *const *W, int64_t HHp,
                           void *stream);

/* Weight prefetch of any row format [API, Buffer.prefetch_weight: packed
 * MXFP4 weights are uint8; optional block-scale tensors follow the same
 * leading E + B row convention and come as a complete gate/up/down set].
 * tensors[t] (t < n_tensors <= 8) is a device pointer to an [E + R*B] array
 * of rows of row_bytes[t] bytes each (packed MXFP4 [H, H'/2] bytes, E8M0
 * block scales [H, H'/32] bytes, bf16 [H, H'] as 2*H*H' bytes, ...).  For
 * every slot with experts_to_copy[j][b] = e >= 0 and every tensor: row
 * E + j*B + b = row e, byte for byte.  Unused slots are not touched.  A
 * tensor whose rows are 16-byte multiples on a 16-byte aligned base moves
 * 16-byte vectors, any other single bytes (correct, slower).  Pass the whole
 * set in one call: one launch covers every tensor.  `tensors` and
 * `row_bytes` are host arrays; a tensor with row_bytes 0 is skipped (its
 * pointer may be NULL). */
int moonep_prefetch_rows(moonep_ctx *ctx, const moonep_comm_plan *plan,
                         int n_tensors, void *const *tensors,
                         const int64_t *row_bytes, void *stream);

/* Decode-path preparation [vLLM, MoonEPPrepareAndFinalize: prepare() and
 * _pad_to_capacity]: the step's batch is padded to the context's static
 * capacity S, and invalid (negative) expert ids become expert 0 with zero
 * route weight (the planner has no sentinel for them), in place:
 *   num_tokens  HOST array [R]: valid tokens of each rank, 0 <= n <= S
 *               (NULL: S for every rank, only invalid ids are mapped)
 *   hidden      [R, S, H] bf16 or NULL, 16-byte aligned: rows s >= n of rank
 *               r are set to 0
 *   topk        [R, S, K] int32: ids < 0, and every id of rows s >= n, set
 *               to 0; ids >= E are left for the planner to report
 *   w_sk        [R, S, K] fp32 or NULL: the weights of those routes set to 0
 *   tokens_per_expert  [R, E] int32 out or NULL: per-rank counts of the
 *               prepared ids below E (the planner's tokens_per_expert)
 * Only padding rows and invalid routes are written. */
int moonep_prepare(moonep_ctx *ctx, const int32_t *num_tokens, uint16_t *hidden,
                   int32_t *topk, float *w_sk, int32_t *tokens_per_expert,
                   void *stream);

/* Gradient reduce of the redundant experts [API, Buffer.reduce_grad; README,
 * Weight buffer].  Gh[p] -> [E, HHp] fp32 home-expert gradients, Gs[p] ->
 * [R*B, HHp] fp32 slot gradients (the [R, B, H, H'] reduce buffer).  For
 * every expert e held by at least one slot:
 *   Gh[e] = Gh[e] + Gs[slot_1] + Gs[slot_2] + ...   (fp32, slots in
 *           ascending (rank, slot) order)
 * then every used slot is set to 0; unused slots are not touched.  `Gh` and
 * `Gs` are host arrays of n_proj (<= 4) device pointers. */
int moonep_reduce_redundant_grad(moonep_ctx *ctx, const moonep_comm_plan *plan,
                                 int n_proj, float *const *Gh,
                                 float *const *Gs, int64_t HHp, void *stream);

/* Zero-copy aliases [API, Buffer.hidden_nvsh_buffer_view and
 * router_weight_buffer_view]: device address of rank `rank`'s [NvS, H] bf16
 * window (row rank*NvS of the context's hidden buffer) and of its [NvS] fp32
 * weight window.  NULL if the context was created without views or the rank
 * is out of range.  Later calls overwrite what they hold. */
void *moonep_hidden_view(moonep_ctx *ctx, int rank);
void *moonep_weight_view(moonep_ctx *ctx, int rank);

/* Synchronise `stream`, return the first error any kernel latched since the
 * last call in *device_status (0 if none) and clear it.  After
 * MOONEP_ERR_TIMEOUT it also clears the planner's cross-block counters and
 * accumulators (a wait that ran out may leave them out of step), so the
 * context plans correctly again; re-plan before reusing a plan from that
 * call.  The return value is the host-side status of the query itself. */
int moonep_get_status(moonep_ctx *ctx, int *device_status, void *stream);

/* Static text for a status code. */
const char *moonep_strerror(int code);

/* Number of SMs the copy kernels use for this context. */
int moonep_num_sms(const moonep_ctx *ctx);

#ifdef __cplusplus
}
#endif
#endif /* MOONEP_H */
