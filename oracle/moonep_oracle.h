/*
 * moonep_oracle.h -- plain, slow, single-threaded CPU oracle for the
 * MoonEP-style balanced expert-parallel hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links or calls this
 * library; only the test-suite, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * Conventions (all arrays are plain row-major host arrays):
 *   R ranks, E experts (L = E/R home experts per rank, expert e lives on rank
 *   e / L), K routes per token, S tokens per rank, C = S*K routes per rank,
 *   B prefetch slots per rank, tp = token_padding,
 *   NvS = roundup(C + (L+B)*(tp-1), tp) dispatched rows per rank.
 *   Global dispatched row of rank j, local row w:  g = j*NvS + w.
 *   bf16 values travel as their uint16 bit patterns.
 */
#ifndef MOONEP_ORACLE_H
#define MOONEP_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MO_OK = 0,
  MO_ERR_INVALID_ARG = -1,
  MO_ERR_BAD_EXPERT = -2,
  MO_ERR_HIST_MISMATCH = -3,
  MO_ERR_SLOTS = -4,
  MO_ERR_NOMEM = -5
};

/* NvS for a configuration, or a negative error. */
int64_t mo_nvs(int R, int E, int K, int S, int B, int tp);

/*
 * Balanced plan.  Inputs: topk [R,S,K] expert ids, tpe [R,E] (may be NULL).
 * Outputs (caller-allocated):
 *   dst [R,S*K]                signed global row (primary g, duplicate -(g+1))
 *   experts_to_copy [R,B]      expert id per prefetch slot or -1
 *   cu_seqlens [R,E+B]         inclusive padded end offsets (rank-local rows)
 *   zero_fill_ranges [R,E+B,2] [start,end) rank-local padding rows
 *   remote_stats [R,2]         {routes received from a remote group, slots used}
 *   dup_counts [R,2]           {duplicate routes, duplicate groups}
 *   dup_groups [R,NvS,3]       (primary row, first dup index, dup count), may be NULL
 *   dup_loffs [R,NvS]          duplicate rows grouped by group, may be NULL
 * Entries of dup_groups / dup_loffs beyond the counts are set to -1.
 * Returns MO_OK or a negative error (outputs then unspecified).
 */
int mo_plan(int R, int E, int K, int S, int B, int tp,
            const int32_t *topk, const int32_t *tpe,
            int32_t *dst, int32_t *experts_to_copy, int32_t *cu_seqlens,
            int32_t *zero_fill_ranges, int32_t *remote_stats,
            int32_t *dup_counts, int32_t *dup_groups, int32_t *dup_loffs);

/*
 * Dispatch over hidden columns [c0, c1) of rows with stride H elements.
 * hidden [R*S, H] bf16 bits, w_sk [R*S*K] fp32 (may be NULL),
 * out [R*NvS, H] bf16 bits, w_out [R*NvS] (may be NULL).
 */
void mo_dispatch(int R, int S, int K, int E, int B, int64_t NvS, int64_t H,
                 int64_t c0, int64_t c1, const int32_t *dst,
                 const int32_t *zero_fill_ranges, const uint16_t *hidden,
                 const float *w_sk, uint16_t *out, float *w_out);

/*
 * Combine for ntok tokens (global token ids r*S+s in `tokens`, or all R*S
 * tokens when tokens == NULL), hidden columns [c0, c1).
 * y [R*NvS, H] bf16 bits; out [ntok, H] bf16 bits (row i = tokens[i]),
 * w_nvs [R*NvS] / w_out [ntok, K] may be NULL.
 */
void mo_combine(int R, int S, int K, int64_t NvS, int64_t H, int64_t c0,
                int64_t c1, const int32_t *dst, const int64_t *tokens,
                int64_t ntok, const uint16_t *y, const float *w_nvs,
                uint16_t *out, float *w_out);

/* Deduplicated combine path: the duplicate prologue (primary rows become the
 * bf16 RNE of the fp32 k-order sum of the token's rows on their rank; y
 * modified in place) and the combine over primary routes only. */
void mo_fold_duplicates(int R, int S, int K, int64_t NvS, int64_t H, int64_t c0, int64_t c1,
                        const int32_t *dst, uint16_t *y);
void mo_combine_primaries(int R, int S, int K, int64_t NvS, int64_t H, int64_t c0, int64_t c1,
                          const int32_t *dst, const int64_t *tokens, int64_t ntok,
                          const uint16_t *y, const float *w_nvs, uint16_t *out, float *w_out);

/* Decode-path preparation, in place: ids < 0 -> expert 0 with weight 0;
 * rows s >= ntok[r] (ntok NULL: none) -> zero hidden row, expert 0, weight 0;
 * tpe [R,E] (optional) = per-rank counts of the resulting ids < E.
 * hidden [R,S,H] bf16 bits or NULL, topk [R,S,K], w [R,S,K] or NULL. */
void mo_prepare(int R, int S, int K, int E, int64_t H, const int32_t *ntok,
                uint16_t *hidden, int32_t *topk, float *w, int32_t *tpe);

/* Weight prefetch, one projection, columns [c0, c1) of rows of HHp elements.
 * W [E + R*B, HHp] bf16 bits. */
void mo_prefetch(int R, int E, int B, const int32_t *experts_to_copy,
                 int64_t HHp, int64_t c0, int64_t c1, uint16_t *W);

/* Weight prefetch of rows of any format (packed MXFP4 uint8, block scales,
 * bf16 seen as bytes): bytes [c0, c1) of rows of row_bytes bytes.
 * W [E + R*B, row_bytes] bytes. */
void mo_prefetch_bytes(int R, int E, int B, const int32_t *experts_to_copy,
                       int64_t row_bytes, int64_t c0, int64_t c1, uint8_t *W);

/* Gradient reduce, one projection, columns [c0, c1).
 * Gh [E, HHp] fp32, Gs [R*B, HHp] fp32. */
void mo_reduce(int R, int E, int B, const int32_t *experts_to_copy,
               int64_t HHp, int64_t c0, int64_t c1, float *Gh, float *Gs);

/* IEEE round-to-nearest-even of an fp32 value to bf16 (bits). */
uint16_t mo_f32_to_bf16(float f);

#ifdef __cplusplus
}
#endif
#endif
