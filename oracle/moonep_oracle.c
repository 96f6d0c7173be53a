/*
 * moonep_oracle.c -- plain, slow, single-threaded CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product path.  Written for a
 * reader who checks it against the pages by eye: no blocking, no fusion, one
 * step per loop, in the order the method states them.  Compile with
 * -ffp-contract=off (there are no multiplies, but keep adds unfused anyway).
 *
 * Sources:
 *   [API]    "MoonEP Public API Visual Guide" -- sections Notation,
 *            Buffer(...), Buffer.dispatch(...), Buffer.prefetch_weight(...),
 *            Buffer.combine(...), Buffer.reduce_grad(...),
 *            MoonEPCommPlan and MoonEPCommPlan.clone().
 *   [README] "MoonshotAI/MoonEP" README -- items 1-3 (perfect balance, online
 *            planning, zero copy), "Weight buffer", "How to set B".
 *   [vLLM]   "vllm...fused_moe.prepare_finalize.moonep" -- prepare() (the
 *            tokens_per_expert bincount and diff(cu_seqlens) segment sizes),
 *            finalize() (combine performs an unweighted K-sum),
 *            MoonEPExpertWeightLayout (unused slots are -1 and never re-zeroed).
 *
 * The pages fix the planner's invariants but not its algorithm.  This file
 * follows one deterministic rule (the "chain" rule), step by step:
 *   1. P_e = routes to expert e ordered by (source rank r, s, k); T_e = |P_e|.
 *      Q_j = P_{jL} || ... || P_{jL+L-1} (home group of rank j, expert order).
 *   2. rem[j] = |Q_j|.  While some rank has rem < C: receiver = lowest rank
 *      with rem < C, donor = lowest rank with rem > C, d = C - rem[receiver];
 *      record piece (donor -> receiver, d); rem[donor] -= d; rem[receiver] = C.
 *   3. keep_j = |Q_j| - (routes rank j donated); rank j keeps Q_j[0, keep_j).
 *   4. Donor l's pieces, in recording order, take consecutive runs of Q_l
 *      starting at keep_l.
 *   5. On a receiver, the experts present in its run get slots 0,1,.. in
 *      ascending id (experts_to_copy); other slots are -1.  More than B
 *      distinct experts is an error (cannot happen when B >= E/R).
 *   6. Segments x = 0..E+B-1 on rank j: x = e for home experts (kept routes),
 *      x = E+b for slot b (received routes), else empty.  Padded length =
 *      ceil(n/tp)*tp; cu_seqlens = inclusive prefix sum; padding rows are
 *      [start+n, end).
 *   7. Rows inside a segment follow Q order.
 *   8. dst = j*NvS + row for the first route of a token that lands on rank j;
 *      a later route of the same token on the same rank is a local duplicate,
 *      encoded -(g+1).
 */
#include "moonep_oracle.h"

#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ bf16 */

/* IEEE 754 round-to-nearest-even of binary32 to the 16-bit bfloat16 format:
 * keep the top 16 bits, rounding on the 16 dropped bits; ties go to the even
 * result.  NaNs stay NaN (quiet bit forced, sign and top payload kept). */
uint16_t mo_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t upper = u >> 16;
  uint32_t lower = u & 0xffffu;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
  return (uint16_t)upper;
}

static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* ------------------------------------------------------------------ sizes */

/* NvS is a row capacity [API, Notation]: the S*K real rows plus the padding
 * of the segments [README, Usage notation].  A rank holds at most L home segments and
 * B slot segments, each padded by at most tp-1 rows. */
int64_t mo_nvs(int R, int E, int K, int S, int B, int tp) {
  if (R < 1 || E < 1 || K < 1 || S < 0 || B < 0 || tp < 1 || E % R) return -1;
  int64_t L = E / R;
  int64_t raw = (int64_t)S * K + (L + B) * (int64_t)(tp - 1);
  return (raw + tp - 1) / tp * tp;
}

/* ------------------------------------------------------------------ plan */

typedef struct { int donor, recv, d, run_start; } piece_t;

int mo_plan(int R, int E, int K, int S, int B, int tp,
            const int32_t *topk, const int32_t *tpe,
            int32_t *dst, int32_t *etc, int32_t *cu, int32_t *zfr,
            int32_t *remote_stats, int32_t *dup_counts,
            int32_t *dup_groups, int32_t *dup_loffs) {
  int64_t NvS = mo_nvs(R, E, K, S, B, tp);
  if (NvS < 0) return MO_ERR_INVALID_ARG;
  const int L = E / R;
  const int64_t C = (int64_t)S * K;
  const int64_t N = (int64_t)R * C;
  const int EB = E + B;
  int status = MO_OK;

  /* Expert ids must name an expert: the planner has no sentinel for invalid
   * ids [vLLM, _pad_to_capacity]. */
  for (int64_t i = 0; i < N; i++)
    if (topk[i] < 0 || topk[i] >= E) return MO_ERR_BAD_EXPERT;

  /* tokens_per_expert is the source rank's histogram [API, Buffer.dispatch;
   * vLLM prepare(): bincount of topk].  Recount and compare. */
  int64_t *cnt = calloc((size_t)R * E, sizeof *cnt);
  int64_t *T = calloc((size_t)E, sizeof *T);
  int64_t *G = calloc((size_t)R, sizeof *G);
  int64_t *qoff = calloc((size_t)E, sizeof *qoff);
  int64_t *Qstart = calloc((size_t)R + 1, sizeof *Qstart);
  int64_t *Q = malloc((size_t)(N ? N : 1) * sizeof *Q);       /* route ids */
  int64_t *fill = calloc((size_t)E, sizeof *fill);
  piece_t *pieces = calloc((size_t)R + 1, sizeof *pieces);
  int64_t *rem = calloc((size_t)R, sizeof *rem);
  int64_t *donated = calloc((size_t)R, sizeof *donated);
  int64_t *keep = calloc((size_t)R, sizeof *keep);
  int *recv_piece = malloc((size_t)R * sizeof *recv_piece);
  int64_t *nseg = calloc((size_t)R * EB, sizeof *nseg);
  int64_t *segstart = calloc((size_t)R * EB, sizeof *segstart);
  int64_t *segfill = calloc((size_t)R * EB, sizeof *segfill);
  int *route_rank = malloc((size_t)(N ? N : 1) * sizeof *route_rank);
  int64_t *route_row = malloc((size_t)(N ? N : 1) * sizeof *route_row);
  if (!cnt || !T || !G || !qoff || !Qstart || !Q || !fill || !pieces || !rem ||
      !donated || !keep || !recv_piece || !nseg || !segstart || !segfill ||
      !route_rank || !route_row) {
    status = MO_ERR_NOMEM;
    goto out;
  }

  for (int r = 0; r < R; r++)
    for (int64_t i = 0; i < C; i++) cnt[(int64_t)r * E + topk[r * C + i]]++;
  if (tpe)
    for (int64_t i = 0; i < (int64_t)R * E; i++)
      if ((int64_t)tpe[i] != cnt[i]) { status = MO_ERR_HIST_MISMATCH; goto out; }

  /* Step 1: T_e, G_j, the offset of P_e inside Q_home(e), and Q itself.
   * Walking routes in (r, s, k) order and appending to their expert's run
   * orders every P_e by (source rank, s, k). */
  for (int e = 0; e < E; e++)
    for (int r = 0; r < R; r++) T[e] += cnt[(int64_t)r * E + e];
  for (int j = 0; j < R; j++) {
    int64_t acc = 0;
    for (int e = j * L; e < (j + 1) * L; e++) { qoff[e] = acc; acc += T[e]; }
    G[j] = acc;
  }
  for (int j = 0; j < R; j++) Qstart[j + 1] = Qstart[j] + G[j];
  for (int r = 0; r < R; r++)
    for (int s = 0; s < S; s++)
      for (int k = 0; k < K; k++) {
        int64_t id = (int64_t)r * C + (int64_t)s * K + k;
        int e = topk[id];
        int h = e / L;
        Q[Qstart[h] + qoff[e] + fill[e]] = id;
        fill[e]++;
      }

  /* Step 2: every rank ends with exactly C routes [README item 1].  Each
   * round fills one receiver to C from one donor, so a receiver only ever
   * hosts one remote home group [README, How to set B]. */
  int npieces = 0;
  for (int j = 0; j < R; j++) { rem[j] = G[j]; recv_piece[j] = -1; }
  for (int round = 0; round <= R; round++) {
    int recv = -1, donor = -1;
    for (int j = 0; j < R; j++) if (rem[j] < C) { recv = j; break; }
    if (recv < 0) break;
    for (int j = 0; j < R; j++) if (rem[j] > C) { donor = j; break; }
    if (donor < 0 || npieces >= R) { status = MO_ERR_INVALID_ARG; goto out; }
    int64_t d = C - rem[recv];
    pieces[npieces].donor = donor;
    pieces[npieces].recv = recv;
    pieces[npieces].d = (int)d;
    recv_piece[recv] = npieces;
    npieces++;
    rem[donor] -= d;
    rem[recv] = C;
    donated[donor] += d;
  }

  /* Step 3 and 4: the kept prefix, then each donor's runs in recording order. */
  for (int j = 0; j < R; j++) keep[j] = G[j] - donated[j];
  {
    int64_t *cursor = calloc((size_t)R, sizeof *cursor);
    if (!cursor) { status = MO_ERR_NOMEM; goto out; }
    for (int j = 0; j < R; j++) cursor[j] = keep[j];
    for (int p = 0; p < npieces; p++) {
      pieces[p].run_start = (int)cursor[pieces[p].donor];
      cursor[pieces[p].donor] += pieces[p].d;
    }
    free(cursor);
  }

  /* Step 5: slots.  experts_to_copy[rank] maps each slot to a global expert,
   * -1 when unused [API, Buffer.prefetch_weight]. */
  for (int64_t i = 0; i < (int64_t)R * B; i++) etc[i] = -1;
  for (int j = 0; j < R; j++) { remote_stats[2 * j] = 0; remote_stats[2 * j + 1] = 0; }
  for (int p = 0; p < npieces; p++) {
    int l = pieces[p].donor, j = pieces[p].recv, nslots = 0, last = -1;
    for (int64_t q = pieces[p].run_start; q < pieces[p].run_start + pieces[p].d; q++) {
      int e = topk[Q[Qstart[l] + q]];
      if (e != last) {
        if (nslots >= B) { status = MO_ERR_SLOTS; goto out; }
        etc[(int64_t)j * B + nslots] = e;
        nslots++;
        last = e;
      }
    }
    remote_stats[2 * j] = pieces[p].d;
    remote_stats[2 * j + 1] = nslots;
  }

  /* Step 6: segment sizes, cu_seqlens (padded end offset of every physical
   * group [API, Buffer.dispatch table]; diff with a leading 0 gives the
   * segment sizes [vLLM, prepare]) and padding ranges. */
  for (int j = 0; j < R; j++) {
    for (int64_t q = 0; q < keep[j]; q++) nseg[(int64_t)j * EB + topk[Q[Qstart[j] + q]]]++;
    int p = recv_piece[j];
    if (p >= 0) {
      int l = pieces[p].donor;
      for (int64_t q = pieces[p].run_start; q < pieces[p].run_start + pieces[p].d; q++) {
        int e = topk[Q[Qstart[l] + q]];
        int b = 0;
        while (etc[(int64_t)j * B + b] != e) b++;
        nseg[(int64_t)j * EB + E + b]++;
      }
    }
    int64_t end = 0;
    for (int x = 0; x < EB; x++) {
      int64_t n = nseg[(int64_t)j * EB + x];
      int64_t padded = (n + tp - 1) / tp * tp;
      segstart[(int64_t)j * EB + x] = end;
      zfr[((int64_t)j * EB + x) * 2 + 0] = (int32_t)(end + n);
      end += padded;
      zfr[((int64_t)j * EB + x) * 2 + 1] = (int32_t)end;
      cu[(int64_t)j * EB + x] = (int32_t)end;
    }
  }

  /* Step 7: rows in Q order inside each segment. */
  for (int j = 0; j < R; j++) {
    for (int64_t q = 0; q < keep[j]; q++) {
      int64_t id = Q[Qstart[j] + q];
      int64_t sx = (int64_t)j * EB + topk[id];
      route_rank[id] = j;
      route_row[id] = segstart[sx] + segfill[sx];
      segfill[sx]++;
    }
    int p = recv_piece[j];
    if (p >= 0) {
      int l = pieces[p].donor;
      for (int64_t q = pieces[p].run_start; q < pieces[p].run_start + pieces[p].d; q++) {
        int64_t id = Q[Qstart[l] + q];
        int e = topk[id];
        int b = 0;
        while (etc[(int64_t)j * B + b] != e) b++;
        int64_t sx = (int64_t)j * EB + E + b;
        route_rank[id] = j;
        route_row[id] = segstart[sx] + segfill[sx];
        segfill[sx]++;
      }
    }
  }

  /* Step 8: dst and its positive/negative encoding [API, Buffer.combine],
   * plus the duplicate-route metadata [API, MoonEPCommPlan]. */
  for (int j = 0; j < R; j++) { dup_counts[2 * j] = 0; dup_counts[2 * j + 1] = 0; }
  for (int r = 0; r < R; r++)
    for (int s = 0; s < S; s++) {
      int64_t base = (int64_t)r * C + (int64_t)s * K;
      for (int k = 0; k < K; k++) {
        int j = route_rank[base + k];
        int64_t g = (int64_t)j * NvS + route_row[base + k];
        int primary = 1;
        for (int k2 = 0; k2 < k; k2++)
          if (route_rank[base + k2] == j) primary = 0;
        dst[base + k] = primary ? (int32_t)g : (int32_t)(-(g + 1));
        if (!primary) dup_counts[2 * j]++;
      }
      for (int k = 0; k < K; k++) {
        int j = route_rank[base + k];
        int first = 1, ndup = 0;
        for (int k2 = 0; k2 < k; k2++) if (route_rank[base + k2] == j) first = 0;
        if (!first) continue;
        for (int k2 = k + 1; k2 < K; k2++) if (route_rank[base + k2] == j) ndup++;
        if (ndup) dup_counts[2 * j + 1]++;
      }
    }

  /* Duplicate groups per rank: one record (primary row, first index into
   * dup_loffs, number of duplicates) per primary that has duplicates, in
   * ascending primary row; the duplicates' rows follow in k order. */
  if (dup_groups || dup_loffs) {
    if (dup_groups) for (int64_t i = 0; i < (int64_t)R * NvS * 3; i++) dup_groups[i] = -1;
    if (dup_loffs) for (int64_t i = 0; i < (int64_t)R * NvS; i++) dup_loffs[i] = -1;
    /* prim_tok[j*NvS + row] = route id of the primary that owns `row`. */
    int64_t *prim_tok = malloc((size_t)R * NvS * sizeof *prim_tok);
    if (!prim_tok) { status = MO_ERR_NOMEM; goto out; }
    for (int64_t i = 0; i < (int64_t)R * NvS; i++) prim_tok[i] = -1;
    for (int64_t id = 0; id < N; id++)
      if (dst[id] >= 0) prim_tok[dst[id]] = id;
    for (int j = 0; j < R; j++) {
      int64_t ngroup = 0, ndup = 0;
      for (int64_t w = 0; w < NvS; w++) {
        int64_t id = prim_tok[(int64_t)j * NvS + w];
        if (id < 0) continue;
        int64_t base = id - id % K;
        int count = 0;
        for (int k2 = (int)(id % K) + 1; k2 < K; k2++)
          if (route_rank[base + k2] == j) {
            if (dup_loffs) dup_loffs[(int64_t)j * NvS + ndup + count] = (int32_t)route_row[base + k2];
            count++;
          }
        if (!count) continue;
        if (dup_groups) {
          int32_t *rec = dup_groups + ((int64_t)j * NvS + ngroup) * 3;
          rec[0] = (int32_t)w;
          rec[1] = (int32_t)ndup;
          rec[2] = count;
        }
        ngroup++;
        ndup += count;
      }
    }
    free(prim_tok);
  }

out:
  free(cnt); free(T); free(G); free(qoff); free(Qstart); free(Q); free(fill);
  free(pieces); free(rem); free(donated); free(keep); free(recv_piece);
  free(nseg); free(segstart); free(segfill); free(route_rank); free(route_row);
  return status;
}

/* ------------------------------------------------------------- prepare */

/* Decode-path preparation, per rank r, following the padding step of the
 * vLLM prepare/finalize page [vLLM, MoonEPPrepareAndFinalize._pad_to_capacity
 * and prepare()]: (1) an invalid (negative) expert id becomes expert 0 with
 * zero route weight; (2) the batch is padded to the static capacity S: rows
 * s >= ntok[r] get a zero hidden row, expert 0 and zero weight; (3)
 * tokens_per_expert is the per-rank count of the resulting ids (ids >= E are
 * left for the planner to report and are not counted).  hidden, w and tpe
 * may be NULL. */
void mo_prepare(int R, int S, int K, int E, int64_t H, const int32_t *ntok,
                uint16_t *hidden, int32_t *topk, float *w, int32_t *tpe) {
  for (int r = 0; r < R; r++) {
    const int n = ntok ? ntok[r] : S;
    for (int s = 0; s < S; s++) {
      const int64_t t = (int64_t)r * S + s;
      for (int k = 0; k < K; k++) {
        const int64_t i = t * K + k;
        if (topk[i] < 0) {
          topk[i] = 0;
          if (w) w[i] = 0.0f;
        }
      }
      if (s >= n) {
        if (hidden)
          for (int64_t c = 0; c < H; c++) hidden[t * H + c] = 0;
        for (int k = 0; k < K; k++) {
          topk[t * K + k] = 0;
          if (w) w[t * K + k] = 0.0f;
        }
      }
    }
    if (tpe) {
      for (int e = 0; e < E; e++) tpe[(int64_t)r * E + e] = 0;
      for (int64_t i = (int64_t)r * S * K; i < (int64_t)(r + 1) * S * K; i++)
        if (topk[i] < E) tpe[(int64_t)r * E + topk[i]]++;
    }
  }
}

/* ------------------------------------------------------------ dispatch */

static int64_t decode_row(int32_t d) { return d >= 0 ? (int64_t)d : -(int64_t)d - 1; }

/* Every route's hidden row lands on its dispatched row, every route weight is
 * scattered, and padding rows are zero-filled [API, Buffer.dispatch].  On one
 * device the locally deduplicated routes are written directly rather than
 * expanded in an epilogue; the bytes that land are the same. */
void mo_dispatch(int R, int S, int K, int E, int B, int64_t NvS, int64_t H,
                 int64_t c0, int64_t c1, const int32_t *dst,
                 const int32_t *zfr, const uint16_t *hidden,
                 const float *w_sk, uint16_t *out, float *w_out) {
  int64_t C = (int64_t)S * K;
  for (int r = 0; r < R; r++)
    for (int s = 0; s < S; s++)
      for (int k = 0; k < K; k++) {
        int64_t id = (int64_t)r * C + (int64_t)s * K + k;
        int64_t g = decode_row(dst[id]);
        for (int64_t c = c0; c < c1; c++)
          out[g * H + c] = hidden[((int64_t)r * S + s) * H + c];
        if (w_sk && w_out) w_out[g] = w_sk[id];
      }
  int EB = E + B;
  for (int j = 0; j < R; j++)
    for (int x = 0; x < EB; x++) {
      int64_t a = zfr[((int64_t)j * EB + x) * 2], b = zfr[((int64_t)j * EB + x) * 2 + 1];
      for (int64_t w = a; w < b; w++) {
        int64_t g = (int64_t)j * NvS + w;
        for (int64_t c = c0; c < c1; c++) out[g * H + c] = 0;
        if (w_out) w_out[g] = 0.0f;
      }
    }
}

/* ------------------------------------------------------------- combine */

/* Gather the K routed rows of every token through dst and sum them: an
 * unweighted K-sum, since route weights are applied inside the expert compute
 * [vLLM, finalize; API, Buffer.combine].  fp32 adds in k order starting from
 * the k = 0 row, one rounding to bf16 at the end.  Weights travel back as bit
 * copies through the same encoding. */
void mo_combine(int R, int S, int K, int64_t NvS, int64_t H, int64_t c0,
                int64_t c1, const int32_t *dst, const int64_t *tokens,
                int64_t ntok, const uint16_t *y, const float *w_nvs,
                uint16_t *out, float *w_out) {
  (void)NvS;
  if (!tokens) ntok = (int64_t)R * S;
  for (int64_t i = 0; i < ntok; i++) {
    int64_t t = tokens ? tokens[i] : i;
    const int32_t *d = dst + t * K;
    for (int64_t c = c0; c < c1; c++) {
      float acc = bf16_to_f32(y[decode_row(d[0]) * H + c]);
      for (int k = 1; k < K; k++) acc = acc + bf16_to_f32(y[decode_row(d[k]) * H + c]);
      out[i * H + c] = mo_f32_to_bf16(acc);
    }
    if (w_nvs && w_out)
      for (int k = 0; k < K; k++) w_out[i * K + k] = w_nvs[decode_row(d[k])];
  }
}

/* ------------------------------------------- deduplicated combine path */

/* Duplicate prologue [API, Buffer.combine: a prologue accumulates duplicate
 * physical rows into their primary rows in fp32, then the main kernel
 * gathers and reduces]: for every token and every rank holding more than one
 * of its routes, the primary row (the token's first route on that rank, the
 * one with dst >= 0) becomes the bf16 RNE rounding of the fp32 sum, in k
 * order, of the token's rows on that rank.  Duplicate rows are left as they
 * are.  y [R*NvS, H] bf16 bits, modified in place; columns [c0, c1). */
void mo_fold_duplicates(int R, int S, int K, int64_t NvS, int64_t H, int64_t c0, int64_t c1,
                        const int32_t *dst, uint16_t *y) {
  for (int64_t t = 0; t < (int64_t)R * S; t++) {
    const int32_t *d = dst + t * K;
    for (int k = 0; k < K; k++) {
      if (d[k] < 0) continue;  /* primary route */
      const int64_t g = d[k];
      const int64_t j = g / NvS;
      int dups = 0;
      for (int k2 = k + 1; k2 < K; k2++)
        if (d[k2] < 0 && decode_row(d[k2]) / NvS == j) dups++;
      if (!dups) continue;
      for (int64_t c = c0; c < c1; c++) {
        float acc = bf16_to_f32(y[g * H + c]);
        for (int k2 = k + 1; k2 < K; k2++)
          if (d[k2] < 0 && decode_row(d[k2]) / NvS == j)
            acc = acc + bf16_to_f32(y[decode_row(d[k2]) * H + c]);
        y[g * H + c] = mo_f32_to_bf16(acc);
      }
    }
  }
}

/* The main combine of the deduplicated path: out[t] = bf16 RNE of the fp32
 * sum, in k order, over the token's primary routes only (each one already
 * holds its rank's fold).  Weights are gathered for every route as in
 * mo_combine.  out [ntok, H] for the tokens listed (all when tokens is NULL). */
void mo_combine_primaries(int R, int S, int K, int64_t NvS, int64_t H, int64_t c0, int64_t c1,
                          const int32_t *dst, const int64_t *tokens, int64_t ntok,
                          const uint16_t *y, const float *w_nvs, uint16_t *out, float *w_out) {
  (void)NvS;
  if (!tokens) ntok = (int64_t)R * S;
  for (int64_t i = 0; i < ntok; i++) {
    const int64_t t = tokens ? tokens[i] : i;
    const int32_t *d = dst + t * K;
    for (int64_t c = c0; c < c1; c++) {
      float acc = bf16_to_f32(y[(int64_t)d[0] * H + c]);  /* route 0 is always primary */
      for (int k = 1; k < K; k++)
        if (d[k] >= 0) acc = acc + bf16_to_f32(y[(int64_t)d[k] * H + c]);
      out[i * H + c] = mo_f32_to_bf16(acc);
    }
    if (w_nvs && w_out)
      for (int k = 0; k < K; k++) w_out[i * K + k] = w_nvs[decode_row(d[k])];
  }
}

/* ------------------------------------------------------------ prefetch */

/* Copy expert e's weight into every slot that names it; unused slots (-1) are
 * skipped and keep their stale contents [API, Buffer.prefetch_weight; vLLM,
 * MoonEPExpertWeightLayout]. */
void mo_prefetch(int R, int E, int B, const int32_t *etc, int64_t HHp,
                 int64_t c0, int64_t c1, uint16_t *W) {
  for (int j = 0; j < R; j++)
    for (int b = 0; b < B; b++) {
      int e = etc[j * B + b];
      if (e < 0) continue;
      int64_t slot = (int64_t)E + (int64_t)j * B + b;
      for (int64_t c = c0; c < c1; c++) W[slot * HHp + c] = W[(int64_t)e * HHp + c];
    }
}

/* Byte-row prefetch: the same slot fill for any row format, rows of
 * row_bytes bytes, bytes [c0, c1) of each row.  Packed MXFP4 weights are
 * uint8 (two 4-bit codes per byte) and their optional block-scale tensors
 * share the leading E + B row convention, so a slot row receives its source
 * row's bytes unchanged [API, Buffer.prefetch_weight: packed MXFP4 weights
 * use uint8; block scales as a complete gate/up/down set]. */
void mo_prefetch_bytes(int R, int E, int B, const int32_t *etc, int64_t row_bytes,
                       int64_t c0, int64_t c1, uint8_t *W) {
  for (int j = 0; j < R; j++)
    for (int b = 0; b < B; b++) {
      int e = etc[j * B + b];
      if (e < 0) continue;
      const int64_t dst_row = (int64_t)E + (int64_t)j * B + b;
      for (int64_t c = c0; c < c1; c++) W[dst_row * row_bytes + c] = W[(int64_t)e * row_bytes + c];
    }
}

/* -------------------------------------------------------------- reduce */

/* For every expert with at least one slot copy: start from its own gradient,
 * add each matching slot gradient in (rank, slot) order, write the sum back;
 * then clear every consumed slot [API, Buffer.reduce_grad; README, Weight
 * buffer (reduce buffer)]. */
void mo_reduce(int R, int E, int B, const int32_t *etc, int64_t HHp,
               int64_t c0, int64_t c1, float *Gh, float *Gs) {
  for (int e = 0; e < E; e++) {
    int used = 0;
    for (int i = 0; i < R * B; i++) if (etc[i] == e) used = 1;
    if (!used) continue;
    for (int64_t c = c0; c < c1; c++) {
      float acc = Gh[(int64_t)e * HHp + c];
      for (int j = 0; j < R; j++)
        for (int b = 0; b < B; b++)
          if (etc[j * B + b] == e) acc = acc + Gs[((int64_t)j * B + b) * HHp + c];
      Gh[(int64_t)e * HHp + c] = acc;
    }
  }
  for (int i = 0; i < R * B; i++) {
    if (etc[i] < 0) continue;
    for (int64_t c = c0; c < c1; c++) Gs[(int64_t)i * HHp + c] = 0.0f;
  }
}
