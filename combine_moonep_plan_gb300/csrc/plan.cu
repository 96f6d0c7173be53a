// Online planner: S*K routes per rank -> a perfectly balanced plan.
//
// "MoonEP Public API Visual Guide", Buffer.dispatch(...): the planning step
// maps every route to its destination row (the dst map), lays out E+B padded
// segments per rank and records the local duplicates.  "MoonshotAI/MoonEP" README,
// items 1-2: every rank receives exactly S*K routes; a GPU planning kernel;
// "How to set B": the redundant experts of a rank come from at most one remote
// home group.
//
// The rule (deterministic):
//   P_e = routes to expert e ordered by (source rank r, s, k); Q_j = the routes
//   of rank j's home experts, expert by expert.  Ranks with more than C = S*K
//   routes donate: repeatedly the lowest-index rank below C is filled up to C
//   by the lowest-index rank above C (one piece per receiver).  A donor keeps a
//   prefix of Q_j; its pieces are consecutive runs after that prefix.  On a
//   receiver the experts of its run take slots 0,1,... in ascending id.
//   Segments: x = e (home expert, kept routes), x = E + b (slot b), each
//   padded to token_padding; rows inside a segment follow Q order.  A later
//   route of a token that lands on a rank already holding one of its routes
//   is a local duplicate, encoded -(g+1).
//
// Kernels:
//   plan_fused_kernel<IT>  the usual path, one cooperative launch: tile CTAs
//                          count and order their routes, all CTAs meet once,
//                          each runs the balance step's routing stage on its
//                          own copy of the per-rank totals and assigns its
//                          routes; two extra CTAs write the plan's tables
//                          and the experts-with-copies list.
//   The tile path (tables too large for one CTA, more than 64 ranks, or more
//   tiles than SMs):
//   K1 plan_hist_kernel    per 2048-route tile: per-expert counts and each
//                          route's ordinal among same-expert routes of the tile
//                          (warp-aggregated with one ballot per key bit, stable).
//   K2 plan_balance_kernel one CTA: column scans of the tile counts (the
//                          position of every tile inside every P_e), the chain
//                          balance, slots, segments, cu_seqlens, padding and
//                          the experts-with-copies list.
//   K3 plan_assign_kernel  one thread per token: Q position -> (rank, row),
//                          duplicate encoding, dup_counts.
//   K4 plan_dup_count_kernel, plan_dup_write_kernel (optional, either path)
//                          one CTA per (1024-row tile, rank): the tile's group
//                          and duplicate counts, then compact duplicate
//                          records in ascending primary row.
#include <map>
#include <mutex>

#include "moonep_internal.cuh"

namespace moonep {
namespace {

struct PlanDims {
  int R, E, K, S, B, tp, L, C, EB, NvS, TPR, G;
  int Bm;  // usable slots per rank: min(B, L)
};

struct PlanOut {
  int32_t *dst, *etc, *cu, *zfr, *remote_stats, *dup_counts, *dup_groups, *dup_loffs;
};

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Lanes of the warp holding the same key (0 <= key < 2^nbits), from one
// ballot per key bit: a fixed cost however many distinct keys the warp holds
// (match.any slows down as the number of distinct values grows).
__device__ __forceinline__ unsigned match_key(int key, int nbits) {
  unsigned m = 0xffffffffu;
  for (int b = 0; b < nbits; b++) {
    const bool bit = (key >> b) & 1;
    const unsigned bb = __ballot_sync(0xffffffffu, bit);
    m &= bit ? bb : ~bb;
  }
  return m;
}

// Bits needed for keys 0..E (E itself marks an invalid route).
__host__ __device__ __forceinline__ int key_bits(int E) {
  int b = 1;
  while ((1 << b) <= E) b++;
  return b;
}

// ------------------------------------------------------------------ K1

__global__ void __launch_bounds__(kPlanThreads)
plan_hist_kernel(const int32_t *__restrict__ topk, PlanDims d, int32_t *__restrict__ hist,
                 int32_t *__restrict__ ord, int32_t *meta, int32_t *status) {
  extern __shared__ int32_t sh[];  // [warps][E] running counts
  constexpr int kWarps = kPlanThreads / 32;
  const int g = blockIdx.x;
  const int r = g / d.TPR, t = g % d.TPR;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kWarps * d.E; i += kPlanThreads) sh[i] = 0;
  __syncthreads();

  int32_t *h = sh + warp * d.E;
  const int32_t *src = topk + (int64_t)r * d.C;
  const unsigned lt = lanemask_lt();
  const int nbits = key_bits(d.E);
  int e_reg[kPlanItems], o_reg[kPlanItems];
  bool bad = false;
#pragma unroll
  for (int c = 0; c < kPlanItems; c++) {
    const int i = t * kTile + warp * (32 * kPlanItems) + c * 32 + lane;
    int e = -1;
    if (i < d.C) {
      e = __ldg(src + i);
      if (e < 0 || e >= d.E) {
        bad = true;
        e = -1;
      }
    }
    const unsigned m = match_key(e >= 0 ? e : d.E, nbits);
    int base = 0;
    if (e >= 0) base = h[e];
    __syncwarp();
    if (e >= 0 && (m & lt) == 0) h[e] = base + __popc(m);
    __syncwarp();
    e_reg[c] = e;
    o_reg[c] = base + __popc(m & lt);
  }
  if (bad) {
    atomicOr(meta + kMetaErr, kErrBadExpert);
    set_status(status, MOONEP_ERR_BAD_EXPERT);
  }
  __syncthreads();
  // Exclusive scan over warps (warp w's routes precede warp w+1's).
  for (int e = threadIdx.x; e < d.E; e += kPlanThreads) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < kWarps; w++) {
      const int v = sh[w * d.E + e];
      sh[w * d.E + e] = run;
      run += v;
    }
    hist[(int64_t)e * d.G + g] = run;
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < kPlanItems; c++) {
    const int i = t * kTile + warp * (32 * kPlanItems) + c * 32 + lane;
    if (i < d.C) ord[(int64_t)r * d.C + i] = e_reg[c] >= 0 ? h[e_reg[c]] + o_reg[c] : 0;
  }
}

// ------------------------------------------------------------------ K2

constexpr int kBalThreads = 1024;
constexpr int kMaxR = kMaxRanks;

// Per-rank and per-piece state of the balance step (shared memory).
struct BalSmall {
  int G[kMaxR];           // routes of rank j's home group
  int keep[kMaxR];        // prefix of Q_j the home rank keeps
  int recv_piece[kMaxR];  // piece (chain order) rank j receives, -1 if none
  int nslots[kMaxR];      // slots rank j uses
  int donor[kMaxR], recv[kMaxR], len[kMaxR], start[kMaxR];  // pieces, chain order
  int pf[kMaxR], pc[kMaxR];             // per donor: first entry and count below
  int ps[kMaxR], pl[kMaxR], pr[kMaxR];  // pieces grouped by donor: Q start, length, receiver
  int part[2][32];                      // per-warp partial sums of the block scans
  int np, err, U;
};

// Tables of the balance step, one entry per expert, per (rank, donor-local
// expert), per slot or per segment.  Segments are numbered rank by rank: the
// rank's L home experts, then its Bm = min(B, L) usable slots (a rank
// receives one piece, from one home group, so it never fills more than L
// slots).  All pointers are generic: shared memory, or global memory when the
// tables are too large.
struct BalTables {
  int32_t *T;        // [E] routes per expert
  int32_t *Q;        // [E] offset of P_e inside Q_home(e)
  int32_t *home_rb;  // [E] row of Q position 0 of expert e on its home rank
  int32_t *slot_b;   // [R*L] slot of (receiver j, donor-local expert u), -1 if none
  int32_t *slot_rb;  // [R*L] row of Q position 0 of that slot's expert on rank j
  int32_t *etc;      // [R*Bm] expert held by slot b of rank j, -1 if none
  int32_t *n;        // [R*(L+Bm)] valid rows per segment
  int32_t *start;    // [R*(L+Bm)+1] padded rows, then their exclusive prefix
  int32_t *padx;     // [R*(L+Bm)+1] padding rows, then their exclusive prefix
  int32_t *rcnt;     // [E+1] slot copies per expert, then first index in the reduce list
  int32_t *rhas;     // [E+1] expert has copies, then its index among such experts
};

__device__ __forceinline__ BalTables bal_tables(int32_t *base, const PlanDims &d) {
  const int nseg = d.E + d.R * d.Bm;
  BalTables t;
  t.T = base;
  t.Q = t.T + d.E;
  t.home_rb = t.Q + d.E;
  t.slot_b = t.home_rb + d.E;
  t.slot_rb = t.slot_b + d.E;
  t.etc = t.slot_rb + d.E;
  t.n = t.etc + d.R * d.Bm;
  t.start = t.n + nseg;
  t.padx = t.start + nseg + 1;
  t.rcnt = t.padx + nseg + 1;
  t.rhas = t.rcnt + d.E + 1;
  return t;
}

// Exclusive prefix sums of a[0..cnt) and b[0..cnt) in place, by a whole block
// of kBalThreads threads (each thread takes a contiguous run, then the runs
// are scanned); a[cnt] and b[cnt] receive the totals when `totals` is set.
// With tp > 0, a[i] is first replaced by n rounded up to tp and b[i] by the
// rounding's padding, where n = a[i].
__device__ void block_scan2(int32_t *a, int32_t *b, int cnt, int tp, bool totals,
                            int (*part)[32]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (cnt + kBalThreads - 1) / kBalThreads;
  const int b0 = min(cnt, tid * per), b1 = min(cnt, b0 + per);
  int sa = 0, sb = 0;
  for (int i = b0; i < b1; i++) {
    int va = a[i], vb = b[i];
    if (tp > 0) {
      const int p = (va + tp - 1) / tp * tp;
      vb = p - va;
      va = p;
      a[i] = va;
      b[i] = vb;
    }
    sa += va;
    sb += vb;
  }
  const int ia = warp_incl_scan(sa), ib = warp_incl_scan(sb);
  if (lane == 31) {
    part[0][warp] = ia;
    part[1][warp] = ib;
  }
  __syncthreads();
  if (warp == 0) {
    const int wa = part[0][lane], wb = part[1][lane];
    const int xa = warp_incl_scan(wa), xb = warp_incl_scan(wb);
    part[0][lane] = xa - wa;
    part[1][lane] = xb - wb;
    if (lane == 31 && totals) {
      a[cnt] = xa;
      b[cnt] = xb;
    }
  }
  __syncthreads();
  int ra = part[0][warp] + ia - sa, rb = part[1][warp] + ib - sb;
  for (int i = b0; i < b1; i++) {
    const int va = a[i], vb = b[i];
    a[i] = ra;
    b[i] = rb;
    ra += va;
    rb += vb;
  }
  __syncthreads();
}

// Stage 1 of the balance step, from the per-expert totals t.T: offsets inside
// the home groups, the chain balance (pieces), slots, segment sizes, their
// padded starts, and the row bases the route assignment needs.  Called by a
// whole block of kBalThreads threads; err_in holds the error bits found so
// far.  Writes only t and s.
// The balance step's initial table values (no input needed, so a caller may
// run this early, before the per-expert totals are known).
__device__ __forceinline__ void balance_init(const PlanDims &d, const BalTables &t, BalSmall &s) {
  const int tid = threadIdx.x;
  const int R = d.R, L = d.L, Bm = d.Bm, LB = L + Bm;
  for (int i = tid; i < R * L; i += kBalThreads) {
    t.slot_b[i] = -1;
    t.slot_rb[i] = 0;
  }
  for (int i = tid; i < R * Bm; i += kBalThreads) t.etc[i] = -1;
  for (int i = tid; i < R * LB; i += kBalThreads) {
    t.n[i] = 0;
    t.start[i] = 0;
  }
  for (int j = tid; j < R; j += kBalThreads) {
    s.recv_piece[j] = -1;
    s.nslots[j] = 0;
  }
}

// inited: balance_init already ran, and a block barrier followed it.
__device__ void balance_route(const PlanDims &d, const BalTables &t, BalSmall &s, int err_in,
                              bool inited = false) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kBalThreads / 32;
  const int R = d.R, E = d.E, L = d.L, B = d.B, Bm = d.Bm, LB = L + Bm, C = d.C;

  if (tid == 0) {
    s.err = err_in;
    s.np = 0;
  }
  if (!inited) balance_init(d, t, s);
  // Phase B: offset of P_e inside Q_home(e) (one warp per home group), G_j.
  for (int j = warp; j < R; j += kWarps) {
    int carry = 0;
    for (int u0 = 0; u0 < L; u0 += 32) {
      const int u = u0 + lane;
      const int v = u < L ? t.T[j * L + u] : 0;
      const int incl = warp_incl_scan(v);
      if (u < L) t.Q[j * L + u] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s.G[j] = carry;
  }
  __syncthreads();

  // Phase C: the chain balance on one warp (lane j holds rank j, and j + 32
  // when R > 32):
  // each round fills the lowest-index rank below C from the lowest-index rank
  // above C; at most R rounds.
  if (warp == 0 && R <= 32) {
    // lane j holds rank j; the loop body is uniform (no branch around a
    // warp vote), which keeps a round to a few votes
    int rem = lane < R ? s.G[lane] : C, don = 0, np = 0;
    for (int round = 0; round <= R; round++) {
      const unsigned rb = __ballot_sync(0xffffffffu, rem < C);
      if (!rb) break;
      const unsigned db = __ballot_sync(0xffffffffu, rem > C);
      if (!db || np >= R) {  // only reachable from a broken histogram
        if (lane == 0) s.err |= kErrHist;
        break;
      }
      const int recv = __ffs(rb) - 1, donor = __ffs(db) - 1;
      const int dd = C - __shfl_sync(0xffffffffu, rem, recv);
      if (lane == 0) {
        s.donor[np] = donor;
        s.recv[np] = recv;
        s.len[np] = dd;
        s.recv_piece[recv] = np;
      }
      np++;
      if (lane == donor) {
        rem -= dd;
        don += dd;
      }
      if (lane == recv) rem = C;
    }
    if (lane < R) s.keep[lane] = s.G[lane] - don;
    if (lane == 0) s.np = np;
  } else if (warp == 0) {
    int rem0 = lane < R ? s.G[lane] : C, rem1 = lane + 32 < R ? s.G[lane + 32] : C;
    int don0 = 0, don1 = 0, np = 0;
    for (int round = 0; round <= R; round++) {
      const unsigned rb0 = __ballot_sync(0xffffffffu, rem0 < C);
      const unsigned rb1 = __ballot_sync(0xffffffffu, rem1 < C);
      if (!rb0 && !rb1) break;
      const unsigned db0 = __ballot_sync(0xffffffffu, rem0 > C);
      const unsigned db1 = __ballot_sync(0xffffffffu, rem1 > C);
      if ((!db0 && !db1) || np >= R) {  // only reachable from a broken histogram
        if (lane == 0) s.err |= kErrHist;
        break;
      }
      const int recv = rb0 ? __ffs(rb0) - 1 : 32 + __ffs(rb1) - 1;
      const int donor = db0 ? __ffs(db0) - 1 : 32 + __ffs(db1) - 1;
      const int rr = recv < 32 ? __shfl_sync(0xffffffffu, rem0, recv)
                               : __shfl_sync(0xffffffffu, rem1, recv - 32);
      const int dd = C - rr;
      if (lane == 0) {
        s.donor[np] = donor;
        s.recv[np] = recv;
        s.len[np] = dd;
        s.recv_piece[recv] = np;
      }
      np++;
      if (lane == (donor & 31)) {
        if (donor < 32) {
          rem0 -= dd;
          don0 += dd;
        } else {
          rem1 -= dd;
          don1 += dd;
        }
      }
      if (lane == (recv & 31)) {
        if (recv < 32)
          rem0 = C;
        else
          rem1 = C;
      }
    }
    if (lane < R) s.keep[lane] = s.G[lane] - don0;
    if (lane + 32 < R) s.keep[lane + 32] = s.G[lane + 32] - don1;
    if (lane == 0) s.np = np;
  }
  __syncthreads();

  // Phase D: per donor, its range in the donor-grouped piece list; per piece
  // (one warp each): where its run starts (after the donor's kept prefix and
  // its earlier pieces), its place in that list, and the receiver's slots;
  // per home expert: its kept routes.
  const int np_all = s.np;
  for (int l = tid; l < R; l += kBalThreads) {
    int first = 0, count = 0;
    for (int q = 0; q < np_all; q++) {
      first += s.donor[q] < l;
      count += s.donor[q] == l;
    }
    s.pf[l] = first;
    s.pc[l] = count;
  }
  for (int p = warp; p < np_all; p += kWarps) {
    const int l = s.donor[p], j = s.recv[p], dd = s.len[p];
    int a = s.keep[l], pos = 0;
    for (int q = 0; q < np_all; q++) {
      if (q < p && s.donor[q] == l) a += s.len[q];
      pos += s.donor[q] < l || (s.donor[q] == l && q < p);
    }
    if (lane == 0) {
      s.start[p] = a;
      s.ps[pos] = a;
      s.pl[pos] = dd;
      s.pr[pos] = j;
    }
    int nslots = 0;
    for (int u0 = 0; u0 < L; u0 += 32) {
      const int u = u0 + lane;
      const int e = l * L + u;
      bool present = false;
      int lo = 0, hi = 0;
      if (u < L) {
        lo = max(a, t.Q[e]);
        hi = min(a + dd, t.Q[e] + t.T[e]);
        present = t.T[e] > 0 && hi > lo;
      }
      const unsigned bal = __ballot_sync(0xffffffffu, present);
      const int b = nslots + __popc(bal & lanemask_lt());
      if (present) {
        if (b < B) {  // b < L, so b < Bm
          t.etc[j * Bm + b] = e;
          t.n[j * LB + L + b] = hi - lo;
          t.start[j * LB + L + b] = hi - lo;
          t.slot_b[j * L + u] = b;
        } else {
          atomicOr(&s.err, kErrSlots);
        }
      }
      nslots += __popc(bal);
    }
    if (lane == 0) s.nslots[j] = min(nslots, B);
  }
  for (int e = tid; e < E; e += kBalThreads) {
    const int j = e / L;
    const int v = min(max(s.keep[j] - t.Q[e], 0), t.T[e]);
    t.n[j * LB + (e - j * L)] = v;
    t.start[j * LB + (e - j * L)] = v;
  }
  __syncthreads();

  // Phase E: every segment rounded up to token_padding; starts and padding
  // rows as prefix sums over all ranks' segments in order.
  block_scan2(t.start, t.padx, R * LB, d.tp, true, s.part);

  // Row bases: the row of Q position 0 of each expert on its home rank and in
  // each slot (rank-local rows).
  for (int e = tid; e < E; e += kBalThreads) {
    const int j = e / L;
    t.home_rb[e] = t.start[j * LB + (e - j * L)] - t.start[j * LB] - t.Q[e];
  }
  for (int i = tid; i < R * L; i += kBalThreads) {
    const int j = i / L, u = i - j * L;
    const int b = t.slot_b[i];
    const int p = s.recv_piece[j];
    if (b >= 0 && p >= 0)
      t.slot_rb[i] = t.start[j * LB + L + b] - t.start[j * LB] - max(s.start[p], t.Q[s.donor[p] * L + u]);
  }
  __syncthreads();
}

// Stage 2 of the balance step, in two parts that may run on two blocks.
// balance_tables: experts_to_copy, cu_seqlens, zero_fill_ranges,
// remote_stats, the padding prefix and the meta words P, U and valid; a
// neutral plan (every later kernel a no-op) when the balance failed or `ok`
// is false.  Called by one whole block after balance_route.
__device__ void balance_tables(const PlanDims &d, const BalTables &t, BalSmall &s, PlanOut o,
                               int32_t *in, const PlanLayout &lay, int32_t *status, bool ok) {
  const int tid = threadIdx.x;
  const int R = d.R, E = d.E, L = d.L, B = d.B, Bm = d.Bm, LB = L + Bm, EB = d.EB, tp = d.tp;
  const int err = s.err;
  if (!ok || err != 0) {
    if (tid == 0) {
      in[kMetaValid] = 0;
      in[kMetaP] = 0;
      in[kMetaU] = 0;
      if (ok)
        set_status(status, (err & kErrBadExpert) ? MOONEP_ERR_BAD_EXPERT
                           : (err & kErrHist)    ? MOONEP_ERR_HIST_MISMATCH
                                                 : MOONEP_ERR_SLOTS);
    }
    for (int i = tid; i < R * B; i += kBalThreads) o.etc[i] = -1;
    for (int i = tid; i < R * EB; i += kBalThreads) {
      o.cu[i] = 0;
      o.zfr[2 * i] = 0;
      o.zfr[2 * i + 1] = 0;
    }
    for (int i = tid; i <= R * EB; i += kBalThreads) in[lay.pad_prefix + i] = 0;
    for (int i = tid; i < 2 * R; i += kBalThreads) o.remote_stats[i] = 0;
    return;
  }
  for (int i = tid; i < R * B; i += kBalThreads) {
    const int j = i / B, b = i - j * B;
    o.etc[i] = b < Bm ? t.etc[j * Bm + b] : -1;
  }
  for (int j = tid; j < R; j += kBalThreads) {
    const int p = s.recv_piece[j];
    o.remote_stats[2 * j] = p >= 0 ? s.len[p] : 0;
    o.remote_stats[2 * j + 1] = s.nslots[j];
  }
  // cu_seqlens, zero-fill ranges and the padding prefix of every (rank,
  // segment): a segment that is neither a home expert nor a usable slot of
  // the rank is empty and sits where the rank's running prefix stands.
  for (int i = tid; i < R * EB; i += kBalThreads) {
    const int j = i / EB, x = i - j * EB;
    const int base = j * LB;
    int c, nn = 0;
    if (x < E) {
      if (x / L == j) {
        c = base + (x - j * L);
        nn = t.n[c];
      } else {
        c = x < j * L ? base : base + L;
      }
    } else if (x - E < Bm) {
      c = base + L + (x - E);
      nn = t.n[c];
    } else {
      c = base + LB;
    }
    const int st = t.start[c] - t.start[base];
    const int end = st + (nn + tp - 1) / tp * tp;
    o.cu[i] = end;
    o.zfr[2 * i] = st + nn;
    o.zfr[2 * i + 1] = end;
    in[lay.pad_prefix + i] = t.padx[c];
  }
  if (tid == 0) {
    int u = 0;
    for (int j = 0; j < R; j++) u += s.nslots[j];
    in[lay.pad_prefix + R * EB] = t.padx[R * LB];
    in[kMetaP] = t.padx[R * LB];
    in[kMetaU] = u;
    in[kMetaValid] = 1;
  }
}

// balance_lists: the list the prefetch and the gradient reduce walk (experts
// with copies in ascending id, their slots in ascending rank) and the meta
// word D; D = 0 when the balance failed or `ok` is false.
// Called by one whole block after balance_route.
__device__ void balance_lists(const PlanDims &d, const BalTables &t, BalSmall &s, int32_t *in,
                              const PlanLayout &lay, bool ok) {
  const int tid = threadIdx.x;
  const int R = d.R, E = d.E, L = d.L, B = d.B, Bm = d.Bm;
  if (!ok || s.err != 0) {
    if (tid == 0) in[kMetaD] = 0;
    return;
  }
  // slot copies per expert (a receiver holds an expert at most once)
  for (int e = tid; e < E; e += kBalThreads) {
    const int l = e / L, u = e - l * L;
    int cnt = 0;
    for (int j = 0; j < R; j++) {
      const int p = s.recv_piece[j];
      if (p >= 0 && s.donor[p] == l && t.slot_b[j * L + u] >= 0) cnt++;
    }
    t.rcnt[e] = cnt;
    t.rhas[e] = cnt > 0;
  }
  __syncthreads();
  block_scan2(t.rcnt, t.rhas, E, 0, true, s.part);
  const int ncopies = t.rcnt[E], nexperts = t.rhas[E];
  for (int e = tid; e < E; e += kBalThreads) {
    const int first = t.rcnt[e];
    if (t.rcnt[e + 1] == first) continue;
    const int di = t.rhas[e];
    const int l = e / L, u = e - l * L;
    in[lay.red_expert + di] = e;
    in[lay.red_first + di] = first;
    int c = 0;
    for (int j = 0; j < R; j++) {
      const int p = s.recv_piece[j];
      if (p >= 0 && s.donor[p] == l && t.slot_b[j * L + u] >= 0)
        in[lay.red_slot + first + c++] = j * B + t.slot_b[j * L + u];
    }
  }
  if (tid == 0) {
    in[lay.red_first + nexperts] = ncopies;
    in[kMetaD] = nexperts;
  }
}

// Tile path: one CTA scans every expert's tile counts (where each tile's
// routes start inside P_e), runs the balance step, and leaves the tables the
// route assignment needs in the plan's internal area.
__global__ void __launch_bounds__(kBalThreads, 1)
plan_balance_kernel(PlanDims d, const int32_t *__restrict__ tpe, int32_t *hist, PlanOut o,
                    int32_t *in, PlanLayout lay, int32_t *status, int tables_shared) {
  extern __shared__ int32_t sm[];
  __shared__ BalSmall bs;
  __shared__ int sErr0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kBalThreads / 32;
  const int R = d.R, E = d.E, G = d.G, L = d.L;
  const BalTables t = bal_tables(tables_shared ? sm : in + lay.bal, d);
  if (tid == 0) sErr0 = in[kMetaErr];
  // Each warp scans whole columns; the column's values are loaded 128 at a
  // time (four per lane) before the scan so the loads overlap.
  for (int e = warp; e < E; e += kWarps) {
    int carry = 0;
    int32_t *col = hist + (int64_t)e * G;
    for (int b0 = 0; b0 < G; b0 += 128) {
      int v[4];
#pragma unroll
      for (int q = 0; q < 4; q++) {
        const int idx = b0 + 32 * q + lane;
        v[q] = idx < G ? col[idx] : 0;
      }
#pragma unroll
      for (int q = 0; q < 4; q++) {
        const int idx = b0 + 32 * q + lane;
        const int incl = warp_incl_scan(v[q]);
        if (idx < G) col[idx] = carry + incl - v[q];
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    __syncwarp();
    if (lane == 0) t.T[e] = carry;
    if (tpe != nullptr) {
      for (int r = lane; r < R; r += 32) {
        int cnt = 0;
        if (G > 0) {
          const int a = col[r * d.TPR];
          const int b = (r + 1 < R) ? col[(r + 1) * d.TPR] : carry;
          cnt = b - a;
        }
        if (cnt != tpe[(int64_t)r * E + e]) set_status(status, MOONEP_ERR_HIST_MISMATCH);
      }
    }
  }
  __syncthreads();
  balance_route(d, t, bs, sErr0);
  // tables of the route assignment kernel
  for (int e = tid; e < E; e += kBalThreads) {
    in[lay.qoff + e] = t.Q[e];
    in[lay.home_rowbase + e] = t.home_rb[e];
  }
  for (int i = tid; i < R * L; i += kBalThreads) in[lay.slot_rowbase + i] = t.slot_rb[i];
  for (int j = tid; j < R; j += kBalThreads) {
    in[lay.keep + j] = bs.keep[j];
    in[lay.piece_first + j] = bs.pf[j];
    in[lay.piece_count + j] = bs.pc[j];
    in[lay.piece_start + j] = bs.ps[j];
    in[lay.piece_len + j] = bs.pl[j];
    in[lay.piece_recv + j] = bs.pr[j];
  }
  for (int i = tid; i < 2 * R; i += kBalThreads) o.dup_counts[i] = 0;
  balance_tables(d, t, bs, o, in, lay, status, true);
  __syncthreads();
  balance_lists(d, t, bs, in, lay, true);
}

// ------------------------------------------------------------------ K3

constexpr int kAssignThreads = 256;
constexpr int kMaxK = 32;

template <int KT>
__global__ void __launch_bounds__(kAssignThreads)
plan_assign_kernel(PlanDims d, const int32_t *__restrict__ topk, const int32_t *__restrict__ ord,
                   const int32_t *__restrict__ tileoff, const int32_t *__restrict__ in,
                   PlanLayout lay, int32_t *__restrict__ dst, int32_t *dup_counts,
                   int32_t *dupflag) {
  extern __shared__ int32_t sm[];
  const int E = d.E, R = d.R, L = d.L;
  int32_t *sQoff = sm;                 // [E]
  int32_t *sHomeRb = sQoff + E;        // [E]
  int32_t *sSlotRb = sHomeRb + E;      // [R*L]
  int32_t *sKeep = sSlotRb + R * L;    // [R]
  int32_t *sPF = sKeep + R;            // piece_first [R]
  int32_t *sPC = sPF + R;              // piece_count [R]
  int32_t *sPS = sPC + R;              // piece_start [R]
  int32_t *sPL = sPS + R;              // piece_len [R]
  int32_t *sPR = sPL + R;              // piece_recv [R]
  int32_t *sDup = sPR + R;             // [R][2]
  for (int i = threadIdx.x; i < E; i += blockDim.x) {
    sQoff[i] = in[lay.qoff + i];
    sHomeRb[i] = in[lay.home_rowbase + i];
  }
  for (int i = threadIdx.x; i < R * L; i += blockDim.x) sSlotRb[i] = in[lay.slot_rowbase + i];
  for (int i = threadIdx.x; i < R; i += blockDim.x) {
    sKeep[i] = in[lay.keep + i];
    sPF[i] = in[lay.piece_first + i];
    sPC[i] = in[lay.piece_count + i];
    sPS[i] = in[lay.piece_start + i];
    sPL[i] = in[lay.piece_len + i];
    sPR[i] = in[lay.piece_recv + i];
  }
  for (int i = threadIdx.x; i < 2 * R; i += blockDim.x) sDup[i] = 0;
  __syncthreads();
  const bool valid = in[kMetaValid] != 0;
  const int K = KT > 0 ? KT : d.K;
  const int64_t tok = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (tok < (int64_t)R * d.S) {
    const int r = (int)(tok / d.S), s = (int)(tok % d.S);
    const int64_t base = (int64_t)r * d.C + (int64_t)s * K;
    int jr[KT > 0 ? KT : kMaxK];
    int gr[KT > 0 ? KT : kMaxK];
#pragma unroll
    for (int k = 0; k < (KT > 0 ? KT : kMaxK); k++) {
      if (KT == 0 && k >= K) break;
      int j = 0, row = 0;
      if (valid) {
        const int e = topk[base + k];
        const int i = s * K + k;
        const int gidx = r * d.TPR + i / kTile;
        const int p = sQoff[e] + tileoff[(int64_t)e * d.G + gidx] + ord[base + k];
        const int l = e / L;
        if (p < sKeep[l]) {
          j = l;
          row = sHomeRb[e] + p;
        } else {
          const int q0 = sPF[l], qn = sPC[l];
          for (int q = q0; q < q0 + qn; q++)
            if (p < sPS[q] + sPL[q]) {
              j = sPR[q];
              row = sSlotRb[j * L + (e - l * L)] + p;
              break;
            }
        }
      }
      jr[k] = j;
      gr[k] = j * d.NvS + row;
    }
#pragma unroll
    for (int k = 0; k < (KT > 0 ? KT : kMaxK); k++) {
      if (KT == 0 && k >= K) break;
      bool primary = true, has_dup = false;
#pragma unroll
      for (int k2 = 0; k2 < (KT > 0 ? KT : kMaxK); k2++) {
        if (KT == 0 && k2 >= K) break;
        if (k2 < k && jr[k2] == jr[k]) primary = false;
        if (k2 > k && jr[k2] == jr[k]) has_dup = true;
      }
      dst[base + k] = primary ? gr[k] : -(gr[k] + 1);
      if (valid) {
        if (!primary) atomicAdd(&sDup[2 * jr[k]], 1);
        if (primary && has_dup) {
          atomicAdd(&sDup[2 * jr[k] + 1], 1);
          if (dupflag) dupflag[gr[k]] = (int)(base + k) + 1;
        }
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 2 * R; i += blockDim.x)
    if (sDup[i]) atomicAdd(dup_counts + i, sDup[i]);
}

// ------------------------------------------------------------- fused
//
// The whole planner in one cooperative launch: G tile blocks of 1024
// threads, R*ceil(S*K/(32*IT*lpc)) of them (lpc = floor(32/K)*K routes per
// warp chunk), one per tile of a source rank, plus a table block and a list
// block:
//   1. each warp of a tile block walks IT chunks of consecutive routes and
//      counts them per expert (warp-aggregated, stable ordinals kept in
//      registers);
//   2. per-expert offsets of the warps; the tile's histogram to global; the
//      tile's counts added to its rank's totals;
//   3. every block waits until all have arrived (bounded by a time limit),
//      reads the per-rank totals and runs the balance step's first stage in
//      its own shared memory (each block computes the same tables from the
//      same totals);
//   4. each tile block adds the earlier tiles of its rank to its offsets, maps
//      its routes to (rank, row), marks duplicates with warp shuffles inside
//      each token's K lanes, and writes dst; meanwhile the table block writes
//      cu_seqlens, zero_fill_ranges, experts_to_copy, remote_stats and the
//      padding prefix, and the list block the experts-with-copies list;
//   5. the tile blocks add their duplicate counts straight into the plan
//      (the table block zeroed them before the meeting); the table block
//      clears the other set of per-rank totals, which the next call uses.
// A warp's chunk holds floor(32 / K) whole tokens, so a token's routes never
// straddle two chunks.  Used when the blocks fit on the SMs at once and the
// tables fit in shared memory; otherwise the three-kernel tile path runs.

constexpr int kFusedThreads = 1024;
constexpr int kFusedWarps = kFusedThreads / 32;
constexpr int kFusedMaxItems = 8;  // routes per thread: 1, 2, 4 or 8

// Routes per warp chunk: whole tokens only (floor(32 / K) * K).
__host__ __device__ __forceinline__ int fused_lanes(int K) { return 32 - 32 % K; }

struct FusedArgs {
  PlanDims d;
  const int32_t *topk, *tpe;
  int32_t *hist;    // [G, E] tile counts
  // Per-rank totals and error bits, two sets used by alternate calls (the
  // parity of the call count): a call adds into its own set, which the
  // previous call's table block left at zero, and clears the other set.
  int32_t *totals;  // [2][R, E] routes per (rank, expert)
  int32_t *errw;    // [2] error bits
  PlanOut o;
  int32_t *in;
  PlanLayout lay;
  int32_t *status;
  // [0] arrivals: grows by G + 2 per call
  unsigned long long *sync;
  int32_t *dupflag;
  int tpr, G;         // tiles per rank, tile blocks (R * tpr; tpr for one rank)
  // Rank-local planning (src_rank >= 0): the launch holds only that source
  // rank's routes (topk points at its [S, K]) and takes the per-rank totals
  // from hist_all, the [R, E] histograms every rank contributed (an
  // all-gather across GPUs); its own recount only checks hist_all[src_rank].
  // Every rank derives the same tables from the same totals and assigns
  // only its own routes.  totals/errw then point at a set of one row.
  int src_rank;
  const int32_t *hist_all;
  int unreachable;    // test hook: the arrival wait can never be satisfied
  long long wait_ns;  // limit of each wait
  // The launch is one thread-block cluster: its blocks meet at the cluster's
  // hardware barrier instead of polling the arrival counter (which still
  // counts the calls).
  int cluster;
};

__device__ __forceinline__ long long globaltimer_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Spin (thread 0) until *p reaches target or the limit passes; true if reached.
__device__ bool wait_counter(const unsigned long long *p, unsigned long long target,
                             long long limit_ns) {
  const long long t0 = globaltimer_ns();
  while (ld_acquire(p) < target) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
    __nanosleep(64);
  }
  return true;
}

size_t fused_smem_words(int R, int E, int B) {
  return (size_t)kFusedWarps * E + (size_t)E * R + (size_t)E + bal_tables_words(R, E, B) +
         (size_t)E;
}

// A word of block `rank`'s shared memory (distributed shared memory of the
// cluster), at the address `p` has in this block.
__device__ __forceinline__ int ld_cluster(const int32_t *p, unsigned rank) {
  const unsigned la = static_cast<unsigned>(__cvta_generic_to_shared(p));
  unsigned ra;
  int v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(ra) : "memory");
  return v;
}

// IT routes per thread (1, 2, 4 or 8; tile = 1024 * IT routes).  A compile-time
// count keeps only the routes' registers live across the balance step.
template <int IT>
__global__ void __launch_bounds__(kFusedThreads, 1) plan_fused_kernel(FusedArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ int32_t sm[];
  __shared__ BalSmall bs;
  __shared__ int s_bad, s_ok, s_err, s_par;
  __shared__ int sDup[2 * kMaxR];  // duplicate counts of this block
  const PlanDims d = a.d;
  const int R = d.R, E = d.E, L = d.L, C = d.C;
  const int g = blockIdx.x;
  const int nblk = a.G + 2;  // tile blocks, then the table block and the list block
  const bool tile = g < a.G, table_block = g == a.G, list_block = g == a.G + 1;
  const bool local = a.src_rank >= 0;
  const int r = local ? a.src_rank : (tile ? g / a.tpr : 0), t = tile ? g % a.tpr : 0;
  const int trows = local ? 1 : R;     // rows of a totals set
  const int trow = local ? 0 : r;      // this block's row in it
  const int gbase = local ? 0 : r * a.tpr;  // this rank's first tile in the launch
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t *h = sm;                     // [warps][E]
  int32_t *sCnt = h + kFusedWarps * E;  // [R*E]
  int32_t *sSrc = sCnt + E * R;         // [E]
  const BalTables tb = bal_tables(sSrc + E, d);
  int32_t *sTile = sSrc + E + bal_tables_words(R, E, d.B);  // [E] this tile's counts
  // One cluster (whole-problem plans of at most 16 blocks): the blocks read
  // each other's tile counts and error flags from shared memory after the
  // cluster barrier, instead of through global totals.
  const bool dsm = a.cluster && !local;

  const int32_t *src = a.topk + (local ? 0 : (int64_t)r * C);
  const unsigned lt = lanemask_lt();
  const int nbits = key_bits(E);
  constexpr int items = IT;
  // a warp's chunk holds whole tokens: lpc = floor(32 / K) * K routes (all 32
  // lanes when K divides 32; the lanes past lpc carry no route)
  const int lpc = fused_lanes(d.K);
  const int wbase = t * kFusedWarps * items * lpc + warp * lpc * items;
  int e_reg[items], o_reg[items];
  if (tid == 0) {
    s_bad = 0;
    // parity of this call: the arrival counter reads between this call's
    // first and last arrival (no block of it has seen all arrive yet)
    s_par = dsm ? 0 : (int)((ld_acquire(a.sync) / (unsigned long long)nblk) & 1ull);
  }
  if (table_block) {
    // the tile blocks add their duplicate counts after the meeting
    for (int i = tid; i < 2 * R; i += kFusedThreads) a.o.dup_counts[i] = 0;
    __threadfence();
  }
  // the balance step's initial tables, off its critical path (the barriers
  // before the balance step order these writes before its reads)
  balance_init(d, tb, bs);
  if (tile) {
    // this tile's routes, loaded first so that their latency overlaps the
    // zeroing of the counts
#pragma unroll
    for (int c = 0; c < items; c++) {
      const int i = wbase + c * lpc + lane;
      e_reg[c] = lane < lpc && i < C ? __ldg(src + i) : -1;
    }
    for (int i = tid; i < kFusedWarps * E; i += kFusedThreads) h[i] = 0;
    __syncthreads();

    // 1. counts and in-warp ordinals
    int32_t *hw = h + warp * E;
    bool bad = false;
#pragma unroll
    for (int c = 0; c < items; c++) {
      const int i = wbase + c * lpc + lane;
      const bool route = lane < lpc && i < C;
      int e = e_reg[c];
      if (route && (e < 0 || e >= E)) bad = true;
      if (!route || e < 0 || e >= E) e = -1;
      const unsigned m = match_key(e >= 0 ? e : E, nbits);
      int base = 0;
      if (e >= 0) base = hw[e];
      __syncwarp();
      if (e >= 0 && (m & lt) == 0) hw[e] = base + __popc(m);
      __syncwarp();
      e_reg[c] = e;
      o_reg[c] = base + __popc(m & lt);
    }
    if (bad) atomicOr(&s_bad, 1);
    __syncthreads();
    if (tid == 0 && s_bad) {
      if (!dsm) atomicOr(a.errw + s_par, kErrBadExpert);
      set_status(a.status, MOONEP_ERR_BAD_EXPERT);
    }
    // 2. warp offsets per expert; the tile's histogram; the rank's totals
    for (int e = tid; e < E; e += kFusedThreads) {
      int run = 0;
      for (int w = 0; w < kFusedWarps; w++) {
        const int v = h[w * E + e];
        h[w * E + e] = run;
        run += v;
      }
      if (dsm) {
        sTile[e] = run;
      } else {
        a.hist[(int64_t)g * E + e] = run;
        if (run) atomicAdd(a.totals + ((int64_t)s_par * trows + trow) * E + e, run);
      }
    }
    if (!dsm) __threadfence();  // this thread's histogram entries and totals, before the arrival
  }
  __syncthreads();

  // this block's first tokens_per_expert word to check, loaded now so that
  // its latency overlaps the meeting
  const int i_tpe = g * kFusedThreads + tid;
  const int tpe0 = (a.tpe != nullptr && !local && i_tpe < R * E) ? __ldg(a.tpe + i_tpe) : 0;

  // 3. all blocks arrive; each waits for the rest
  if (tid == 0 && dsm) s_ok = 1;
  if (tid == 0 && !dsm) {
    __threadfence();
    const unsigned long long n = (unsigned long long)nblk;
    const unsigned long long old = atomicAdd(a.sync, 1ull);
    const unsigned long long target = old - old % n + n;
    s_ok = a.cluster ? 1 : wait_counter(a.sync, target + (a.unreachable ? 1 : 0), a.wait_ns);
    if (!s_ok) set_status(a.status, MOONEP_ERR_TIMEOUT);
  }
  if (a.cluster) {
    // every thread of every block of the cluster; the release/acquire pair
    // orders the blocks' histogram, totals and error-bit writes before the
    // reads that follow
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  }
  if (dsm) {
    // error flags of the tile blocks, one lane per block
    if (warp == 0) {
      const int b = lane < a.G ? ld_cluster(&s_bad, lane) : 0;
      const unsigned m = __ballot_sync(0xffffffffu, b != 0);
      if (lane == 0) s_err = m ? kErrBadExpert : 0;
    }
  } else if (tid == 0) {
    s_err = s_ok ? __ldcg(a.errw + s_par) : 0;
  }
  __syncthreads();
  const bool ok = s_ok;
  if (ok) {
    const int32_t *tot_in = a.totals + (int64_t)s_par * trows * E;
    if (local) {
      // the gathered histograms are the totals; this rank's recount checks
      // its own row, a slice per block (a mismatch latches its error; the
      // tables stay those of the gathered counts, which every rank shares)
      for (int i = tid; i < R * E; i += kFusedThreads) sCnt[i] = __ldg(a.hist_all + i);
      for (int e = g * kFusedThreads + tid; e < E; e += nblk * kFusedThreads)
        if (__ldcg(tot_in + e) != __ldg(a.hist_all + (int64_t)r * E + e))
          set_status(a.status, MOONEP_ERR_HIST_MISMATCH);
    } else if (dsm) {
      // rank j's totals: the sum of its tiles' counts (blocks j*tpr ...)
      for (int i = tid; i < R * E; i += kFusedThreads) {
        const int j = i / E, e = i - j * E;
        int v = 0;
        for (int tt = 0; tt < a.tpr; tt++) v += ld_cluster(sTile + e, j * a.tpr + tt);
        sCnt[i] = v;
      }
    } else {
      for (int i = tid; i < R * E; i += kFusedThreads) sCnt[i] = __ldcg(tot_in + i);
    }
    __syncthreads();
    for (int e = tid; e < E; e += kFusedThreads) {
      int tot = 0, before = 0;
      for (int j = 0; j < R; j++) {
        const int v = sCnt[j * E + e];
        before += j < r ? v : 0;
        tot += v;
      }
      tb.T[e] = tot;
      sSrc[e] = before;
    }
    // tokens_per_expert against the recount, a slice per block: a mismatch
    // latches its error but the plan stands (it is built from the recount)
    if (a.tpe != nullptr && !local)
      for (int i = i_tpe; i < R * E; i += nblk * kFusedThreads)
        if (sCnt[i] != (i == i_tpe ? tpe0 : __ldg(a.tpe + i)))
          set_status(a.status, MOONEP_ERR_HIST_MISMATCH);
    __syncthreads();
  }
  if (ok) {
    // where this tile's routes start inside P_e: sSrc holds the earlier
    // ranks' routes; add the rank's earlier tiles (all loads in flight at
    // once; balance_route's barriers order the adds before their use)
    for (int i = tid; i < E * t; i += kFusedThreads) {
      const int e = i % E, tt = i / E;
      atomicAdd(&sSrc[e], dsm ? ld_cluster(sTile + e, gbase + tt)
                              : __ldcg(a.hist + (int64_t)(gbase + tt) * E + e));
    }
  }
  // this block has read the others' shared memory (the values are in use,
  // so the reads are done: no ordering needed); each block waits for every
  // block's arrival before it exits, so its counts outlive the reads
  if (dsm) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  if (ok) balance_route(d, tb, bs, s_err, true);

  if (list_block) {
    balance_lists(d, tb, bs, a.in, a.lay, ok);
    if (dsm) asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    return;
  }
  if (table_block) {
    balance_tables(d, tb, bs, a.o, a.in, a.lay, a.status, ok);
    // the other set of totals and error bits, used by the next call, back to
    // zero (the previous call, its last user, has completed)
    int32_t *other = a.totals + (int64_t)(1 - s_par) * trows * E;
    for (int i = tid; i < trows * E; i += kFusedThreads) other[i] = 0;
    if (tid == 0) a.errw[1 - s_par] = 0;
    if (dsm) asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    return;
  }

  // 4. this tile's routes -> (rank, row), duplicate marks, dst
  for (int i = tid; i < 2 * R; i += kFusedThreads) sDup[i] = 0;
  __syncthreads();
  const bool valid = ok && bs.err == 0;
  const int K = d.K;
  // A token's K routes sit in K consecutive lanes.  Routes of one token that
  // land on the same rank share the key (token lane group, rank); the lanes
  // past lpc form a group of their own.
  const int dkey_bits = key_bits(((32 + K - 1) / K) * (R + 1));
  const int rkey_bits = key_bits(R);
  int32_t *dst = a.o.dst + (int64_t)r * C;
#pragma unroll
  for (int c = 0; c < items; c++) {
    const int i = wbase + c * lpc + lane;
    const bool in_range = lane < lpc && i < C;
    int j = R, row = 0;
    if (in_range) {
      j = 0;
      if (valid) {
        const int e = e_reg[c];
        const int p = tb.Q[e] + sSrc[e] + h[warp * E + e] + o_reg[c];
        const int l = e / L;
        if (p < bs.keep[l]) {
          j = l;
          row = tb.home_rb[e] + p;
        } else {
          const int q0 = bs.pf[l], qn = bs.pc[l];
          for (int pc = q0; pc < q0 + qn; pc++)
            if (p < bs.ps[pc] + bs.pl[pc]) {
              j = bs.pr[pc];
              row = tb.slot_rb[j * L + (e - l * L)] + p;
              break;
            }
        }
      }
    }
    const unsigned same = match_key((lane / K) * (R + 1) + j, dkey_bits);
    const bool primary = (same & lt) == 0;
    const bool has_dup = (same & ~lt & ~(1u << lane)) != 0;
    const bool cnt_dup = in_range && valid && !primary;
    const bool cnt_grp = in_range && valid && primary && has_dup;
    if (in_range) {
      const int gr = j * d.NvS + row;
      dst[i] = primary ? gr : -(gr + 1);
      if (cnt_grp && a.dupflag) a.dupflag[gr] = (int)((int64_t)r * C + i) + 1;
    }
    // dup_counts: the lowest lane of each receiving rank adds for its rank
    const unsigned md = __ballot_sync(0xffffffffu, cnt_dup);
    const unsigned mg = __ballot_sync(0xffffffffu, cnt_grp);
    if (md | mg) {
      const int rk = (cnt_dup || cnt_grp) ? j : R;
      const unsigned mr = match_key(rk, rkey_bits);
      if (rk < R && (mr & lt) == 0) {
        const int nd = __popc(mr & md), ng = __popc(mr & mg);
        if (nd) atomicAdd(&sDup[2 * rk], nd);
        if (ng) atomicAdd(&sDup[2 * rk + 1], ng);
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < 2 * R; i += kFusedThreads)
    if (sDup[i]) atomicAdd(a.o.dup_counts + i, sDup[i]);
  if (dsm) asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ K4

constexpr int kDupThreads = kDupTile;

// The group of row w of rank j: has = 1 when w is a primary row with
// duplicates on its rank (dupflag names its route), cnt = their number.
__device__ __forceinline__ void dup_row(const PlanDims &d, const int32_t *__restrict__ dst,
                                        const int32_t *__restrict__ dupflag, int j, int w,
                                        int &has, int &cnt, int64_t &tb, int &k) {
  has = cnt = 0;
  tb = 0;
  k = 0;
  if (w >= d.NvS) return;
  const int rid = dupflag[(int64_t)j * d.NvS + w] - 1;
  if (rid < 0) return;
  k = rid % d.K;
  tb = rid - k;
  for (int k2 = k + 1; k2 < d.K; k2++) {
    const int v = dst[tb + k2];
    const int64_t g = v >= 0 ? v : -(int64_t)v - 1;
    if (g / d.NvS == j) cnt++;
  }
  has = 1;
}

// Block-wide exclusive scan of two counters (1024 threads); returns the
// totals through tot.
__device__ __forceinline__ void dup_block_scan(int has, int cnt, int &hx, int &cx, int (&tot)[2]) {
  __shared__ int wsum[2][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int hi = warp_incl_scan(has), ci = warp_incl_scan(cnt);
  if (lane == 31) {
    wsum[0][warp] = hi;
    wsum[1][warp] = ci;
  }
  __syncthreads();
  if (warp == 0) {
    wsum[0][lane] = warp_incl_scan(wsum[0][lane]);
    wsum[1][lane] = warp_incl_scan(wsum[1][lane]);
  }
  __syncthreads();
  hx = (warp ? wsum[0][warp - 1] : 0) + hi - has;
  cx = (warp ? wsum[1][warp - 1] : 0) + ci - cnt;
  tot[0] = wsum[0][31];
  tot[1] = wsum[1][31];
}

// Pass 1: per (tile, rank) block, the tile's group and duplicate counts.
__global__ void __launch_bounds__(kDupThreads)
plan_dup_count_kernel(PlanDims d, const int32_t *__restrict__ dst,
                      const int32_t *__restrict__ dupflag, int32_t *__restrict__ tiles) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x, j = blockIdx.y, T = gridDim.x;
  int has, cnt, k;
  int64_t tb;
  dup_row(d, dst, dupflag, j, t * kDupTile + threadIdx.x, has, cnt, tb, k);
  int hx, cx, tot[2];
  dup_block_scan(has, cnt, hx, cx, tot);
  if (threadIdx.x == 0) {
    tiles[((int64_t)j * T + t) * 2] = tot[0];
    tiles[((int64_t)j * T + t) * 2 + 1] = tot[1];
  }
}

// Pass 2: every block adds up the counts of the rank's earlier tiles, then
// writes its groups (ascending primary row) and their duplicate rows (k order).
__global__ void __launch_bounds__(kDupThreads)
plan_dup_write_kernel(PlanDims d, const int32_t *__restrict__ dst,
                      const int32_t *__restrict__ dupflag, const int32_t *__restrict__ tiles,
                      int32_t *__restrict__ dup_groups, int32_t *__restrict__ dup_loffs) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int base[2][32];
  const int t = blockIdx.x, j = blockIdx.y, T = gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int sg = 0, sd = 0;
  for (int i = tid; i < t; i += kDupThreads) {
    sg += tiles[((int64_t)j * T + i) * 2];
    sd += tiles[((int64_t)j * T + i) * 2 + 1];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sg += __shfl_xor_sync(0xffffffffu, sg, o);
    sd += __shfl_xor_sync(0xffffffffu, sd, o);
  }
  if (lane == 0) {
    base[0][warp] = sg;
    base[1][warp] = sd;
  }
  const int w = t * kDupTile + tid;
  int has, cnt, k;
  int64_t tb;
  dup_row(d, dst, dupflag, j, w, has, cnt, tb, k);
  int hx, cx, tot[2];
  dup_block_scan(has, cnt, hx, cx, tot);  // its barriers also publish base[][]
  int g0 = 0, d0 = 0;
  for (int i = 0; i < kDupThreads / 32; i++) {
    g0 += base[0][i];
    d0 += base[1][i];
  }
  if (!has) return;
  const int64_t rowbase = (int64_t)j * d.NvS;
  const int gi = g0 + hx, di = d0 + cx;
  int32_t *rec = dup_groups + (rowbase + gi) * 3;
  rec[0] = w;
  rec[1] = di;
  rec[2] = cnt;
  int c = 0;
  for (int k2 = k + 1; k2 < d.K; k2++) {
    const int v = dst[tb + k2];
    const int64_t g = v >= 0 ? v : -(int64_t)v - 1;
    if (g / d.NvS == j) dup_loffs[rowbase + di + c++] = (int)(g - rowbase);
  }
}

}  // namespace

// Routes per thread of the single-launch planner: the fewest (most tiles,
// most SMs at work) for which every tile block and the two table blocks fit on
// the SMs at once; 0 if none.
int plan_fused_tiles(int C, int K, int items) {
  const int per_tile = kFusedWarps * items * fused_lanes(K);
  const int tpr = (C + per_tile - 1) / per_tile;
  return tpr > 0 ? tpr : 1;
}

int plan_fused_items(int R, int C, int K, int sms) {
  for (int items = 1; items <= kFusedMaxItems; items *= 2)
    if ((int64_t)R * plan_fused_tiles(C, K, items) + 2 <= sms) return items;
  return 0;
}

// Tiles of any planner launch (the histogram area holds E words per tile):
// the tile path, the single-launch planner over every rank, or over one rank.
int plan_hist_tiles(int R, int C, int K, int sms) {
  const int tile_path = R * ((C + kTile - 1) / kTile);
  const int items = plan_fused_items(R, C, K, sms);
  const int fused = items ? R * plan_fused_tiles(C, K, items) : 0;
  const int items1 = plan_fused_items(1, C, K, sms);
  const int local = items1 ? plan_fused_tiles(C, K, items1) : 0;
  const int m = tile_path > fused ? tile_path : fused;
  return m > local ? m : local;
}

int64_t plan_totals_offset(int R, int E, int C, int K, int sms) {
  return (int64_t)E * plan_hist_tiles(R, C, K, sms);
}

// After the totals: the rank-local planner's two [E] sets and error words.
int64_t plan_rank_totals_offset(int R, int E, int C, int K, int sms) {
  return plan_totals_offset(R, E, C, K, sms) + 2 * (int64_t)R * E + 8;
}

int64_t plan_scratch_words(int R, int E, int C, int K, int sms) {
  return plan_rank_totals_offset(R, E, C, K, sms) + 2 * (int64_t)E + 8;
}

// Shared memory the planner kernels may use.
constexpr size_t kPlanSmemLimit = 200 * 1024;

int plan_fused_choice(int R, int E, int K, int B, int C, int sms) {
  if (K < 1 || K > kMaxK || R > kMaxR || plan_fused_items(R, C, K, sms) == 0) return 0;
  return fused_smem_words(R, E, B) * sizeof(int32_t) <= kPlanSmemLimit ? K : 0;
}

static bool bal_in_shared(int R, int E, int B) {
  return bal_tables_words(R, E, B) * sizeof(int32_t) <= kPlanSmemLimit;
}

// Raise a kernel's dynamic shared memory limit to at least `bytes` (never
// lower it: contexts of different shapes share the kernels).  The default
// limit is 48 KB minus the kernel's static shared memory, so any size is set
// explicitly.
static cudaError_t raise_dyn_smem(const void *f, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void *>, int> limit;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  int &cur = limit[{dev, f}];
  if (bytes <= cur) return cudaSuccess;
  e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) cur = bytes;
  return e;
}

cudaError_t plan_configure(int R, int E, int B) {
  const int hist_smem = (kPlanThreads / 32) * E * (int)sizeof(int32_t);
  const int assign_smem = (3 * E + 8 * R) * (int)sizeof(int32_t);
  const int bal_smem =
      bal_in_shared(R, E, B) ? (int)(bal_tables_words(R, E, B) * sizeof(int32_t)) : 0;
  cudaError_t e = raise_dyn_smem((const void *)plan_hist_kernel, hist_smem);
  if (e == cudaSuccess) e = raise_dyn_smem((const void *)plan_balance_kernel, bal_smem);
  const void *as[] = {(const void *)plan_assign_kernel<0>, (const void *)plan_assign_kernel<1>,
                      (const void *)plan_assign_kernel<2>, (const void *)plan_assign_kernel<4>,
                      (const void *)plan_assign_kernel<6>, (const void *)plan_assign_kernel<8>};
  for (const void *f : as)
    if (e == cudaSuccess) e = raise_dyn_smem(f, assign_smem);
  if (e == cudaSuccess && plan_fused_choice(R, E, 1, B, 0, 1 << 30)) {
    const int fsmem = (int)(fused_smem_words(R, E, B) * sizeof(int32_t));
    const void *fs[] = {(const void *)plan_fused_kernel<1>, (const void *)plan_fused_kernel<2>,
                        (const void *)plan_fused_kernel<4>, (const void *)plan_fused_kernel<8>};
    for (const void *f : fs)
      if (e == cudaSuccess) e = raise_dyn_smem(f, fsmem);
  }
  return e;
}

static PlanDims plan_dims(const moonep_ctx *ctx) {
  const moonep_config &c = ctx->cfg;
  PlanDims d;
  d.R = c.R;
  d.E = c.E;
  d.K = c.K;
  d.S = c.S;
  d.B = c.B;
  d.tp = c.token_padding;
  d.L = ctx->L;
  d.C = ctx->C;
  d.EB = ctx->EB;
  d.NvS = ctx->NvS;
  d.TPR = ctx->TPR;
  d.G = ctx->G;
  d.Bm = usable_slots(d.R, d.E, d.B);
  return d;
}

static PlanOut plan_out(const moonep_comm_plan *plan) {
  return PlanOut{plan->dst, plan->experts_to_copy, plan->cu_seqlens, plan->zero_fill_ranges,
                 plan->remote_stats, plan->dup_counts, plan->dup_groups, plan->dup_loffs};
}

static cudaError_t launch_fused(const FusedArgs &fa, int items, cudaStream_t st) {
  const size_t smem = fused_smem_words(fa.d.R, fa.d.E, fa.d.B) * sizeof(int32_t);
  const dim3 grid(fa.G + 2), block(kFusedThreads);
  // one cluster of G + 2 blocks (co-resident by construction), else a
  // cooperative launch
  const bool coop = fa.cluster == 0;
  const int cl = fa.cluster ? fa.G + 2 : 1;
  return items == 1   ? launch_pdl_ex(plan_fused_kernel<1>, grid, block, smem, st, coop, cl, fa)
         : items == 2 ? launch_pdl_ex(plan_fused_kernel<2>, grid, block, smem, st, coop, cl, fa)
         : items == 4 ? launch_pdl_ex(plan_fused_kernel<4>, grid, block, smem, st, coop, cl, fa)
                      : launch_pdl_ex(plan_fused_kernel<8>, grid, block, smem, st, coop, cl, fa);
}

// Largest cluster a launch may ask for (non-portable sizes above 8).
constexpr int kMaxPlanCluster = 16;

int plan_cluster_blocks(const moonep_ctx *ctx) {
  const moonep_config &c = ctx->cfg;
  if (ctx->test_planner_timeout || !ctx->d_sync) return 0;
  if (plan_fused_choice(c.R, c.E, c.K, c.B, ctx->C, ctx->sms_device) == 0) return 0;
  const int items = plan_fused_items(c.R, ctx->C, c.K, ctx->sms_device);
  const int nblk = c.R * plan_fused_tiles(ctx->C, c.K, items) + 2;
  if (nblk > kMaxPlanCluster) return 0;
  const void *f = items == 1   ? (const void *)plan_fused_kernel<1>
                  : items == 2 ? (const void *)plan_fused_kernel<2>
                  : items == 4 ? (const void *)plan_fused_kernel<4>
                               : (const void *)plan_fused_kernel<8>;
  if (nblk > 8 &&
      cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nblk);
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = fused_smem_words(c.R, c.E, c.B) * sizeof(int32_t);
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = nblk;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, f, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return clusters >= 1 ? nblk : 0;
}

int plan_rank_supported(const moonep_ctx *ctx) {
  const moonep_config &c = ctx->cfg;
  if (c.K < 1 || c.K > kMaxK || c.R > kMaxR) return 0;
  if (fused_smem_words(c.R, c.E, c.B) * sizeof(int32_t) > kPlanSmemLimit) return 0;
  return plan_fused_items(1, ctx->C, c.K, ctx->sms_device) > 0;
}

int launch_plan_rank(moonep_ctx *ctx, int rank, const int32_t *topk_r, const int32_t *hist_all,
                     moonep_comm_plan *plan, cudaStream_t st) {
  const PlanDims d = plan_dims(ctx);
  FusedArgs fa;
  fa.d = d;
  fa.src_rank = rank;
  fa.hist_all = hist_all;
  fa.topk = topk_r;
  fa.tpe = nullptr;
  fa.hist = ctx->d_hist;
  const int items = plan_fused_items(1, d.C, d.K, ctx->sms_device);
  fa.tpr = plan_fused_tiles(d.C, d.K, items);
  fa.G = fa.tpr;
  fa.totals = ctx->d_hist + plan_rank_totals_offset(d.R, d.E, d.C, d.K, ctx->sms_device);
  fa.errw = fa.totals + 2 * (int64_t)d.E;
  fa.o = plan_out(plan);
  fa.in = plan->internal;
  fa.lay = PlanLayout::make(d.R, d.E, d.B, d.NvS, false);
  fa.status = ctx->d_status;
  fa.sync = ctx->d_sync + kSyncRankLocal;  // the rank-local calls' own arrival counter
  fa.dupflag = nullptr;
  fa.unreachable = ctx->test_planner_timeout;
  fa.wait_ns = ctx->test_planner_timeout ? 200000000LL : 1000000000LL;
  fa.cluster = 0;
  cudaError_t e = launch_fused(fa, items, st);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(cudaGetLastError());
}

int launch_plan(moonep_ctx *ctx, const int32_t *topk, const int32_t *tpe,
                moonep_comm_plan *plan, cudaStream_t st) {
  const PlanDims d = plan_dims(ctx);
  const bool dup = (plan->flags & MOONEP_PLAN_DUP_RECORDS) != 0;
  PlanLayout lay = PlanLayout::make(d.R, d.E, d.B, d.NvS, dup);
  int32_t *in = plan->internal;
  int32_t *dupflag = dup ? in + lay.dupflag : nullptr;
  cudaError_t e;
  if (dup) {
    e = cudaMemsetAsync(dupflag, 0, (size_t)d.R * d.NvS * sizeof(int32_t), st);
    if (e != cudaSuccess) return cuda_status(e);
  }
  const PlanOut o = plan_out(plan);
  const int fused_k = plan_fused_choice(d.R, d.E, d.K, d.B, d.C, ctx->sms_device);
  if (fused_k > 0 && ctx->d_sync != nullptr) {
    FusedArgs fa;
    fa.src_rank = -1;
    fa.hist_all = nullptr;
    fa.d = d;
    fa.topk = topk;
    fa.tpe = tpe;
    fa.hist = ctx->d_hist;
    const int items = plan_fused_items(d.R, d.C, d.K, ctx->sms_device);
    fa.tpr = plan_fused_tiles(d.C, d.K, items);
    fa.G = d.R * fa.tpr;
    fa.totals = ctx->d_hist + plan_totals_offset(d.R, d.E, d.C, d.K, ctx->sms_device);
    fa.errw = fa.totals + 2 * (int64_t)d.R * d.E;
    fa.o = o;
    fa.in = in;
    fa.lay = lay;
    fa.status = ctx->d_status;
    fa.sync = ctx->d_sync;
    fa.dupflag = dupflag;
    fa.unreachable = ctx->test_planner_timeout;
    fa.wait_ns = ctx->test_planner_timeout ? 200000000LL : 1000000000LL;
    fa.cluster = ctx->plan_cluster == fa.G + 2 ? 1 : 0;
    e = launch_fused(fa, items, st);
    if (e != cudaSuccess) return cuda_status(e);
  } else {
    e = cudaMemsetAsync(in, 0, kMetaWords * sizeof(int32_t), st);
    if (e != cudaSuccess) return cuda_status(e);
    if (d.G > 0) {
      const size_t smem = (size_t)(kPlanThreads / 32) * d.E * sizeof(int32_t);
      plan_hist_kernel<<<d.G, kPlanThreads, smem, st>>>(topk, d, ctx->d_hist, ctx->d_ord, in,
                                                         ctx->d_status);
    }
    const bool bal_shared = bal_in_shared(d.R, d.E, d.B);
    plan_balance_kernel<<<1, kBalThreads,
                          bal_shared ? bal_tables_words(d.R, d.E, d.B) * sizeof(int32_t) : 0, st>>>(
        d, tpe, ctx->d_hist, o, in, lay, ctx->d_status, bal_shared ? 1 : 0);
    if ((int64_t)d.R * d.S > 0) {
      const int64_t ntok = (int64_t)d.R * d.S;
      const int grid = (int)((ntok + kAssignThreads - 1) / kAssignThreads);
      const size_t smem = (size_t)(2 * d.E + d.R * d.L + 8 * d.R) * sizeof(int32_t);
#define MOONEP_ASSIGN(KV)                                                                \
  plan_assign_kernel<KV><<<grid, kAssignThreads, smem, st>>>(d, topk, ctx->d_ord,         \
                                                             ctx->d_hist, in, lay,        \
                                                             plan->dst, plan->dup_counts, \
                                                             dupflag)
      switch (d.K) {
        case 1: MOONEP_ASSIGN(1); break;
        case 2: MOONEP_ASSIGN(2); break;
        case 4: MOONEP_ASSIGN(4); break;
        case 6: MOONEP_ASSIGN(6); break;
        case 8: MOONEP_ASSIGN(8); break;
        default: MOONEP_ASSIGN(0); break;
      }
#undef MOONEP_ASSIGN
    }
  }
  if (dup && d.NvS > 0) {
    const dim3 grid(dup_tiles_per_rank(d.NvS), d.R);
    cudaError_t e2 = launch_pdl(plan_dup_count_kernel, grid, kDupThreads, 0, st, false, d,
                                (const int32_t *)plan->dst, (const int32_t *)(in + lay.dupflag),
                                in + lay.dup_tiles);
    if (e2 == cudaSuccess)
      e2 = launch_pdl(plan_dup_write_kernel, grid, kDupThreads, 0, st, false, d,
                      (const int32_t *)plan->dst, (const int32_t *)(in + lay.dupflag),
                      (const int32_t *)(in + lay.dup_tiles), plan->dup_groups, plan->dup_loffs);
    if (e2 != cudaSuccess) return cuda_status(e2);
  }
  return cuda_status(cudaGetLastError());
}

}  // namespace moonep
