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
//   K1 plan_hist_kernel    per 2048-route tile: per-expert counts and each
//                          route's ordinal among same-expert routes of the tile
//                          (warp-aggregated with __match_any_sync, stable).
//   K2 plan_balance_kernel one CTA: column scans of the tile counts (the
//                          position of every tile inside every P_e), the chain
//                          balance, slots, segments, cu_seqlens, padding and
//                          the copy / reduce lists.
//   K3 plan_assign_kernel  one thread per token: Q position -> (rank, row),
//                          duplicate encoding, dup_counts.
//   K4 plan_dup_kernel     (optional) one CTA per rank: compact duplicate
//                          records in ascending primary row.
#include "moonep_internal.cuh"

namespace moonep {
namespace {

struct PlanDims {
  int R, E, K, S, B, tp, L, C, EB, NvS, TPR, G;
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
constexpr int kMaxR = 64;

// Shared-memory working set of the balance step (all pointers generic: nseg
// and pad may live in global memory when R*(E+B) is too large for shared
// memory).
struct BalTables {
  int32_t *T;       // [E] routes per expert
  int32_t *Q;       // [E] offset of P_e inside Q_home(e)
  int32_t *slot_b;  // [R*L] slot of (receiver j, donor-local expert u), -1 if none
  int32_t *etc;     // [R*B] experts_to_copy
  int32_t *rcnt;    // [E] slot copies per expert, then first index in the reduce list
  int32_t *rhas;    // [E] expert has copies, then its index among such experts
  int32_t *nseg;    // [R*(E+B)] valid rows, then segment starts
  int32_t *pad;     // [R*(E+B)] padding rows, then their prefix inside the rank
};

inline size_t bal_tables_words(int R, int E, int B, bool nseg_shared) {
  return (size_t)5 * E + (size_t)R * B + (nseg_shared ? 2 * (size_t)R * (E + B) : 0);
}

__device__ __forceinline__ BalTables bal_tables(int32_t *base, const PlanDims &d,
                                                int32_t *nseg_global, int32_t *pad_global,
                                                bool nseg_shared) {
  BalTables t;
  t.T = base;
  t.Q = t.T + d.E;
  t.slot_b = t.Q + d.E;
  t.etc = t.slot_b + d.R * d.L;
  t.rcnt = t.etc + d.R * d.B;
  t.rhas = t.rcnt + d.E;
  t.nseg = nseg_shared ? t.rhas + d.E : nseg_global;
  t.pad = nseg_shared ? t.nseg + d.R * d.EB : pad_global;
  return t;
}

// Exclusive prefix sum of v[0..n) in place, by a whole block of kBalThreads
// threads (each thread sums a contiguous run, then the runs are scanned);
// returns the total to every thread.
__device__ int block_exclusive_scan(int32_t *v, int n) {
  __shared__ int wsum[32];
  __shared__ int total;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (n + kBalThreads - 1) / kBalThreads;
  const int b0 = min(n, tid * per), b1 = min(n, b0 + per);
  int local = 0;
  for (int i = b0; i < b1; i++) local += v[i];
  const int incl = warp_incl_scan(local);
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = wsum[lane];
    const int wi = warp_incl_scan(w);
    wsum[lane] = wi - w;
    if (lane == 31) total = wi;
  }
  __syncthreads();
  int run = wsum[warp] + incl - local;
  for (int i = b0; i < b1; i++) {
    const int x = v[i];
    v[i] = run;
    run += x;
  }
  const int tot = total;
  __syncthreads();
  return tot;
}

// Everything after the per-expert totals: group offsets, the chain balance,
// slots, segments and cu_seqlens, padding prefix, row bases, copy and reduce
// lists.  Called by one whole block of kBalThreads threads with t.T filled;
// err holds the error bits found so far.
// When `ready` is given, the tables the route assignment needs (group
// offsets, kept prefixes, pieces, row bases, the valid flag) are published
// there as soon as they are written (ready = target), and the rest (padding
// prefix, copy and reduce lists, experts_to_copy, counts) is finished while
// the other CTAs already assign routes.
__device__ void balance_tail(const PlanDims &d, const BalTables &t, PlanOut o, int32_t *in,
                             const PlanLayout &lay, int32_t *status, int err_in,
                             unsigned long long *ready = nullptr,
                             unsigned long long target = 0) {
  __shared__ int sG[kMaxR], sKeep[kMaxR], sRecvPiece[kMaxR], sNslots[kMaxR], sRankPad[kMaxR];
  __shared__ int pDonor[kMaxR], pRecv[kMaxR], pLen[kMaxR], pStart[kMaxR];
  __shared__ int sNp, sErr, sP, sU;
  __shared__ int sPadOff[kMaxR], sSlotOff[kMaxR];
  __shared__ int sPart[2][32];  // per-warp partial sums of a rank's segments
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kBalThreads / 32;
  const int R = d.R, E = d.E, L = d.L, B = d.B, EB = d.EB, C = d.C;
  int32_t *sT = t.T, *sQ = t.Q, *slot_b = t.slot_b, *setc = t.etc, *nseg = t.nseg;

  if (tid == 0) {
    sErr = err_in;
    sNp = 0;
  }
  for (int i = tid; i < R * B; i += kBalThreads) setc[i] = -1;
  for (int i = tid; i < R * EB; i += kBalThreads) nseg[i] = 0;
  for (int i = tid; i < R * L; i += kBalThreads) slot_b[i] = -1;
  for (int j = tid; j < R; j += kBalThreads) {
    sRecvPiece[j] = -1;
    sNslots[j] = 0;
  }
  for (int i = tid; i < 2 * R; i += kBalThreads) {
    o.remote_stats[i] = 0;
    o.dup_counts[i] = 0;
  }
  // Phase B: offset of P_e inside Q_home(e) (one warp per home group), G_j.
  for (int j = warp; j < R; j += kWarps) {
    int carry = 0;
    for (int u0 = 0; u0 < L; u0 += 32) {
      const int u = u0 + lane;
      const int v = u < L ? sT[j * L + u] : 0;
      const int incl = warp_incl_scan(v);
      if (u < L) {
        sQ[j * L + u] = carry + incl - v;
        in[lay.qoff + j * L + u] = carry + incl - v;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) sG[j] = carry;
  }
  __syncthreads();

  // Phase C: the chain balance on one warp (lane j holds rank j and j + 32):
  // each round fills the lowest-index rank below C from the lowest-index rank
  // above C; at most R rounds.
  if (warp == 0 && R <= 32) {
    // lane j holds rank j
    int rem = lane < R ? sG[lane] : C, don = 0, np = 0;
    for (int round = 0; round <= R; round++) {
      const unsigned rb = __ballot_sync(0xffffffffu, rem < C);
      if (!rb) break;
      const unsigned db = __ballot_sync(0xffffffffu, rem > C);
      if (!db || np >= R) {  // only reachable from a broken histogram
        if (lane == 0) sErr |= kErrHist;
        break;
      }
      const int recv = __ffs(rb) - 1, donor = __ffs(db) - 1;
      const int dd = C - __shfl_sync(0xffffffffu, rem, recv);
      if (lane == 0) {
        pDonor[np] = donor;
        pRecv[np] = recv;
        pLen[np] = dd;
        sRecvPiece[recv] = np;
      }
      np++;
      if (lane == donor) {
        rem -= dd;
        don += dd;
      }
      if (lane == recv) rem = C;
    }
    if (lane < R) {
      sKeep[lane] = sG[lane] - don;
      in[lay.keep + lane] = sKeep[lane];
    }
    if (lane == 0) sNp = np;
  } else if (warp == 0) {
    const int C_ = C;
    int rem0 = lane < R ? sG[lane] : C_, rem1 = lane + 32 < R ? sG[lane + 32] : C_;
    int don0 = 0, don1 = 0, np = 0;
    for (int round = 0; round <= R; round++) {
      const unsigned rb0 = __ballot_sync(0xffffffffu, rem0 < C_);
      const unsigned rb1 = __ballot_sync(0xffffffffu, rem1 < C_);
      if (!rb0 && !rb1) break;
      const unsigned db0 = __ballot_sync(0xffffffffu, rem0 > C_);
      const unsigned db1 = __ballot_sync(0xffffffffu, rem1 > C_);
      if ((!db0 && !db1) || np >= R) {  // only reachable from a broken histogram
        if (lane == 0) sErr |= kErrHist;
        break;
      }
      const int recv = rb0 ? __ffs(rb0) - 1 : 32 + __ffs(rb1) - 1;
      const int donor = db0 ? __ffs(db0) - 1 : 32 + __ffs(db1) - 1;
      const int rr = recv < 32 ? __shfl_sync(0xffffffffu, rem0, recv)
                               : __shfl_sync(0xffffffffu, rem1, recv - 32);
      const int dd = C_ - rr;
      if (lane == 0) {
        pDonor[np] = donor;
        pRecv[np] = recv;
        pLen[np] = dd;
        sRecvPiece[recv] = np;
      }
      np++;
      if (lane == (donor & 31)) {
        if (donor < 32) { rem0 -= dd; don0 += dd; } else { rem1 -= dd; don1 += dd; }
      }
      if (lane == (recv & 31)) {
        if (recv < 32) rem0 = C_; else rem1 = C_;
      }
    }
    for (int h2 = 0; h2 < 2; h2++) {
      const int j = lane + 32 * h2;
      if (j < R) {
        sKeep[j] = sG[j] - (h2 ? don1 : don0);
        in[lay.keep + j] = sKeep[j];
      }
    }
    if (lane == 0) sNp = np;
  }
  __syncthreads();

  // Phase D: per piece (one warp each): where its run starts (after the
  // donor's kept prefix and its earlier pieces), its place in the
  // donor-grouped piece list, and the receiver's slots; per donor: its piece
  // list range; per home expert: its kept routes.
  const int np_all = sNp;
  for (int l = tid; l < R; l += kBalThreads) {
    int first = 0, count = 0;
    for (int q = 0; q < np_all; q++) {
      first += pDonor[q] < l;
      count += pDonor[q] == l;
    }
    in[lay.piece_first + l] = first;
    in[lay.piece_count + l] = count;
  }
  for (int p = warp; p < np_all; p += kWarps) {
    const int l = pDonor[p], j = pRecv[p], dd = pLen[p];
    int a = sKeep[l], pos = 0;
    for (int q = 0; q < np_all; q++) {
      if (q < p && pDonor[q] == l) a += pLen[q];
      pos += pDonor[q] < l || (pDonor[q] == l && q < p);
    }
    if (lane == 0) {
      pStart[p] = a;
      in[lay.piece_start + pos] = a;
      in[lay.piece_len + pos] = dd;
      in[lay.piece_recv + pos] = j;
    }
    int nslots = 0;
    for (int u0 = 0; u0 < L; u0 += 32) {
      const int u = u0 + lane;
      const int e = l * L + u;
      bool present = false;
      int lo = 0, hi = 0;
      if (u < L) {
        lo = max(a, sQ[e]);
        hi = min(a + dd, sQ[e] + sT[e]);
        present = sT[e] > 0 && hi > lo;
      }
      const unsigned bal = __ballot_sync(0xffffffffu, present);
      const int b = nslots + __popc(bal & lanemask_lt());
      if (present) {
        if (b < B) {
          setc[j * B + b] = e;
          nseg[j * EB + E + b] = hi - lo;
          slot_b[j * L + u] = b;
        } else {
          atomicOr(&sErr, kErrSlots);
        }
      }
      nslots += __popc(bal);
    }
    if (lane == 0) {
      sNslots[j] = min(nslots, B);
      o.remote_stats[2 * j] = dd;
      o.remote_stats[2 * j + 1] = min(nslots, B);
    }
  }
  for (int e = tid; e < E; e += kBalThreads) {
    const int j = e / L;
    nseg[j * EB + e] = min(max(sKeep[j] - sQ[e], 0), sT[e]);
  }
  __syncthreads();

  // Phase E: per rank, padded segment lengths -> cu_seqlens, padding ranges,
  // segment starts (kept in nseg) and padding prefix inside the rank (pad).
  // With R < 32 each rank's E+B segments are split over wpr warps: partial
  // sums first, then each warp rescans its part from its offset.
  const int wpr = R >= kWarps ? 1 : kWarps / R;  // warps per rank (R * wpr <= 32)
  const int part = (EB + wpr - 1) / wpr;
  if (wpr > 1 && warp < R * wpr) {
    const int pj = warp / wpr, pw = warp % wpr;
    const int x_lo = min(EB, pw * part), x_hi = min(EB, x_lo + part);
    int sum = 0, psum = 0;
    for (int x = x_lo + lane; x < x_hi; x += 32) {
      const int n = nseg[pj * EB + x];
      const int padded = (n + d.tp - 1) / d.tp * d.tp;
      sum += padded;
      psum += padded - n;
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) {
      sum += __shfl_xor_sync(0xffffffffu, sum, o2);
      psum += __shfl_xor_sync(0xffffffffu, psum, o2);
    }
    if (lane == 0) {
      sPart[0][warp] = sum;
      sPart[1][warp] = psum;
    }
  }
  __syncthreads();
  for (int task = warp; task < R * wpr; task += kWarps) {
    const int pj = task / wpr, pw = task % wpr;
    const int x_lo = min(EB, pw * part), x_hi = min(EB, x_lo + part);
    int carry = 0, pcarry = 0;
    for (int q = 0; q < pw; q++) {
      carry += sPart[0][pj * wpr + q];
      pcarry += sPart[1][pj * wpr + q];
    }
    for (int x0 = x_lo; x0 < x_hi; x0 += 32) {
      const int x = x0 + lane;
      const int n = x < x_hi ? nseg[pj * EB + x] : 0;
      const int padded = (n + d.tp - 1) / d.tp * d.tp;
      const int pc = padded - n;
      const int incl = warp_incl_scan(padded);
      const int pincl = warp_incl_scan(pc);
      if (x < x_hi) {
        const int end = carry + incl;
        const int start = end - padded;
        o.cu[pj * EB + x] = end;
        o.zfr[2 * (pj * EB + x)] = start + n;
        o.zfr[2 * (pj * EB + x) + 1] = end;
        nseg[pj * EB + x] = start;
        t.pad[pj * EB + x] = pcarry + pincl - pc;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
      pcarry += __shfl_sync(0xffffffffu, pincl, 31);
    }
    if (lane == 0 && pw == wpr - 1) sRankPad[pj] = pcarry;
  }
  __syncthreads();
  // row bases the route assignment needs
  for (int e = tid; e < E; e += kBalThreads)
    in[lay.home_rowbase + e] = nseg[(e / L) * EB + e] - sQ[e];
  for (int i = tid; i < R * L; i += kBalThreads) {
    const int j = i / L, u = i % L;
    const int b = slot_b[i];
    const int p = sRecvPiece[j];
    if (b >= 0 && p >= 0) {
      const int e = pDonor[p] * L + u;
      in[lay.slot_rowbase + i] = nseg[j * EB + E + b] - max(pStart[p], sQ[e]);
    }
  }
  if (ready != nullptr) {
    if (tid == 0) in[kMetaValid] = sErr == 0 ? 1 : 0;
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      atomicExch(ready, target);
    }
  }
  // slot copies per expert (a receiver holds an expert at most once)
  for (int e = tid; e < E; e += kBalThreads) {
    const int l = e / L, u = e % L;
    int cnt = 0;
    for (int j = 0; j < R; j++) {
      const int p = sRecvPiece[j];
      if (p >= 0 && pDonor[p] == l && slot_b[j * L + u] >= 0) cnt++;
    }
    t.rcnt[e] = cnt;
    t.rhas[e] = cnt > 0;
  }
  __syncthreads();

  // Phase F: rank offsets of padding rows and of used slots; reduce-list
  // positions.
  if (tid == 0) {
    int p = 0, u = 0;
    for (int j = 0; j < R; j++) {
      sPadOff[j] = p;
      p += sRankPad[j];
      sSlotOff[j] = u;
      u += sNslots[j];
    }
    sP = p;
    sU = u;
    in[lay.pad_prefix + R * EB] = p;
  }
  const int ncopies = block_exclusive_scan(t.rcnt, E);
  const int nexperts = block_exclusive_scan(t.rhas, E);

  // Phase G: global padding prefix, row bases, copy list, reduce list,
  // experts_to_copy.
  for (int i = tid; i < R * EB; i += kBalThreads)
    in[lay.pad_prefix + i] = t.pad[i] + sPadOff[i / EB];
  for (int i = tid; i < R * B; i += kBalThreads) {
    const int j = i / B, b = i % B;
    o.etc[i] = setc[i];
    if (b < sNslots[j]) {
      in[lay.copy_slot + sSlotOff[j] + b] = i;
      in[lay.copy_expert + sSlotOff[j] + b] = setc[i];
    }
  }
  // experts with copies in ascending id; their slots in ascending rank
  for (int e = tid; e < E; e += kBalThreads) {
    const int first = t.rcnt[e];
    const int next = e + 1 < E ? t.rcnt[e + 1] : ncopies;
    if (next == first) continue;
    const int di = t.rhas[e];
    const int l = e / L, u = e % L;
    in[lay.red_expert + di] = e;
    in[lay.red_first + di] = first;
    int c = 0;
    for (int j = 0; j < R; j++) {
      const int p = sRecvPiece[j];
      if (p >= 0 && pDonor[p] == l && slot_b[j * L + u] >= 0)
        in[lay.red_slot + first + c++] = j * B + slot_b[j * L + u];
    }
  }
  if (tid == 0) {
    in[lay.red_first + nexperts] = ncopies;
    in[kMetaD] = nexperts;
  }
  __syncthreads();

  // Phase H: publish, or neutralise the plan on error.  The error word is
  // left at zero for the next plan.
  const int err = sErr;
  if (err == 0) {
    if (tid == 0) {
      in[kMetaP] = sP;
      in[kMetaU] = sU;
      in[kMetaValid] = 1;
      in[kMetaErr] = 0;
    }
    return;
  }
  if (tid == 0) {
    in[kMetaErr] = 0;
    in[kMetaValid] = 0;
    in[kMetaP] = 0;
    in[kMetaU] = 0;
    in[kMetaD] = 0;
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
}

// Tile path: one CTA scans every expert's tile counts (where each tile's
// routes start inside P_e), then runs the balance tail.
__global__ void __launch_bounds__(kBalThreads)
plan_balance_kernel(PlanDims d, const int32_t *__restrict__ tpe, int32_t *hist, PlanOut o,
                    int32_t *in, PlanLayout lay, int32_t *status, int nseg_shared) {
  extern __shared__ int32_t sm[];
  __shared__ int sErr0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kBalThreads / 32;
  const int R = d.R, E = d.E, G = d.G;
  const BalTables t = bal_tables(sm, d, in + lay.nseg, in + lay.padw, nseg_shared != 0);
  if (tid == 0) sErr0 = in[kMetaErr];
  __syncthreads();
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
    if (lane == 0) {
      t.T[e] = carry;
      in[lay.T + e] = carry;
    }
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
  balance_tail(d, t, o, in, lay, status, sErr0);
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
// The whole planner in one cooperative launch of R*ceil(S*K/8192) blocks of
// 1024 threads, one per 8192-route tile of a source rank:
//   1. each warp walks 8 chunks of 32 consecutive routes and counts them per
//      expert (warp-aggregated, stable ordinals kept in registers);
//   2. per-expert offsets of the warps; the tile's histogram to global;
//   3. the last block to arrive sums the tiles per rank, checks
//      tokens_per_expert, scans over ranks and runs the balance step for every
//      rank, then publishes; the others wait for that (bounded by a time
//      limit);
//   4. every block adds the earlier tiles of its rank to its offsets, maps its
//      routes to (rank, row), marks duplicates with warp shuffles inside each
//      token's K lanes, and writes dst.
// Used when K divides 32 (a token's routes then never straddle a 32-route
// chunk), the tiles fit on the SMs at once and the tables fit in shared
// memory; otherwise the three-kernel tile path runs.

constexpr int kFusedThreads = 1024;
constexpr int kFusedWarps = kFusedThreads / 32;
constexpr int kFusedMaxItems = 8;  // routes per thread: 1, 2, 4 or 8 (tile = 1024 * items)

struct FusedArgs {
  PlanDims d;
  const int32_t *topk, *tpe;
  int32_t *hist;      // [G, E] tile counts, then [R, E] where each rank starts in P_e
  PlanOut o;
  int32_t *in;
  PlanLayout lay;
  int32_t *status;
  unsigned long long *sync;  // [0] arrivals, [1] last published arrival target
  int32_t *dupflag;
  int32_t *totals;    // [R, E] routes per (rank, expert): zero between calls
  int32_t *rank_off;  // [R, E] where each rank's routes start inside P_e
  int items;          // routes per thread; tile = 1024 * items routes
  int tpr, G;         // tiles per rank, R * tpr
  int nseg_shared;
  int publish;        // 0 only when a test makes the wait run out
  long long wait_ns;  // limit of the wait for the balance step
};

__device__ __forceinline__ long long globaltimer_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

size_t fused_smem_words(int R, int E, int B, bool nseg_shared) {
  return (size_t)kFusedWarps * E + 4 * (size_t)E + 8 * (size_t)R + (size_t)E * R +
         bal_tables_words(R, E, B, nseg_shared);
}

// IT routes per thread (1, 2, 4 or 8; tile = 1024 * IT routes).  A compile-time
// count keeps only the routes' registers live across the balance step.
template <int IT>
__global__ void __launch_bounds__(kFusedThreads, 1) plan_fused_kernel(FusedArgs a) {
  extern __shared__ int32_t sm[];
  const PlanDims d = a.d;
  const int R = d.R, E = d.E, L = d.L, C = d.C;
  const int g = blockIdx.x;
  const int r = g / a.tpr, t = g % a.tpr;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t *h = sm;                       // [warps][E]
  int32_t *sQoff = h + kFusedWarps * E;  // [E]
  int32_t *sHomeRb = sQoff + E;          // [E]
  int32_t *sSrc = sHomeRb + E;           // [E]
  int32_t *sSlotRb = sSrc + E;           // [R*L]
  int32_t *sR = sSlotRb + R * L;         // keep, first, count, start, len, recv [R each], dups [2R]
  int32_t *sCnt = sR + 8 * R;            // [R*E] (balance block)
  int32_t *sBal = sCnt + E * R;          // balance tables
  __shared__ int s_last, s_timeout, s_valid, s_bad, s_err;
  __shared__ unsigned long long s_target;

  const int32_t *src = a.topk + (int64_t)r * C;
  const unsigned lt = lanemask_lt();
  const int nbits = key_bits(E);
  for (int i = tid; i < kFusedWarps * E; i += kFusedThreads) h[i] = 0;
  if (tid == 0) {
    s_bad = 0;
    s_err = 0;
    s_timeout = 0;
  }
  __syncthreads();

  // 1. counts and in-warp ordinals
  int32_t *hw = h + warp * E;
  constexpr int items = IT;
  const int wbase = t * kFusedThreads * items + warp * 32 * items;
  int e_reg[items], o_reg[items];
  bool bad = false;
#pragma unroll
  for (int c = 0; c < items; c++) {
    const int i = wbase + c * 32 + lane;
    e_reg[c] = i < C ? __ldg(src + i) : -1;
  }
#pragma unroll
  for (int c = 0; c < items; c++) {
    const int i = wbase + c * 32 + lane;
    int e = e_reg[c];
    if (i < C && (e < 0 || e >= E)) bad = true;
    if (i >= C || e < 0 || e >= E) e = -1;
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
    atomicOr(a.in + kMetaErr, kErrBadExpert);
    set_status(a.status, MOONEP_ERR_BAD_EXPERT);
  }
  // 2. warp offsets per expert; the tile's histogram
  for (int e = tid; e < E; e += kFusedThreads) {
    int run = 0;
    for (int w = 0; w < kFusedWarps; w++) {
      const int v = h[w * E + e];
      h[w * E + e] = run;
      run += v;
    }
    a.hist[(int64_t)g * E + e] = run;
    if (run) atomicAdd(a.totals + (int64_t)r * E + e, run);
  }
  __threadfence();  // this thread's histogram entries, before the arrival
  __syncthreads();

  // 3. the last block to arrive balances; the others wait for it
  if (tid == 0) {
    __threadfence();
    const unsigned long long G = (unsigned long long)a.G;
    const unsigned long long old = atomicAdd(a.sync, 1ull);
    s_last = old % G == G - 1;
    s_target = old - old % G + G;
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    // per-rank counts (summed by the tiles' atomics); cleared for the next call
    for (int i = tid; i < R * E; i += kFusedThreads) {
      const int v = __ldcg(a.totals + i);
      a.totals[i] = 0;
      sCnt[i] = v;
    }
    __syncthreads();
    const BalTables tb = bal_tables(sBal, d, a.in + a.lay.nseg, a.in + a.lay.padw, a.nseg_shared != 0);
    // where each rank's routes start inside P_e, and T_e
    for (int e = tid; e < E; e += kFusedThreads) {
      int run = 0;
      for (int j = 0; j < R; j++) {
        a.rank_off[(int64_t)j * E + e] = run;
        run += sCnt[j * E + e];
      }
      tb.T[e] = run;
      a.in[a.lay.T + e] = run;
    }
    __syncthreads();
    // publishes the routing tables part-way through (unless a test withholds it)
    balance_tail(d, tb, a.o, a.in, a.lay, a.status, s_err | __ldcg(a.in + kMetaErr),
                 a.publish ? a.sync + 1 : nullptr, s_target);
    // tokens_per_expert against the recount, after the publication: a
    // mismatch latches its error but the plan stands (it is built from the
    // recount)
    if (a.tpe != nullptr)
      for (int i = tid; i < R * E; i += kFusedThreads)
        if (sCnt[i] != __ldg(a.tpe + i)) set_status(a.status, MOONEP_ERR_HIST_MISMATCH);
  } else {
    if (tid == 0) {
      const long long t0 = globaltimer_ns();
      const volatile unsigned long long *ready = a.sync + 1;
      while (*ready < s_target) {
        if (globaltimer_ns() - t0 > a.wait_ns) {
          s_timeout = 1;
          set_status(a.status, MOONEP_ERR_TIMEOUT);
          break;
        }
        __nanosleep(256);
      }
      __threadfence();
    }
    __syncthreads();
  }

  // 4. this tile's routes -> (rank, row), duplicate marks, dst
  for (int e = tid; e < E; e += kFusedThreads) {
    sQoff[e] = __ldcg(a.in + a.lay.qoff + e);
    sHomeRb[e] = __ldcg(a.in + a.lay.home_rowbase + e);
    // where this tile's routes start inside P_e: the rank's start plus the
    // rank's earlier tiles
    int off = __ldcg(a.rank_off + (int64_t)r * E + e);
#pragma unroll 4
    for (int tt = 0; tt < t; tt++) off += __ldcg(a.hist + (int64_t)(r * a.tpr + tt) * E + e);
    sSrc[e] = off;
  }
  for (int i = tid; i < R * L; i += kFusedThreads) sSlotRb[i] = __ldcg(a.in + a.lay.slot_rowbase + i);
  for (int j = tid; j < R; j += kFusedThreads) {
    sR[j] = __ldcg(a.in + a.lay.keep + j);
    sR[R + j] = __ldcg(a.in + a.lay.piece_first + j);
    sR[2 * R + j] = __ldcg(a.in + a.lay.piece_count + j);
    sR[3 * R + j] = __ldcg(a.in + a.lay.piece_start + j);
    sR[4 * R + j] = __ldcg(a.in + a.lay.piece_len + j);
    sR[5 * R + j] = __ldcg(a.in + a.lay.piece_recv + j);
  }
  for (int i = tid; i < 2 * R; i += kFusedThreads) sR[6 * R + i] = 0;
  if (tid == 0) s_valid = (__ldcg(a.in + kMetaValid) != 0) && !s_timeout;
  __syncthreads();
  const bool valid = s_valid;
  const int K = d.K;
  // A token's K routes sit in K consecutive lanes.  Routes of one token that
  // land on the same rank share the key (token lane group, rank).
  const int dkey_bits = key_bits((32 / K) * (R + 1));
  const int rkey_bits = key_bits(R);
  const unsigned lt_mask = lanemask_lt();
  int32_t *dst = a.o.dst + (int64_t)r * C;
#pragma unroll
  for (int c = 0; c < items; c++) {
    const int i = wbase + c * 32 + lane;
    const bool in_range = i < C;
    int j = R, row = 0;
    if (in_range) {
      j = 0;
      if (valid) {
        const int e = e_reg[c];
        const int p = sQoff[e] + sSrc[e] + h[warp * E + e] + o_reg[c];
        const int l = e / L;
        if (p < sR[l]) {
          j = l;
          row = sHomeRb[e] + p;
        } else {
          const int q0 = sR[R + l], qn = sR[2 * R + l];
          for (int pc = q0; pc < q0 + qn; pc++)
            if (p < sR[3 * R + pc] + sR[4 * R + pc]) {
              j = sR[5 * R + pc];
              row = sSlotRb[j * L + (e - l * L)] + p;
              break;
            }
        }
      }
    }
    const unsigned same = match_key((lane / K) * (R + 1) + j, dkey_bits);
    const bool primary = (same & lt_mask) == 0;
    const bool has_dup = (same & ~lt_mask & ~(1u << lane)) != 0;
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
      if (rk < R && (mr & lt_mask) == 0) {
        const int nd = __popc(mr & md), ng = __popc(mr & mg);
        if (nd) atomicAdd(&sR[6 * R + 2 * rk], nd);
        if (ng) atomicAdd(&sR[6 * R + 2 * rk + 1], ng);
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < 2 * R; i += kFusedThreads)
    if (sR[6 * R + i]) atomicAdd(a.o.dup_counts + i, sR[6 * R + i]);
}

// ------------------------------------------------------------------ K4

constexpr int kDupThreads = 1024;

__global__ void __launch_bounds__(kDupThreads)
plan_dup_kernel(PlanDims d, const int32_t *__restrict__ dst, const int32_t *__restrict__ dupflag,
                int32_t *__restrict__ dup_groups, int32_t *__restrict__ dup_loffs) {
  __shared__ int wsum[2][32];
  __shared__ int carry[2];
  const int j = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t rowbase = (int64_t)j * d.NvS;
  if (tid == 0) carry[0] = carry[1] = 0;
  __syncthreads();
  for (int w0 = 0; w0 < d.NvS; w0 += kDupThreads) {
    const int w = w0 + tid;
    int has = 0, cnt = 0, rid = -1;
    if (w < d.NvS) {
      rid = dupflag[rowbase + w] - 1;
      if (rid >= 0) {
        const int k = rid % d.K;
        const int64_t tb = rid - k;
        for (int k2 = k + 1; k2 < d.K; k2++) {
          const int v = dst[tb + k2];
          const int64_t g = v >= 0 ? v : -(int64_t)v - 1;
          if (g / d.NvS == j) cnt++;
        }
        has = 1;
      }
    }
    // block exclusive scans of has and cnt
    int hi = warp_incl_scan(has), ci = warp_incl_scan(cnt);
    if (lane == 31) {
      wsum[0][warp] = hi;
      wsum[1][warp] = ci;
    }
    __syncthreads();
    if (warp == 0) {
      const int a = warp_incl_scan(wsum[0][lane]);
      const int b = warp_incl_scan(wsum[1][lane]);
      wsum[0][lane] = a;
      wsum[1][lane] = b;
    }
    __syncthreads();
    const int gi = carry[0] + (warp ? wsum[0][warp - 1] : 0) + hi - has;
    const int di = carry[1] + (warp ? wsum[1][warp - 1] : 0) + ci - cnt;
    if (has) {
      int32_t *rec = dup_groups + (rowbase + gi) * 3;
      rec[0] = w;
      rec[1] = di;
      rec[2] = cnt;
      const int k = rid % d.K;
      const int64_t tb = rid - k;
      int c = 0;
      for (int k2 = k + 1; k2 < d.K; k2++) {
        const int v = dst[tb + k2];
        const int64_t g = v >= 0 ? v : -(int64_t)v - 1;
        if (g / d.NvS == j) dup_loffs[rowbase + di + c++] = (int)(g - rowbase);
      }
    }
    __syncthreads();
    if (tid == 0) {
      carry[0] += wsum[0][31];
      carry[1] += wsum[1][31];
    }
    __syncthreads();
  }
}

}  // namespace

// Fused path if K divides 32, a warp walks at most 64 chunks of 32 routes,
// and its tables fit in shared memory.  Returns K (template) or 0.
// Routes per thread of the single-launch planner: the fewest (most tiles,
// most SMs at work) for which every tile fits on the SMs at once; 0 if none.
int plan_fused_items(int R, int C, int sms) {
  for (int items = 1; items <= kFusedMaxItems; items *= 2) {
    const int tpr = (C + kFusedThreads * items - 1) / (kFusedThreads * items);
    if ((int64_t)R * (tpr > 0 ? tpr : 1) <= sms) return items;
  }
  return 0;
}

// Tiles of either planner path: the histogram area holds E words per tile,
// then the fused path's [R, E] totals and [R, E] rank starts.
int plan_hist_tiles(int R, int C, int sms) {
  const int tile_path = R * ((C + kTile - 1) / kTile);
  const int items = plan_fused_items(R, C, sms);
  const int fused = items ? R * ((C + kFusedThreads * items - 1) / (kFusedThreads * items)) : 0;
  return tile_path > fused ? tile_path : fused;
}

int plan_fused_tiles(int C, int items) {
  const int tpr = (C + kFusedThreads * items - 1) / (kFusedThreads * items);
  return tpr > 0 ? tpr : 1;
}

int plan_fused_choice(int R, int E, int K, int B, int C, int sms, bool *nseg_shared) {
  if (32 % K != 0 || R > kMaxR || plan_fused_items(R, C, sms) == 0) return 0;
  const size_t limit = 200 * 1024 / sizeof(int32_t);
  if (fused_smem_words(R, E, B, true) <= limit) {
    *nseg_shared = true;
    return K;
  }
  if (fused_smem_words(R, E, B, false) <= limit) {
    *nseg_shared = false;
    return K;
  }
  return 0;
}

cudaError_t plan_configure(int R, int E, int B) {
  const int hist_smem = (kPlanThreads / 32) * E * (int)sizeof(int32_t);
  const int assign_smem = (3 * E + 8 * R) * (int)sizeof(int32_t);
  const bool bal_shared = bal_tables_words(R, E, B, true) * sizeof(int32_t) <= 160 * 1024;
  const int bal_smem = (int)(bal_tables_words(R, E, B, bal_shared) * sizeof(int32_t));
  cudaError_t e = cudaSuccess;
  if (hist_smem > 48 * 1024)
    e = cudaFuncSetAttribute(plan_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             hist_smem);
  if (e == cudaSuccess && bal_smem > 48 * 1024)
    e = cudaFuncSetAttribute(plan_balance_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bal_smem);
  if (e == cudaSuccess && assign_smem > 48 * 1024) {
    const void *fs[] = {(const void *)plan_assign_kernel<0>, (const void *)plan_assign_kernel<1>,
                        (const void *)plan_assign_kernel<2>, (const void *)plan_assign_kernel<4>,
                        (const void *)plan_assign_kernel<6>, (const void *)plan_assign_kernel<8>};
    for (const void *f : fs)
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, assign_smem);
  }
  bool ns = false;
  if (e == cudaSuccess && plan_fused_choice(R, E, 1, B, 0, 1 << 30, &ns)) {
    const int fsmem = (int)(fused_smem_words(R, E, B, ns) * sizeof(int32_t));
    if (fsmem > 48 * 1024) {
      const void *fs[] = {(const void *)plan_fused_kernel<1>, (const void *)plan_fused_kernel<2>,
                          (const void *)plan_fused_kernel<4>, (const void *)plan_fused_kernel<8>};
      for (const void *f : fs)
        if (e == cudaSuccess)
          e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, fsmem);
    }
  }
  return e;
}

int launch_plan(moonep_ctx *ctx, const int32_t *topk, const int32_t *tpe,
                moonep_comm_plan *plan, cudaStream_t st) {
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
  const bool dup = (plan->flags & MOONEP_PLAN_DUP_RECORDS) != 0;
  PlanLayout lay = PlanLayout::make(d.R, d.E, d.B, d.NvS, dup);
  int32_t *in = plan->internal;
  int32_t *dupflag = dup ? in + lay.dupflag : nullptr;
  cudaError_t e;
  if (dup) {
    e = cudaMemsetAsync(dupflag, 0, (size_t)d.R * d.NvS * sizeof(int32_t), st);
    if (e != cudaSuccess) return cuda_status(e);
  }
  PlanOut o{plan->dst, plan->experts_to_copy, plan->cu_seqlens, plan->zero_fill_ranges,
            plan->remote_stats, plan->dup_counts, plan->dup_groups, plan->dup_loffs};
  bool nseg_shared = false;
  const int fused_k = plan_fused_choice(d.R, d.E, d.K, d.B, d.C, ctx->sms_device, &nseg_shared);
  if (fused_k > 0 && ctx->d_sync != nullptr) {
    FusedArgs fa;
    fa.d = d;
    fa.topk = topk;
    fa.tpe = tpe;
    fa.hist = ctx->d_hist;
    fa.items = plan_fused_items(d.R, d.C, ctx->sms_device);
    fa.tpr = plan_fused_tiles(d.C, fa.items);
    fa.G = d.R * fa.tpr;
    fa.totals = ctx->d_hist + (int64_t)d.E * plan_hist_tiles(d.R, d.C, ctx->sms_device);
    fa.rank_off = fa.totals + (int64_t)d.R * d.E;
    fa.o = o;
    fa.in = in;
    fa.lay = lay;
    fa.status = ctx->d_status;
    fa.sync = ctx->d_sync;
    fa.dupflag = dupflag;
    fa.nseg_shared = nseg_shared ? 1 : 0;
    fa.publish = ctx->test_unpublished_plan ? 0 : 1;
    fa.wait_ns = ctx->test_unpublished_plan ? 200000000LL : 1000000000LL;
    void *args[] = {&fa};
    const size_t smem = fused_smem_words(d.R, d.E, d.B, nseg_shared) * sizeof(int32_t);
    const void *kern = fa.items == 1   ? (const void *)plan_fused_kernel<1>
                       : fa.items == 2 ? (const void *)plan_fused_kernel<2>
                       : fa.items == 4 ? (const void *)plan_fused_kernel<4>
                                       : (const void *)plan_fused_kernel<8>;
    e = cudaLaunchCooperativeKernel(kern, dim3(fa.G), dim3(kFusedThreads), args, smem, st);
    if (e != cudaSuccess) return cuda_status(e);
  } else {
    e = cudaMemsetAsync(in, 0, kMetaWords * sizeof(int32_t), st);
    if (e != cudaSuccess) return cuda_status(e);
    if (d.G > 0) {
      const size_t smem = (size_t)(kPlanThreads / 32) * d.E * sizeof(int32_t);
      plan_hist_kernel<<<d.G, kPlanThreads, smem, st>>>(topk, d, ctx->d_hist, ctx->d_ord, in,
                                                         ctx->d_status);
    }
    const bool bal_shared = bal_tables_words(d.R, d.E, d.B, true) * sizeof(int32_t) <= 160 * 1024;
    plan_balance_kernel<<<1, kBalThreads,
                          bal_tables_words(d.R, d.E, d.B, bal_shared) * sizeof(int32_t), st>>>(
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
  if (dup)
    plan_dup_kernel<<<d.R, kDupThreads, 0, st>>>(d, plan->dst, in + lay.dupflag,
                                                 plan->dup_groups, plan->dup_loffs);
  return cuda_status(cudaGetLastError());
}

}  // namespace moonep
