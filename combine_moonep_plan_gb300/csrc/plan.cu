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
    const unsigned m = __match_any_sync(0xffffffffu, e);
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

__global__ void __launch_bounds__(kBalThreads)
plan_balance_kernel(PlanDims d, const int32_t *__restrict__ tpe, int32_t *hist, PlanOut o,
                    int32_t *in, PlanLayout lay, int32_t *status) {
  extern __shared__ int32_t sm[];  // T[E], Q[E]
  int32_t *sT = sm;
  int32_t *sQ = sm + d.E;
  __shared__ int sG[kMaxR], sKeep[kMaxR], sRecvPiece[kMaxR], sNslots[kMaxR], sRankPad[kMaxR];
  __shared__ int pDonor[kMaxR], pRecv[kMaxR], pLen[kMaxR], pStart[kMaxR];
  __shared__ int sNp, sErr, sP, sU;
  __shared__ int sPadOff[kMaxR], sSlotOff[kMaxR];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kBalThreads / 32;
  const int R = d.R, E = d.E, L = d.L, B = d.B, EB = d.EB, C = d.C, G = d.G;
  int32_t *Tg = in + lay.T, *qoffg = in + lay.qoff, *nseg = in + lay.nseg;
  int32_t *slot_rb = in + lay.slot_rowbase;
  int32_t *slot_b = in + lay.slot_b;
  if (tid == 0) {
    sErr = in[kMetaErr];
    sNp = 0;
  }
  __syncthreads();

  // Phase A: for every expert, exclusive scan of its tile counts over all
  // (rank, tile) in order -> where each tile's routes start inside P_e.
  for (int e = warp; e < E; e += kWarps) {
    int carry = 0;
    int32_t *col = hist + (int64_t)e * G;
    for (int b0 = 0; b0 < G; b0 += 32) {
      const int idx = b0 + lane;
      const int v = idx < G ? col[idx] : 0;
      const int incl = warp_incl_scan(v);
      if (idx < G) col[idx] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    __syncwarp();
    if (lane == 0) {
      sT[e] = carry;
      Tg[e] = carry;
    }
    if (tpe != nullptr) {
      for (int r = lane; r < R; r += 32) {
        int cnt = 0;
        if (G > 0) {
          const int a = col[r * d.TPR];
          const int b = (r + 1 < R) ? col[(r + 1) * d.TPR] : carry;
          cnt = b - a;
        }
        if (cnt != tpe[(int64_t)r * E + e]) atomicOr(&sErr, kErrHist);
      }
    }
  }
  // Defaults for the slot tables.
  for (int i = tid; i < R * B; i += kBalThreads) o.etc[i] = -1;
  for (int i = tid; i < R * EB; i += kBalThreads) nseg[i] = 0;
  for (int i = tid; i < R * L; i += kBalThreads) slot_b[i] = -1;
  for (int i = tid; i < 2 * R; i += kBalThreads) {
    o.remote_stats[i] = 0;
    o.dup_counts[i] = 0;
  }
  __syncthreads();

  // Phase B: offset of P_e inside Q_home(e), and G_j = |Q_j|.
  for (int j = tid; j < R; j += kBalThreads) {
    int acc = 0;
    for (int e = j * L; e < (j + 1) * L; e++) {
      sQ[e] = acc;
      qoffg[e] = acc;
      acc += sT[e];
    }
    sG[j] = acc;
  }
  __syncthreads();

  // Phase C: the chain balance (at most R rounds, each fills one receiver).
  if (tid == 0) {
    int rem[kMaxR], donated[kMaxR];
    for (int j = 0; j < R; j++) {
      rem[j] = sG[j];
      donated[j] = 0;
      sRecvPiece[j] = -1;
    }
    int np = 0;
    for (int round = 0; round <= R; round++) {
      int recv = -1, donor = -1;
      for (int j = 0; j < R; j++)
        if (rem[j] < C) { recv = j; break; }
      if (recv < 0) break;
      for (int j = 0; j < R; j++)
        if (rem[j] > C) { donor = j; break; }
      if (donor < 0 || np >= R) {  // only reachable from a broken histogram
        sErr |= kErrHist;
        break;
      }
      const int dd = C - rem[recv];
      pDonor[np] = donor;
      pRecv[np] = recv;
      pLen[np] = dd;
      sRecvPiece[recv] = np;
      np++;
      rem[donor] -= dd;
      rem[recv] = C;
      donated[donor] += dd;
    }
    int cursor[kMaxR];
    for (int j = 0; j < R; j++) {
      sKeep[j] = sG[j] - donated[j];
      cursor[j] = sKeep[j];
      in[lay.keep + j] = sKeep[j];
    }
    for (int p = 0; p < np; p++) {
      pStart[p] = cursor[pDonor[p]];
      cursor[pDonor[p]] += pLen[p];
    }
    // pieces grouped by donor, recording order inside a donor
    int n = 0;
    for (int l = 0; l < R; l++) {
      in[lay.piece_first + l] = n;
      int c = 0;
      for (int p = 0; p < np; p++)
        if (pDonor[p] == l) {
          in[lay.piece_start + n] = pStart[p];
          in[lay.piece_len + n] = pLen[p];
          in[lay.piece_recv + n] = pRecv[p];
          n++;
          c++;
        }
      in[lay.piece_count + l] = c;
    }
    sNp = np;
  }
  __syncthreads();

  // Phase D: slots of every receiver (one warp per piece) and home counts.
  for (int p = warp; p < sNp; p += kWarps) {
    const int l = pDonor[p], j = pRecv[p], a = pStart[p], dd = pLen[p];
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
          o.etc[j * B + b] = e;
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
  for (int j = tid; j < R; j += kBalThreads)
    if (sRecvPiece[j] < 0) sNslots[j] = 0;
  for (int e = tid; e < E; e += kBalThreads) {
    const int j = e / L;
    nseg[j * EB + e] = min(max(sKeep[j] - sQ[e], 0), sT[e]);
  }
  __syncthreads();

  // Phase E: per rank, padded segment lengths -> cu_seqlens, padding ranges,
  // segment starts (kept in nseg) and the rank's padding-row prefix.
  for (int j = warp; j < R; j += kWarps) {
    int carry = 0, pcarry = 0;
    for (int x0 = 0; x0 < EB; x0 += 32) {
      const int x = x0 + lane;
      const int n = x < EB ? nseg[j * EB + x] : 0;
      const int padded = (n + d.tp - 1) / d.tp * d.tp;
      const int pc = padded - n;
      const int incl = warp_incl_scan(padded);
      const int pincl = warp_incl_scan(pc);
      if (x < EB) {
        const int end = carry + incl;
        const int start = end - padded;
        o.cu[j * EB + x] = end;
        o.zfr[2 * (j * EB + x)] = start + n;
        o.zfr[2 * (j * EB + x) + 1] = end;
        nseg[j * EB + x] = start;
        in[lay.pad_prefix + j * EB + x] = pcarry + pincl - pc;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
      pcarry += __shfl_sync(0xffffffffu, pincl, 31);
    }
    if (lane == 0) sRankPad[j] = pcarry;
  }
  __syncthreads();

  // Phase F: rank offsets of padding rows and of used slots.
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
  __syncthreads();

  // Phase G: global padding prefix, row bases, copy list, reduce list.
  for (int i = tid; i < R * EB; i += kBalThreads) in[lay.pad_prefix + i] += sPadOff[i / EB];
  for (int e = tid; e < E; e += kBalThreads)
    in[lay.home_rowbase + e] = nseg[(e / L) * EB + e] - sQ[e];
  for (int i = tid; i < R * L; i += kBalThreads) {
    const int j = i / L, u = i % L;
    const int b = slot_b[i];
    const int p = sRecvPiece[j];
    if (b >= 0 && p >= 0) {
      const int e = pDonor[p] * L + u;
      slot_rb[i] = nseg[j * EB + E + b] - max(pStart[p], sQ[e]);
    }
  }
  for (int i = tid; i < R * B; i += kBalThreads) {
    const int j = i / B, b = i % B;
    if (b < sNslots[j]) {
      in[lay.copy_slot + sSlotOff[j] + b] = i;
      in[lay.copy_expert + sSlotOff[j] + b] = o.etc[i];
    }
  }
  if (warp == 0) {
    // experts with copies in ascending id; their slots in ascending rank
    // (a receiver holds an expert at most once, in slot slot_b[j][u]).
    int dcarry = 0, scarry = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      int cnt = 0;
      if (e < E) {
        const int l = e / L, u = e % L;
        for (int j = 0; j < R; j++) {
          const int p = sRecvPiece[j];
          if (p >= 0 && pDonor[p] == l && slot_b[j * L + u] >= 0) cnt++;
        }
      }
      const bool has = cnt > 0;
      const unsigned bal = __ballot_sync(0xffffffffu, has);
      const int di = dcarry + __popc(bal & lanemask_lt());
      const int sincl = warp_incl_scan(cnt);
      const int first = scarry + sincl - cnt;
      if (has) {
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
      dcarry += __popc(bal);
      scarry += __shfl_sync(0xffffffffu, sincl, 31);
    }
    if (lane == 0) {
      in[lay.red_first + dcarry] = scarry;
      in[kMetaD] = dcarry;
    }
  }
  __syncthreads();

  // Phase H: publish, or neutralise the plan on error.
  const int err = sErr;
  if (err == 0) {
    if (tid == 0) {
      in[kMetaP] = sP;
      in[kMetaU] = sU;
      in[kMetaValid] = 1;
    }
    return;
  }
  if (tid == 0) {
    in[kMetaErr] = err;
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

cudaError_t plan_configure(int R, int E) {
  const int hist_smem = (kPlanThreads / 32) * E * (int)sizeof(int32_t);
  const int assign_smem = (3 * E + 8 * R) * (int)sizeof(int32_t);
  const int bal_smem = 2 * E * (int)sizeof(int32_t);
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
  return e;
}

int launch_plan(moonep_ctx *ctx, const int32_t *topk, const int32_t *tpe, moonep_comm_plan *plan,
                cudaStream_t st) {
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
  cudaError_t e = cudaMemsetAsync(in, 0, kMetaWords * sizeof(int32_t), st);
  if (e != cudaSuccess) return cuda_status(e);
  if (dup) {
    e = cudaMemsetAsync(in + lay.dupflag, 0, (size_t)d.R * d.NvS * sizeof(int32_t), st);
    if (e != cudaSuccess) return cuda_status(e);
  }
  if (d.G > 0) {
    const size_t smem = (size_t)(kPlanThreads / 32) * d.E * sizeof(int32_t);
    plan_hist_kernel<<<d.G, kPlanThreads, smem, st>>>(topk, d, ctx->d_hist, ctx->d_ord, in,
                                                       ctx->d_status);
  }
  PlanOut o{plan->dst, plan->experts_to_copy, plan->cu_seqlens, plan->zero_fill_ranges,
            plan->remote_stats, plan->dup_counts, plan->dup_groups, plan->dup_loffs};
  plan_balance_kernel<<<1, kBalThreads, 2 * d.E * sizeof(int32_t), st>>>(
      d, tpe, ctx->d_hist, o, in, lay, ctx->d_status);
  if ((int64_t)d.R * d.S > 0) {
    const int64_t ntok = (int64_t)d.R * d.S;
    const int grid = (int)((ntok + kAssignThreads - 1) / kAssignThreads);
    const size_t smem = (size_t)(2 * d.E + d.R * d.L + 8 * d.R) * sizeof(int32_t);
    int32_t *dupflag = dup ? in + lay.dupflag : nullptr;
#define MOONEP_ASSIGN(KV)                                                              \
  plan_assign_kernel<KV><<<grid, kAssignThreads, smem, st>>>(d, topk, ctx->d_ord,       \
                                                             ctx->d_hist, in, lay,      \
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
  if (dup)
    plan_dup_kernel<<<d.R, kDupThreads, 0, st>>>(d, plan->dst, in + lay.dupflag,
                                                 plan->dup_groups, plan->dup_loffs);
  return cuda_status(cudaGetLastError());
}

}  // namespace moonep
