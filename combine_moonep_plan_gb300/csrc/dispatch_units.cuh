// The dispatch's unit loop, shared by the stand-alone dispatch kernel and the
// small-batch plan+dispatch kernel.
//
// "MoonEP Public API Visual Guide", Buffer.dispatch(...): every route's token
// row lands on its destination row |dst|, every routing weight beside it,
// and padding rows are zero.  The work is cut into units: first one unit per
// padding row (found by a 32-way search over the plan's padding prefix),
// then units of (token, chunk of 32*kU 16-byte vectors), strided over every
// warp of the grid.  A token unit loads its chunk of the source row once
// (the load issued before its dst entries are decoded, so the two round
// trips overlap) and stores it to all K destination rows.
#pragma once

#include "copy_common.cuh"
#include "moonep_internal.cuh"

namespace moonep {

struct DispatchArgs {
  const uint4 *hidden;
  const float *w_sk;
  const int32_t *dst;
  const int32_t *pad_prefix;
  const int32_t *zfr;
  int32_t *status;
  int64_t ntok;       // tokens of the launch: R*S, or S (rank-local)
  int64_t total_rows; // R*NvS
  int K, H8, nchunk, NvS, EB;
  int seg_lo, seg_hi;  // the (rank, segment) entries whose padding rows this launch zeroes
  int primaries_only;  // rows of duplicate routes are left for the expand epilogue
  int interleave;      // number warps across blocks first (small batches)
};

// Destination addressing of global row g = j*NvS + w.  Flat: one [R*NvS, H]
// buffer.  Windows: rank j's [NvS, H] rows start at row[j] (and its route
// weights at w[j]), each window its own allocation.
struct FlatRows {
  uint4 *out;
  float *w_out;
  __device__ __forceinline__ uint4 *row(int64_t g, int H8, int) const { return out + g * H8; }
  __device__ __forceinline__ float *weight(int64_t g, int) const { return w_out + g; }
  __device__ __forceinline__ bool has_weights() const { return w_out != nullptr; }
};

struct WindowRows {
  uint4 *out[kMaxRanks];
  float *w_out[kMaxRanks];
  __device__ __forceinline__ uint4 *row(int64_t g, int H8, int NvS) const {
    const int j = (int)(g / NvS);
    return out[j] + (g - (int64_t)j * NvS) * H8;
  }
  __device__ __forceinline__ float *weight(int64_t g, int NvS) const {
    const int j = (int)(g / NvS);
    return w_out[j] + (g - (int64_t)j * NvS);
  }
  __device__ __forceinline__ bool has_weights() const { return w_out[0] != nullptr; }
};

// The arguments of a dispatch of ntok tokens starting at source rank r0
// (plan->dst row r0 on), zeroing the padding rows of (rank, segment) entries
// [seg_lo, seg_hi), in units of 32*U 16-byte vectors.
DispatchArgs dispatch_args(const moonep_ctx *ctx, const moonep_comm_plan *plan,
                           const uint16_t *hidden, const float *w_sk, int64_t ntok, int r0,
                           int seg_lo, int seg_hi, int U);

// A word of the plan: through the read-only path when an earlier kernel
// wrote it, through L2 when another block of the same launch did.
template <bool kSameLaunch>
__device__ __forceinline__ int32_t plan_word(const int32_t *p) {
  return kSameLaunch ? __ldcg(p) : __ldg(p);
}

// Units wid, wid + nw, ... of the launch (wid: this warp, nw: warps of the
// grid), whole-warp code.  kU: 16-byte vectors per lane per token unit.
// kSameLaunch: the plan was written by other blocks of this launch.
template <int KT, int kU, class Rows, bool kSameLaunch = false>
__device__ __forceinline__ void dispatch_units(const DispatchArgs &a, const Rows &rows,
                                               int64_t wid, int64_t nw) {
  constexpr int kChunk = 32 * kU;  // vectors per unit
  const int lane = threadIdx.x & 31;
  const int K = KT > 0 ? KT : a.K;
  const int64_t tok_units = a.ntok * a.nchunk;
  // padding rows of the launch's segments (all of them, or one rank's)
  const int64_t q0 = plan_word<kSameLaunch>(a.pad_prefix + a.seg_lo);
  const int64_t P = plan_word<kSameLaunch>(a.pad_prefix + a.seg_hi) - q0;
  const int64_t units = P + tok_units;  // padding rows first, then token units
  const bool wts = rows.has_weights();
  // The warp's next token unit's dst entries are loaded one unit ahead.
  int32_t d_next = 0;
  {
    int64_t w0 = wid - P;
    if (w0 < 0) w0 += ((-w0 + nw - 1) / nw) * nw;
    if (w0 < tok_units && lane < K)
      d_next = plan_word<kSameLaunch>(a.dst + (w0 / a.nchunk) * K + lane);
  }
  for (int64_t uu = wid; uu < units; uu += nw) {
    const int64_t u = uu - P;
    if (u >= 0) {
      const int64_t t = u / a.nchunk;
      const int c = (int)(u - t * a.nchunk);
      const int32_t d_cur = d_next;
      if (u + nw < tok_units && lane < K)
        d_next = plan_word<kSameLaunch>(a.dst + ((u + nw) / a.nchunk) * K + lane);
      const uint4 *src = a.hidden + t * a.H8;
      const int v0 = c * kChunk + lane;
      uint4 x[kU];
#pragma unroll
      for (int i = 0; i < kU; i++) {
        const int v = v0 + 32 * i;
        if (v < a.H8) x[i] = ld_stream(src + v);
      }
      float wv = 0.0f;
      if (c == 0 && lane < K && wts) wv = __ldg(a.w_sk + t * K + lane);
      int64_t g = -1;
      if (lane < K) {
        const int64_t gg = decode_row(d_cur);
        if (gg < a.total_rows) {
          g = gg;
        } else {
          set_status(a.status, MOONEP_ERR_PLAN);
        }
        if (c == 0 && g >= 0 && wts) *rows.weight(g, a.NvS) = wv;
        if (a.primaries_only && d_cur < 0) g = -1;
      }
      if (KT > 0) {
#pragma unroll
        for (int k = 0; k < (KT > 0 ? KT : 1); k++) {
          const int64_t gk = __shfl_sync(0xffffffffu, g, k);
          if (gk < 0) continue;
          uint4 *dp = rows.row(gk, a.H8, a.NvS);
#pragma unroll
          for (int i = 0; i < kU; i++) {
            const int v = v0 + 32 * i;
            if (v < a.H8) st_global(dp + v, x[i]);
          }
        }
      } else {
        for (int k = 0; k < K; k++) {
          const int64_t gk = __shfl_sync(0xffffffffu, g, k);
          if (gk < 0) continue;
          uint4 *dp = rows.row(gk, a.H8, a.NvS);
#pragma unroll
          for (int i = 0; i < kU; i++) {
            const int v = v0 + 32 * i;
            if (v < a.H8) st_global(dp + v, x[i]);
          }
        }
      }
    } else {
      // padding row q: segment = last s with pad_prefix[s] <= q, found by a
      // 32-way search (each round the lanes probe 32 points of the range:
      // three dependent loads for a few thousand segments, not a dozen)
      const int64_t q = q0 + uu;
      int lo = a.seg_lo, hi = a.seg_hi;
      while (hi - lo > 1) {
        const int step = (hi - lo + 31) >> 5;
        const int idx = lo + lane * step;
        const bool le = idx < hi && plan_word<kSameLaunch>(a.pad_prefix + idx) <= q;
        const unsigned m = __ballot_sync(0xffffffffu, le);
        lo += (31 - __clz(m)) * step;
        hi = min(hi, lo + step);
      }
      const int j = lo / a.EB;
      const int64_t row = plan_word<kSameLaunch>(a.zfr + 2 * lo) +
                          (q - plan_word<kSameLaunch>(a.pad_prefix + lo));
      const int64_t g = (int64_t)j * a.NvS + row;
      if (g >= a.total_rows) {
        set_status(a.status, MOONEP_ERR_PLAN);
        continue;
      }
      uint4 *dp = rows.row(g, a.H8, a.NvS);
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (int v = lane; v < a.H8; v += 32) st_global(dp + v, z);
      if (lane == 0 && wts) *rows.weight(g, a.NvS) = 0.0f;
    }
  }
}

}  // namespace moonep
