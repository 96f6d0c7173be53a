// The deduplicated data flow's two local steps.
//
// "MoonEP Public API Visual Guide", Buffer.dispatch(...): a token routed to
// several experts on one destination rank crosses the link once (its primary
// route, dst >= 0); the dispatch epilogue on that rank expands the primary row
// into the rows of the token's later routes there (dst < 0).
// Buffer.combine(...): the duplicate prologue first accumulates every rank's
// duplicate rows of a token into the primary row in fp32 (one bf16 rounding),
// so the gather again moves one row per (token, rank).
// MoonEPCommPlan: dup_groups / dup_loffs list, per rank, each primary row with
// the rank-local rows of its duplicates (in k order) -- the work lists of both
// steps.
//
// Units of (group, chunk of a row) are split into one contiguous run per warp
// of a persistent grid; the global group index is mapped to its rank through a
// per-warp prefix over dup_counts[j][1].  Expand reads the primary chunk once
// and stores it to every duplicate row; fold loads the primary with the first
// two duplicate chunks (then two at a time), adds them in k order in fp32 and
// stores one bf16 RNE result.
// HBM bytes per call (D duplicate routes, Gr groups, row = H*2 bytes):
// expand reads Gr rows and writes D rows; fold reads Gr + D rows and writes Gr.
#include "copy_common.cuh"
#include "moonep_internal.cuh"

namespace moonep {
namespace {

constexpr int kExpandThreads = 256;
constexpr int kFoldThreads = 128;
constexpr int kExpandU = 8;  // 16-byte vectors per lane per unit (4 KB)
constexpr int kFoldU = 4;    // 2 KB per row per unit
constexpr int kFoldBatch = 2;

struct Args {
  uint4 *rows;                // [R*NvS, H8]
  const int32_t *dup_counts;  // [R, 2]
  const int32_t *groups;      // [R, NvS, 3]
  const int32_t *loffs;       // [R, NvS]
  int32_t *status;
  int R, NvS, K, H8, nchunk;
};

__device__ __forceinline__ int warp_scan_incl(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

__device__ __forceinline__ void add8(float (&acc)[8], const uint4 &v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    acc[2 * i] += __uint_as_float(w[i] << 16);
    acc[2 * i + 1] += __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ void set8(float (&acc)[8], const uint4 &v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    acc[2 * i] = __uint_as_float(w[i] << 16);
    acc[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint4 pack8(const float (&acc)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i]));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i + 1]));
    w[i] = lo | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// One group of rank j, decoded and checked: primary row and duplicate rows
// (lane k < cnt holds the k-th duplicate's rank-local row).  Returns false
// (and flags the plan as invalid) when a record points outside the rank.
struct Group {
  int64_t base;  // j*NvS
  int prim, cnt, dup;
};

__device__ __forceinline__ bool load_group(const Args &a, int j, int i, Group &g) {
  const int lane = threadIdx.x & 31;
  const int32_t *rec = a.groups + ((int64_t)j * a.NvS + i) * 3;
  const int v = lane < 3 ? __ldg(rec + lane) : 0;
  g.base = (int64_t)j * a.NvS;
  g.prim = __shfl_sync(0xffffffffu, v, 0);
  const int first = __shfl_sync(0xffffffffu, v, 1);
  g.cnt = __shfl_sync(0xffffffffu, v, 2);
  bool ok = g.prim >= 0 && g.prim < a.NvS && g.cnt >= 1 && g.cnt < a.K && first >= 0 &&
            first <= a.NvS - g.cnt;
  g.dup = 0;
  if (ok && lane < g.cnt) {
    g.dup = __ldg(a.loffs + g.base + first + lane);
    if (g.dup < 0 || g.dup >= a.NvS) ok = false;
  }
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && lane == 0) set_status(a.status, MOONEP_ERR_PLAN);
  return ok;
}

template <bool FOLD>
__global__ void __launch_bounds__(FOLD ? kFoldThreads : kExpandThreads, FOLD ? 4 : 3)
dedup_kernel(Args a) {
  constexpr int kThreads = FOLD ? kFoldThreads : kExpandThreads;
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t wid = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * kThreads) >> 5;
  // groups per rank (R <= 64: two ranks per lane), inclusive prefix p0 for
  // rank lane, p1 for rank lane + 32
  int c0 = lane < a.R ? __ldg(a.dup_counts + 2 * lane + 1) : 0;
  int c1 = lane + 32 < a.R ? __ldg(a.dup_counts + 2 * (lane + 32) + 1) : 0;
  if (c0 < 0 || c0 > a.NvS || c1 < 0 || c1 > a.NvS) {
    set_status(a.status, MOONEP_ERR_PLAN);
    c0 = c1 = 0;
  }
  const int p0 = warp_scan_incl(c0);
  const int p1 = warp_scan_incl(c1) + __shfl_sync(0xffffffffu, p0, 31);
  const int total = __shfl_sync(0xffffffffu, p1, 31);
  const int64_t units = (int64_t)total * a.nchunk;
  // Each warp takes a contiguous run of units, so consecutive units share a
  // group and its record (three dependent loads) is read once per group, not
  // once per chunk.
  const int64_t per = (units + nw - 1) / nw;
  const int64_t ub = wid * per;
  const int64_t ue = ub + per < units ? ub + per : units;
  int cur = -1;
  bool ok = false;
  Group g;
  for (int64_t u = ub; u < ue; u++) {
    const int gi = (int)(u / a.nchunk);
    const int c = (int)(u - (int64_t)gi * a.nchunk);
    if (gi != cur) {
      cur = gi;
      // rank of group gi = number of ranks whose inclusive prefix is <= gi
      const int j = __popc(__ballot_sync(0xffffffffu, p0 <= gi)) +
                    __popc(__ballot_sync(0xffffffffu, p1 <= gi));
      const int jm = (j - 1) & 31;
      const int e0 = __shfl_sync(0xffffffffu, p0, jm), e1 = __shfl_sync(0xffffffffu, p1, jm);
      const int excl = j == 0 ? 0 : (j - 1 < 32 ? e0 : e1);
      ok = load_group(a, j, gi - excl, g);
    }
    if (!ok) continue;
    const uint4 *prow = a.rows + (g.base + g.prim) * a.H8;
    if (!FOLD) {
      const int v0 = c * 32 * kExpandU + lane;
      uint4 x[kExpandU];
#pragma unroll
      for (int i = 0; i < kExpandU; i++) {
        const int v = v0 + 32 * i;
        if (v < a.H8) x[i] = ld_stream(prow + v);
      }
      for (int k = 0; k < g.cnt; k++) {
        uint4 *dp = a.rows + (g.base + __shfl_sync(0xffffffffu, g.dup, k)) * a.H8;
#pragma unroll
        for (int i = 0; i < kExpandU; i++) {
          const int v = v0 + 32 * i;
          if (v < a.H8) st_global(dp + v, x[i]);
        }
      }
    } else {
      // primary and the first two duplicates are loaded together (most
      // groups have one or two), later duplicates two at a time; the adds
      // run in k order
      const int v0 = c * 32 * kFoldU + lane;
      float acc[kFoldU][8];
      for (int k0 = 0; k0 < g.cnt; k0 += kFoldBatch) {
        uint4 x[kFoldU], y[kFoldBatch][kFoldU];
#pragma unroll
        for (int i = 0; i < kFoldU; i++) {
          const int v = v0 + 32 * i;
          x[i] = make_uint4(0, 0, 0, 0);
          if (k0 == 0 && v < a.H8) x[i] = ld_stream(prow + v);
        }
#pragma unroll
        for (int kk = 0; kk < kFoldBatch; kk++) {
          const int dr = __shfl_sync(0xffffffffu, g.dup, (k0 + kk) & 31);
          const uint4 *row = a.rows + (g.base + dr) * a.H8;
#pragma unroll
          for (int i = 0; i < kFoldU; i++) {
            const int v = v0 + 32 * i;
            y[kk][i] = make_uint4(0, 0, 0, 0);
            if (k0 + kk < g.cnt && v < a.H8) y[kk][i] = ld_stream(row + v);
          }
        }
        if (k0 == 0) {
#pragma unroll
          for (int i = 0; i < kFoldU; i++) set8(acc[i], x[i]);
        }
#pragma unroll
        for (int kk = 0; kk < kFoldBatch; kk++) {
          if (k0 + kk >= g.cnt) break;
#pragma unroll
          for (int i = 0; i < kFoldU; i++) add8(acc[i], y[kk][i]);
        }
      }
      uint4 *op = a.rows + (g.base + g.prim) * a.H8;
#pragma unroll
      for (int i = 0; i < kFoldU; i++) {
        const int v = v0 + 32 * i;
        if (v < a.H8) st_global(op + v, pack8(acc[i]));
      }
    }
  }
}

int launch_dedup(moonep_ctx *ctx, const moonep_comm_plan *plan, uint16_t *rows, bool fold,
                 cudaStream_t st) {
  const moonep_config &c = ctx->cfg;
  if (!(plan->flags & MOONEP_PLAN_DUP_RECORDS) || !plan->dup_groups || !plan->dup_loffs)
    return MOONEP_ERR_INVALID_ARG;
  Args a;
  a.rows = reinterpret_cast<uint4 *>(rows);
  a.dup_counts = plan->dup_counts;
  a.groups = plan->dup_groups;
  a.loffs = plan->dup_loffs;
  a.status = ctx->d_status;
  a.R = c.R;
  a.NvS = ctx->NvS;
  a.K = c.K;
  a.H8 = c.H / 8;
  const int U = fold ? kFoldU : kExpandU;
  a.nchunk = (a.H8 + 32 * U - 1) / (32 * U);
  if (a.H8 == 0 || c.K < 2 || (int64_t)c.R * c.S == 0) return MOONEP_OK;
  const cudaError_t e =
      fold ? launch_pdl(dedup_kernel<true>, ctx->sms * ctx->blocks_fold, kFoldThreads, 0, st,
                        false, a)
           : launch_pdl(dedup_kernel<false>, ctx->sms * ctx->blocks_expand, kExpandThreads, 0, st,
                        false, a);
  return cuda_status(e);
}

}  // namespace

int occupancy_dedup(bool fold) {
  int n = 0;
  const cudaError_t e =
      fold ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dedup_kernel<true>, kFoldThreads, 0)
           : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dedup_kernel<false>,
                                                           kExpandThreads, 0);
  if (e != cudaSuccess) n = 1;
  return n > 0 ? n : 1;
}

int launch_expand(moonep_ctx *ctx, const moonep_comm_plan *plan, uint16_t *rows,
                  cudaStream_t st) {
  return launch_dedup(ctx, plan, rows, false, st);
}

int launch_fold(moonep_ctx *ctx, const moonep_comm_plan *plan, uint16_t *rows, cudaStream_t st) {
  return launch_dedup(ctx, plan, rows, true, st);
}

}  // namespace moonep
