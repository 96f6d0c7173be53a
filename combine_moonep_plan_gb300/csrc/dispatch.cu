// Fused-permute dispatch.
//
// "MoonEP Public API Visual Guide", Buffer.dispatch(...): decode route
// i = s*K + k, copy the token's hidden row to its destination row, scatter
// every routing weight, zero-fill padding, expand locally deduplicated routes.
// "MoonshotAI/MoonEP" README item 3: tokens are written straight to their
// expert-grouped positions (no permute in, no permute out).
//
// On one GPU every destination row is local HBM, so duplicates are expanded by
// writing the row to every |dst| directly: each source row is read once and
// written K times.  The work is cut into units of (token, 4 KB chunk of its
// row; 2 KB when the batch is too small to occupy every warp) followed by
// whole padding rows, strided over every warp of a persistent grid, so the
// tail is balanced whatever the token count.
// HBM bytes per call: read R*S*H*2 + N*8 (dst, weights); write
// (N + P)*(H*2 + 4), P = padding rows.
//
// The rank-local form (one source rank's tokens, destination rows in R
// separately allocated rank windows, the padding of that rank's own window)
// is the same kernel with another row addressing: the per-GPU shape of the
// dispatch when each rank is a GPU and a remote window is a peer pointer.
#include "copy_common.cuh"
#include "moonep_internal.cuh"

namespace moonep {
namespace {

constexpr int kThreads = 256;

struct Args {
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

// kU: 16-byte vectors per lane per unit (8: 4 KB units; 4: 2 KB units for
// batches too small to give every warp of the grid a 4 KB unit).
template <int KT, int kU, class Rows>
__global__ void __launch_bounds__(kThreads) dispatch_kernel(Args a, Rows rows) {
  constexpr int kChunk = 32 * kU;  // vectors per unit
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t wid = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * kThreads) >> 5;
  const int K = KT > 0 ? KT : a.K;
  const int64_t tok_units = a.ntok * a.nchunk;
  // padding rows of the launch's segments (all of them, or one rank's)
  const int64_t q0 = __ldg(a.pad_prefix + a.seg_lo);
  const int64_t P = __ldg(a.pad_prefix + a.seg_hi) - q0;
  const int64_t units = tok_units + P;  // then one unit per padding row
  const bool wts = rows.has_weights();
  // The next token unit's dst entries are loaded one unit ahead.
  int32_t d_next = 0;
  if (wid < tok_units && lane < K) d_next = __ldg(a.dst + (wid / a.nchunk) * K + lane);
  for (int64_t u = wid; u < units; u += nw) {
    if (u < tok_units) {
      const int64_t t = u / a.nchunk;
      const int c = (int)(u - t * a.nchunk);
      const int32_t d_cur = d_next;
      if (u + nw < tok_units && lane < K)
        d_next = __ldg(a.dst + ((u + nw) / a.nchunk) * K + lane);
      int64_t g = -1;
      if (lane < K) {
        const int64_t gg = decode_row(d_cur);
        if (gg < a.total_rows) {
          g = gg;
        } else {
          set_status(a.status, MOONEP_ERR_PLAN);
        }
        if (c == 0 && g >= 0 && wts) *rows.weight(g, a.NvS) = __ldg(a.w_sk + t * K + lane);
        if (a.primaries_only && d_cur < 0) g = -1;
      }
      const uint4 *src = a.hidden + t * a.H8;
      const int v0 = c * kChunk + lane;
      uint4 x[kU];
#pragma unroll
      for (int i = 0; i < kU; i++) {
        const int v = v0 + 32 * i;
        if (v < a.H8) x[i] = ld_stream(src + v);
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
      const int64_t q = q0 + (u - tok_units);
      int lo = a.seg_lo, hi = a.seg_hi;
      while (hi - lo > 1) {
        const int step = (hi - lo + 31) >> 5;
        const int idx = lo + lane * step;
        const bool le = idx < hi && __ldg(a.pad_prefix + idx) <= q;
        const unsigned m = __ballot_sync(0xffffffffu, le);
        lo += (31 - __clz(m)) * step;
        hi = min(hi, lo + step);
      }
      const int j = lo / a.EB;
      const int64_t row = __ldg(a.zfr + 2 * lo) + (q - __ldg(a.pad_prefix + lo));
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

template <int KT>
void *kernel_ptr() {
  return (void *)dispatch_kernel<KT, 8, FlatRows>;
}

template <int KT, class Rows>
cudaError_t launch(const Args &a, const Rows &rows, int u, int grid, cudaStream_t st) {
  return u == 4 ? launch_pdl(dispatch_kernel<KT, 4, Rows>, grid, kThreads, 0, st, false, a, rows)
                : launch_pdl(dispatch_kernel<KT, 8, Rows>, grid, kThreads, 0, st, false, a, rows);
}

template <class Rows>
cudaError_t launch_k(const Args &a, const Rows &rows, int u, int grid, cudaStream_t st) {
  switch (a.K) {
    case 1: return launch<1>(a, rows, u, grid, st);
    case 2: return launch<2>(a, rows, u, grid, st);
    case 4: return launch<4>(a, rows, u, grid, st);
    case 8: return launch<8>(a, rows, u, grid, st);
    default: return launch<0>(a, rows, u, grid, st);
  }
}

// Arguments shared by both forms; ntok tokens starting at source rank r0.
Args make_args(const moonep_ctx *ctx, const moonep_comm_plan *plan, const uint16_t *hidden,
               const float *w_sk, int64_t ntok, int r0, int seg_lo, int seg_hi) {
  const moonep_config &c = ctx->cfg;
  PlanLayout lay = PlanLayout::make(c.R, c.E, c.B, ctx->NvS,
                                    (plan->flags & MOONEP_PLAN_DUP_RECORDS) != 0);
  Args a;
  a.hidden = reinterpret_cast<const uint4 *>(hidden);
  a.w_sk = w_sk;
  a.dst = plan->dst + (int64_t)r0 * ctx->C;
  a.pad_prefix = plan->internal + lay.pad_prefix;
  a.zfr = plan->zero_fill_ranges;
  a.status = ctx->d_status;
  a.ntok = ntok;
  a.total_rows = (int64_t)c.R * ctx->NvS;
  a.K = c.K;
  a.H8 = c.H / 8;
  a.NvS = ctx->NvS;
  a.EB = ctx->EB;
  a.seg_lo = seg_lo;
  a.seg_hi = seg_hi;
  a.primaries_only = 0;
  return a;
}

// 2 KB units when 4 KB units would leave warps of the grid idle (decode-
// sized batches: 16.7 us instead of 21.5 us at 1024 tokens of 8 KB; at
// large batches 4 KB units are 2 % faster)
int unit_vectors(const Args &a, int grid) {
  const int64_t warps = (int64_t)grid * (kThreads / 32);
  return a.ntok * ((a.H8 + 255) / 256) < warps ? 4 : 8;
}

}  // namespace

int occupancy_dispatch(int K) {
  int n = 0;
  void *f = K == 1 ? kernel_ptr<1>() : K == 2 ? kernel_ptr<2>() : K == 4 ? kernel_ptr<4>()
          : K == 8 ? kernel_ptr<8>() : kernel_ptr<0>();
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, kThreads, 0) != cudaSuccess) n = 1;
  return n > 0 ? n : 1;
}

int launch_dispatch(moonep_ctx *ctx, const moonep_comm_plan *plan, const uint16_t *hidden,
                    const float *w_sk, uint16_t *out, float *w_out, cudaStream_t st,
                    bool primaries_only) {
  const moonep_config &c = ctx->cfg;
  Args a = make_args(ctx, plan, hidden, w_sk, (int64_t)c.R * c.S, 0, 0, c.R * ctx->EB);
  a.primaries_only = primaries_only ? 1 : 0;
  const int grid = ctx->sms * ctx->blocks_dispatch;
  const int u = unit_vectors(a, grid);
  a.nchunk = (a.H8 + 32 * u - 1) / (32 * u);
  if (a.H8 == 0) return MOONEP_OK;
  FlatRows rows{reinterpret_cast<uint4 *>(out), w_out};
  return cuda_status(launch_k(a, rows, u, grid, st));
}

int launch_dispatch_rank(moonep_ctx *ctx, const moonep_comm_plan *plan, int rank,
                         const uint16_t *hidden_r, const float *w_r, uint16_t *const *windows,
                         float *const *w_windows, cudaStream_t st) {
  const moonep_config &c = ctx->cfg;
  Args a = make_args(ctx, plan, hidden_r, w_r, c.S, rank, rank * ctx->EB, (rank + 1) * ctx->EB);
  const int grid = ctx->sms * ctx->blocks_dispatch;
  const int u = unit_vectors(a, grid);
  a.nchunk = (a.H8 + 32 * u - 1) / (32 * u);
  if (a.H8 == 0) return MOONEP_OK;
  WindowRows rows;
  for (int j = 0; j < kMaxRanks; j++) {
    rows.out[j] = j < c.R ? reinterpret_cast<uint4 *>(windows[j]) : nullptr;
    rows.w_out[j] = (w_windows && j < c.R) ? w_windows[j] : nullptr;
  }
  return cuda_status(launch_k(a, rows, u, grid, st));
}

}  // namespace moonep
