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
// written K times.  The work is cut into whole padding rows followed by units
// of (token, 4 KB chunk of its row; 2 KB when the batch is too small to
// occupy every warp), strided over every warp of a persistent grid, so the
// tail is balanced whatever the token count (dispatch_units.cuh).
// HBM bytes per call: read R*S*H*2 + N*8 (dst, weights); write
// (N + P)*(H*2 + 4), P = padding rows.
//
// The rank-local form (one source rank's tokens, destination rows in R
// separately allocated rank windows, the padding of that rank's own window)
// is the same kernel with another row addressing: the per-GPU shape of the
// dispatch when each rank is a GPU and a remote window is a peer pointer.
#include "dispatch_units.cuh"

namespace moonep {
namespace {

constexpr int kThreads = 256;
using Args = DispatchArgs;

// kU: 16-byte vectors per lane per unit (8: 4 KB units; 4: 2 KB units for
// batches too small to give every warp of the grid a 4 KB unit).
template <int KT, int kU, class Rows>
__global__ void __launch_bounds__(kThreads) dispatch_kernel(Args a, Rows rows) {
  pdl_wait();
  pdl_launch_dependents();
  // small batches (a few units per warp): warps numbered across blocks
  // first, so the units of the last round spread over every SM; large
  // batches keep a block's warps on consecutive units (neighbouring chunks
  // of one token's rows written together)
  const int64_t wid = a.interleave ? (int64_t)(threadIdx.x >> 5) * gridDim.x + blockIdx.x
                                   : ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * kThreads) >> 5;
  dispatch_units<KT, kU>(a, rows, wid, nw);
}

template <int KT, int U = 8>
void *kernel_ptr() {
  return (void *)dispatch_kernel<KT, U, FlatRows>;
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

// 2 KB units when 4 KB units would leave warps of the grid idle (decode-
// sized batches: 16.7 us instead of 21.5 us at 1024 tokens of 8 KB; at
// large batches 4 KB units are 2 % faster)
int unit_vectors(int64_t ntok, int H8, int grid) {
  const int64_t warps = (int64_t)grid * (kThreads / 32);
  return ntok * ((H8 + 255) / 256) < warps ? 4 : 8;
}

}  // namespace

DispatchArgs dispatch_args(const moonep_ctx *ctx, const moonep_comm_plan *plan,
                           const uint16_t *hidden, const float *w_sk, int64_t ntok, int r0,
                           int seg_lo, int seg_hi, int U) {
  const moonep_config &c = ctx->cfg;
  PlanLayout lay = PlanLayout::make(c.R, c.E, c.B, ctx->NvS,
                                    (plan->flags & MOONEP_PLAN_DUP_RECORDS) != 0);
  DispatchArgs a;
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
  a.nchunk = (a.H8 + 32 * U - 1) / (32 * U);
  a.NvS = ctx->NvS;
  a.EB = ctx->EB;
  a.seg_lo = seg_lo;
  a.seg_hi = seg_hi;
  a.primaries_only = 0;
  const int64_t units = ntok * a.nchunk;
  a.interleave = units <= 4 * (int64_t)ctx->sms * ctx->blocks_dispatch * (kThreads / 32);
  return a;
}

// Resident blocks per SM of the 4 KB-unit kernel (small_units: the 2 KB-unit
// kernel, which needs fewer registers, so more of its blocks fit).
int occupancy_dispatch(int K, bool small_units) {
  int n = 0;
  void *f = small_units
                ? (K == 1 ? kernel_ptr<1, 4>() : K == 2 ? kernel_ptr<2, 4>()
                   : K == 4 ? kernel_ptr<4, 4>() : K == 8 ? kernel_ptr<8, 4>()
                            : kernel_ptr<0, 4>())
                : (K == 1 ? kernel_ptr<1>() : K == 2 ? kernel_ptr<2>() : K == 4 ? kernel_ptr<4>()
                   : K == 8 ? kernel_ptr<8>() : kernel_ptr<0>());
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, kThreads, 0) != cudaSuccess) n = 1;
  return n > 0 ? n : 1;
}

int launch_dispatch(moonep_ctx *ctx, const moonep_comm_plan *plan, const uint16_t *hidden,
                    const float *w_sk, uint16_t *out, float *w_out, cudaStream_t st,
                    bool primaries_only) {
  const moonep_config &c = ctx->cfg;
  const int64_t ntok = (int64_t)c.R * c.S;
  const int u = unit_vectors(ntok, c.H / 8, ctx->sms * ctx->blocks_dispatch);
  const int grid = ctx->sms * (u == 4 ? ctx->blocks_dispatch_small : ctx->blocks_dispatch);
  Args a = dispatch_args(ctx, plan, hidden, w_sk, ntok, 0, 0, c.R * ctx->EB, u);
  a.primaries_only = primaries_only ? 1 : 0;
  if (a.H8 == 0) return MOONEP_OK;
  FlatRows rows{reinterpret_cast<uint4 *>(out), w_out};
  return cuda_status(launch_k(a, rows, u, grid, st));
}

int launch_dispatch_rank(moonep_ctx *ctx, const moonep_comm_plan *plan, int rank,
                         const uint16_t *hidden_r, const float *w_r, uint16_t *const *windows,
                         float *const *w_windows, cudaStream_t st) {
  const moonep_config &c = ctx->cfg;
  const int u = unit_vectors(c.S, c.H / 8, ctx->sms * ctx->blocks_dispatch);
  const int grid = ctx->sms * (u == 4 ? ctx->blocks_dispatch_small : ctx->blocks_dispatch);
  Args a = dispatch_args(ctx, plan, hidden_r, w_r, c.S, rank, rank * ctx->EB,
                         (rank + 1) * ctx->EB, u);
  if (a.H8 == 0) return MOONEP_OK;
  WindowRows rows;
  for (int j = 0; j < kMaxRanks; j++) {
    rows.out[j] = j < c.R ? reinterpret_cast<uint4 *>(windows[j]) : nullptr;
    rows.w_out[j] = (w_windows && j < c.R) ? w_windows[j] : nullptr;
  }
  return cuda_status(launch_k(a, rows, u, grid, st));
}

}  // namespace moonep
