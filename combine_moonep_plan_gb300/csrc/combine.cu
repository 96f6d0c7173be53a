// Combine: the reverse data movement of dispatch.
//
// "MoonEP Public API Visual Guide", Buffer.combine(...): follow plan.dst, read
// the valid rows and perform the top-k reduction of every original token;
// routing weights are gathered back through the same positive/negative
// encoding.  The vLLM integration's finalize() fixes the reduction as an
// unweighted K-sum (weights are applied inside the expert compute).
//
// out[t, :] = bf16_rne( y[|dst(t,0)|,:] + y[|dst(t,1)|,:] + ... ) with the adds
// in fp32 in k order.  The page's version first folds duplicate rows into
// their primaries (to save link bytes between GPUs); on one GPU every row is
// read directly, so there is a single rounding at the end.
// Units of (token, chunk of 32*U 16-byte vectors) are strided over the warps
// of a persistent grid; each lane keeps K*U 16-byte loads in flight.  Every
// unit reads 2 KB contiguous from each of its K rows: with K = 8 and 1 KB per
// row the reads were scattered enough to hold HBM near 70 %; 2 KB per row (in
// two batches of four rows, 128-thread blocks) reaches the copy bandwidth.
// HBM bytes per call: read N*H*2 + N*4 (dst) [+ N*4 weights]; write
// R*S*H*2 [+ N*4].
//
// The rank-local form (one source rank's tokens, its K rows read from R
// separately allocated rank windows) is the same kernel with another row
// addressing: the per-GPU shape of the combine when each rank is a GPU and
// the owner pulls its rows from its peers.
#include "copy_common.cuh"
#include "moonep_internal.cuh"

namespace moonep {
namespace {


struct Args {
  const int32_t *dst;
  uint4 *out;
  float *w_out;
  int32_t *status;
  int64_t ntok;
  int64_t total_rows;
  int K, H8, nchunk, NvS;
  int interleave;  // number warps across blocks first (small batches)
};

// Source addressing of global row g = j*NvS + w: one [R*NvS, H] buffer, or
// rank j's [NvS, H] rows at row[j] (its [NvS] weights at w[j]).
struct FlatRows {
  static constexpr bool kPrimaries = true;  // also instantiated for the deduplicated combine
  const uint4 *y;
  const float *w_nvs;
  __device__ __forceinline__ const uint4 *row(int64_t g, int H8, int) const { return y + g * H8; }
  __device__ __forceinline__ const float *weight(int64_t g, int) const { return w_nvs + g; }
};

struct WindowRows {
  static constexpr bool kPrimaries = false;
  const uint4 *y[kMaxRanks];
  const float *w_nvs[kMaxRanks];
  __device__ __forceinline__ const uint4 *row(int64_t g, int H8, int NvS) const {
    const int j = (int)(g / NvS);
    return y[j] + (g - (int64_t)j * NvS) * H8;
  }
  __device__ __forceinline__ const float *weight(int64_t g, int NvS) const {
    const int j = (int)(g / NvS);
    return w_nvs[j] + (g - (int64_t)j * NvS);
  }
};

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4 &v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    acc[2 * i] += __uint_as_float(w[i] << 16);
    acc[2 * i + 1] += __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ void set_bf16x8(float (&acc)[8], const uint4 &v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    acc[2 * i] = __uint_as_float(w[i] << 16);
    acc[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&acc)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i]));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i + 1]));
    w[i] = lo | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// KT: compile-time K (0 = runtime K, up to 32).  U: vectors per lane per unit.
// BT: threads per block (128 for the specialised K: with 80-170 registers per
// thread, small blocks leave room for more resident warps).  KB: rows loaded
// per batch.  Per K, chosen by measurement: K = 8 reads 2 KB of each row per
// unit in two batches of four rows; K = 2 reads 4 KB of both rows at once
// (0.98 of the copy bandwidth on the Mixtral shape, 0.95 with 2 KB); K = 3
// reads 4 KB of one row at a time, K = 4 2 KB of two rows, K = 6 2 KB of three
// rows (1.00-1.04 of the copy bandwidth each, where a runtime-K kernel gave
// 0.66-0.78), K = 10 4 KB of one row at a time (0.85); any other K takes the
// runtime-K kernel, four rows per batch.  PRIM: sum the primary
// routes only (dst >= 0; the duplicates were folded into them), a separate
// instantiation so that the direct kernel carries none of its code.
template <int KT, int U, int BT, int KB, bool PRIM, class Rows>
__global__ void __launch_bounds__(BT) combine_kernel(Args a, Rows rows) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  // small batches (a few units per warp): warps numbered across blocks
  // first, so the units of the last round spread over every SM
  const int64_t wid = a.interleave ? (int64_t)(threadIdx.x >> 5) * gridDim.x + blockIdx.x
                                   : ((int64_t)blockIdx.x * BT + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * BT) >> 5;
  const int K = KT > 0 ? KT : a.K;
  const int64_t units = a.ntok * a.nchunk;
  // The next unit's dst entries are loaded one unit ahead, so their latency
  // overlaps the current unit's row loads.
  int32_t d_next = 0;
  if (wid < units && lane < K) d_next = __ldg(a.dst + (wid / a.nchunk) * K + lane);
  for (int64_t u = wid; u < units; u += nw) {
    const int64_t t = u / a.nchunk;
    const int c = (int)(u - t * a.nchunk);
    const int32_t d_cur = d_next;
    if (u + nw < units && lane < K) d_next = __ldg(a.dst + ((u + nw) / a.nchunk) * K + lane);
    int64_t g = 0;
    // duplicate routes that the prologue folded into their primaries (the
    // same for every lane: route k's sign, broadcast)
    const unsigned dupm = PRIM ? __ballot_sync(0xffffffffu, lane < K && d_cur < 0) : 0u;
    if (lane < K) {
      g = decode_row(d_cur);
      if (g >= a.total_rows) {
        set_status(a.status, MOONEP_ERR_PLAN);
        g = 0;
      }
      if (c == 0 && a.w_out) a.w_out[t * K + lane] = __ldg(rows.weight(g, a.NvS));
    }
    const int v0 = c * 32 * U + lane;
    float acc[U][8];
    if (KT > 0) {
      constexpr int KK = KT > 0 ? KT : 1;
#pragma unroll
      for (int k0 = 0; k0 < KK; k0 += KB) {
        uint4 x[KB][U];
#pragma unroll
        for (int kk = 0; kk < KB; kk++) {
          const uint4 *row = rows.row(__shfl_sync(0xffffffffu, g, k0 + kk), a.H8, a.NvS);
          const bool skip = (dupm >> (k0 + kk)) & 1u;
#pragma unroll
          for (int i = 0; i < U; i++) {
            const int v = v0 + 32 * i;
            if (v < a.H8 && !skip) x[kk][i] = ld_stream(row + v);
          }
        }
#pragma unroll
        for (int i = 0; i < U; i++) {
#pragma unroll
          for (int kk = 0; kk < KB; kk++) {
            if ((dupm >> (k0 + kk)) & 1u) continue;
            if (k0 + kk == 0) set_bf16x8(acc[i], x[kk][i]);
            else add_bf16x8(acc[i], x[kk][i]);
          }
        }
      }
    } else {
      // runtime K: batches of KB rows, the last one partial
      for (int k0 = 0; k0 < K; k0 += KB) {
        uint4 x[KB][U];
#pragma unroll
        for (int kk = 0; kk < KB; kk++) {
          const int k = k0 + kk;
          const uint4 *row = rows.row(__shfl_sync(0xffffffffu, g, k & 31), a.H8, a.NvS);
          const bool use = k < K && !((dupm >> (k & 31)) & 1u);
#pragma unroll
          for (int i = 0; i < U; i++) {
            const int v = v0 + 32 * i;
            if (use && v < a.H8) x[kk][i] = ld_stream(row + v);
          }
        }
#pragma unroll
        for (int i = 0; i < U; i++) {
#pragma unroll
          for (int kk = 0; kk < KB; kk++) {
            const int k = k0 + kk;
            if (k >= K || ((dupm >> (k & 31)) & 1u)) continue;
            if (k == 0) set_bf16x8(acc[i], x[kk][i]);
            else add_bf16x8(acc[i], x[kk][i]);
          }
        }
      }
    }
    uint4 *op = a.out + t * a.H8;
#pragma unroll
    for (int i = 0; i < U; i++) {
      const int v = v0 + 32 * i;
      if (v < a.H8) st_global(op + v, pack_bf16x8(acc[i]));
    }
  }
}

template <int KT, int U, int BT, int KB, class Rows>
cudaError_t launch(const Args &a, const Rows &rows, bool prim, int grid, cudaStream_t st) {
  if constexpr (Rows::kPrimaries) {
    if (prim)
      return launch_pdl(combine_kernel<KT, U, BT, KB, true, Rows>, grid, BT, 0, st, false, a,
                        rows);
  }
  return launch_pdl(combine_kernel<KT, U, BT, KB, false, Rows>, grid, BT, 0, st, false, a, rows);
}

// Batch shape per K (vectors per lane, threads per block, rows per batch),
// the instantiations occupancy_combine measures.
template <class Rows>
cudaError_t launch_k(const Args &a, const Rows &rows, bool prim, int grid, cudaStream_t st) {
  switch (a.K) {
    case 1: return launch<1, 4, 256, 1>(a, rows, prim, grid, st);
    case 2: return launch<2, 8, 128, 2>(a, rows, prim, grid, st);
    case 3: return launch<3, 8, 128, 1>(a, rows, prim, grid, st);
    case 4: return launch<4, 4, 128, 2>(a, rows, prim, grid, st);
    case 6: return launch<6, 4, 128, 3>(a, rows, prim, grid, st);
    case 8: return launch<8, 4, 128, 4>(a, rows, prim, grid, st);
    case 10: return launch<10, 8, 128, 1>(a, rows, prim, grid, st);
    default: return launch<0, 4, 128, 4>(a, rows, prim, grid, st);
  }
}

int unit_vectors(int K) { return (K == 2 || K == 3 || K == 10) ? 8 : 4; }

Args make_args(const moonep_ctx *ctx, const moonep_comm_plan *plan, int64_t ntok, int r0,
               uint16_t *out, float *w_out) {
  const moonep_config &c = ctx->cfg;
  Args a;
  a.dst = plan->dst + (int64_t)r0 * ctx->C;
  a.out = reinterpret_cast<uint4 *>(out);
  a.w_out = w_out;
  a.status = ctx->d_status;
  a.ntok = ntok;
  a.total_rows = (int64_t)c.R * ctx->NvS;
  a.K = c.K;
  a.H8 = c.H / 8;
  const int U = unit_vectors(c.K);
  a.nchunk = (a.H8 + 32 * U - 1) / (32 * U);
  a.NvS = ctx->NvS;
  const int bt = c.K == 1 ? 256 : 128;
  a.interleave = ntok * a.nchunk <= 4 * (int64_t)ctx->sms * ctx->blocks_combine * (bt / 32);
  return a;
}

}  // namespace

int occupancy_combine(int K) {
  int n = 0;
  void *f = K == 1 ? (void *)combine_kernel<1, 4, 256, 1, false, FlatRows>
          : K == 2 ? (void *)combine_kernel<2, 8, 128, 2, false, FlatRows>
          : K == 3 ? (void *)combine_kernel<3, 8, 128, 1, false, FlatRows>
          : K == 4 ? (void *)combine_kernel<4, 4, 128, 2, false, FlatRows>
          : K == 6 ? (void *)combine_kernel<6, 4, 128, 3, false, FlatRows>
          : K == 8 ? (void *)combine_kernel<8, 4, 128, 4, false, FlatRows>
          : K == 10 ? (void *)combine_kernel<10, 8, 128, 1, false, FlatRows>
                    : (void *)combine_kernel<0, 4, 128, 4, false, FlatRows>;
  const int bt = K == 1 ? 256 : 128;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, bt, 0) != cudaSuccess) n = 1;
  return n > 0 ? n : 1;
}

int launch_combine(moonep_ctx *ctx, const moonep_comm_plan *plan, const uint16_t *y,
                   const float *w_nvs, uint16_t *out, float *w_out, cudaStream_t st,
                   bool primaries_only) {
  const moonep_config &c = ctx->cfg;
  Args a = make_args(ctx, plan, (int64_t)c.R * c.S, 0, out, w_out);
  if (a.ntok == 0 || a.H8 == 0) return MOONEP_OK;
  FlatRows rows{reinterpret_cast<const uint4 *>(y), w_nvs};
  return cuda_status(launch_k(a, rows, primaries_only, ctx->sms * ctx->blocks_combine, st));
}

int launch_combine_rank(moonep_ctx *ctx, const moonep_comm_plan *plan, int rank,
                        const uint16_t *const *y_windows, const float *const *w_windows,
                        uint16_t *out_r, float *w_out_r, cudaStream_t st) {
  const moonep_config &c = ctx->cfg;
  Args a = make_args(ctx, plan, c.S, rank, out_r, w_out_r);
  if (a.ntok == 0 || a.H8 == 0) return MOONEP_OK;
  WindowRows rows;
  for (int j = 0; j < kMaxRanks; j++) {
    rows.y[j] = j < c.R ? reinterpret_cast<const uint4 *>(y_windows[j]) : nullptr;
    rows.w_nvs[j] = (w_windows && j < c.R) ? w_windows[j] : nullptr;
  }
  return cuda_status(launch_k(a, rows, false, ctx->sms * ctx->blocks_combine, st));
}

}  // namespace moonep
