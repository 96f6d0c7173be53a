// Decode-path preparation: padding to the static token capacity.
//
// vLLM "fused_moe.prepare_finalize.moonep" page, MoonEPPrepareAndFinalize:
// prepare() picks a buffer whose capacity S fits the step's token count,
// pads the batch to S (zero hidden rows, expert 0, zero route weight) and
// maps invalid (negative) expert ids to expert 0 with zero weight, since the
// planner has no sentinel for them (_pad_to_capacity); tokens_per_expert is
// the count of the padded ids.
//
// Here the batch already sits in capacity-sized [R, S, ...] buffers (rank r's
// first num_tokens[r] rows valid), and the preparation runs in place: only
// padding rows and invalid routes are written, so a full batch costs one read
// of the ids and weights.  Blocks [0, R) each take one rank's S*K routes,
// eight per thread with their loads in flight together (sanitise, count per
// expert in shared memory, write tokens_per_expert); the remaining blocks
// zero the padding rows of the hidden tensor, one warp per 2 KB of a row
// with 16-byte stores.
#include "copy_common.cuh"
#include "moonep_internal.cuh"

namespace moonep {
namespace {

constexpr int kThreads = 512;
constexpr int kZeroVec = 128;  // 16-byte vectors per zeroing unit (2 KB of a row)
constexpr int kMaxRanks = 64;
constexpr int kBatch = 8;  // routes per thread whose loads are in flight together

struct PrepArgs {
  int32_t ntok[kMaxRanks];  // valid tokens of each rank
  int32_t pad_first[kMaxRanks + 1];  // first padding row (flattened) of each rank
  uint4 *hidden;            // [R*S, H8] or null
  int32_t *topk;            // [R*S*K]
  float *w;                 // [R*S*K] or null
  int32_t *tpe;             // [R*E] or null
  int R, S, K, E, H8;
};

__global__ void __launch_bounds__(kThreads) prepare_kernel(PrepArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ int32_t hist[];  // [E], route blocks only
  const int tid = threadIdx.x, lane = tid & 31;
  if ((int)blockIdx.x < a.R) {
    const int r = blockIdx.x;
    const int n = a.ntok[r];
    if (a.tpe)
      for (int e = tid; e < a.E; e += kThreads) hist[e] = 0;
    __syncthreads();
    const int64_t C = (int64_t)a.S * a.K;
    int32_t *ids = a.topk + r * C;
    float *ws = a.w ? a.w + r * C : nullptr;
    // few experts: the routes of a warp share counters, so they are added
    // once per distinct id (match), not once per route
    const bool few = a.E <= 32;
    for (int64_t i0 = 0; i0 < C; i0 += (int64_t)kThreads * kBatch) {
      int ev[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; b++) {
        const int64_t i = i0 + (int64_t)b * kThreads + tid;
        ev[b] = i < C ? ids[i] : 0;
      }
#pragma unroll
      for (int b = 0; b < kBatch; b++) {
        const int64_t i = i0 + (int64_t)b * kThreads + tid;
        int e = ev[b];
        if (i < C) {
          const int s = (int)(i / a.K);
          if (s >= n || e < 0) {
            if (e != 0) ids[i] = 0;
            if (ws) ws[i] = 0.0f;
            e = 0;
          }
        } else {
          e = -1;
        }
        if (a.tpe) {
          if (few) {
            const unsigned m = __match_any_sync(0xffffffffu, e);
            if (e >= 0 && e < a.E && lane == __ffs(m) - 1) atomicAdd(&hist[e], __popc(m));
          } else if (e >= 0 && e < a.E) {
            atomicAdd(&hist[e], 1);
          }
        }
      }
    }
    __syncthreads();
    if (a.tpe)
      for (int e = tid; e < a.E; e += kThreads) a.tpe[(int64_t)r * a.E + e] = hist[e];
    return;
  }
  // zero the padding rows: one warp per 2 KB of a row (flattened over the
  // ranks' padding rows)
  const int nch = (a.H8 + kZeroVec - 1) / kZeroVec;
  const int64_t units = (int64_t)a.pad_first[a.R] * nch;
  const int64_t warps = ((int64_t)(gridDim.x - a.R) * kThreads) >> 5;
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int64_t u = ((int64_t)(blockIdx.x - a.R) * kThreads + tid) >> 5; u < units; u += warps) {
    const int64_t q = u / nch;
    const int c = (int)(u - q * nch);
    int r = 0;
    while (r + 1 < a.R && a.pad_first[r + 1] <= q) r++;
    const int64_t s = a.ntok[r] + (q - a.pad_first[r]);
    uint4 *row = a.hidden + ((int64_t)r * a.S + s) * a.H8;
    const int v1 = min(a.H8, (c + 1) * kZeroVec);
    for (int v = c * kZeroVec + lane; v < v1; v += 32) st_global(row + v, z);
  }
}

}  // namespace

int launch_prepare(moonep_ctx *ctx, const int32_t *num_tokens, uint16_t *hidden,
                   int32_t *topk, float *w, int32_t *tpe, cudaStream_t st) {
  const moonep_config &c = ctx->cfg;
  PrepArgs a{};
  int64_t pad_rows = 0;
  for (int r = 0; r < c.R; r++) {
    const int n = num_tokens ? num_tokens[r] : c.S;
    a.ntok[r] = n;
    a.pad_first[r] = (int32_t)pad_rows;
    pad_rows += c.S - n;
  }
  a.pad_first[c.R] = (int32_t)pad_rows;
  a.hidden = reinterpret_cast<uint4 *>(hidden);
  a.topk = topk;
  a.w = w;
  a.tpe = tpe;
  a.R = c.R;
  a.S = c.S;
  a.K = c.K;
  a.E = c.E;
  a.H8 = c.H / 8;
  // one warp per 2 KB of a padding row, at most four blocks per SM
  const int64_t zunits = hidden ? pad_rows * ((a.H8 + kZeroVec - 1) / kZeroVec) : 0;
  int64_t zb = (zunits * 32 + kThreads - 1) / kThreads;
  const int64_t cap = (int64_t)ctx->sms * 4;
  if (zb > cap) zb = cap;
  if (!hidden) a.pad_first[c.R] = 0;
  const size_t smem = tpe ? (size_t)c.E * sizeof(int32_t) : 0;
  return cuda_status(
      launch_pdl(prepare_kernel, dim3((unsigned)(c.R + zb)), dim3(kThreads), smem, st, false, a));
}

}  // namespace moonep
