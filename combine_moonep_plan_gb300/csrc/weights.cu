// Redundant-expert weight prefetch and gradient reduce.
//
// "MoonEP Public API Visual Guide", Buffer.prefetch_weight(...): each used slot
// of plan.experts_to_copy receives its source expert's [H, H'] weight; -1
// slots are skipped.  Buffer.reduce_grad(...): every owned expert seeds an
// accumulator with its own fp32 gradient, adds the matching slot gradients of
// every rank, writes the sum back, and the consumed slots are cleared.
// "MoonshotAI/MoonEP" README, "Weight buffer": the [E+B, H, H'] tensors and the
// [R, B, H, H'] reduce buffer.
//
// One device holds every rank's slots: the weight tensor is [E + R*B, HHp]
// (rank j's slot b is row E + j*B + b) and the slot gradients are [R*B, HHp].
// The planner leaves compact lists on the device (used slots; experts with
// copies and their slots in (rank, slot) order), so both kernels walk only the
// rows that move.  Work units are chunks of an expert's row, strided over a
// persistent grid: prefetch reads the chunk once and writes it to every slot
// holding the expert; reduce reads each slot element once, adds it, and
// zeroes it in the same thread, so no barrier separates the reduce and the
// clear.
// HBM bytes (D experts with copies, U used slots): prefetch (D + U)*row_bytes
// per tensor (row_bytes = H*H'*2 for bf16, H*H'/2 for packed MXFP4, H*H'/32
// for its block scales); reduce (2*D + 2*U)*HHp*4.
#include "copy_common.cuh"
#include "moonep_internal.cuh"

namespace moonep {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxProj = 4;
constexpr int kMaxTensors = 8;   // prefetch: e.g. gate/up/down and their block scales
constexpr int kChunkVec = 2048;  // 16-byte vectors per unit (32 KB)
constexpr int kPU = 4;           // vectors per thread per step (prefetch)

// Prefetch of n tensors whose expert rows have row_bytes[t] bytes each
// (bf16 weights, packed MXFP4 bytes, block scales, ...).  A tensor whose
// rows are 16-byte multiples on a 16-byte aligned base moves 16-byte vectors;
// any other moves single bytes.  Units walk the experts that have copies (the
// reduce list: expert, then its slots in (rank, slot) order): a chunk of the
// expert's row is read once and stored to every slot holding it.
struct PrefetchArgs {
  uint8_t *T[kMaxTensors];
  int64_t row_bytes[kMaxTensors];
  int64_t nchunk[kMaxTensors];  // 32 KB units per row
  unsigned vec_mask;            // bit t: tensor t moves 16-byte vectors
  const int32_t *meta, *red_expert, *red_first, *red_slot;
  int n, E;
};

constexpr int kMaxCopies = 64;  // slots holding one expert: at most one per rank

__global__ void __launch_bounds__(kThreads) prefetch_kernel(PrefetchArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int s_dst[kMaxCopies];  // slot rows of the staged expert
  __shared__ int s_n;
  const int64_t D = a.meta[kMetaD];
  int64_t units = 0;
  for (int t = 0; t < a.n; t++) units += D * a.nchunk[t];
  int64_t staged = -1;  // expert index of the staged slot list
  for (int64_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
    // unit -> (tensor, expert with copies, chunk); tensors in order
    int t = 0;
    int64_t rem = unit;
    while (t + 1 < a.n && rem >= D * a.nchunk[t]) {
      rem -= D * a.nchunk[t];
      t++;
    }
    const int64_t di = rem / a.nchunk[t];
    const int64_t c = rem - di * a.nchunk[t];
    if (di != staged) {
      __syncthreads();  // the previous list is no longer read
      const int f0 = a.red_first[di], f1 = a.red_first[di + 1];
      if (threadIdx.x == 0) s_n = min(f1 - f0, kMaxCopies);
      for (int q = threadIdx.x; q < f1 - f0 && q < kMaxCopies; q += kThreads)
        s_dst[q] = a.E + a.red_slot[f0 + q];
      __syncthreads();
      staged = di;
    }
    const int n = s_n;
    const int64_t rb = a.row_bytes[t];
    uint8_t *base = a.T[t];
    const uint8_t *src = base + (int64_t)a.red_expert[di] * rb;
    if ((a.vec_mask >> t) & 1u) {
      const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
      const int64_t v_begin = c * kChunkVec;
      const int64_t v_end = min(v_begin + kChunkVec, rb / 16);
      for (int64_t v = v_begin + threadIdx.x; v < v_end; v += kThreads * kPU) {
        uint4 x[kPU];
#pragma unroll
        for (int i = 0; i < kPU; i++)
          if (v + i * kThreads < v_end) x[i] = ld_stream(s4 + v + i * kThreads);
        for (int q = 0; q < n; q++) {
          uint4 *d4 = reinterpret_cast<uint4 *>(base + (int64_t)s_dst[q] * rb);
#pragma unroll
          for (int i = 0; i < kPU; i++)
            if (v + i * kThreads < v_end) st_global(d4 + v + i * kThreads, x[i]);
        }
      }
    } else {
      const int64_t b_begin = c * kChunkVec * 16;
      const int64_t b_end = min(b_begin + (int64_t)kChunkVec * 16, rb);
      for (int64_t v = b_begin + threadIdx.x; v < b_end; v += kThreads) {
        const uint8_t x = src[v];
        for (int q = 0; q < n; q++) base[(int64_t)s_dst[q] * rb + v] = x;
      }
    }
  }
}

struct ReduceArgs {
  float4 *Gh[kMaxProj];
  float4 *Gs[kMaxProj];
  const int32_t *meta, *red_expert, *red_first, *red_slot;
  int n_proj;
  int64_t vec_per_row;  // HHp / 4
  int64_t nchunk;
};

constexpr int kRedChunk = 2048;  // float4 per unit (32 KB of the home row)
constexpr int kMaxSlotsPerExpert = 256;

// Columns [v_begin, v_end) of one expert: acc = home, then each slot in list
// order (acc = acc + slot), slot elements zeroed, home = acc.  A thread holds
// RV columns and loads the home element and up to NS slot elements of each
// together (RV * (1 + NS) loads in flight), so one round trip to memory
// covers several rows of the column.
template <int RV, int NS>
__device__ __forceinline__ void reduce_columns(float4 *home, float4 *const *slot, int n,
                                               int64_t v_begin, int64_t v_end) {
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t v = v_begin + threadIdx.x; v < v_end; v += RV * kThreads) {
    bool ok[RV];
    float4 acc[RV];
#pragma unroll
    for (int i = 0; i < RV; i++) {
      ok[i] = v + i * kThreads < v_end;
      if (ok[i]) acc[i] = ld_once_f4(home + v + i * kThreads);
    }
    for (int f = 0; f < n; f += NS) {
      float4 x[NS][RV];
#pragma unroll
      for (int q = 0; q < NS; q++) {
        if (f + q < n) {
#pragma unroll
          for (int i = 0; i < RV; i++)
            if (ok[i]) x[q][i] = ld_once_f4(slot[f + q] + v + i * kThreads);
        }
      }
#pragma unroll
      for (int q = 0; q < NS; q++) {
        if (f + q < n) {
#pragma unroll
          for (int i = 0; i < RV; i++) {
            if (!ok[i]) continue;
            acc[i].x = acc[i].x + x[q][i].x;
            acc[i].y = acc[i].y + x[q][i].y;
            acc[i].z = acc[i].z + x[q][i].z;
            acc[i].w = acc[i].w + x[q][i].w;
            st_global_f4(slot[f + q] + v + i * kThreads, zero);
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < RV; i++)
      if (ok[i]) st_global_f4(home + v + i * kThreads, acc[i]);
  }
}

// One unit = one 32 KB chunk of one expert's row (and of its slot rows).  A
// thread takes four columns and two slot rows at a time: 8 loads in flight
// for an expert with one copy, 12 for more; within 64 registers, so four
// blocks fit on an SM.  The slot list of the unit's expert is staged in
// shared memory once per expert.
__global__ void __launch_bounds__(kThreads, 4) reduce_kernel(ReduceArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float4 *s_slot[kMaxSlotsPerExpert];
  __shared__ float4 *s_home;
  __shared__ int s_n;
  const int64_t D = a.meta[kMetaD];
  const int64_t per_proj = D * a.nchunk;
  const int64_t units = per_proj * a.n_proj;
  int64_t staged = -1;  // p * D + di of the staged slot list
  for (int64_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
    const int p = (int)(unit / per_proj);
    const int64_t rem = unit - p * per_proj;
    const int64_t di = rem / a.nchunk;
    const int64_t c = rem - di * a.nchunk;
    if (p * D + di != staged) {
      __syncthreads();  // the previous expert's list is no longer read
      const int f0 = a.red_first[di], f1 = a.red_first[di + 1];
      if (threadIdx.x == 0) {
        s_n = min(f1 - f0, kMaxSlotsPerExpert);
        s_home = a.Gh[p] + (int64_t)a.red_expert[di] * a.vec_per_row;
      }
      for (int q = threadIdx.x; q < f1 - f0 && q < kMaxSlotsPerExpert; q += kThreads)
        s_slot[q] = a.Gs[p] + (int64_t)a.red_slot[f0 + q] * a.vec_per_row;
      __syncthreads();
      staged = p * D + di;
    }
    const int n = s_n;
    const int64_t v_begin = c * kRedChunk;
    const int64_t v_end = min(v_begin + kRedChunk, a.vec_per_row);
    reduce_columns<4, 2>(s_home, s_slot, n, v_begin, v_end);
  }
}

}  // namespace

int occupancy_copy() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, prefetch_kernel, kThreads, 0) !=
      cudaSuccess)
    n = 1;
  return n > 0 ? n : 1;
}

int occupancy_reduce() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, reduce_kernel, kThreads, 0) !=
      cudaSuccess)
    n = 1;
  return n > 0 ? n : 1;
}

int launch_prefetch(moonep_ctx *ctx, const moonep_comm_plan *plan, int n, void *const *T,
                    const int64_t *row_bytes, cudaStream_t st) {
  const moonep_config &c = ctx->cfg;
  if (n < 1 || n > kMaxTensors) return MOONEP_ERR_INVALID_ARG;
  PlanLayout lay = PlanLayout::make(c.R, c.E, c.B, ctx->NvS,
                                    (plan->flags & MOONEP_PLAN_DUP_RECORDS) != 0);
  PrefetchArgs a{};
  bool any = false;
  for (int t = 0; t < n; t++) {
    const int64_t rb = row_bytes[t];
    a.T[t] = static_cast<uint8_t *>(T[t]);
    a.row_bytes[t] = rb;
    if (rb % 16 == 0 && aligned16(T[t])) a.vec_mask |= 1u << t;
    a.nchunk[t] = (rb + (int64_t)kChunkVec * 16 - 1) / ((int64_t)kChunkVec * 16);
    any = any || rb > 0;
  }
  a.meta = plan->internal;
  a.red_expert = plan->internal + lay.red_expert;
  a.red_first = plan->internal + lay.red_first;
  a.red_slot = plan->internal + lay.red_slot;
  a.n = n;
  a.E = c.E;
  if (!any || c.B == 0) return MOONEP_OK;
  const int grid = ctx->sms * ctx->blocks_copy;
  return cuda_status(launch_pdl(prefetch_kernel, grid, kThreads, 0, st, false, a));
}

int launch_reduce(moonep_ctx *ctx, const moonep_comm_plan *plan, int n_proj, float *const *Gh,
                  float *const *Gs, int64_t HHp, cudaStream_t st) {
  const moonep_config &c = ctx->cfg;
  if (n_proj < 1 || n_proj > kMaxProj) return MOONEP_ERR_INVALID_ARG;
  PlanLayout lay = PlanLayout::make(c.R, c.E, c.B, ctx->NvS,
                                    (plan->flags & MOONEP_PLAN_DUP_RECORDS) != 0);
  ReduceArgs a{};
  for (int p = 0; p < n_proj; p++) {
    a.Gh[p] = reinterpret_cast<float4 *>(Gh[p]);
    a.Gs[p] = reinterpret_cast<float4 *>(Gs[p]);
  }
  a.meta = plan->internal;
  a.red_expert = plan->internal + lay.red_expert;
  a.red_first = plan->internal + lay.red_first;
  a.red_slot = plan->internal + lay.red_slot;
  a.n_proj = n_proj;
  a.vec_per_row = HHp / 4;
  a.nchunk = (a.vec_per_row + kRedChunk - 1) / kRedChunk;
  if (a.vec_per_row == 0 || c.B == 0) return MOONEP_OK;
  return cuda_status(
      launch_pdl(reduce_kernel, ctx->sms * ctx->blocks_reduce, kThreads, 0, st, false, a));
}

}  // namespace moonep
