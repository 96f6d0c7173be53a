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
#include <mutex>

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
          if (k0 + kk >= KK) continue;  // the last batch of a K that KB does not divide
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
            if (k0 + kk >= KK || ((dupm >> (k0 + kk)) & 1u)) continue;
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

// ------------------------------------------------ staged combine (any K)
//
// For a K without a register-tuned batch shape: one warp per block; every
// unit's K row chunks (2 KB each) are copied into shared memory by the bulk
// copy engine (cp.async.bulk, completion counted on an mbarrier), two stages
// deep, so the next unit's K chunks are in flight while the warp sums the
// current one from shared memory.  Bytes in flight no longer depend on
// registers: K * 2 KB per warp and stage.  Same arithmetic as combine_kernel:
// fp32 adds in k order from the k = 0 row, one RNE rounding.

constexpr int kStageChunk = 2048;  // bytes of a row per unit

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t mbar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(mbar), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for a stage's copies; gives up after limit_ns (the copies of valid
// addresses always complete, so this only bounds a broken run).
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity, long long limit_ns) {
  if (mbar_try_wait(mbar, parity)) return true;
  long long t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  while (!mbar_try_wait(mbar, parity)) {
    long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > limit_ns) return false;
  }
  return true;
}

template <class Rows>
__global__ void __launch_bounds__(32) combine_staged_kernel(Args a, Rows rows) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ __align__(128) uint8_t stage_mem[];
  const int lane = threadIdx.x;
  const int K = a.K;
  const int stage_bytes = K * kStageChunk;
  const uint32_t buf0 = smem_u32(stage_mem);
  const uint32_t mbar0 = buf0 + 2 * stage_bytes;  // two mbarriers after the two stages
  if (lane == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbar0) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbar0 + 8) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  const int64_t row_bytes = (int64_t)a.H8 * 16;
  const int nchunk = a.nchunk;
  const int64_t units = a.ntok * nchunk;
  const int64_t nw = gridDim.x;  // one warp per block
  const int64_t u0 = blockIdx.x;
  const long long limit_ns = 1000000000LL;
  unsigned pending = 0;  // bit s: stage s has copies in flight

  // issue unit u's K chunk copies into stage s (d: this lane's dst entry)
  auto issue = [&](int64_t u, int st, int32_t d) {
    const int64_t t = u / nchunk;
    const int c = (int)(u - t * nchunk);
    const int64_t off = (int64_t)c * kStageChunk;
    const int bytes = (int)min((int64_t)kStageChunk, row_bytes - off);
    const uint32_t mbar = mbar0 + 8 * st;
    if (lane == 0)
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar),
                   "r"(bytes * K)
                   : "memory");
    __syncwarp();
    if (lane < K) {
      int64_t g = decode_row(d);
      if (g >= a.total_rows) {
        set_status(a.status, MOONEP_ERR_PLAN);
        g = 0;
      }
      const uint8_t *src = reinterpret_cast<const uint8_t *>(rows.row(g, a.H8, a.NvS)) + off;
      const uint32_t dst = buf0 + st * stage_bytes + lane * kStageChunk;
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
          ::"r"(dst), "l"(src), "r"(bytes), "r"(mbar)
          : "memory");
    }
    pending |= 1u << st;
  };

  int32_t d_cur = 0, d_nxt = 0;
  if (u0 < units && lane < K) d_cur = __ldg(a.dst + (u0 / nchunk) * K + lane);
  if (u0 < units) issue(u0, 0, d_cur);
  if (u0 + nw < units && lane < K) d_nxt = __ldg(a.dst + ((u0 + nw) / nchunk) * K + lane);
  uint32_t phase = 0;  // bit s: parity of stage s's next completion
  int s = 0;
  for (int64_t u = u0; u < units; u += nw) {
    const int64_t un = u + nw;
    if (un < units) issue(un, s ^ 1, d_nxt);
    int32_t d_far = 0;
    if (un + nw < units && lane < K) d_far = __ldg(a.dst + ((un + nw) / nchunk) * K + lane);
    if (!mbar_wait(mbar0 + 8 * s, (phase >> s) & 1u, limit_ns)) {
      set_status(a.status, MOONEP_ERR_TIMEOUT);
      break;
    }
    pending &= ~(1u << s);
    phase ^= 1u << s;
    const int64_t t = u / nchunk;
    const int c = (int)(u - t * nchunk);
    if (c == 0 && a.w_out && lane < K) {
      int64_t g = decode_row(d_cur);
      if (g >= a.total_rows) g = 0;
      a.w_out[t * K + lane] = __ldg(rows.weight(g, a.NvS));
    }
    // this lane's 16-byte vectors of the chunk: lane + 32 * i
    const uint8_t *stage = stage_mem + s * stage_bytes;
    const int vmax = (int)(min((int64_t)kStageChunk, row_bytes - (int64_t)c * kStageChunk) / 16);
    uint4 *op = a.out + t * a.H8 + (int64_t)c * (kStageChunk / 16);
#pragma unroll
    for (int i = 0; i < kStageChunk / 512; i++) {
      const int v = lane + 32 * i;
      if (v >= vmax) continue;
      float acc[8];
      set_bf16x8(acc, *reinterpret_cast<const uint4 *>(stage + v * 16));
      for (int k = 1; k < K; k++)
        add_bf16x8(acc, *reinterpret_cast<const uint4 *>(stage + k * kStageChunk + v * 16));
      st_global(op + v, pack_bf16x8(acc));
    }
    // the generic-proxy reads of this stage come before the copies that
    // refill it (issued at the next iteration)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    d_cur = d_nxt;
    d_nxt = d_far;
    s ^= 1;
  }
  // a wait that gave up leaves copies in flight into this block's shared
  // memory: wait for them (bounded) before the block exits
  for (int st = 0; st < 2; st++)
    if (pending & (1u << st)) mbar_wait(mbar0 + 8 * st, (phase >> st) & 1u, limit_ns);
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

// The staged kernel's shared memory for K rows: two stages of K 2 KB chunks
// and two mbarriers; blocks per SM (one warp each), cached per K.
size_t staged_smem(int K) { return (size_t)2 * K * kStageChunk + 16; }

template <class Rows>
int staged_blocks_per_sm(int K) {
  static int cache[33];  // K up to 32
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[K] == 0) {
    const size_t smem = staged_smem(K);
    int n = 0;
    // the limit is set once for the largest K (a per-K setting would lower
    // it below what an earlier K needs)
    if (cudaFuncSetAttribute(combine_staged_kernel<Rows>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)staged_smem(32)) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, combine_staged_kernel<Rows>, 32,
                                                      smem) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cache[K] = n > 0 ? n : -1;
  }
  return cache[K];
}

// K with a register-tuned batch shape (combine_kernel); every other K up to
// 32 takes the staged kernel (direct combine only).
bool staged_k(int K) {
  return !(K == 1 || K == 2 || K == 3 || K == 4 || K == 6 || K == 8 || K == 10);
}

template <class Rows>
cudaError_t launch_staged(const Args &a, const Rows &rows, int sms, cudaStream_t st) {
  const int per_sm = staged_blocks_per_sm<Rows>(a.K);
  if (per_sm <= 0) return cudaErrorInvalidConfiguration;
  Args b = a;
  b.nchunk = (int)((int64_t)a.H8 * 16 + kStageChunk - 1) / kStageChunk;
  return launch_pdl(combine_staged_kernel<Rows>, sms * per_sm, 32, staged_smem(a.K), st, false,
                    b, rows);
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
  if (!primaries_only && staged_k(c.K)) return cuda_status(launch_staged(a, rows, ctx->sms, st));
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
  if (staged_k(c.K)) return cuda_status(launch_staged(a, rows, ctx->sms, st));
  return cuda_status(launch_k(a, rows, false, ctx->sms * ctx->blocks_combine, st));
}

}  // namespace moonep
