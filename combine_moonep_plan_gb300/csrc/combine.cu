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
  int64_t nw;      // staged kernel: blocks (one warp each) that take units
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
// 0.66-0.78).  The direct combine of any other K takes the staged kernel
// below; the primaries-only sum takes K = 10 as 4 KB of one row at a time and
// the rest through the runtime-K kernel, four rows per batch.  PRIM: sum the primary
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
// unit's K row chunks (kChunk bytes each) are copied into shared memory by
// the bulk copy engine (cp.async.bulk, completion counted on an mbarrier),
// kStages deep, so the next units' K chunks are in flight while the warp sums
// the current one from shared memory.  Bytes in flight no longer depend on
// registers: (kStages - 1) * K * kChunk per warp.  Same arithmetic as
// combine_kernel: fp32 adds in k order from the k = 0 row, one RNE rounding.

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

template <int kChunk, int kStages, class Rows>
__global__ void __launch_bounds__(32) combine_staged_kernel(Args a, Rows rows) {
  static_assert(kChunk % 512 == 0 && kStages >= 2 && kStages <= 8, "stage shape");
  pdl_wait();
  pdl_launch_dependents();
  if (blockIdx.x >= a.nw) return;
  extern __shared__ __align__(128) uint8_t stage_mem[];
  const int lane = threadIdx.x;
  const int K = a.K;
  const int stage_bytes = K * kChunk;
  const uint32_t buf0 = smem_u32(stage_mem);
  const uint32_t mbar0 = buf0 + kStages * stage_bytes;  // one mbarrier per stage after them
  if (lane == 0) {
    for (int q = 0; q < kStages; q++)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbar0 + 8 * q) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  const int64_t row_bytes = (int64_t)a.H8 * 16;
  const int nchunk = a.nchunk;
  const int64_t units = a.ntok * nchunk;
  const int64_t nw = a.nw;  // one warp per block
  const int64_t u0 = blockIdx.x;
  const long long limit_ns = 1000000000LL;
  unsigned pending = 0;  // bit q: stage q has copies in flight

  // this lane's dst entry of unit u (route k = lane)
  auto dst_of = [&](int64_t u) -> int32_t {
    return (u < units && lane < K) ? __ldg(a.dst + (u / nchunk) * K + lane) : 0;
  };
  // issue unit u's K chunk copies into stage q (d: this lane's dst entry)
  auto issue = [&](int64_t u, int q, int32_t d) {
    const int64_t t = u / nchunk;
    const int c = (int)(u - t * nchunk);
    const int64_t off = (int64_t)c * kChunk;
    const int bytes = (int)min((int64_t)kChunk, row_bytes - off);
    const uint32_t mbar = mbar0 + 8 * q;
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
      const uint32_t dst = buf0 + q * stage_bytes + lane * kChunk;
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
          ::"r"(dst), "l"(src), "r"(bytes), "r"(mbar)
          : "memory");
    }
    pending |= 1u << q;
  };

  // kStages - 1 units in flight ahead of the one being summed; the dst
  // entries of the next unit to issue are loaded one iteration ahead
  for (int p = 0; p < kStages - 1; p++)
    if (u0 + p * nw < units) issue(u0 + p * nw, p, dst_of(u0 + p * nw));
  int32_t d_pre = dst_of(u0 + (int64_t)(kStages - 1) * nw);
  uint32_t phase = 0;  // bit q: parity of stage q's next completion
  int q = 0;
  for (int64_t u = u0; u < units; u += nw) {
    const int64_t ua = u + (int64_t)(kStages - 1) * nw;
    if (ua < units) issue(ua, q == 0 ? kStages - 1 : q - 1, d_pre);
    d_pre = dst_of(ua + nw);
    if (!mbar_wait(mbar0 + 8 * q, (phase >> q) & 1u, limit_ns)) {
      set_status(a.status, MOONEP_ERR_TIMEOUT);
      break;
    }
    pending &= ~(1u << q);
    phase ^= 1u << q;
    const int64_t t = u / nchunk;
    const int c = (int)(u - t * nchunk);
    if (c == 0 && a.w_out && lane < K) {
      int64_t g = decode_row(__ldg(a.dst + t * K + lane));
      if (g >= a.total_rows) g = 0;
      a.w_out[t * K + lane] = __ldg(rows.weight(g, a.NvS));
    }
    // this lane's 16-byte vectors of the chunk: lane + 32 * i
    const uint8_t *stage = stage_mem + q * stage_bytes;
    const int vmax = (int)(min((int64_t)kChunk, row_bytes - (int64_t)c * kChunk) / 16);
    uint4 *op = a.out + t * a.H8 + (int64_t)c * (kChunk / 16);
#pragma unroll
    for (int i = 0; i < kChunk / 512; i++) {
      const int v = lane + 32 * i;
      if (v >= vmax) continue;
      float acc[8];
      set_bf16x8(acc, *reinterpret_cast<const uint4 *>(stage + v * 16));
      for (int k = 1; k < K; k++)
        add_bf16x8(acc, *reinterpret_cast<const uint4 *>(stage + k * kChunk + v * 16));
      st_global(op + v, pack_bf16x8(acc));
    }
    // the generic-proxy reads of this stage come before the copies that
    // refill it (issued at the next iteration)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    q = q + 1 == kStages ? 0 : q + 1;
  }
  // a wait that gave up leaves copies in flight into this block's shared
  // memory: wait for them (bounded) before the block exits
  for (int p = 0; p < kStages; p++)
    if (pending & (1u << p)) mbar_wait(mbar0 + 8 * p, (phase >> p) & 1u, limit_ns);
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

// Stage shape of the staged kernel per K (chunk bytes, stages).
struct StageShape {
  int chunk, stages;
};

// Measured at H = 7168 over K = 5..32 and chunks of 1-2 KB with 2-4 stages:
// two stages of 2 KB chunks reach 0.99-1.04 of the copy bandwidth up to
// K = 13; from K = 14 on, 2 KB chunks leave three blocks or fewer per SM
// (0.67-0.90), and 1 KB chunks, twice the blocks, reach 0.96-1.01 (0.85 at
// K = 32).  More stages gained nothing (0.85-0.98).
StageShape stage_shape(int K) { return K <= 13 ? StageShape{2048, 2} : StageShape{1024, 2}; }

size_t staged_smem(int K, StageShape sh) { return (size_t)sh.stages * K * sh.chunk + 8 * sh.stages; }

template <int kChunk, int kStages, class Rows>
cudaError_t launch_staged_shape(const Args &a, const Rows &rows, int sms, cudaStream_t st) {
  auto f = combine_staged_kernel<kChunk, kStages, Rows>;
  const size_t smem = staged_smem(a.K, {kChunk, kStages});
  // blocks per SM (one warp each), cached per K; the limit is set once for
  // the largest K (a per-K setting would lower it below what an earlier K
  // needs)
  static int cache[33];
  static std::mutex mu;
  int per_sm;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (cache[a.K] == 0) {
      int n = 0;
      if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)staged_smem(32, {kChunk, kStages})) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, 32, smem) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
      }
      cache[a.K] = n > 0 ? n : -1;
    }
    per_sm = cache[a.K];
  }
  if (per_sm <= 0) return cudaErrorInvalidConfiguration;
  Args b = a;
  b.nchunk = (int)(((int64_t)a.H8 * 16 + kChunk - 1) / kChunk);
  // Units are strided over the blocks; when their count is a multiple of the
  // chunks per row, each block would take the same chunk of every row it
  // visits, which measured 0.69-0.77 of the copy bandwidth against 0.96-1.05
  // otherwise (top-5, 7, 10, 14 and 15 at H = 7168): one block then sits out.
  b.nw = (int64_t)sms * per_sm;
  if (b.nchunk > 1 && b.nw % b.nchunk == 0) b.nw -= 1;
  return launch_pdl(f, sms * per_sm, 32, smem, st, false, b, rows);
}

// K with a register-tuned batch shape (combine_kernel); every other K up to
// 32 takes the staged kernel (direct combine only).
bool staged_k(int K) { return !(K == 1 || K == 2 || K == 3 || K == 4 || K == 6 || K == 8); }

template <class Rows>
cudaError_t launch_staged(const Args &a, const Rows &rows, int sms, cudaStream_t st) {
  const StageShape sh = stage_shape(a.K);
  if (sh.chunk == 1024) return launch_staged_shape<1024, 2>(a, rows, sms, st);
  return launch_staged_shape<2048, 2>(a, rows, sms, st);
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

// Small batches with K = 8 (a few units per warp, the decode step): units of
// 1 KB of each row, in batches of two rows.  The kernel then needs 72
// registers instead of 168, so seven blocks fit per SM instead of three; at
// the decode shape the combine inside the step drops from 16.4 to 12.5 us and
// the plan->dispatch->combine chain from 35.5 to 33.7 us (1 KB units in
// batches of four rows, five blocks per SM: 14.3 and 34.7 us).
constexpr int kSmallU = 2;

template <class Rows>
cudaError_t launch_small_k8(Args a, const Rows &rows, bool prim, int grid, cudaStream_t st) {
  a.nchunk = (a.H8 + 32 * kSmallU - 1) / (32 * kSmallU);
  return launch<8, kSmallU, 128, 2>(a, rows, prim, grid, st);
}

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
  a.nw = 0;
  return a;
}

}  // namespace

int occupancy_combine_small(int K) {
  if (K != 8) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &n, combine_kernel<8, kSmallU, 128, 2, false, FlatRows>, 128, 0) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

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
  if (c.K == 8 && a.interleave && ctx->blocks_combine_small > 0)
    return cuda_status(
        launch_small_k8(a, rows, primaries_only, ctx->sms * ctx->blocks_combine_small, st));
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
  if (c.K == 8 && a.interleave && ctx->blocks_combine_small > 0)
    return cuda_status(launch_small_k8(a, rows, false, ctx->sms * ctx->blocks_combine_small, st));
  return cuda_status(launch_k(a, rows, false, ctx->sms * ctx->blocks_combine, st));
}

}  // namespace moonep
