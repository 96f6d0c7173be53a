// Internal declarations shared by the translation units of libmoonep.
// Not part of the public ABI (include/moonep.h is).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moonep.h"

namespace moonep {

// Ranks a configuration may have (the balance step keeps per-rank state in
// shared memory; the rank-local copy kernels take one window per rank).
constexpr int kMaxRanks = 64;

// The planner's arrival counters (ctx->d_sync), each on its own 128-byte
// line: whole-problem calls at word 0, rank-local calls at kSyncRankLocal.
constexpr int kSyncWords = 32;  // 64-bit words
constexpr int kSyncRankLocal = 16;

// Routes handled by one planner tile: 8 warps x 32 lanes x 8 routes.
constexpr int kPlanThreads = 256;
constexpr int kPlanItems = 8;
constexpr int kTile = kPlanThreads * kPlanItems;

// Bits of the plan-local error word (meta[kMetaErr]).
constexpr int kErrBadExpert = 1;
constexpr int kErrHist = 2;
constexpr int kErrSlots = 4;

// Scalar words at the head of plan->internal.
enum {
  kMetaErr = 0,    // error bits found while planning
  kMetaValid = 1,  // 1 when the plan's tables are usable
  kMetaP = 2,      // padding rows over all ranks
  kMetaU = 3,      // used prefetch slots over all ranks
  kMetaD = 4,      // experts with at least one slot copy
  kMetaWords = 16
};

// Word offsets of the tables inside plan->internal (see PlanLayout::make).
// Usable prefetch slots per rank: a rank receives at most one piece, from one
// home group, so it never fills more than L = E/R slots.
__host__ __device__ inline int usable_slots(int R, int E, int B) { return B < E / R ? B : E / R; }

// Words of the balance step's tables (shared memory, or the plan's internal
// area when they do not fit): per expert T, Q, home row base, slot copies and
// their index (+1 each), per (rank, donor-local expert) slot and row base,
// experts_to_copy of the usable slots, and per segment (E + R*Bm) valid rows
// plus two prefix sums.
__host__ __device__ inline size_t bal_tables_words(int R, int E, int B) {
  const size_t Bm = (size_t)usable_slots(R, E, B);
  const size_t nseg = (size_t)E + (size_t)R * Bm;
  return 7 * (size_t)E + 2 + (size_t)R * Bm + nseg + 2 * (nseg + 1);
}

// Layout of plan->internal (int32 words after the meta words).
// Rows of a rank handled by one block of the duplicate-record builder.
constexpr int kDupTile = 1024;
inline int dup_tiles_per_rank(int NvS) { return (NvS + kDupTile - 1) / kDupTile; }

struct PlanLayout {
  int64_t qoff, home_rowbase, keep, piece_first, piece_count, piece_start, piece_len,
      piece_recv, slot_rowbase, bal, pad_prefix, red_expert, red_first,
      red_slot, dupflag, dup_tiles, total;
  static PlanLayout make(int R, int E, int B, int NvS, bool dup_records) {
    PlanLayout l;
    const int L = E / R, EB = E + B;
    int64_t o = kMetaWords;
    auto take = [&o](int64_t n) { int64_t at = o; o += (n + 3) / 4 * 4; return at; };
    l.qoff = take(E);
    l.home_rowbase = take(E);
    l.keep = take(R);
    l.piece_first = take(R);
    l.piece_count = take(R);
    l.piece_start = take(R);
    l.piece_len = take(R);
    l.piece_recv = take(R);
    l.slot_rowbase = take((int64_t)R * L);
    l.bal = take((int64_t)bal_tables_words(R, E, B));
    l.pad_prefix = take((int64_t)R * EB + 1);
    l.red_expert = take(E);
    l.red_first = take(E + 1);
    l.red_slot = take((int64_t)R * B);
    l.dupflag = dup_records ? take((int64_t)R * NvS) : -1;
    // per rank and tile of kDupTile rows: {groups, duplicate routes}
    l.dup_tiles = dup_records ? take((int64_t)R * dup_tiles_per_rank(NvS) * 2) : -1;
    l.total = o;
    return l;
  }
};

}  // namespace moonep

struct moonep_ctx {
  moonep_config cfg;
  int device;
  int sms;         // SMs the copy kernels may use
  int sms_device;  // SMs of the device
  int L, C, EB, NvS, TPR, G;  // E/R, S*K, E+B, rows per rank, tiles per rank, R*TPR
  int destroyed;
  int32_t *d_status;   // sticky first error
  int32_t *d_hist;     // planner scratch: tile histograms, [R, E] totals, duplicate counts, error bits
  int32_t *d_ord;      // [R*C] ordinal of a route among its tile's routes to the same expert
  uint16_t *d_hidden_view;  // optional [R*NvS, H] bf16
  float *d_weight_view;     // optional [R*NvS] fp32
  unsigned long long *d_sync;  // [kSyncWords] the planner's counters (kSync*)
  int test_planner_timeout;    // test hook: the planner's arrival wait never completes
  int plan_cluster;            // blocks of the whole-problem planner launched as one
                               // cluster (0: a cooperative launch)
  int blocks_dispatch, blocks_dispatch_small, blocks_combine, blocks_combine_small, blocks_copy, blocks_reduce, blocks_expand,
      blocks_fold;  // resident blocks per SM
};

namespace moonep {

int check_ctx(const moonep_ctx *ctx);
int check_plan(const moonep_ctx *ctx, const moonep_comm_plan *plan);
inline bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
int cuda_status(cudaError_t e);

// Launchers (one per translation unit).
int launch_plan(moonep_ctx *ctx, const int32_t *topk, const int32_t *tpe,
                moonep_comm_plan *plan, cudaStream_t st);
// The rank-local planner (one source rank's routes, gathered [R, E]
// histograms), and whether the configuration allows it (the single-launch
// planner's tables fit in shared memory and one rank's tiles fit on the SMs).
int launch_plan_rank(moonep_ctx *ctx, int rank, const int32_t *topk_r, const int32_t *hist_all,
                     moonep_comm_plan *plan, cudaStream_t st);
int plan_rank_supported(const moonep_ctx *ctx);
int launch_dispatch(moonep_ctx *ctx, const moonep_comm_plan *plan, const uint16_t *hidden,
                    const float *w_sk, uint16_t *out, float *w_out, cudaStream_t st,
                    bool primaries_only = false);
int launch_combine(moonep_ctx *ctx, const moonep_comm_plan *plan, const uint16_t *y,
                   const float *w_nvs, uint16_t *out, float *w_out, cudaStream_t st,
                   bool primaries_only = false);
// Rank-local forms: source rank `rank`'s tokens, rows in R rank windows
// (windows[j] = rank j's [NvS, H] rows, w_windows[j] its [NvS] weights).
int launch_dispatch_rank(moonep_ctx *ctx, const moonep_comm_plan *plan, int rank,
                         const uint16_t *hidden_r, const float *w_r, uint16_t *const *windows,
                         float *const *w_windows, cudaStream_t st);
int launch_combine_rank(moonep_ctx *ctx, const moonep_comm_plan *plan, int rank,
                        const uint16_t *const *y_windows, const float *const *w_windows,
                        uint16_t *out_r, float *w_out_r, cudaStream_t st);
// The deduplicated data flow's local steps: copy every primary row to its
// duplicates (dispatch epilogue), or fold every rank's duplicate rows of a
// token into its primary row (combine prologue).
int launch_expand(moonep_ctx *ctx, const moonep_comm_plan *plan, uint16_t *rows, cudaStream_t st);
int launch_fold(moonep_ctx *ctx, const moonep_comm_plan *plan, uint16_t *rows, cudaStream_t st);
int launch_prefetch(moonep_ctx *ctx, const moonep_comm_plan *plan, int n, void *const *T,
                    const int64_t *row_bytes, cudaStream_t st);
int launch_prepare(moonep_ctx *ctx, const int32_t *num_tokens, uint16_t *hidden,
                   int32_t *topk, float *w, int32_t *tpe, cudaStream_t st);
int launch_reduce(moonep_ctx *ctx, const moonep_comm_plan *plan, int n_proj, float *const *Gh,
                  float *const *Gs, int64_t HHp, cudaStream_t st);
// Opt the planner kernels into the dynamic shared memory E experts need.
cudaError_t plan_configure(int R, int E, int B);
// Blocks of the single-launch planner when they can run as one thread-block
// cluster on this device (at most 16), else 0.
int plan_cluster_blocks(const moonep_ctx *ctx);
// K when the single-launch planner handles this shape (0: the tile path).
int plan_fused_choice(int R, int E, int K, int B, int C, int sms);
// Tiles the histogram area must hold (either planner path).
int plan_hist_tiles(int R, int C, int K, int sms);
// The planner's scratch (ctx->d_hist): E words per tile, then two sets of
// [R, E] totals (at plan_totals_offset) and two error words, used by
// alternate calls, zero before a call uses them.
int64_t plan_totals_offset(int R, int E, int C, int K, int sms);
// After those: the rank-local planner's two [E] totals sets and error words.
int64_t plan_rank_totals_offset(int R, int E, int C, int K, int sms);
int64_t plan_scratch_words(int R, int E, int C, int K, int sms);
int occupancy_dispatch(int K, bool small_units);
int occupancy_combine(int K);
int occupancy_combine_small(int K);
int occupancy_copy();
int occupancy_reduce();
int occupancy_dedup(bool fold);

// Programmatic dependent launch: every kernel of the library is launched
// with launch_pdl, so it may be scheduled while the kernel before it on the
// stream is still running.  Its first statement is pdl_wait(): it waits until
// that kernel has completed and its memory is visible, before touching any
// memory; then pdl_launch_dependents() lets the next kernel be scheduled.
// Back-to-back launches (the decode path's plan -> dispatch -> combine) then
// overlap one kernel's launch latency with the previous one's tail.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// cluster > 1: the grid is one or more thread-block clusters of that many
// blocks (every block of a cluster is resident at once, on one GPC).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, bool cooperative, int cluster, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[3];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  n++;
  if (cooperative) {
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = 1;
    n++;
  }
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    n++;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, bool cooperative, Args &&...args) {
  return launch_pdl_ex(kernel, grid, block, smem, st, cooperative, 1,
                       std::forward<Args>(args)...);
}

// Latch the first error code into the status word.
__device__ __forceinline__ void set_status(int32_t *status, int code) {
  atomicCAS(status, 0, code);
}

}  // namespace moonep
