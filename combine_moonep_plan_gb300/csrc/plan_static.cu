// moonep_plan_noalloc: the planner for callers that cannot allocate device
// memory.
//
// Some callers cannot call cudaMalloc: a framework whose caching allocator
// owns every byte of device memory and accounts for it (a foreign cudaMalloc
// both escapes that accounting and can fail when the pool has reserved the
// device), or a latency-critical host path that cannot afford cudaMalloc's
// implicit device synchronisation.  moonep_plan needs a context (created with
// cudaMalloc) and a plan (also cudaMalloc'd); this entry point needs neither.
// The caller passes the inputs and every output array; the planner's
// intermediate tables (per-tile histograms, ordinals, balance tables) live in
// one file-scope __device__ array of fixed size, which every GPU that loads
// the library holds until the process exits.
#include <mutex>

#include "moonep_internal.cuh"

namespace moonep {
namespace {

// 4 MiB of planner scratch: enough for R*S*K up to ~900k routes at E = 384.
constexpr int64_t kNoAllocScratchWords = int64_t(1) << 20;
__device__ __align__(256) int32_t g_plan_scratch[kNoAllocScratchWords];

constexpr int kMaxDevices = 256;
std::mutex g_setup_mu;
int32_t *g_scratch_addr[kMaxDevices];  // device address of g_plan_scratch, per device

int64_t round_words(int64_t w) { return (w + 63) / 64 * 64; }

// Once per device, with that device current: the device address of the
// scratch array (the host-side symbol is only a stand-in, not a device
// address).  On every call: the planner kernels' shared-memory limits for
// this (R, E, B).  Their tables grow with E*R and with B, not with E alone,
// so a limit set for an earlier shape may be too low for this one;
// plan_configure only raises a limit (never lowers it, other shapes share the
// kernels) and returns at once when it is already high enough.
int setup(int device, int R, int E, int B, int32_t **scratch) {
  if (device < 0 || device >= kMaxDevices) return MOONEP_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_addr[device]) {
    void *ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_plan_scratch);
    if (e != cudaSuccess || !ptr) {
      cudaGetLastError();
      return MOONEP_ERR_CUDA;
    }
    g_scratch_addr[device] = static_cast<int32_t *>(ptr);
  }
  if (plan_configure(R, E, B) != cudaSuccess) {
    cudaGetLastError();
    return MOONEP_ERR_CUDA;
  }
  *scratch = g_scratch_addr[device];
  return MOONEP_OK;
}

}  // namespace
}  // namespace moonep

using namespace moonep;

extern "C" int moonep_plan_noalloc(const moonep_config *cfg, const int32_t *topk,
                                   const int32_t *tpe, int32_t *dst,
                                   int32_t *experts_to_copy, int32_t *cu_seqlens,
                                   int32_t *zero_fill_ranges, int32_t *remote_stats,
                                   int32_t *dup_counts, int32_t *status, void *stream) {
  if (!cfg) return MOONEP_ERR_INVALID_ARG;
  const moonep_config &c = *cfg;
  if (c.R < 1 || c.R > 64 || c.E < 1 || c.E % c.R != 0 || c.E > 4096 || c.K < 1 ||
      c.K > 32 || c.S < 0 || c.B < 0 || c.token_padding < 1)
    return MOONEP_ERR_INVALID_ARG;
  const int64_t L = c.E / c.R, tp = c.token_padding;
  const int64_t C = (int64_t)c.S * c.K;
  const int64_t nvs = (C + (L + c.B) * (tp - 1) + tp - 1) / tp * tp;
  if ((int64_t)c.R * nvs >= (int64_t)INT32_MAX - 1 || (int64_t)c.R * C >= (int64_t)INT32_MAX)
    return MOONEP_ERR_INVALID_ARG;
  if (!status || (!experts_to_copy && c.B > 0) || !cu_seqlens || !zero_fill_ranges ||
      !remote_stats || !dup_counts || (C > 0 && (!topk || !dst)))
    return MOONEP_ERR_INVALID_ARG;

  int device = 0, sms = 0;
  if (cudaGetDevice(&device) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
    cudaGetLastError();
    return MOONEP_ERR_CUDA;
  }
  // scratch: planner sync words, the planner's scratch (histograms of either
  // path, [R, E] totals, duplicate counts, error word), ordinals [R*S*K],
  // plan tables
  const int64_t tpr = (C + kTile - 1) / kTile;
  const int64_t sync_words = 64;
  const int64_t totals_off = plan_totals_offset(c.R, c.E, (int)C, c.K, sms);
  const int64_t hist_words = round_words(plan_scratch_words(c.R, c.E, (int)C, c.K, sms));
  const int64_t ord_words = round_words((int64_t)c.R * C);
  const PlanLayout lay = PlanLayout::make(c.R, c.E, c.B, (int)nvs, false);
  if (sync_words + hist_words + ord_words + lay.total > kNoAllocScratchWords)
    return MOONEP_ERR_INVALID_ARG;

  int32_t *scratch = nullptr;
  int st = setup(device, c.R, c.E, c.B, &scratch);
  if (st) return st;

  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return MOONEP_ERR_CUDA;
  // The planner's counters, per-rank totals, duplicate counts and error word
  // must start at zero: clear them on every call (the scratch serves every
  // shape).
  if (cudaMemsetAsync(scratch, 0, sync_words * sizeof(int32_t), s) != cudaSuccess ||
      cudaMemsetAsync(scratch + sync_words + totals_off, 0,
                      (size_t)(plan_scratch_words(c.R, c.E, (int)C, c.K, sms) - totals_off) *
                          sizeof(int32_t),
                      s) != cudaSuccess)
    return MOONEP_ERR_CUDA;

  // A context and a plan that only point: no member owns memory.
  moonep_ctx ctx{};
  ctx.cfg = c;
  ctx.device = device;
  ctx.L = (int)L;
  ctx.C = (int)C;
  ctx.EB = c.E + c.B;
  ctx.NvS = (int)nvs;
  ctx.TPR = (int)tpr;
  ctx.sms = ctx.sms_device = sms;
  ctx.G = (int)(c.R * tpr);
  ctx.d_status = status;
  ctx.d_sync = reinterpret_cast<unsigned long long *>(scratch);
  ctx.d_hist = scratch + sync_words;
  ctx.d_ord = scratch + sync_words + hist_words;
  moonep_comm_plan plan{};
  plan.dst = dst;
  plan.experts_to_copy = experts_to_copy;
  plan.cu_seqlens = cu_seqlens;
  plan.zero_fill_ranges = zero_fill_ranges;
  plan.remote_stats = remote_stats;
  plan.dup_counts = dup_counts;
  plan.internal = scratch + sync_words + hist_words + ord_words;
  plan.internal_bytes = lay.total * sizeof(int32_t);
  plan.N = (int)C;
  plan.R = c.R;
  plan.E = c.E;
  plan.B = c.B;
  plan.K = c.K;
  plan.S = c.S;
  plan.NvS = plan.NvS_padded = (int)nvs;
  plan.flags = 0;
  if (cudaMemsetAsync(plan.internal, 0, kMetaWords * sizeof(int32_t), s) != cudaSuccess)
    return MOONEP_ERR_CUDA;
  return launch_plan(&ctx, topk, tpe, &plan, s);
}
