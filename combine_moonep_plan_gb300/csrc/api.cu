// C ABI entry points: argument checks, resource lifetime, launches.
//
// "MoonEP Public API Visual Guide": Buffer(...) validates the topology and
// derives the capacities; Buffer.destroy() synchronises and releases
// everything, idempotently; MoonEPCommPlan.clone() deep-copies the plan;
// Buffer.hidden_nvsh_buffer_view / router_weight_buffer_view expose rank
// windows of the persistent buffers without copying.
#include <stdlib.h>
#include <string.h>

#include "moonep_internal.cuh"

namespace moonep {

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOONEP_OK : MOONEP_ERR_CUDA; }

int check_ctx(const moonep_ctx *ctx) {
  if (!ctx) return MOONEP_ERR_INVALID_ARG;
  if (ctx->destroyed) return MOONEP_ERR_DESTROYED;
  return MOONEP_OK;
}

int check_plan(const moonep_ctx *ctx, const moonep_comm_plan *p) {
  if (!p || !p->dst || !p->internal) return MOONEP_ERR_INVALID_ARG;
  const moonep_config &c = ctx->cfg;
  if (p->R != c.R || p->E != c.E || p->B != c.B || p->K != c.K || p->S != c.S ||
      p->NvS != ctx->NvS)
    return MOONEP_ERR_INVALID_ARG;
  return MOONEP_OK;
}

static int64_t nvs_of(const moonep_config &c) {
  const int64_t L = c.E / c.R, tp = c.token_padding;
  const int64_t raw = (int64_t)c.S * c.K + (L + c.B) * (tp - 1);
  return (raw + tp - 1) / tp * tp;
}

static int validate(const moonep_config *c) {
  if (!c) return MOONEP_ERR_INVALID_ARG;
  if (c->R < 1 || c->R > 64 || c->E < 1 || c->E % c->R != 0 || c->K < 1 || c->K > 32 ||
      c->S < 0 || c->H < 0 || c->H % 8 != 0 || c->B < 0 || c->token_padding < 1)
    return MOONEP_ERR_INVALID_ARG;
  // shared-memory tables of the planner (per-warp histograms: 8 * E words)
  if (c->E > 4096) return MOONEP_ERR_INVALID_ARG;
  const int64_t nvs = nvs_of(*c);
  if ((int64_t)c->R * nvs >= (int64_t)INT32_MAX - 1) return MOONEP_ERR_INVALID_ARG;
  if ((int64_t)c->R * c->S * c->K >= (int64_t)INT32_MAX) return MOONEP_ERR_INVALID_ARG;
  return MOONEP_OK;
}

static size_t scratch_bytes_of(const moonep_config &c) {
  const int64_t C = (int64_t)c.S * c.K;
  // planner tiles of either path: at most R * ceil(S*K / 1024)
  const int64_t tiles = (int64_t)c.R * ((C + 1023) / 1024 > 0 ? (C + 1023) / 1024 : 1);
  // planner tiles of every launch form, two [R, E] and two [E] totals sets
  const int64_t local = (C + 543) / 544 > 0 ? (C + 543) / 544 : 1;
  const int64_t t = tiles > local ? tiles : local;
  return (size_t)(c.E * (t + 2 * c.R + 2) + c.R * C) * sizeof(int32_t) + 1024;
}

}  // namespace moonep

using namespace moonep;

extern "C" {

int moonep_query_sizes(const moonep_config *cfg, int *NvS, int *NvS_padded,
                       size_t *scratch_bytes) {
  int st = validate(cfg);
  if (st) return st;
  const int64_t nvs = nvs_of(*cfg);
  if (NvS) *NvS = (int)nvs;
  if (NvS_padded) *NvS_padded = (int)nvs;
  if (scratch_bytes) *scratch_bytes = scratch_bytes_of(*cfg);
  return MOONEP_OK;
}

int moonep_ctx_create(const moonep_config *cfg, int alloc_views, moonep_ctx **out) {
  if (!out) return MOONEP_ERR_INVALID_ARG;
  *out = nullptr;
  int st = validate(cfg);
  if (st) return st;
  moonep_ctx *ctx = (moonep_ctx *)calloc(1, sizeof(moonep_ctx));
  if (!ctx) return MOONEP_ERR_NOMEM;
  ctx->cfg = *cfg;
  const moonep_config &c = ctx->cfg;
  cudaError_t e = cudaGetDevice(&ctx->device);
  int sms = 0;
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, ctx->device);
  if (e != cudaSuccess) {
    free(ctx);
    return MOONEP_ERR_CUDA;
  }
  // SM cap: the config's num_sms, else the MOONEP_NUM_SMS environment
  // variable, else every SM
  int cap = c.num_sms;
  if (cap <= 0) {
    const char *env = getenv("MOONEP_NUM_SMS");
    cap = env ? atoi(env) : 0;
  }
  ctx->sms = (cap > 0 && cap < sms) ? cap : sms;
  ctx->sms_device = sms;
  ctx->L = c.E / c.R;
  ctx->C = c.S * c.K;
  ctx->EB = c.E + c.B;
  ctx->NvS = (int)nvs_of(c);
  ctx->TPR = (ctx->C + kTile - 1) / kTile;
  ctx->G = c.R * ctx->TPR;
  ctx->blocks_dispatch = occupancy_dispatch(c.K, false);
  ctx->blocks_dispatch_small = occupancy_dispatch(c.K, true);
  ctx->blocks_combine = occupancy_combine(c.K);
  ctx->blocks_combine_small = occupancy_combine_small(c.K);
  ctx->blocks_copy = occupancy_copy();
  ctx->blocks_reduce = occupancy_reduce();
  ctx->blocks_expand = occupancy_dedup(false);
  ctx->blocks_fold = occupancy_dedup(true);
  const size_t hist =
      (size_t)plan_scratch_words(c.R, c.E, ctx->C, c.K, ctx->sms_device) * sizeof(int32_t);
  const size_t ord = (size_t)c.R * ctx->C * sizeof(int32_t);
  e = cudaMalloc(&ctx->d_status, 256);
  if (e == cudaSuccess) e = cudaMemset(ctx->d_status, 0, 256);
  if (e == cudaSuccess) e = cudaMalloc(&ctx->d_sync, kSyncWords * sizeof(unsigned long long));
  if (e == cudaSuccess) e = cudaMemset(ctx->d_sync, 0, kSyncWords * sizeof(unsigned long long));
  if (e == cudaSuccess && hist) e = cudaMalloc(&ctx->d_hist, hist);
  if (e == cudaSuccess && hist) e = cudaMemset(ctx->d_hist, 0, hist);
  if (e == cudaSuccess && ord) e = cudaMalloc(&ctx->d_ord, ord);
  if (e == cudaSuccess && alloc_views) {
    const size_t rows = (size_t)c.R * ctx->NvS;
    e = cudaMalloc(&ctx->d_hidden_view, rows * c.H * sizeof(uint16_t) + 16);
    if (e == cudaSuccess) e = cudaMalloc(&ctx->d_weight_view, rows * sizeof(float) + 16);
  }
  if (e == cudaSuccess) e = plan_configure(c.R, c.E, c.B);
  {
    const char *t = getenv("MOONEP_TEST_PLANNER_TIMEOUT");
    ctx->test_planner_timeout = (t && t[0] == '1') ? 1 : 0;
  }
  if (e == cudaSuccess) ctx->plan_cluster = plan_cluster_blocks(ctx);
  if (e != cudaSuccess) {
    cudaFree(ctx->d_status);
    cudaFree(ctx->d_sync);
    cudaFree(ctx->d_hist);
    cudaFree(ctx->d_ord);
    cudaFree(ctx->d_hidden_view);
    cudaFree(ctx->d_weight_view);
    free(ctx);
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? MOONEP_ERR_NOMEM : MOONEP_ERR_CUDA;
  }
  *out = ctx;
  return MOONEP_OK;
}

int moonep_ctx_destroy(moonep_ctx *ctx) {
  if (!ctx || ctx->destroyed) return MOONEP_OK;
  cudaError_t e = cudaDeviceSynchronize();
  cudaFree(ctx->d_status);
  cudaFree(ctx->d_sync);
  ctx->d_sync = nullptr;
  cudaFree(ctx->d_hist);
  cudaFree(ctx->d_ord);
  cudaFree(ctx->d_hidden_view);
  cudaFree(ctx->d_weight_view);
  ctx->d_status = nullptr;
  ctx->d_hist = ctx->d_ord = nullptr;
  ctx->d_hidden_view = nullptr;
  ctx->d_weight_view = nullptr;
  ctx->destroyed = 1;
  return cuda_status(e);
}

void moonep_ctx_free(moonep_ctx *ctx) {
  if (!ctx) return;
  moonep_ctx_destroy(ctx);
  free(ctx);
}

int moonep_ctx_destroyed(const moonep_ctx *ctx) { return ctx ? ctx->destroyed : 1; }

int moonep_num_sms(const moonep_ctx *ctx) { return ctx ? ctx->sms : 0; }

int moonep_plan_create(moonep_ctx *ctx, int flags, moonep_comm_plan *plan) {
  int st = check_ctx(ctx);
  if (st) return st;
  if (!plan || (flags & ~MOONEP_PLAN_DUP_RECORDS)) return MOONEP_ERR_INVALID_ARG;
  const moonep_config &c = ctx->cfg;
  memset(plan, 0, sizeof(*plan));
  const bool dup = (flags & MOONEP_PLAN_DUP_RECORDS) != 0;
  const PlanLayout lay = PlanLayout::make(c.R, c.E, c.B, ctx->NvS, dup);
  const size_t n_dst = (size_t)c.R * ctx->C, n_etc = (size_t)c.R * c.B;
  const size_t n_cu = (size_t)c.R * ctx->EB;
  const size_t n_dg = dup ? (size_t)c.R * ctx->NvS * 3 : 0, n_dl = dup ? (size_t)c.R * ctx->NvS : 0;
  // one allocation, each array 256-byte aligned
  auto up = [](size_t words) { return (words * sizeof(int32_t) + 255) / 256 * 256; };
  const size_t bytes = up(n_dst) + up(n_etc) + up(n_cu) + up(2 * n_cu) + up(2 * c.R) +
                       up(2 * c.R) + up(n_dg) + up(n_dl) + up(lay.total);
  char *base = nullptr;
  cudaError_t e = cudaMalloc(&base, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? MOONEP_ERR_NOMEM : MOONEP_ERR_CUDA;
  }
  e = cudaMemset(base, 0, bytes);
  char *p = base;
  auto carve = [&p, &up](size_t words) {
    int32_t *r = words ? (int32_t *)p : nullptr;
    p += up(words);
    return r;
  };
  plan->dst = carve(n_dst);
  if (!plan->dst) plan->dst = (int32_t *)base;  // S == 0: keep a non-null handle
  plan->experts_to_copy = carve(n_etc);
  plan->cu_seqlens = carve(n_cu);
  plan->zero_fill_ranges = carve(2 * n_cu);
  plan->remote_stats = carve(2 * c.R);
  plan->dup_counts = carve(2 * c.R);
  plan->dup_groups = carve(n_dg);
  plan->dup_loffs = carve(n_dl);
  plan->internal = carve(lay.total);
  plan->internal_bytes = lay.total * sizeof(int32_t);
  plan->N = ctx->C;
  plan->R = c.R;
  plan->E = c.E;
  plan->B = c.B;
  plan->K = c.K;
  plan->S = c.S;
  plan->NvS = ctx->NvS;
  plan->NvS_padded = ctx->NvS;
  plan->flags = flags;
  // base pointer for destroy: the first carved array sits at `base`
  (void)bytes;
  return cuda_status(e);
}

static void *plan_base(const moonep_comm_plan *plan) {
  // dst is always the first array of the allocation
  return plan->dst;
}

int moonep_plan_destroy(moonep_comm_plan *plan) {
  if (!plan || !plan->internal) return MOONEP_OK;
  cudaError_t e = cudaDeviceSynchronize();
  cudaFree(plan_base(plan));
  memset(plan, 0, sizeof(*plan));
  return cuda_status(e);
}

int moonep_plan_clone(const moonep_comm_plan *src, moonep_comm_plan *dst, void *stream) {
  if (!src || !dst || !src->internal || !dst->internal) return MOONEP_ERR_INVALID_ARG;
  if (src->R != dst->R || src->E != dst->E || src->B != dst->B || src->K != dst->K ||
      src->S != dst->S || src->NvS != dst->NvS || src->flags != dst->flags)
    return MOONEP_ERR_INVALID_ARG;
  // both plans are single allocations with identical layouts
  const char *sb = (const char *)plan_base(src);
  char *db = (char *)plan_base(dst);
  const size_t bytes = (size_t)((const char *)src->internal - sb) + src->internal_bytes;
  cudaError_t e = cudaMemcpyAsync(db, sb, bytes, cudaMemcpyDeviceToDevice, (cudaStream_t)stream);
  return cuda_status(e);
}

int moonep_plan(moonep_ctx *ctx, const int32_t *topk, const int32_t *tpe, moonep_comm_plan *plan,
                void *stream) {
  int st = check_ctx(ctx);
  if (st) return st;
  if ((st = check_plan(ctx, plan))) return st;
  if (ctx->C > 0 && !topk) return MOONEP_ERR_INVALID_ARG;
  return launch_plan(ctx, topk, tpe, plan, (cudaStream_t)stream);
}

int moonep_plan_rank(moonep_ctx *ctx, int rank, const int32_t *topk_r, const int32_t *hist_all,
                     moonep_comm_plan *plan, void *stream) {
  int st = check_ctx(ctx);
  if (st) return st;
  if ((st = check_plan(ctx, plan))) return st;
  if (rank < 0 || rank >= ctx->cfg.R || !hist_all || (ctx->C > 0 && !topk_r))
    return MOONEP_ERR_INVALID_ARG;
  if ((plan->flags & MOONEP_PLAN_DUP_RECORDS) || !plan_rank_supported(ctx))
    return MOONEP_ERR_INVALID_ARG;
  return launch_plan_rank(ctx, rank, topk_r, hist_all, plan, (cudaStream_t)stream);
}

// The R window pointers of a rank-local call: all given and 16-byte aligned
// (weights: all given or the array NULL, 4-byte aligned).
static int check_windows(const moonep_ctx *ctx, const void *const *rows, const void *const *w,
                         bool need_w) {
  const int R = ctx->cfg.R;
  if (!rows) return MOONEP_ERR_INVALID_ARG;
  for (int j = 0; j < R; j++)
    if (!rows[j] || !aligned16(rows[j])) return MOONEP_ERR_INVALID_ARG;
  if (need_w != (w != nullptr)) return MOONEP_ERR_INVALID_ARG;
  if (w)
    for (int j = 0; j < R; j++)
      if (!w[j] || ((uintptr_t)w[j] & 3)) return MOONEP_ERR_INVALID_ARG;
  return MOONEP_OK;
}

int moonep_dispatch_rank(moonep_ctx *ctx, const moonep_comm_plan *plan, int rank,
                         const uint16_t *hidden_r, const float *w_r, uint16_t *const *windows,
                         float *const *w_windows, void *stream) {
  int st = check_ctx(ctx);
  if (st) return st;
  if ((st = check_plan(ctx, plan))) return st;
  if (rank < 0 || rank >= ctx->cfg.R) return MOONEP_ERR_INVALID_ARG;
  if (ctx->cfg.S > 0 && !hidden_r) return MOONEP_ERR_INVALID_ARG;
  if (!aligned16(hidden_r) || ((uintptr_t)w_r & 3)) return MOONEP_ERR_INVALID_ARG;
  if ((st = check_windows(ctx, (const void *const *)windows, (const void *const *)w_windows,
                          w_r != nullptr)))
    return st;
  return launch_dispatch_rank(ctx, plan, rank, hidden_r, w_r, windows, w_windows,
                              (cudaStream_t)stream);
}

int moonep_combine_rank(moonep_ctx *ctx, const moonep_comm_plan *plan, int rank,
                        const uint16_t *const *y_windows, const float *const *w_windows,
                        uint16_t *out_r, float *w_out_r, void *stream) {
  int st = check_ctx(ctx);
  if (st) return st;
  if ((st = check_plan(ctx, plan))) return st;
  if (rank < 0 || rank >= ctx->cfg.R) return MOONEP_ERR_INVALID_ARG;
  if (ctx->cfg.S > 0 && !out_r) return MOONEP_ERR_INVALID_ARG;
  if (!aligned16(out_r) || ((uintptr_t)w_out_r & 3)) return MOONEP_ERR_INVALID_ARG;
  if ((st = check_windows(ctx, (const void *const *)y_windows, (const void *const *)w_windows,
                          w_out_r != nullptr)))
    return st;
  return launch_combine_rank(ctx, plan, rank, y_windows, w_windows, out_r, w_out_r,
                             (cudaStream_t)stream);
}

int moonep_dispatch(moonep_ctx *ctx, const moonep_comm_plan *plan, const uint16_t *hidden,
                    const float *w_sk, uint16_t *hidden_nvsh, float *w_nvs, void *stream) {
  int st = check_ctx(ctx);
  if (st) return st;
  if ((st = check_plan(ctx, plan))) return st;
  const int64_t ntok = (int64_t)ctx->cfg.R * ctx->cfg.S;
  if (!hidden_nvsh || (ntok > 0 && !hidden)) return MOONEP_ERR_INVALID_ARG;
  if (ntok > 0 && (w_sk == nullptr) != (w_nvs == nullptr)) return MOONEP_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(hidden_nvsh) || ((uintptr_t)w_sk & 3) ||
      ((uintptr_t)w_nvs & 3))
    return MOONEP_ERR_INVALID_ARG;
  return launch_dispatch(ctx, plan, hidden, w_sk, hidden_nvsh, w_nvs, (cudaStream_t)stream);
}

int moonep_combine(moonep_ctx *ctx, const moonep_comm_plan *plan, const uint16_t *y_nvsh,
                   const float *w_nvs, uint16_t *out_sh, float *w_sk_out, void *stream) {
  int st = check_ctx(ctx);
  if (st) return st;
  if ((st = check_plan(ctx, plan))) return st;
  const int64_t ntok = (int64_t)ctx->cfg.R * ctx->cfg.S;
  if (ntok > 0 && (!y_nvsh || !out_sh)) return MOONEP_ERR_INVALID_ARG;
  if (ntok > 0 && (w_nvs == nullptr) != (w_sk_out == nullptr)) return MOONEP_ERR_INVALID_ARG;
  if (!aligned16(y_nvsh) || !aligned16(out_sh) || ((uintptr_t)w_nvs & 3) ||
      ((uintptr_t)w_sk_out & 3))
    return MOONEP_ERR_INVALID_ARG;
  return launch_combine(ctx, plan, y_nvsh, w_nvs, out_sh, w_sk_out, (cudaStream_t)stream);
}

int moonep_dispatch_dedup(moonep_ctx *ctx, const moonep_comm_plan *plan, const uint16_t *hidden,
                          const float *w_sk, uint16_t *hidden_nvsh, float *w_nvs, void *stream) {
  int st = check_ctx(ctx);
  if (st) return st;
  if ((st = check_plan(ctx, plan))) return st;
  if (!(plan->flags & MOONEP_PLAN_DUP_RECORDS)) return MOONEP_ERR_INVALID_ARG;
  const int64_t ntok = (int64_t)ctx->cfg.R * ctx->cfg.S;
  if (!hidden_nvsh || (ntok > 0 && !hidden)) return MOONEP_ERR_INVALID_ARG;
  if (ntok > 0 && (w_sk == nullptr) != (w_nvs == nullptr)) return MOONEP_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(hidden_nvsh) || ((uintptr_t)w_sk & 3) ||
      ((uintptr_t)w_nvs & 3))
    return MOONEP_ERR_INVALID_ARG;
  const cudaStream_t s = (cudaStream_t)stream;
  if ((st = launch_dispatch(ctx, plan, hidden, w_sk, hidden_nvsh, w_nvs, s, true))) return st;
  return launch_expand(ctx, plan, hidden_nvsh, s);
}

int moonep_combine_dedup(moonep_ctx *ctx, const moonep_comm_plan *plan, uint16_t *y_nvsh,
                         const float *w_nvs, uint16_t *out_sh, float *w_sk_out, void *stream) {
  int st = check_ctx(ctx);
  if (st) return st;
  if ((st = check_plan(ctx, plan))) return st;
  if (!(plan->flags & MOONEP_PLAN_DUP_RECORDS)) return MOONEP_ERR_INVALID_ARG;
  const int64_t ntok = (int64_t)ctx->cfg.R * ctx->cfg.S;
  if (ntok > 0 && (!y_nvsh || !out_sh)) return MOONEP_ERR_INVALID_ARG;
  if (ntok > 0 && (w_nvs == nullptr) != (w_sk_out == nullptr)) return MOONEP_ERR_INVALID_ARG;
  if (!aligned16(y_nvsh) || !aligned16(out_sh) || ((uintptr_t)w_nvs & 3) ||
      ((uintptr_t)w_sk_out & 3))
    return MOONEP_ERR_INVALID_ARG;
  const cudaStream_t s = (cudaStream_t)stream;
  if ((st = launch_fold(ctx, plan, y_nvsh, s))) return st;
  return launch_combine(ctx, plan, y_nvsh, w_nvs, out_sh, w_sk_out, s, true);
}

int moonep_prefetch_weight(moonep_ctx *ctx, const moonep_comm_plan *plan, int n_proj,
                           uint16_t *const *W, int64_t HHp, void *stream) {
  int st = check_ctx(ctx);
  if (st) return st;
  if ((st = check_plan(ctx, plan))) return st;
  if (!W || n_proj < 1 || n_proj > 4 || HHp < 0 || HHp % 8 != 0) return MOONEP_ERR_INVALID_ARG;
  for (int p = 0; p < n_proj; p++)
    if (!W[p] || !aligned16(W[p])) return MOONEP_ERR_INVALID_ARG;
  void *T[4];
  int64_t rb[4];
  for (int p = 0; p < n_proj; p++) {
    T[p] = W[p];
    rb[p] = HHp * 2;
  }
  return launch_prefetch(ctx, plan, n_proj, T, rb, (cudaStream_t)stream);
}

int moonep_prefetch_rows(moonep_ctx *ctx, const moonep_comm_plan *plan, int n_tensors,
                         void *const *tensors, const int64_t *row_bytes, void *stream) {
  int st = check_ctx(ctx);
  if (st) return st;
  if ((st = check_plan(ctx, plan))) return st;
  if (!tensors || !row_bytes || n_tensors < 1 || n_tensors > 8) return MOONEP_ERR_INVALID_ARG;
  for (int t = 0; t < n_tensors; t++)
    if (row_bytes[t] < 0 || (row_bytes[t] > 0 && !tensors[t])) return MOONEP_ERR_INVALID_ARG;
  return launch_prefetch(ctx, plan, n_tensors, tensors, row_bytes, (cudaStream_t)stream);
}

int moonep_prepare(moonep_ctx *ctx, const int32_t *num_tokens, uint16_t *hidden,
                   int32_t *topk, float *w_sk, int32_t *tokens_per_expert, void *stream) {
  int st = check_ctx(ctx);
  if (st) return st;
  const moonep_config &c = ctx->cfg;
  if ((int64_t)c.S * c.K > 0 && !topk) return MOONEP_ERR_INVALID_ARG;
  if (hidden && !aligned16(hidden)) return MOONEP_ERR_INVALID_ARG;
  if (num_tokens)
    for (int r = 0; r < c.R; r++)
      if (num_tokens[r] < 0 || num_tokens[r] > c.S) return MOONEP_ERR_INVALID_ARG;
  if ((int64_t)c.R * c.S == 0) return MOONEP_OK;
  return launch_prepare(ctx, num_tokens, hidden, topk, w_sk, tokens_per_expert,
                        (cudaStream_t)stream);
}

int moonep_reduce_redundant_grad(moonep_ctx *ctx, const moonep_comm_plan *plan, int n_proj,
                                 float *const *Gh, float *const *Gs, int64_t HHp,
                                 void *stream) {
  int st = check_ctx(ctx);
  if (st) return st;
  if ((st = check_plan(ctx, plan))) return st;
  if (!Gh || !Gs || n_proj < 1 || n_proj > 4 || HHp < 0 || HHp % 4 != 0)
    return MOONEP_ERR_INVALID_ARG;
  for (int p = 0; p < n_proj; p++)
    if (!Gh[p] || !Gs[p] || !aligned16(Gh[p]) || !aligned16(Gs[p])) return MOONEP_ERR_INVALID_ARG;
  return launch_reduce(ctx, plan, n_proj, Gh, Gs, HHp, (cudaStream_t)stream);
}

void *moonep_hidden_view(moonep_ctx *ctx, int rank) {
  if (check_ctx(ctx) || !ctx->d_hidden_view || rank < 0 || rank >= ctx->cfg.R) return nullptr;
  return ctx->d_hidden_view + (size_t)rank * ctx->NvS * ctx->cfg.H;
}

void *moonep_weight_view(moonep_ctx *ctx, int rank) {
  if (check_ctx(ctx) || !ctx->d_weight_view || rank < 0 || rank >= ctx->cfg.R) return nullptr;
  return ctx->d_weight_view + (size_t)rank * ctx->NvS;
}

int moonep_get_status(moonep_ctx *ctx, int *device_status, void *stream) {
  int st = check_ctx(ctx);
  if (st) return st;
  if (!device_status) return MOONEP_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int32_t v = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(&v, ctx->d_status, sizeof(v), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(ctx->d_status, 0, sizeof(int32_t));
  // A planner wait that ran out may have left its counters and accumulators
  // out of step: start them again from zero.
  if (e == cudaSuccess && v == MOONEP_ERR_TIMEOUT) {
    const moonep_config &c = ctx->cfg;
    const int64_t off = plan_totals_offset(c.R, c.E, ctx->C, c.K, ctx->sms_device);
    const int64_t words = plan_scratch_words(c.R, c.E, ctx->C, c.K, ctx->sms_device) - off;
    e = cudaMemset(ctx->d_sync, 0, kSyncWords * sizeof(unsigned long long));
    if (e == cudaSuccess) e = cudaMemset(ctx->d_hist + off, 0, (size_t)words * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
  }
  if (e != cudaSuccess) return MOONEP_ERR_CUDA;
  *device_status = v;
  return MOONEP_OK;
}

const char *moonep_strerror(int code) {
  switch (code) {
    case MOONEP_OK: return "ok";
    case MOONEP_ERR_INVALID_ARG: return "invalid argument";
    case MOONEP_ERR_BAD_EXPERT: return "expert id outside [0, E)";
    case MOONEP_ERR_HIST_MISMATCH: return "tokens_per_expert does not match topk";
    case MOONEP_ERR_SLOTS: return "a rank needs more than B prefetch slots";
    case MOONEP_ERR_CUDA: return "CUDA error";
    case MOONEP_ERR_DESTROYED: return "context destroyed";
    case MOONEP_ERR_PLAN: return "plan row outside the dispatched buffer";
    case MOONEP_ERR_NOMEM: return "device allocation failed";
    case MOONEP_ERR_TIMEOUT: return "a planner block gave up waiting for the balance step";
    default: return "unknown status";
  }
}

}  // extern "C"
