// C ABI of libtokenselect: argument validation, context and cache lifetime,
// and the stream-ordered composition of one decode step.
#include <cmath>
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "ts_internal.h"

using namespace ts;

namespace {

template <typename T>
cudaError_t alloc(T** p, size_t n) {
  *p = nullptr;
  if (n == 0) n = 1;
  return cudaMalloc(reinterpret_cast<void**>(p), n * sizeof(T));
}

void free_ctx_buffers(ts_ctx* c) {
  for (auto& b : c->prof) {
    if (b.begin) cudaEventDestroy(b.begin);
    if (b.end) cudaEventDestroy(b.end);
    b.begin = b.end = nullptr;
  }
  cudaFree(c->status);
  cudaFree(c->logits);
  cudaFree(c->partials);
  cudaFree(c->stats);
  cudaFree(c->counters);
  cudaFree(c->sel_state);
  cudaFree(c->hist);
  cudaFree(c->mass_hist);
  cudaFree(c->chunk_counts);
  cudaFree(c->attn_part);
  cudaFree(c->vote);
  cudaFree(c->hit);
  cudaFree(c->qmean);
  cudaFree(c->blk_len);
  cudaFree(c->blk_idx);
  cudaFree(c->sel_rows);
  cudaFree(c->step_partials);
  cudaFree(c->step_hist);
  cudaFree(c->step_mass);
  cudaFree(c->cand_n);
  cudaFree(c->cands);
  cudaFree(c->cta_cnt);
  cudaFree(c->apart);
  cudaFree(c->step_wpart);
  cudaFree(c->gsync);
  cudaFree(c->phase_ns);
}

float resolve_scale(const ts_ctx* ctx, float scale) {
  return scale == 0.f ? 1.f / std::sqrt((float)ctx->cfg.head_dim) : scale;
}

bool valid_params(const ts_select_params* p) {
  if (!p) return false;
  if (p->mode != TS_SELECT_TOPK && p->mode != TS_SELECT_TOPP) return false;
  if (p->k < 0 || p->n_sink < 0 || p->n_local < 0) return false;
  if (p->mode == TS_SELECT_TOPP && !(p->top_p > 0.f)) return false;
  if (std::isnan(p->theta) || std::isnan(p->softmax_scale)) return false;
  if (p->score_fn != TS_SCORE_HEAD_SOFT_VOTE && p->score_fn != TS_SCORE_LOGIT_SUM &&
      p->score_fn != TS_SCORE_HEAD_HARD_VOTE)
    return false;
  // the ablation selection functions are ranked by top-k only (top-p's mass is the soft vote's)
  if (p->score_fn != TS_SCORE_HEAD_SOFT_VOTE && p->mode != TS_SELECT_TOPK) return false;
  return true;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

int ts_version(void) { return 100; }

const char* ts_status_str(ts_status s) {
  switch (s) {
    case TS_OK: return "ok";
    case TS_ERR_INVALID_ARG: return "invalid argument";
    case TS_ERR_SHAPE: return "shape outside the context's limits";
    case TS_ERR_UNSUPPORTED: return "head geometry not compiled";
    case TS_ERR_CUDA: return "CUDA runtime error";
    case TS_ERR_PAGE_OOB: return "page-table entry outside the pool";
    case TS_ERR_CAPACITY: return "selection larger than its output buffer";
    case TS_ERR_TIMEOUT: return "a bounded device wait ran out";
    case TS_ERR_COOP_UNAVAILABLE: return "cooperative launch refused";
    case TS_ERR_SEQ_LEN: return "sequence length outside [0, max tokens]";
    case TS_ERR_SCRATCH_LIMIT: return "size beyond the fixed scratch of the no-alloc call";
  }
  return "unknown status";
}

ts_status ts_create(ts_ctx** out, const ts_config* cfg) {
  if (!out || !cfg) return TS_ERR_INVALID_ARG;
  *out = nullptr;
  const ts_config& c = *cfg;
  if (c.n_q_heads < 1 || c.n_kv_heads < 1 || c.n_q_heads % c.n_kv_heads != 0) return TS_ERR_INVALID_ARG;
  if (c.max_batch < 1 || c.max_pages_per_seq < 1 || c.num_pages < 1 || c.head_dim < 1) return TS_ERR_INVALID_ARG;
  if (c.kv_dtype != TS_KV_F32 && c.kv_dtype != TS_KV_BF16) return TS_ERR_INVALID_ARG;
  if (c.page_size != kPage && c.page_size != 1) return TS_ERR_UNSUPPORTED;
  if (c.n_kv_heads > kCounterSlots - 2 || c.n_q_heads > 256) return TS_ERR_UNSUPPORTED;
  if ((int64_t)c.max_pages_per_seq * c.page_size > (int64_t)1 << 30) return TS_ERR_SHAPE;
  if (!score_supported(c)) return TS_ERR_UNSUPPORTED;

  ts_ctx* ctx = new (std::nothrow) ts_ctx();
  if (!ctx) return TS_ERR_CUDA;
  ctx->cfg = c;
  // environment switches, read here once (never per call):
  // TOKENSELECT_MULTI_KERNEL=1 keeps ts_decode_step on the multi-kernel path (tests, comparisons)
  if (const char* env = std::getenv("TOKENSELECT_MULTI_KERNEL")) ctx->use_step = !(env[0] == '1');
  // the persistent kernel's TMA page tiles are 16 tokens: a token-granular pool (one token per
  // page) takes the multi-kernel path
  if (c.page_size != kPage) ctx->use_step = false;
  ctx->page_shift = c.page_size == kPage ? 4 : 0;
  ctx->debug = std::getenv("TS_DEBUG") != nullptr;
  if (const char* env = std::getenv("TOKENSELECT_NO_TC")) ctx->no_tc = env[0] == '1';
  if (const char* env = std::getenv("TOKENSELECT_SCAN_CLAIM")) ctx->scan_claim = env[0] == '1';
  // TOKENSELECT_TOPP_ATTEND=gather / range / range_tc: the persistent kernel's top-p attention
  // always shares the selected tokens out over the CTAs, or always attends each CTA's own range
  // (when it may), with P.V on CUDA cores or on the tensor cores (bf16, d = 128)
  if (const char* env = std::getenv("TOKENSELECT_TOPP_ATTEND")) {
    if (std::strcmp(env, "gather") == 0) ctx->range_attend = 0;
    if (std::strcmp(env, "range") == 0) ctx->range_attend = 2;
    if (std::strcmp(env, "range_tc") == 0) {
      ctx->range_attend = 2;
      ctx->range_tc = true;
    }
  }
  if (const char* env = std::getenv("TOKENSELECT_L2_BUDGET_MB")) {
    const long mb = std::strtol(env, nullptr, 10);
    if (mb > 0) ctx->l2_budget = (int64_t)mb << 20;
  }
  if (cudaGetDevice(&ctx->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device) != cudaSuccess) {
    delete ctx;
    return TS_ERR_CUDA;
  }
  const size_t B = c.max_batch, H = c.n_q_heads, HKV = c.n_kv_heads, G = H / HKV, D = c.head_dim;
  ctx->max_tokens = c.max_pages_per_seq * c.page_size;
  ctx->score_max_chunks = (ctx->max_tokens + kScorePagesPerCta * kPage - 1) / (kScorePagesPerCta * kPage);
  ctx->sel_max_chunks = (ctx->max_tokens + kSelChunk - 1) / kSelChunk;
  ctx->attn_splits = kAttnMaxSplits;
  const size_t T = ctx->max_tokens;
  cudaError_t e = cudaSuccess;
  auto chk = [&](cudaError_t r) {
    if (e == cudaSuccess) e = r;
  };
  const size_t NS = (size_t)ctx->num_sms;
  // [B][H][T] logits of the multi-kernel path; the persistent kernel keeps, per CTA, the
  // logits of its page range: at most (B*T/16 + NS) pages, which this also covers
  ctx->logits_floats = (int64_t)(B * H * T + H * NS * 2 * kPage);
  chk(alloc(&ctx->status, 1));
  chk(alloc(&ctx->logits, (size_t)ctx->logits_floats));
  chk(alloc(&ctx->step_partials, B * NS * 2 * H));   // two partial rows per CTA where a tile holds two pages
  chk(alloc(&ctx->step_hist, B * kStepHistPerSeq));
  chk(alloc(&ctx->step_mass, B * kStepHistPerSeq));
  chk(alloc(&ctx->cand_n, B));
  chk(alloc(&ctx->cands, B * 2048));
  chk(alloc(&ctx->cta_cnt, B * NS * 4));
  chk(alloc(&ctx->apart, B * NS * H * (D + 2) + 2 * B * H));   // (max, sum) rows padded to an even count
  // per CTA: [sequence][scan warp][head] (max, sum exp) pairs of the CUDA-core scan
  chk(alloc(&ctx->step_wpart, NS * B * kMaxScanWarps * kMaxScanG * 2));
  chk(alloc(&ctx->gsync, 4));
  if (e == cudaSuccess) chk(cudaMemset(ctx->gsync, 0, 4 * sizeof(unsigned)));   // then kept zero by each launch
  chk(alloc(&ctx->phase_ns, 64));
  chk(alloc(&ctx->partials, B * ctx->score_max_chunks * H));
  chk(alloc(&ctx->stats, B * H));
  chk(alloc(&ctx->counters, B * kCounterSlots));
  chk(alloc(&ctx->sel_state, B));
  chk(alloc(&ctx->hist, B * 2048));
  chk(alloc(&ctx->mass_hist, B * 2048));
  chk(alloc(&ctx->chunk_counts, B * ctx->sel_max_chunks));
  chk(alloc(&ctx->attn_part, B * HKV * kAttnMaxSplits * G * (D + 2)));
  chk(alloc(&ctx->vote, B * T));
  chk(alloc(&ctx->hit, B));
  chk(alloc(&ctx->qmean, B * H * D));
  chk(alloc(&ctx->blk_len, B));
  chk(alloc(&ctx->blk_idx, B * T + B));
  chk(alloc(&ctx->sel_rows, NS * kStepFlagCap));
  if (e == cudaSuccess) chk(cudaMemset(ctx->status, 0, sizeof(int)));
  if (e == cudaSuccess) chk(cudaMemset(ctx->counters, 0, B * kCounterSlots * sizeof(unsigned)));
  if (e == cudaSuccess) chk(cudaMemset(ctx->hist, 0, B * 2048 * sizeof(unsigned)));
  if (e == cudaSuccess) chk(cudaMemset(ctx->mass_hist, 0, B * 2048 * sizeof(unsigned long long)));
  if (e == cudaSuccess) chk(cudaMemset(ctx->hit, 0, B));
  if (e == cudaSuccess) chk(cudaMemset(ctx->phase_ns, 0, 64 * sizeof(unsigned long long)));
  if (e == cudaSuccess) chk(cudaDeviceSynchronize());
  if (e != cudaSuccess) {
    free_ctx_buffers(ctx);
    delete ctx;
    return TS_ERR_CUDA;
  }
  *out = ctx;
  return TS_OK;
}

ts_status ts_destroy(ts_ctx* ctx) {
  if (!ctx) return TS_ERR_INVALID_ARG;
  cudaDeviceSynchronize();
  free_ctx_buffers(ctx);
  delete ctx;
  return TS_OK;
}

ts_status ts_cache_create(ts_ctx* ctx, ts_cache** out, int n_layers, int capacity) {
  if (!ctx || !out || n_layers < 1 || capacity < 1) return TS_ERR_INVALID_ARG;
  *out = nullptr;
  ts_cache* c = new (std::nothrow) ts_cache();
  if (!c) return TS_ERR_CUDA;
  c->ctx = ctx;
  c->n_layers = n_layers;
  c->capacity = capacity;
  const size_t LB = (size_t)n_layers * ctx->cfg.max_batch;
  const size_t HD = (size_t)ctx->cfg.n_q_heads * ctx->cfg.head_dim;
  cudaError_t e = alloc(&c->cq, LB * HD);
  if (e == cudaSuccess) e = alloc(&c->ct, LB * capacity);
  if (e == cudaSuccess) e = alloc(&c->ct_count, LB);
  if (e == cudaSuccess) e = alloc(&c->filled, LB);
  if (e == cudaSuccess) e = cudaMemset(c->filled, 0, LB);
  if (e == cudaSuccess) e = cudaMemset(c->ct_count, 0, LB * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(c->cq);
    cudaFree(c->ct);
    cudaFree(c->ct_count);
    cudaFree(c->filled);
    delete c;
    return TS_ERR_CUDA;
  }
  *out = c;
  return TS_OK;
}

ts_status ts_cache_destroy(ts_cache* c) {
  if (!c) return TS_ERR_INVALID_ARG;
  cudaDeviceSynchronize();
  cudaFree(c->cq);
  cudaFree(c->ct);
  cudaFree(c->ct_count);
  cudaFree(c->filled);
  delete c;
  return TS_OK;
}

ts_status ts_cache_reset(ts_cache* c, void* stream) {
  if (!c) return TS_ERR_INVALID_ARG;
  return launch_cache_reset(c, as_stream(stream));
}

ts_status ts_cache_check(ts_ctx* ctx, ts_cache* cache, int layer, const float* q, int B, float theta,
                         uint8_t* hit, float* cos_out, void* stream) {
  if (!ctx || !cache || !q || !hit || cache->ctx != ctx) return TS_ERR_INVALID_ARG;
  if (layer < 0 || layer >= cache->n_layers || B < 1 || B > ctx->cfg.max_batch) return TS_ERR_SHAPE;
  if (std::isnan(theta)) return TS_ERR_INVALID_ARG;
  return launch_cache_check(ctx, cache, layer, q, B, theta, hit, cos_out, as_stream(stream));
}

ts_status ts_score(ts_ctx* ctx, const float* q, const void* k_pool, const int32_t* page_table,
                   const int32_t* seq_lens, int B, const uint8_t* skip, float scale, float* vote,
                   int64_t vote_stride, void* stream) {
  if (!ctx || !q || !k_pool || !page_table || !seq_lens || !vote) return TS_ERR_INVALID_ARG;
  if (B < 1 || B > ctx->cfg.max_batch || vote_stride < ctx->max_tokens) return TS_ERR_SHAPE;
  if (std::isnan(scale)) return TS_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(k_pool) % 16 != 0) return TS_ERR_INVALID_ARG;
  ScoreCall c{q, k_pool, page_table, seq_lens, skip, B, resolve_scale(ctx, scale), vote, vote_stride};
  return launch_score(ctx, c, as_stream(stream));
}

ts_status ts_score_fn(ts_ctx* ctx, const ts_select_params* params, const float* q, const void* k_pool,
                      const int32_t* page_table, const int32_t* seq_lens, int B, const uint8_t* skip,
                      float* vote, int64_t vote_stride, void* stream) {
  if (!ctx || !q || !k_pool || !page_table || !seq_lens || !vote || !valid_params(params))
    return TS_ERR_INVALID_ARG;
  if (B < 1 || B > ctx->cfg.max_batch || vote_stride < ctx->max_tokens) return TS_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(k_pool) % 16 != 0) return TS_ERR_INVALID_ARG;
  ScoreCall c{q, k_pool, page_table, seq_lens, skip, B, resolve_scale(ctx, params->softmax_scale), vote,
              vote_stride};
  c.fn = params->score_fn;
  c.k = params->k;
  c.n_sink = params->n_sink;
  c.n_local = params->n_local;
  return launch_score(ctx, c, as_stream(stream));
}

ts_status ts_select(ts_ctx* ctx, ts_cache* cache, int layer, const float* q, const float* vote,
                    int64_t vote_stride, const int32_t* seq_lens, int B, const uint8_t* hit,
                    const ts_select_params* params, int32_t* idx, int64_t idx_stride, int32_t* count,
                    void* stream) {
  if (!ctx || !vote || !seq_lens || !idx || !count || !valid_params(params)) return TS_ERR_INVALID_ARG;
  if (B < 1 || B > ctx->cfg.max_batch || vote_stride < ctx->max_tokens || idx_stride < 1) return TS_ERR_SHAPE;
  if (hit && !cache) return TS_ERR_INVALID_ARG;
  if (cache) {
    if (cache->ctx != ctx || !q) return TS_ERR_INVALID_ARG;
    if (layer < 0 || layer >= cache->n_layers) return TS_ERR_SHAPE;
  }
  SelectCall c{cache, layer, q, vote, vote_stride, seq_lens, B, hit, *params, idx, idx_stride, count};
  return launch_select(ctx, c, as_stream(stream));
}

ts_status ts_sparse_attend(ts_ctx* ctx, const float* q, const void* k_pool, const void* v_pool,
                           const int32_t* page_table, const int32_t* idx, int64_t idx_stride,
                           const int32_t* count, int B, float scale, float* out, float* lse, void* stream) {
  if (!ctx || !q || !k_pool || !v_pool || !page_table || !idx || !count || !out) return TS_ERR_INVALID_ARG;
  if (B < 1 || B > ctx->cfg.max_batch || idx_stride < 1) return TS_ERR_SHAPE;
  if (std::isnan(scale)) return TS_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(k_pool) % 16 != 0 || reinterpret_cast<uintptr_t>(v_pool) % 16 != 0)
    return TS_ERR_INVALID_ARG;
  AttendCall c{q, k_pool, v_pool, page_table, idx, idx_stride, count, B, resolve_scale(ctx, scale), out, lse};
  return launch_attend(ctx, c, as_stream(stream));
}

ts_status ts_decode_step(ts_ctx* ctx, ts_cache* cache, int layer, const float* q, const void* k_pool,
                         const void* v_pool, const int32_t* page_table, const int32_t* seq_lens, int B,
                         const ts_select_params* params, float* vote, int64_t vote_stride, int32_t* idx,
                         int64_t idx_stride, int32_t* count, float* out, float* lse, uint8_t* hit,
                         void* stream) {
  if (!ctx || !q || !k_pool || !v_pool || !page_table || !seq_lens || !idx || !count || !out ||
      !valid_params(params))
    return TS_ERR_INVALID_ARG;
  if (B < 1 || B > ctx->cfg.max_batch || idx_stride < 1) return TS_ERR_SHAPE;
  if (cache && (cache->ctx != ctx || layer < 0 || layer >= cache->n_layers)) return TS_ERR_INVALID_ARG;
  if (!vote) {
    vote = ctx->vote;
    vote_stride = ctx->max_tokens;
  }
  if (vote_stride < ctx->max_tokens) return TS_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(k_pool) % 16 != 0 || reinterpret_cast<uintptr_t>(v_pool) % 16 != 0)
    return TS_ERR_INVALID_ARG;
  cudaStream_t s = as_stream(stream);
  const float scale = resolve_scale(ctx, params->softmax_scale);
  const bool use_cache = cache != nullptr && params->theta <= 1.f;
  uint8_t* hbuf = hit ? hit : ctx->hit;
  ts_status st = TS_OK;
  if (ctx->use_step && step_supported(ctx->cfg) && B <= 64 && params->score_fn == TS_SCORE_HEAD_SOFT_VOTE) {
    // one persistent cooperative kernel for the whole step
    if (!use_cache && hit && cudaMemsetAsync(hit, 0, B, s) != cudaSuccess) return TS_ERR_CUDA;
    StepCall sc{};
    sc.phases = kPhaseScore | kPhaseSelect | kPhaseAttend | (use_cache ? kPhaseCheck : 0);
    sc.B = B;
    sc.q = q;
    sc.k_pool = k_pool;
    sc.v_pool = v_pool;
    sc.page_table = page_table;
    sc.seq_lens = seq_lens;
    sc.scale = scale;
    sc.theta = params->theta;
    sc.hit_in = nullptr;
    sc.hit_out = use_cache ? hbuf : nullptr;
    sc.cache = cache;
    sc.layer = layer;
    sc.params = *params;
    sc.vote = vote;
    sc.vote_stride = vote_stride;
    sc.idx = idx;
    sc.idx_stride = idx_stride;
    sc.count = count;
    sc.out = out;
    sc.lse = lse;
    st = launch_step(ctx, sc, s);
    if (ctx->debug) std::fprintf(stderr, "ts decode step: persistent kernel -> %s\n", ts_status_str(st));
    if (st != TS_ERR_COOP_UNAVAILABLE) return st;
    ctx->use_step = false;  // the multi-kernel path below from now on
  }
  if (use_cache) {
    st = launch_cache_check(ctx, cache, layer, q, B, params->theta, hbuf, nullptr, s);
    if (st != TS_OK) return st;
  } else if (hit) {
    if (cudaMemsetAsync(hit, 0, B, s) != cudaSuccess) return TS_ERR_CUDA;
  }
  const uint8_t* skip = use_cache ? hbuf : nullptr;
  ScoreCall sc{q, k_pool, page_table, seq_lens, skip, B, scale, vote, vote_stride};
  sc.fn = params->score_fn;
  sc.k = params->k;
  sc.n_sink = params->n_sink;
  sc.n_local = params->n_local;
  st = launch_score(ctx, sc, s);
  if (st != TS_OK) return st;
  SelectCall sel{cache, layer, q, vote, vote_stride, seq_lens, B, skip, *params, idx, idx_stride, count};
  st = launch_select(ctx, sel, s);
  if (st != TS_OK) return st;
  AttendCall ac{q, k_pool, v_pool, page_table, idx, idx_stride, count, B, scale, out, lse};
  return launch_attend(ctx, ac, s);
}

ts_status ts_prefill_chunk(ts_ctx* ctx, const float* q, int c, const void* k_pool, const void* v_pool,
                           const int32_t* page_table, const int32_t* seq_lens, int B, const ts_select_params* params,
                           float* vote, int64_t vote_stride, int32_t* idx, int64_t idx_stride, int32_t* count,
                           float* out, float* lse, void* stream) {
  if (!ctx || !q || !k_pool || !v_pool || !page_table || !seq_lens || !idx || !count || !out ||
      !valid_params(params))
    return TS_ERR_INVALID_ARG;
  if (params->mode != TS_SELECT_TOPK || params->score_fn != TS_SCORE_HEAD_SOFT_VOTE) return TS_ERR_INVALID_ARG;
  if (c < 1 || B < 1 || B > ctx->cfg.max_batch || idx_stride < 1) return TS_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(k_pool) % 16 != 0 || reinterpret_cast<uintptr_t>(v_pool) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(q) % 16 != 0)
    return TS_ERR_INVALID_ARG;
  if (!chunk_attend_supported(ctx->cfg)) return TS_ERR_UNSUPPORTED;
  if (!vote) {
    vote = ctx->vote;
    vote_stride = ctx->max_tokens;
  }
  if (vote_stride < ctx->max_tokens) return TS_ERR_SHAPE;
  cudaStream_t s = as_stream(stream);
  const float scale = resolve_scale(ctx, params->softmax_scale);
  // (1) the mean query of every chunk
  ts_status st = launch_chunk_mean(ctx, q, c, B, ctx->qmean, s);
  if (st != TS_OK) return st;
  // (2) one selection from it: score, vote and top-k (the persistent kernel without its attention)
  st = TS_ERR_COOP_UNAVAILABLE;
  if (ctx->use_step && step_supported(ctx->cfg) && B <= 64) {
    StepCall sc{};
    sc.phases = kPhaseScore | kPhaseSelect;
    sc.B = B;
    sc.q = ctx->qmean;
    sc.k_pool = k_pool;
    sc.v_pool = v_pool;
    sc.page_table = page_table;
    sc.seq_lens = seq_lens;
    sc.scale = scale;
    sc.theta = 2.f;
    sc.params = *params;
    sc.vote = vote;
    sc.vote_stride = vote_stride;
    sc.idx = idx;
    sc.idx_stride = idx_stride;
    sc.count = count;
    st = launch_step(ctx, sc, s);
    if (st != TS_OK && st != TS_ERR_COOP_UNAVAILABLE) return st;
  }
  if (st != TS_OK) {
    ScoreCall scc{ctx->qmean, k_pool, page_table, seq_lens, nullptr, B, scale, vote, vote_stride};
    st = launch_score(ctx, scc, s);
    if (st != TS_OK) return st;
    SelectCall sel{nullptr, 0, ctx->qmean, vote, vote_stride, seq_lens, B, nullptr, *params, idx, idx_stride, count};
    st = launch_select(ctx, sel, s);
    if (st != TS_OK) return st;
  }
  // (3) the chunk's queries attend causally to the shared selection, on the tensor cores
  ChunkAttendCall ac{q, c, k_pool, v_pool, page_table, seq_lens, idx, idx_stride, count, B, scale, out, lse};
  return launch_chunk_attend(ctx, ac, s);
}

ts_status ts_append_kv(ts_ctx* ctx, const void* k_new, const void* v_new, const int32_t* page_table,
                       const int32_t* seq_lens, int B, void* k_pool, void* v_pool, void* stream) {
  if (!ctx || !k_new || !v_new || !page_table || !seq_lens || !k_pool || !v_pool) return TS_ERR_INVALID_ARG;
  if (B < 1 || B > ctx->cfg.max_batch) return TS_ERR_SHAPE;
  for (const void* p : {k_new, v_new, static_cast<const void*>(k_pool), static_cast<const void*>(v_pool)})
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return TS_ERR_INVALID_ARG;
  return launch_append_kv(ctx, k_new, v_new, page_table, seq_lens, B, k_pool, v_pool, as_stream(stream));
}

ts_status ts_select_blocks(ts_ctx* ctx, const float* vote, int64_t vote_stride, const int32_t* seq_lens, int B,
                           int block, int budget, int32_t* idx, int64_t idx_stride, int32_t* count, void* stream) {
  if (!ctx || !vote || !seq_lens || !idx || !count) return TS_ERR_INVALID_ARG;
  if (block < 1 || budget < 0) return TS_ERR_INVALID_ARG;
  if (B < 1 || B > ctx->cfg.max_batch || vote_stride < ctx->max_tokens || idx_stride < 1) return TS_ERR_SHAPE;
  return launch_select_blocks(ctx, vote, vote_stride, seq_lens, B, block, budget, idx, idx_stride, count,
                              as_stream(stream));
}

ts_status ts_debug_phase_ns(ts_ctx* ctx, uint64_t* out64, void* stream) {
  if (!ctx || !out64) return TS_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return TS_ERR_CUDA;
  if (cudaMemcpy(out64, ctx->phase_ns, 64 * sizeof(uint64_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return TS_ERR_CUDA;
  return cudaMemset(ctx->phase_ns, 0, 64 * sizeof(uint64_t)) == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}

ts_status ts_kernel_count(ts_ctx* ctx, int64_t* out) {
  if (!ctx || !out) return TS_ERR_INVALID_ARG;
  *out = ctx->kernels;
  return TS_OK;
}

ts_status ts_profile_enable(ts_ctx* ctx, int on) {
  if (!ctx) return TS_ERR_INVALID_ARG;
  if (on) {
    for (auto& b : ctx->prof) {
      if (!b.begin && cudaEventCreate(&b.begin) != cudaSuccess) return TS_ERR_CUDA;
      if (!b.end && cudaEventCreate(&b.end) != cudaSuccess) return TS_ERR_CUDA;
    }
  }
  ctx->prof_on = on != 0;
  return TS_OK;
}

ts_status ts_profile_read(ts_ctx* ctx, ts_profile* out, int keep) {
  if (!ctx || !out) return TS_ERR_INVALID_ARG;
  for (int i = 0; i < ctx->prof_used; ++i) {
    ProfBracket& b = ctx->prof[i];
    if (!b.recorded) continue;
    if (cudaEventSynchronize(b.end) != cudaSuccess) return TS_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, b.begin, b.end) != cudaSuccess) return TS_ERR_CUDA;
    out->ms[b.family] += ms;
    out->launches[b.family] += 1;
  }
  if (!keep) ctx->prof_used = 0;
  return TS_OK;
}

ts_status ts_set_wait_limit(ts_ctx* ctx, uint64_t ns) {
  if (!ctx || ns == 0) return TS_ERR_INVALID_ARG;
  ctx->wait_ns = ns;
  return TS_OK;
}

ts_status ts_inject_barrier_skip(ts_ctx* ctx, int cta, int barrier) {
  if (!ctx || cta < 0 || barrier < 0) return TS_ERR_INVALID_ARG;
  ctx->inject_skip_cta = cta;
  ctx->inject_skip_barrier = barrier;
  return TS_OK;
}

ts_status ts_get_status(ts_ctx* ctx, ts_status* device_status, void* stream) {
  if (!ctx || !device_status) return TS_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return TS_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, ctx->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return TS_ERR_CUDA;
  if (cudaMemset(ctx->status, 0, sizeof(int)) != cudaSuccess) return TS_ERR_CUDA;
  *device_status = static_cast<ts_status>(v);
  return TS_OK;
}

}  // extern "C"
