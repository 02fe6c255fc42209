/*
 * tokenselect.h - C ABI of the token-level KV selection decode path (sm_103a).
 *
 * The method: TokenSelect ("TokenSelect: Efficient Long-Context Inference and
 * Length Extrapolation for LLMs via Dynamic Token-Level KV Cache Selection").
 * One decode step of one layer is, per sequence of the batch:
 *
 *   1. Selection Cache check: cos(Q, C_Q) >= theta reuses the cached indices
 *      (deep notes, Appendix Algorithm 1; review, section 3.2).
 *   2. Paged dot product: l[h][i] = alpha <q_h, K_{h/G}[i]> over all N cached
 *      tokens of the paged cache (deep notes, Appendix Algorithm 2).
 *   3. Head soft vote: v[i] = sum_h softmax_h(l[h])[i] (deep notes, "Head soft
 *      vote", equation T_head-soft-vote).
 *   4. Selection: TopK(v) over the candidates [s, N-w), or the shortest
 *      (vote desc, index asc) prefix with mass >= p*H, united with the sinks
 *      [0, s) and the local window [N-w, N) (review, section 4.2, "2K+512").
 *   5. Sparse attention over the selected tokens (deep notes, "Formalising
 *      selective sparse attention", equation for O-hat).
 *
 * Conventions for every call below:
 *  - Tensor arguments are DEVICE pointers owned by the caller. The library
 *    never frees them. A context owns its own device scratch; a cache handle
 *    owns C_Q and C_T. Both are freed by their destroy call.
 *  - Layouts are dense row-major. KV pools are [num_pages][H_kv][P][d] (fp32
 *    or bf16, 16-byte aligned base); token i of sequence b lives in page
 *    page_table[b * max_pages_per_seq + i / P] at slot i % P (page tables are
 *    int32 [B][max_pages_per_seq], entries past a sequence unused). Queries are
 *    fp32 [B][H][d]. Query head h reads KV head h / (H / H_kv).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *    stream) and returns before it runs. Argument and shape errors are
 *    reported synchronously by the return value, before anything is enqueued.
 *    Errors found on the device (a page id outside the pool, an output that
 *    does not fit, a wait that ran out) are recorded in the context's status
 *    word and read back with ts_get_status. Nothing aborts or traps.
 *  - A context is bound to the device current at ts_create and is not thread
 *    safe: calls on one context must be serialised by the caller, and calls
 *    that share a context's scratch must go to one stream (or be ordered).
 */
#ifndef TOKENSELECT_H
#define TOKENSELECT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ts_ctx ts_ctx;     /* opaque; library-owned */
typedef struct ts_cache ts_cache; /* opaque; library-owned */

typedef enum {
  TS_OK = 0,
  TS_ERR_INVALID_ARG = 1,      /* null pointer, bad enum, negative size        */
  TS_ERR_SHAPE = 2,            /* sizes beyond what the context was created for */
  TS_ERR_UNSUPPORTED = 3,      /* head geometry without a compiled kernel       */
  TS_ERR_CUDA = 4,             /* a CUDA runtime call failed                    */
  TS_ERR_PAGE_OOB = 5,         /* device: page-table entry outside the pool     */
  TS_ERR_CAPACITY = 6,         /* device: selection larger than its buffer      */
  TS_ERR_TIMEOUT = 7,          /* device: a bounded wait ran out                */
  TS_ERR_COOP_UNAVAILABLE = 8, /* a cooperative launch was refused              */
  TS_ERR_SEQ_LEN = 9,          /* device: seq_lens[b] < 0 or above the maximum  */
  TS_ERR_SCRATCH_LIMIT = 10    /* beyond the fixed scratch of the no-alloc call */
} ts_status;

enum { TS_KV_F32 = 0, TS_KV_BF16 = 1 };
enum { TS_SELECT_TOPK = 0, TS_SELECT_TOPP = 1 };
/* Selection function whose per-token score the top-k ranks (TokenSelect deep
 * notes, "Evolution of the selection function"; TokenSelect review, section
 * 3.1 and the ablation of section 4.4 / table 4):
 *  HEAD_SOFT_VOTE  v_i = sum_h softmax(scale q_h.K^T)_i  (the method);
 *  LOGIT_SUM       s_i = sum_h scale q_h.k_{g(h),i}: plain TopK(Q.K^T) of the
 *                  concatenated heads, dominated by high-norm heads (signed);
 *  HEAD_HARD_VOTE  c_i = number of query heads whose own top-k over the
 *                  candidates [s, N-w) (ties to the lower index) holds i.
 * The two ablations serve top-k only and run on the multi-kernel path. */
enum { TS_SCORE_HEAD_SOFT_VOTE = 0, TS_SCORE_LOGIT_SUM = 1, TS_SCORE_HEAD_HARD_VOTE = 2 };

/* Shape of the model's attention and of the caller's pools, fixed per context. */
typedef struct {
  int n_q_heads;          /* H                                                  */
  int n_kv_heads;         /* H_kv, divides H                                    */
  int head_dim;           /* d (64 or 128)                                      */
  int page_size;          /* P tokens per page: 16, or 1 for a token-granular   */
                          /* pool (one token per page; separate kernels only)   */
  int kv_dtype;           /* TS_KV_F32 or TS_KV_BF16                            */
  int max_batch;          /* largest B of any call                              */
  int max_pages_per_seq;  /* page-table row stride; max tokens = this * P       */
  int64_t num_pages;      /* pool size in pages; larger page ids are errors     */
} ts_config;

/* Selection parameters (review, section 4.2: k = 2048, 4 sinks, 512 local;
 * deep notes, Algorithm 1: theta = 0.9). */
typedef struct {
  int mode;               /* TS_SELECT_TOPK or TS_SELECT_TOPP                   */
  int k;                  /* top-k budget over the candidates                   */
  int n_sink;             /* s: tokens [0, s) always kept                       */
  int n_local;            /* w: tokens [N-w, N) always kept                     */
  float top_p;            /* mass fraction for TOPP; >= 1 keeps every token     */
  float theta;            /* cache threshold; > 1 never hits                    */
  float softmax_scale;    /* alpha; 0 means 1/sqrt(d)                           */
  int score_fn;           /* TS_SCORE_*; 0 (the head soft vote) by default      */
} ts_select_params;

/* Context: validates and records cfg, allocates the device scratch for
 * max_batch sequences of max_pages_per_seq * page_size tokens on the current
 * device. Returns TS_ERR_UNSUPPORTED for a head geometry with no kernel. */
ts_status ts_create(ts_ctx** out, const ts_config* cfg);
ts_status ts_destroy(ts_ctx* ctx);

/* Selection Cache for n_layers layers of max_batch sequences: per (sequence,
 * layer) a first-query flag, C_Q (fp32 H*d) and C_T (int32, `capacity`
 * entries). Starts empty (every first query misses). */
ts_status ts_cache_create(ts_ctx* ctx, ts_cache** out, int n_layers, int capacity);
ts_status ts_cache_destroy(ts_cache* cache);
/* Marks every (sequence, layer) as empty again; enqueued on `stream`. */
ts_status ts_cache_reset(ts_cache* cache, void* stream);

/* Algorithm 1's test for one layer: hit[b] = 1 iff the entry of (b, layer)
 * is filled, and cos(q_b, C_Q) >= theta over the H*d query (fp32).
 * q [B][H][d]; hit uint8 [B]; cos_out fp32 [B] or NULL (NaN when empty). */
ts_status ts_cache_check(ts_ctx* ctx, ts_cache* cache, int layer, const float* q, int B,
                         float theta, uint8_t* hit, float* cos_out, void* stream);

/* Paged dot product + fused per-head softmax normaliser + head soft vote.
 * For each b with skip == NULL or skip[b] == 0:
 *   vote[b * vote_stride + i] = sum_h exp(l[h][i] - L_h),  i < seq_lens[b],
 * with l = scale * <q_h, K_{h/G}[i]> and L_h = log sum_i exp(l[h][i]).
 * The H x N logits are context scratch and are not returned. scale 0 means
 * 1/sqrt(d). seq_lens int32 [B] on the device, each in [0, max_pages_per_seq
 * * page_size]; vote_stride >= max_pages_per_seq * page_size. Entries past
 * seq_lens[b] and skipped rows are left untouched. */
ts_status ts_score(ts_ctx* ctx, const float* q, const void* k_pool, const int32_t* page_table,
                   const int32_t* seq_lens, int B, const uint8_t* skip, float scale,
                   float* vote, int64_t vote_stride, void* stream);

/* The per-token score of one selection function (params->score_fn, TS_SCORE_*)
 * for the top-k of ts_select: HEAD_SOFT_VOTE computes exactly what ts_score
 * does; LOGIT_SUM writes the signed sums of the per-head logits (rank them by
 * passing the same params to ts_select); HEAD_HARD_VOTE runs one top-k per
 * query head over the candidates [s, N-w) of params (k, n_sink, n_local; ties
 * to the lower index) and writes the vote counts as floats (exact small
 * integers, 0 outside the candidates). Every entry i < seq_lens[b] of a row
 * that is not skipped is written; layout and scale as in ts_score. */
ts_status ts_score_fn(ts_ctx* ctx, const ts_select_params* params, const float* q, const void* k_pool,
                      const int32_t* page_table, const int32_t* seq_lens, int B, const uint8_t* skip,
                      float* vote, int64_t vote_stride, void* stream);

/* Selection (top-k or top-p) united with sinks and window, ascending.
 * For each b: if hit != NULL and hit[b] != 0, the index set is rebuilt from
 * the cache entry (cached part within [s, N-w), plus the current sinks and
 * window); otherwise it is selected from vote and, if cache != NULL, the
 * entry of (b, layer) takes the selected part and q_b (Algorithm 1). Ties in
 * the vote go to the lower index. idx int32 [B][idx_stride] receives the
 * count[b] indices; a count above idx_stride (or a selected part above the
 * cache capacity) records TS_ERR_CAPACITY and writes nothing past the end.
 * q may be NULL when cache is NULL. With params->score_fn == LOGIT_SUM the
 * scores are ranked as signed values; top-p needs the head soft vote (its
 * mass is the vote's), else TS_ERR_INVALID_ARG. */
ts_status ts_select(ts_ctx* ctx, ts_cache* cache, int layer, const float* q, const float* vote,
                    int64_t vote_stride, const int32_t* seq_lens, int B, const uint8_t* hit,
                    const ts_select_params* params, int32_t* idx, int64_t idx_stride,
                    int32_t* count, void* stream);

/* Sparse attention: out[b][h] = softmax_i(scale q_h.K_i) V_i over the count[b]
 * indices idx[b * idx_stride + j] (split over the index list, merged by
 * log-sum-exp). out fp32 [B][H][d]; lse fp32 [B][H] or NULL. An empty index
 * list gives out = 0 and lse = -inf. */
ts_status ts_sparse_attend(ts_ctx* ctx, const float* q, const void* k_pool, const void* v_pool,
                           const int32_t* page_table, const int32_t* idx, int64_t idx_stride,
                           const int32_t* count, int B, float scale, float* out, float* lse,
                           void* stream);

/* Sparse attention for callers that cannot allocate device memory: the same
 * computation and the same kernel as ts_sparse_attend, but with no context.
 * The paper has no counterpart; this exists for callers that run where
 * cudaMalloc is unavailable or forbidden - inside a memory pool or arena they
 * do not own, under a framework allocator that must see every allocation, or
 * in a process that has to keep device memory fixed after start-up - and
 * so cannot create a context (ts_create allocates its scratch).
 * Its scratch (split partials, merge counters, a fallback status slot) is one
 * fixed static device array of 4 MiB + 16 KiB in the library, held by every
 * GPU that loads the library until the process exits. Limits: B <= 48,
 * n_kv_heads <= 64 (one merge counter per (sequence, KV head) in the head of
 * the array) and B * H_kv * G * (d + 2) <= 2^20 floats (one split per
 * (sequence, KV head) at that size); beyond them the call returns
 * TS_ERR_SCRATCH_LIMIT and enqueues nothing. A NaN scale returns
 * TS_ERR_INVALID_ARG, as in ts_sparse_attend. It calls no cudaMalloc/cudaFree. The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) and the
 * SM count: make that first call before any stream capture on that device.
 * Every call clears the merge counters, then uses the shared array: calls
 * that overlap on the GPU (other streams, other threads) race on it and must
 * be serialised by the caller. Geometry: n_q_heads, n_kv_heads, head_dim,
 * kv_dtype as in ts_config; pools of num_pages pages; page_table int32
 * [B][max_pages_per_seq]. status: int32 on the device or NULL; receives the
 * first device error (0 otherwise is left unchanged). Other arguments as in
 * ts_sparse_attend. */
ts_status ts_sparse_attend_noalloc(int n_q_heads, int n_kv_heads, int head_dim, int kv_dtype,
                                   const float* q, const void* k_pool, const void* v_pool,
                                   int64_t num_pages, const int32_t* page_table,
                                   int max_pages_per_seq, const int32_t* idx, int64_t idx_stride,
                                   const int32_t* count, int B, float scale, float* out, float* lse,
                                   int32_t* status, void* stream);

/* One whole decode step of one layer, stream-ordered, no host synchronisation:
 * cache check (when cache != NULL and theta <= 1), score and vote for the
 * sequences that miss, selection (and cache update), sparse attention.
 * hit uint8 [B] (may be NULL) receives the cache decisions. vote receives the
 * votes of the missing sequences (may be NULL: context scratch is used).
 * Supported geometries run as one cooperative launch; repeated calls on the
 * same inputs give bit-identical results. params->score_fn other than the
 * head soft vote (the ablations) runs the multi-kernel path with that
 * selection function (the vote buffer then holds its scores); so does a
 * context with one-token pages. Environment switches, read once by
 * ts_create (comparisons and tests): TOKENSELECT_MULTI_KERNEL=1 keeps the
 * multi-kernel path; TOKENSELECT_NO_TC=1 scans on CUDA cores instead of tensor
 * cores; TOKENSELECT_SCAN_CLAIM=1 lets the CTAs claim scan pages from a shared
 * counter when at most two sequences are scanned (faster where SM bandwidth
 * differs, but no longer bit-identical from run to run);
 * TOKENSELECT_L2_BUDGET_MB sets the logit bytes one CUDA-core scan wave may
 * keep in L2; TOKENSELECT_TOPP_ATTEND=gather / range / range_tc fixes the top-p
 * attention (selected tokens shared out over the CTAs; each CTA's own scanned
 * range from the scan's logits, P.V on CUDA cores or on the tensor cores),
 * otherwise chosen per sequence by how dense the selection is; TS_DEBUG prints
 * launch diagnostics. */
ts_status ts_decode_step(ts_ctx* ctx, ts_cache* cache, int layer, const float* q,
                         const void* k_pool, const void* v_pool, const int32_t* page_table,
                         const int32_t* seq_lens, int B, const ts_select_params* params,
                         float* vote, int64_t vote_stride, int32_t* idx, int64_t idx_stride,
                         int32_t* count, float* out, float* lse, uint8_t* hit, void* stream);

/* Appends the current token's K and V rows to the paged pools before a
 * decode step (the harness step of reading R9: the current token is the last
 * cached position). For each b, k_new / v_new [B][H_kv][d] (device, kv_dtype
 * elements, 16-byte aligned) are written to pool[page][g][slot] of position
 * seq_lens[b] - 1, page = page_table[b][(seq_lens[b] - 1) / page_size]. A
 * length outside [1, max tokens] records TS_ERR_SEQ_LEN, a page outside the
 * pool TS_ERR_PAGE_OOB (nothing is written for that sequence). */
ts_status ts_append_kv(ts_ctx* ctx, const void* k_new, const void* v_new, const int32_t* page_table,
                       const int32_t* seq_lens, int B, void* k_pool, void* v_pool, void* stream);

/* Block-level selection, the granularity the method argues against
 * (TokenSelect review, figure 2(b): InfLLM-style methods keep or drop whole
 * blocks; granularity 1 is token-level selection). From the votes of each
 * sequence (non-negative, e.g. from ts_score): blocks of `block` consecutive
 * tokens (the last one ragged) are scored by their largest vote, the
 * budget / block best blocks are taken (ties to the lower block) and every
 * token of them is written to idx [B][idx_stride] ascending, count [B]; a
 * list longer than idx_stride records TS_ERR_CAPACITY. No sinks, window or
 * cache: it serves the recall comparison of the two granularities. */
ts_status ts_select_blocks(ts_ctx* ctx, const float* vote, int64_t vote_stride, const int32_t* seq_lens, int B,
                           int block, int budget, int32_t* idx, int64_t idx_stride, int32_t* count,
                           void* stream);

/* Chunk-wise prefill selection (TokenSelect deep notes, "Optimising the
 * selection frequency of the prefill stage"; review, section 3.2): the c
 * queries of a prefill chunk, q fp32 [B][c][H][d] (16-byte aligned), are
 * averaged into one query per sequence, (1/c) sum_i q[b][i]; that mean query
 * is scored and selects once (head soft vote, top-k over [s, N-w) united
 * with sinks and window, ties to the lower index; no Selection Cache in
 * prefill), writing vote (or context scratch when NULL), idx [B][idx_stride]
 * ascending and count [B] as ts_decode_step does. The chunk's own tokens must
 * already be cached as the last c of seq_lens[b] tokens: query i attends to
 * the selected tokens at positions <= seq_lens[b] - c + i (causal), giving
 * out fp32 [B][c][H][d] and lse fp32 [B][c][H] (or NULL). The attention runs
 * on the tensor cores for bf16 pools with d = 64 or 128 (else
 * TS_ERR_UNSUPPORTED). params must be top-k with the head soft vote. */
ts_status ts_prefill_chunk(ts_ctx* ctx, const float* q, int c, const void* k_pool, const void* v_pool,
                           const int32_t* page_table, const int32_t* seq_lens, int B,
                           const ts_select_params* params, float* vote, int64_t vote_stride,
                           int32_t* idx, int64_t idx_stride, int32_t* count, float* out, float* lse,
                           void* stream);

/* Failure detection (no counterpart in the pages; the library's own safety
 * net). Every wait of the persistent decode-step kernel - its grid barriers
 * and its copy, tensor-core and accumulator waits - gives up after `ns`
 * nanoseconds (default 1 s): the kernel then records TS_ERR_TIMEOUT, raises an
 * abort word that the other CTAs see at their next barrier, waits (bounded)
 * for its own copies in flight, frees its tensor memory and returns, so the
 * context stays usable. The waits of the separate calls (ts_score,
 * ts_sparse_attend) keep the 1 s bound. ns == 0 is TS_ERR_INVALID_ARG. */
ts_status ts_set_wait_limit(ts_ctx* ctx, uint64_t ns);

/* Fault injection for tests of the time-out path: the NEXT persistent
 * decode-step launch of this context makes CTA `cta` leave at its grid
 * barrier number `barrier` (0 = the first) without arriving, so that every
 * other CTA's bounded wait runs out (TS_ERR_TIMEOUT through ts_get_status).
 * Nothing faults, traps or hangs: the run-out is the ordinary bounded-wait
 * path, and the launch after it starts from clean barrier words. The request
 * is consumed by that one launch; a cta beyond the grid injects nothing. */
ts_status ts_inject_barrier_skip(ts_ctx* ctx, int cta, int barrier);

/* Synchronises `stream`, then reads and clears the device status word.
 * *device_status receives TS_OK or the first device error since the last read. */
ts_status ts_get_status(ts_ctx* ctx, ts_status* device_status, void* stream);

/* Static text for a status code. */
const char* ts_status_str(ts_status s);

/* Kernel timing (tracing). While enabled, every kernel launch of the library is
 * bracketed by a pair of CUDA events on its stream, tagged with its family;
 * inside a CUDA graph capture the events become event-record nodes that each
 * replay re-records. At most 256 brackets are held; later ones are dropped. */
enum {
  TS_PROF_CHECK = 0,   /* Selection Cache test                     */
  TS_PROF_SCORE = 1,   /* paged dot product + per-CTA normaliser    */
  TS_PROF_VOTE = 2,    /* head soft vote                            */
  TS_PROF_SELECT = 3,  /* radix selection, refresh and compaction   */
  TS_PROF_ATTEND = 4,  /* sparse attention + merge                  */
  TS_PROF_STEP = 5,    /* the persistent whole-step kernel          */
  TS_PROF_N = 6
};
typedef struct {
  double ms[TS_PROF_N];        /* summed device time per family */
  int64_t launches[TS_PROF_N]; /* brackets summed per family    */
} ts_profile;
ts_status ts_profile_enable(ts_ctx* ctx, int on);
/* Waits for the recorded brackets and ADDS their durations into *out. With
 * keep == 0 the brackets are released; keep != 0 leaves them registered so a
 * replayed CUDA graph can be read again after each replay. */
ts_status ts_profile_read(ts_ctx* ctx, ts_profile* out, int keep);

/* Number of kernel launches this context has issued (or captured into a CUDA
 * graph) since ts_create, counted on the host at each launch. */
ts_status ts_kernel_count(ts_ctx* ctx, int64_t* out);

/* Tracing: %globaltimer values (ns) at which CTA 0 of the last persistent
 * decode-step kernel reached its phase boundaries (0: start, 1: set-up done,
 * 2+3w / 3+3w / 4+3w: wave w scanned / partials written / barrier passed,
 * 20: scoring done, 21: radix levels done, 22: candidates gathered,
 * 23: selection done, 24: attention done, 25: last barrier passed,
 * 26: outputs merged, 27: end; 32..63 finer points inside the phases, see
 * the kernel source; 0 where not reached). Synchronises `stream`, copies 64
 * values to out64 (host) and clears them. */
ts_status ts_debug_phase_ns(ts_ctx* ctx, uint64_t* out64, void* stream);

/* Library version, e.g. 100 for 0.1.0. */
int ts_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TOKENSELECT_H */
