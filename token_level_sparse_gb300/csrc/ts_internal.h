// Host-side internals of libtokenselect: context, cache and the launchers each
// kernel file exports to the C ABI layer.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/tokenselect.h"

namespace ts {

constexpr int kStepFlagCap = 8192;   // persistent kernel: most tokens of one CTA's page range
constexpr int kPage = 16;            // tokens per page (the only page size compiled)
constexpr int kScorePagesPerCta = 16;  // pages of one sequence per score CTA
constexpr int kSelThreads = 512;     // select kernels: threads per CTA
constexpr int kSelPerThread = 8;     // consecutive tokens per thread
constexpr int kSelChunk = kSelThreads * kSelPerThread;
constexpr int kAttnMaxSplits = 64;   // CTAs per (sequence, KV head) in the attention

// Per-sequence state of the radix selection (device resident).
struct SelState {
  uint32_t prefix;               // fixed high bits of the threshold
  uint32_t mask;                 // which bits of prefix are fixed
  int32_t k_rem;                 // top-k: tokens still to take at/under prefix
  int32_t n_gt;                  // tokens strictly above the prefix range
  unsigned long long mass_rem;   // top-p: fixed-point mass still to reach
  int32_t all;                   // 1: every token of the domain is selected
  int32_t ties;                  // tokens equal to the threshold to take (by index)
};

struct ChunkCount {              // per selection chunk, written by the count pass
  int gt_all, eq_all, gt_cand, eq_cand, eq_pre;
};

}  // namespace ts

namespace ts {
struct ProfBracket {
  cudaEvent_t begin = nullptr, end = nullptr;
  int family = 0;
  bool recorded = false;  // both events were recorded
};
constexpr int kProfMax = 256;
}  // namespace ts

struct ts_ctx {
  ts_config cfg;
  int device = 0;
  int num_sms = 0;
  int max_tokens = 0;            // max_pages_per_seq * page size
  int score_max_chunks = 0;      // score CTAs per sequence (upper bound)
  int sel_max_chunks = 0;        // selection chunks per sequence (upper bound)
  int attn_splits = 0;           // attention CTAs per (sequence, KV head)
  // device scratch
  int* status = nullptr;                 // first device error since last read
  float* logits = nullptr;               // [max_batch][H][max_tokens]
  float2* partials = nullptr;            // [max_batch][score_max_chunks][H]  (max, sum)
  float2* stats = nullptr;               // [max_batch][H]  (max, 1/sum)
  unsigned* counters = nullptr;          // last-CTA counters, kCounterSlots per sequence
  ts::SelState* sel_state = nullptr;     // [max_batch]
  unsigned* hist = nullptr;              // [max_batch][2048]
  unsigned long long* mass_hist = nullptr;  // [max_batch][2048]
  ts::ChunkCount* chunk_counts = nullptr;   // [max_batch][sel_max_chunks]
  float* attn_part = nullptr;            // [max_batch][H_kv][attn_splits][G*(D+2)]
  float* vote = nullptr;                 // [max_batch][max_tokens] (decode step)
  uint8_t* hit = nullptr;                // [max_batch] (decode step)
  float* qmean = nullptr;                // [max_batch][H][d] mean query of a prefill chunk
  int32_t* blk_len = nullptr;            // [max_batch] block counts (block-level selection)
  int32_t* blk_idx = nullptr;            // [max_batch][max_tokens] selected blocks, then [max_batch] counts
  int32_t* sel_rows = nullptr;           // persistent kernel: per CTA, its selected tokens [kStepFlagCap]
  int64_t kernels = 0;           // kernel launches issued
  // persistent decode-step kernel
  int step_grid = 0;                     // CTAs of the cooperative launch (0: not yet sized)
  int64_t logits_floats = 0;             // size of `logits` (also the step kernel's spill area)
  float2* step_partials = nullptr;       // [max_batch][num_sms][tile pages (1 or 2)][H]
  unsigned* step_hist = nullptr;         // [3][max_batch][2048]
  unsigned long long* step_mass = nullptr;  // [3][max_batch][2048]
  unsigned* cand_n = nullptr;            // [max_batch]
  unsigned long long* cands = nullptr;   // [max_batch][2048]
  int* cta_cnt = nullptr;                // [max_batch][num_sms][3]
  float* apart = nullptr;                // attention partials: o [B][H][parts][num_sms][d / parts], (max, sum) [B][H][even]
  struct KMap {                          // encoded TMA tensor maps of recent K and V pools
    const void* pool = nullptr;
    int64_t num_pages = 0;
    alignas(64) unsigned char map[128];
  } kmaps[16];
  int kmap_next = 0;
  float* step_wpart = nullptr;           // per SM: CUDA-core scan (max, sum exp) pairs, see the persistent kernel
  unsigned* gsync = nullptr;             // grid barrier state (4 words)
  unsigned long long* phase_ns = nullptr;  // [64] phase boundary times of the last step kernel
  bool use_step = true;                  // the persistent kernel is available
  int page_shift = 4;                    // log2 of the page size (16 tokens, or 1)
  int range_attend = 1;                  // top-p attention over each CTA's range: 0 never, 1 when dense, 2 always
  bool range_tc = false;                 // ... with P.V on the tensor cores (measured slower: opt-in)
  // settings read once at ts_create (environment) or set through the C ABI
  bool debug = false;                    // TS_DEBUG: launch diagnostics on stderr
  bool no_tc = false;                    // TOKENSELECT_NO_TC=1: CUDA-core scan only
  bool scan_claim = false;               // TOKENSELECT_SCAN_CLAIM=1: scan pages claimed from a counter
  int64_t l2_budget = 0;                 // TOKENSELECT_L2_BUDGET_MB: logits one scan wave keeps in L2 (0: default)
  uint64_t wait_ns = 1000000000ull;      // bound on every wait of the persistent kernel (ts_set_wait_limit)
  int inject_skip_cta = -1;              // ts_inject_barrier_skip: one launch, CTA leaves at a barrier
  int inject_skip_barrier = -1;
  // kernel timing
  bool prof_on = false;
  int prof_used = 0;
  ts::ProfBracket prof[ts::kProfMax];
};

struct ts_cache {
  ts_ctx* ctx = nullptr;
  int n_layers = 0;
  int capacity = 0;
  float* cq = nullptr;           // [n_layers][max_batch][H*d]
  int32_t* ct = nullptr;         // [n_layers][max_batch][capacity]
  int32_t* ct_count = nullptr;   // [n_layers][max_batch]
  uint8_t* filled = nullptr;     // [n_layers][max_batch]
};

namespace ts {

// Counter slots per sequence: [0] score, [1] select, [2 .. 2+H_kv) attention.
constexpr int kCounterSlots = 2 + 64;
constexpr int kMaxScanWarps = 16;  // warps of the persistent step kernel's scan
constexpr int kStepHistPerSeq = 16384 + 128 + 2048 + 64;  // persistent kernel radix histogram bins per sequence
constexpr int kMaxScanG = 8;       // query heads per KV head the persistent kernel supports

struct ScoreCall {
  const float* q;
  const void* k_pool;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const uint8_t* skip;
  int B;
  float scale;
  float* vote;
  int64_t vote_stride;
  int fn = TS_SCORE_HEAD_SOFT_VOTE;   // selection function (TS_SCORE_*)
  int k = 0, n_sink = 0, n_local = 0; // the hard vote's per-head top-k
};

struct SelectCall {
  ts_cache* cache;
  int layer;
  const float* q;
  const float* vote;
  int64_t vote_stride;
  const int32_t* seq_lens;
  int B;
  const uint8_t* hit;
  ts_select_params params;
  int32_t* idx;
  int64_t idx_stride;
  int32_t* count;
};

struct AttendCall {
  const float* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* page_table;
  const int32_t* idx;
  int64_t idx_stride;
  const int32_t* count;
  int B;
  float scale;
  float* out;
  float* lse;
};

struct StepCall {
  int phases;            // TS_PHASE_* bits
  int B;
  const float* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* page_table;
  const int32_t* seq_lens;
  float scale;
  float theta;
  const uint8_t* hit_in;
  uint8_t* hit_out;
  ts_cache* cache;
  int layer;
  ts_select_params params;
  float* vote;
  int64_t vote_stride;
  int32_t* idx;
  int64_t idx_stride;
  int32_t* count;
  float* out;
  float* lse;
};
constexpr int kPhaseCheck = 1, kPhaseScore = 2, kPhaseSelect = 4, kPhaseAttend = 8;

struct ChunkAttendCall {   // causal attention of a prefill chunk's c queries over one index set
  const float* q;          // [B][c][H][d]
  int c;
  const void* k_pool;
  const void* v_pool;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int32_t* idx;
  int64_t idx_stride;
  const int32_t* count;
  int B;
  float scale;
  float* out;              // [B][c][H][d]
  float* lse;              // [B][c][H] or null
};

// Head geometries with a compiled kernel: (kv type flag, element type, d, H_kv, G).
#define TS_STEP_GEOMETRIES(X)             \
  X(TS_KV_F32, float, 64, 4, 1)           \
  X(TS_KV_F32, float, 64, 2, 4)           \
  X(TS_KV_F32, float, 128, 8, 4)          \
  X(TS_KV_BF16, __nv_bfloat16, 128, 8, 4) \
  X(TS_KV_BF16, __nv_bfloat16, 128, 4, 7) \
  X(TS_KV_BF16, __nv_bfloat16, 128, 8, 1) \
  X(TS_KV_BF16, __nv_bfloat16, 64, 4, 2)  \
  X(TS_KV_BF16, __nv_bfloat16, 128, 2, 8)

bool step_supported(const ts_config& c);
ts_status launch_step(ts_ctx* ctx, const StepCall& a, cudaStream_t s);
bool score_supported(const ts_config& c);
ts_status launch_score(ts_ctx* ctx, const ScoreCall& a, cudaStream_t s);
ts_status launch_select(ts_ctx* ctx, const SelectCall& a, cudaStream_t s);
ts_status launch_attend(ts_ctx* ctx, const AttendCall& a, cudaStream_t s);
bool chunk_attend_supported(const ts_config& c);
ts_status launch_append_kv(ts_ctx* ctx, const void* k_new, const void* v_new, const int32_t* page_table,
                           const int32_t* seq_lens, int B, void* k_pool, void* v_pool, cudaStream_t s);
ts_status launch_select_blocks(ts_ctx* ctx, const float* vote, int64_t vote_stride, const int32_t* seq_lens, int B,
                               int block, int budget, int32_t* idx, int64_t idx_stride, int32_t* count,
                               cudaStream_t s);
ts_status launch_chunk_mean(ts_ctx* ctx, const float* q, int c, int B, float* qm, cudaStream_t s);
ts_status launch_chunk_attend(ts_ctx* ctx, const ChunkAttendCall& c, cudaStream_t s);
ts_status launch_cache_check(ts_ctx* ctx, ts_cache* cache, int layer, const float* q, int B,
                             float theta, uint8_t* hit, float* cos_out, cudaStream_t s);
ts_status launch_cache_reset(ts_cache* cache, cudaStream_t s);

inline ts_status cuda_status(cudaError_t e) { return e == cudaSuccess ? TS_OK : TS_ERR_CUDA; }

// Raises one kernel's dynamic shared-memory limit once per device (so no
// attribute call happens inside a stream capture after the first launch on
// that device). Templated on the kernel itself: one flag set per kernel.
// The flag word is atomic: callers on several host threads may race here (the attribute
// call itself is idempotent).
template <auto Kernel>
inline bool ensure_smem(size_t bytes, int device) {
  static std::atomic<unsigned long long> done{0ull};  // one bit per device
  const unsigned long long bit = 1ull << (device & 63);
  if (done.load(std::memory_order_acquire) & bit) return true;
  if (cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
    return false;
  done.fetch_or(bit, std::memory_order_acq_rel);
  return true;
}

// Brackets the launches made during its lifetime with a pair of timing events
// when the context's profiling is on.
class ProfScope {
 public:
  ProfScope(ts_ctx* ctx, int family, cudaStream_t s) : s_(s) {
    if (!ctx->prof_on || ctx->prof_used >= kProfMax) return;
    b_ = &ctx->prof[ctx->prof_used];
    if (!b_->begin || !b_->end) {  // events are made by ts_profile_enable, never during a capture
      b_ = nullptr;
      return;
    }
    ++ctx->prof_used;
    b_->family = family;
    b_->recorded = false;
    // Inside a stream capture only an "external" record becomes an event-record
    // node that each graph replay executes.
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s_, &cs) != cudaSuccess) cs = cudaStreamCaptureStatusNone;
    flags_ = cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
    if (cudaEventRecordWithFlags(b_->begin, s_, flags_) != cudaSuccess) b_ = nullptr;
  }
  ~ProfScope() {
    if (b_) b_->recorded = cudaEventRecordWithFlags(b_->end, s_, flags_) == cudaSuccess;
  }
  ProfScope(const ProfScope&) = delete;
  ProfScope& operator=(const ProfScope&) = delete;

 private:
  ProfBracket* b_ = nullptr;
  cudaStream_t s_;
  unsigned flags_ = cudaEventRecordDefault;
};

}  // namespace ts
