// Paged dot product + per-head softmax normaliser + head soft vote.
//
// TokenSelect deep notes, Appendix Algorithm 2 (Paged Dot Product Kernel):
// per head, the query sits on chip and blocks of cached tokens are brought
// in through the page table to form s = <q, k>. Here one CTA owns a run of
// pages of one sequence. A producer warp streams whole pages (all KV heads,
// 16 tokens, contiguous in the pool) into a shared-memory ring with 1-D bulk
// copies (TMA); eight consumer warps each hold the G queries of one KV head
// in registers, so every K element is read from HBM once and feeds G FMAs.
//
// "Head soft vote" (same page, equation T_head-soft-vote) needs each head's
// normaliser L_h = log sum_i exp(l_hi) over all N tokens before any vote
// exists. Each CTA reduces its tokens to (max, sum) per head; the last CTA of
// a sequence merges them (fixed order, compensated sums) into (M_h, 1/Z_h);
// a second kernel forms v_i = sum_h exp(l_hi - M_h)/Z_h.
#include <cfloat>

#include "ts_common.cuh"

namespace ts {
namespace {

constexpr int cpow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}
constexpr int cclamp(int x, int lo, int hi) { return x < lo ? lo : (x > hi ? hi : x); }

template <typename KT, int D, int HKV, int G>
struct ScoreShape {
  static constexpr int P = kPage;                      // tokens per stage: one 16-token page, or 16 one-token pages
  static constexpr int EPC = KV<KT>::kPerChunk;        // elements per 16-byte chunk
  static constexpr int GP = cpow2(G);                   // heads padded to a power of two
  static constexpr int CPL = (GP * 2 * EPC <= 64) ? 2 : 1;  // chunks per lane (q registers <= 64)
  static constexpr int DPL = EPC * CPL;                 // dims per lane
  static constexpr int LPR = D / DPL;                   // lanes per K row
  static constexpr int RPW = 32 / LPR;                  // rows per warp step
  static constexpr int NCW = 8;                         // consumer warps
  static constexpr int WPH = NCW / HKV;                 // consumer warps per KV head
  static constexpr int ROWS = P / WPH;                  // page rows per consumer warp
  static constexpr int ITERS = ROWS / RPW;
  static constexpr int PPC = kScorePagesPerCta;
  static constexpr int TOK = PPC * P;                   // tokens per CTA
  static constexpr int STAGE_BYTES = HKV * P * D * (int)sizeof(KT);  // 16 tokens, all KV heads
  static constexpr int NST = cclamp(131072 / STAGE_BYTES, 2, 8);
  static constexpr int THREADS = (NCW + 1) * 32;
  static_assert(D % DPL == 0 && 32 % LPR == 0, "row split");
  static_assert(NCW % HKV == 0 && P % WPH == 0 && ROWS % RPW == 0 && ITERS >= 1, "warp split");
  static_assert(GP <= LPR, "head split");
  static_assert(STAGE_BYTES % 16 == 0, "bulk copy size");
  static size_t smem_bytes(int H) {
    return (size_t)NST * STAGE_BYTES + (size_t)H * TOK * sizeof(float) + 2 * NST * sizeof(uint64_t) +
           (NST + 4) * sizeof(int);
  }
};

struct ScoreKArgs {
  const float* q;
  const void* k_pool;
  const int32_t* page_table;
  int pt_stride;
  const int32_t* seq_lens;
  const uint8_t* skip;
  int64_t num_pages;
  float scale;
  int H;
  float* logits;
  int max_tokens;
  float2* partials;
  int max_chunks;
  float2* stats;
  unsigned* counters;
  int* status;
  int page_size;               // 16, or 1 for a token-granular pool
};

template <typename KT, int D, int HKV, int G>
__global__ void __launch_bounds__(ScoreShape<KT, D, HKV, G>::THREADS, 1)
    score_logits_kernel(ScoreKArgs a) {
  using S = ScoreShape<KT, D, HKV, G>;
  extern __shared__ __align__(128) unsigned char smem[];
  const int b = blockIdx.y;
  if (a.skip && a.skip[b]) return;
  const int n = a.seq_lens[b];
  if (n < 0 || n > a.max_tokens) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_error(a.status, TS_ERR_SEQ_LEN);
    return;
  }
  const int n_pages = (n + S::P - 1) / S::P;
  const int n_chunks = (n_pages + S::PPC - 1) / S::PPC;
  const int chunk = blockIdx.x;
  if (chunk >= n_chunks) return;
  const int page0 = chunk * S::PPC;
  const int np = min(S::PPC, n_pages - page0);
  const int tok0 = page0 * S::P;
  const int n_tok = min(n - tok0, np * S::P);
  const int H = a.H;

  unsigned char* stages = smem;
  float* sl = reinterpret_cast<float*>(smem + (size_t)S::NST * S::STAGE_BYTES);  // [H][TOK]
  uint64_t* full = reinterpret_cast<uint64_t*>(sl + (size_t)H * S::TOK);
  uint64_t* empty = full + S::NST;
  int* s_valid = reinterpret_cast<int*>(empty + S::NST);  // [NST]
  int* s_last = s_valid + S::NST;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < S::NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], S::NCW);
    }
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == S::NCW) {
    // ---------------- producer: the warp streams the CTA's stages through the ring (lane 0
    // waits and arms the barrier; with one-token pages each lane fetches one token)
    const unsigned char* pool = static_cast<const unsigned char*>(a.k_pool);
    constexpr uint32_t kRow = D * (uint32_t)sizeof(KT);
    int issued = 0;
    for (int p = 0; p < np; ++p) {
      const int s = p % S::NST;
      int free_ok = 1;
      if (lane == 0 && p >= S::NST) free_ok = mbar_wait(&empty[s], ((p / S::NST) - 1) & 1);
      if (!__shfl_sync(kFull, free_ok, 0)) {
        if (lane == 0) set_error(a.status, TS_ERR_TIMEOUT);
        break;
      }
      unsigned char* dst = stages + (size_t)s * S::STAGE_BYTES;
      if (a.page_size == S::P) {
        // one page: every KV head's 16 rows, contiguous in the pool and in the stage
        if (lane == 0) {
          const int page = a.page_table[(size_t)b * a.pt_stride + page0 + p];
          const bool ok = page >= 0 && (int64_t)page < a.num_pages;
          s_valid[s] = ok;
          if (ok) {
            mbar_arrive_expect_tx(&full[s], S::STAGE_BYTES);
            bulk_g2s(dst, pool + (size_t)page * S::STAGE_BYTES, S::STAGE_BYTES, &full[s]);
          } else {
            set_error(a.status, TS_ERR_PAGE_OOB);
            mbar_arrive(&full[s]);
          }
        }
      } else {
        // token-granular pool (one token per page): the stage's 16 tokens come from their own
        // pages, token r's rows [H_kv][d] (contiguous in its page) to token-major rows (r, g)
        // of the stage; tokens past the sequence are not copied (their logits are masked)
        const int t0 = tok0 + p * S::P;
        const int nr = min(S::P, n - t0);
        int page = -1;
        if (lane < nr) page = a.page_table[(size_t)b * a.pt_stride + t0 + lane];
        const bool ok = page >= 0 && (int64_t)page < a.num_pages;
        const unsigned good = __ballot_sync(kFull, lane < nr && ok);
        if (lane == 0) {
          const bool all = __popc(good) == nr;
          s_valid[s] = all;
          if (!all) set_error(a.status, TS_ERR_PAGE_OOB);
          mbar_arrive_expect_tx(&full[s], (uint32_t)__popc(good) * HKV * kRow);
        }
        __syncwarp();
        if (lane < nr && ok)
          bulk_g2s(dst + (size_t)lane * HKV * kRow, pool + (size_t)page * HKV * kRow, HKV * kRow, &full[s]);
      }
      ++issued;
    }
    // No copy may still be landing in shared memory when the CTA exits.
    if (lane == 0)
      for (int p = max(0, issued - S::NST); p < issued; ++p) {
        if (!mbar_wait(&full[p % S::NST], (p / S::NST) & 1)) set_error(a.status, TS_ERR_TIMEOUT);
      }
  } else {
    // ---------------- consumers: warp -> (KV head g, rows of each page)
    const int g = warp / S::WPH;
    const int row0 = (warp % S::WPH) * S::ROWS;
    const int lrow = lane / S::LPR, lin = lane % S::LPR;
    float qr[S::GP][S::DPL];
#pragma unroll
    for (int j = 0; j < S::GP; ++j) {
      const float* qh = a.q + ((size_t)b * H + g * G + j) * D;
#pragma unroll
      for (int c = 0; c < S::CPL; ++c)
#pragma unroll
        for (int e = 0; e < S::EPC; ++e)
          qr[j][c * S::EPC + e] = (j < G) ? qh[(lin + c * S::LPR) * S::EPC + e] : 0.f;
    }
    const bool writer = (lin & (S::LPR / S::GP - 1)) == 0;
    const bool token_major = a.page_size != S::P;   // one-token pages: stage rows (token, g)
    for (int p = 0; p < np; ++p) {
      const int s = p % S::NST;
      if (!mbar_wait(&full[s], (p / S::NST) & 1)) {
        set_error(a.status, TS_ERR_TIMEOUT);
        break;
      }
      const bool valid = s_valid[s] != 0;
      const KT* st = reinterpret_cast<const KT*>(stages + (size_t)s * S::STAGE_BYTES);
#pragma unroll
      for (int it = 0; it < S::ITERS; ++it) {
        const int row = row0 + it * S::RPW + lrow;
        const KT* rp = st + (token_major ? (size_t)row * HKV + g : (size_t)g * S::P + row) * D;
        float acc0[S::GP], acc1[S::GP];
#pragma unroll
        for (int j = 0; j < S::GP; ++j) acc0[j] = acc1[j] = 0.f;
#pragma unroll
        for (int c = 0; c < S::CPL; ++c) {
          float kf[S::EPC];
          KV<KT>::unpack(lds128(rp + (lin + c * S::LPR) * S::EPC), kf);
#pragma unroll
          for (int j = 0; j < S::GP; ++j)
#pragma unroll
            for (int e = 0; e < S::EPC; ++e) {
              // two independent chains: by chunk when a lane has two, else by parity
              if ((S::CPL == 2 ? c : (e & 1)) == 0)
                acc0[j] = fmaf(qr[j][c * S::EPC + e], kf[e], acc0[j]);
              else
                acc1[j] = fmaf(qr[j][c * S::EPC + e], kf[e], acc1[j]);
            }
        }
        float v[S::GP];
#pragma unroll
        for (int j = 0; j < S::GP; ++j) v[j] = acc0[j] + acc1[j];
        int which;
        const float dot = transpose_reduce<S::GP, S::LPR>(v, lane, which);
        const int tl = p * S::P + row;
        if (writer && which < G)
          sl[(size_t)(g * G + which) * S::TOK + tl] = (valid && tl < n_tok) ? dot * a.scale : -INFINITY;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  __syncthreads();

  // ---------------- per-head (max, sum exp) of this CTA's tokens; logits out
  constexpr int NW = S::NCW + 1;
  for (int h = warp; h < H; h += NW) {
    const float* row = sl + (size_t)h * S::TOK;
    float m = -INFINITY;
    for (int t = lane; t < n_tok; t += 32) m = fmaxf(m, row[t]);
    m = warp_max(m);
    float z = 0.f;
    if (m > -INFINITY)
      for (int t = lane; t < n_tok; t += 32) z += expf(row[t] - m);
    z = warp_sum(z);
    if (lane == 0) a.partials[((size_t)b * a.max_chunks + chunk) * H + h] = make_float2(m, z);
    float* out = a.logits + ((size_t)b * H + h) * a.max_tokens + tok0;
    for (int t = lane; t < n_tok; t += 32) out[t] = row[t];
  }

  // ---------------- the last CTA of the sequence merges the partials
  __threadfence();
  __syncthreads();
  if (tid == 0) *s_last = atomicAdd(&a.counters[(size_t)b * kCounterSlots], 1u) == (unsigned)(n_chunks - 1);
  __syncthreads();
  if (!*s_last) return;
  __threadfence();
  for (int h = warp; h < H; h += NW) {
    const float2* pp = a.partials + (size_t)b * a.max_chunks * H + h;
    float M = -INFINITY;
    for (int c = lane; c < n_chunks; c += 32) M = fmaxf(M, __ldcg(pp + (size_t)c * H).x);
    M = warp_max(M);
    KahanF kz;
    for (int c = lane; c < n_chunks; c += 32) {
      const float2 mz = __ldcg(pp + (size_t)c * H);
      if (mz.y > 0.f) kz.add(mz.y * expf(mz.x - M));
    }
    const float z = warp_sum_comp(kz.s, -kz.c);
    if (lane == 0) a.stats[(size_t)b * H + h] = make_float2(M, 1.f / z);
  }
  if (tid == 0) a.counters[(size_t)b * kCounterSlots] = 0u;
}

struct VoteKArgs {
  const int32_t* seq_lens;
  const uint8_t* skip;
  int H;
  const float* logits;
  int max_tokens;
  const float2* stats;
  float* vote;
  int64_t vote_stride;
  int fn;              // TS_SCORE_*: soft vote, logit sum, or zeros for the hard vote's counts
};

constexpr int kVoteThreads = 256;
constexpr int kVotePerThread = 4;
constexpr int kVoteTile = kVoteThreads * kVotePerThread;
constexpr int kMaxHeads = 256;

// v_i = sum_h exp(l_hi - M_h) / Z_h, compensated over the heads.
__global__ void __launch_bounds__(kVoteThreads) score_vote_kernel(VoteKArgs a) {
  const int b = blockIdx.y;
  if (a.skip && a.skip[b]) return;
  const int n = a.seq_lens[b];
  const int t0 = blockIdx.x * kVoteTile;
  if (n < 0 || n > a.max_tokens || t0 >= n) return;
  __shared__ float sM[kMaxHeads], sIZ[kMaxHeads];
  for (int h = threadIdx.x; h < a.H; h += blockDim.x) {
    const float2 st = a.stats[(size_t)b * a.H + h];
    sM[h] = st.x;
    sIZ[h] = st.y;
  }
  __syncthreads();
  const float* lb = a.logits + (size_t)b * a.H * a.max_tokens;
#pragma unroll
  for (int i = 0; i < kVotePerThread; ++i) {
    const int t = t0 + i * kVoteThreads + threadIdx.x;
    if (t >= n) break;
    KahanF acc;
    if (a.fn == TS_SCORE_HEAD_SOFT_VOTE) {
      for (int h = 0; h < a.H; ++h) acc.add(expf(lb[(size_t)h * a.max_tokens + t] - sM[h]) * sIZ[h]);
    } else if (a.fn == TS_SCORE_LOGIT_SUM) {
      // plain TopK(Q.K^T) over the concatenated heads: the sum of the per-head logits
      for (int h = 0; h < a.H; ++h) acc.add(lb[(size_t)h * a.max_tokens + t]);
    }   // the hard vote's counts start from zero and are added by hard_vote_kernel
    a.vote[(size_t)b * a.vote_stride + t] = acc.s - acc.c;
  }
}

struct HardVoteKArgs {
  const int32_t* seq_lens;
  const uint8_t* skip;
  int H;
  const float* logits;
  int max_tokens;
  int k, n_sink, n_local;
  float* vote;
  int64_t vote_stride;
};

constexpr int kHardThreads = 1024;

// Head hard vote (TokenSelect deep notes, "Evolution of the selection function":
// TopK(sum_h I(i in TopK(Q^h K^h^T)))): CTA (h, b) finds query head h's own top-k over
// the candidates [s_end, ls) of sequence b and adds one vote to each of its tokens.
// The k-th logit is found by a radix select over the order-preserving 32-bit keys,
// 8 bits per pass from the top (shared-memory histograms); tokens above it are taken,
// and tokens equal to it in index order until k are taken. Votes are added as 1.0f:
// sums of small integers are exact in fp32, so the order of the adds does not matter.
__global__ void __launch_bounds__(kHardThreads) hard_vote_kernel(HardVoteKArgs a) {
  const int h = blockIdx.x, b = blockIdx.y;
  if (a.skip && a.skip[b]) return;
  const int n = a.seq_lens[b];
  if (n < 0 || n > a.max_tokens) return;
  int s_end, ls;
  budget_segments(n, a.n_sink, a.n_local, s_end, ls);
  const int lo = s_end, hi = ls, len = hi - lo;
  if (a.k <= 0 || len <= 0) return;
  float* vb = a.vote + (size_t)b * a.vote_stride;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (len <= a.k) {
    for (int i = lo + tid; i < hi; i += blockDim.x) atomicAdd(&vb[i], 1.f);
    return;
  }
  const float* row = a.logits + ((size_t)b * a.H + h) * a.max_tokens;
  __shared__ unsigned hist[256];
  __shared__ unsigned s_prefix, s_krem;
  __shared__ int wcnt[32];
  uint32_t prefix = 0u, mask = 0u;
  unsigned krem = (unsigned)a.k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0u;
    __syncthreads();
    for (int i = lo + tid; i < hi; i += blockDim.x) {
      const uint32_t key = ordered_key(row[i]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // bins from the top: lane L sums bins 255 - 8L .. 248 - 8L, then a prefix over lanes
      unsigned c = 0;
      for (int j = 0; j < 8; ++j) c += hist[255 - 8 * lane - j];
      unsigned inc = c;
      for (int d = 1; d < 32; d <<= 1) {
        const unsigned o = __shfl_up_sync(kFull, inc, d);
        if (lane >= d) inc += o;
      }
      const unsigned ballot = __ballot_sync(kFull, inc - c < krem && inc >= krem);
      const int L = __ffs(ballot) - 1;   // the domain holds more than k tokens: some lane crosses
      if (ballot == 0u && lane == 0) {   // (unreachable) keep the state well defined
        s_prefix = prefix;
        s_krem = krem;
      }
      if (lane == L) {
        unsigned before = inc - c;
        for (int j = 0; j < 8; ++j) {
          const int bin = 255 - 8 * L - j;
          if (before + hist[bin] >= krem) {
            s_prefix = prefix | ((uint32_t)bin << shift);
            s_krem = krem - before;
            break;
          }
          before += hist[bin];
        }
      }
    }
    __syncthreads();
    prefix = s_prefix;
    krem = s_krem;
    mask |= 255u << shift;
    __syncthreads();
  }
  // prefix is the k-th key; krem tokens equal to it are taken, lowest index first
  unsigned taken = 0;
  for (int base = lo; base < hi; base += blockDim.x) {
    const int i = base + tid;
    const uint32_t key = i < hi ? ordered_key(row[i]) : 0u;
    const bool gt = i < hi && key > prefix, eq = i < hi && key == prefix;
    const unsigned bal = __ballot_sync(kFull, eq);
    if (lane == 0) wcnt[warp] = __popc(bal);
    __syncthreads();
    unsigned before = taken;
    for (int w = 0; w < warp; ++w) before += wcnt[w];
    unsigned tot = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += wcnt[w];
    const unsigned rank = before + __popc(bal & ((1u << lane) - 1u));
    if (gt || (eq && rank < krem)) atomicAdd(&vb[i], 1.f);
    taken += tot;
    __syncthreads();
  }
}

template <typename KT, int D, int HKV, int G>
ts_status run_score(ts_ctx* ctx, const ScoreCall& c, cudaStream_t s) {
  using S = ScoreShape<KT, D, HKV, G>;
  const int H = ctx->cfg.n_q_heads;
  const size_t smem = S::smem_bytes(H);
  auto kern = score_logits_kernel<KT, D, HKV, G>;
  if (!ensure_smem<score_logits_kernel<KT, D, HKV, G>>(S::smem_bytes(HKV * G), ctx->device))  // H = H_kv * G
    return TS_ERR_CUDA;
  ScoreKArgs a;
  a.q = c.q;
  a.k_pool = c.k_pool;
  a.page_table = c.page_table;
  a.pt_stride = ctx->cfg.max_pages_per_seq;
  a.seq_lens = c.seq_lens;
  a.skip = c.skip;
  a.num_pages = ctx->cfg.num_pages;
  a.scale = c.scale;
  a.H = H;
  a.logits = ctx->logits;
  a.max_tokens = ctx->max_tokens;
  a.partials = ctx->partials;
  a.max_chunks = ctx->score_max_chunks;
  a.stats = ctx->stats;
  a.counters = ctx->counters;
  a.status = ctx->status;
  a.page_size = ctx->cfg.page_size;
  {
    ProfScope ps(ctx, TS_PROF_SCORE, s);
    kern<<<dim3(ctx->score_max_chunks, c.B), S::THREADS, smem, s>>>(a);
  }
  ctx->kernels += 2;
  VoteKArgs v{c.seq_lens, c.skip, H, ctx->logits, ctx->max_tokens, ctx->stats, c.vote, c.vote_stride, c.fn};
  {
    ProfScope ps(ctx, TS_PROF_VOTE, s);
    score_vote_kernel<<<dim3((ctx->max_tokens + kVoteTile - 1) / kVoteTile, c.B), kVoteThreads, 0, s>>>(v);
    if (c.fn == TS_SCORE_HEAD_HARD_VOTE) {
      HardVoteKArgs hv{c.seq_lens, c.skip, H, ctx->logits, ctx->max_tokens, c.k, c.n_sink, c.n_local,
                       c.vote, c.vote_stride};
      hard_vote_kernel<<<dim3(H, c.B), kHardThreads, 0, s>>>(hv);
      ctx->kernels += 1;
    }
  }
  return cuda_status(cudaGetLastError());
}

}  // namespace

// Head geometries with a compiled scoring kernel: (kv type, d, H_kv, G).
#define TS_SCORE_GEOMETRIES(X)          \
  X(TS_KV_F32, float, 64, 4, 1)         \
  X(TS_KV_F32, float, 64, 2, 4)         \
  X(TS_KV_F32, float, 128, 8, 4)        \
  X(TS_KV_BF16, __nv_bfloat16, 128, 8, 4) \
  X(TS_KV_BF16, __nv_bfloat16, 128, 4, 7) \
  X(TS_KV_BF16, __nv_bfloat16, 128, 8, 1) \
  X(TS_KV_BF16, __nv_bfloat16, 64, 4, 2)  \
  X(TS_KV_BF16, __nv_bfloat16, 128, 2, 8)

bool score_supported(const ts_config& c) {
  const int G = c.n_kv_heads > 0 ? c.n_q_heads / c.n_kv_heads : 0;
#define X(DT, T, D_, HKV_, G_) \
  if (c.kv_dtype == DT && c.head_dim == D_ && c.n_kv_heads == HKV_ && G == G_) return true;
  TS_SCORE_GEOMETRIES(X)
#undef X
  return false;
}

ts_status launch_score(ts_ctx* ctx, const ScoreCall& a, cudaStream_t s) {
  const ts_config& c = ctx->cfg;
  const int G = c.n_q_heads / c.n_kv_heads;
#define X(DT, T, D_, HKV_, G_) \
  if (c.kv_dtype == DT && c.head_dim == D_ && c.n_kv_heads == HKV_ && G == G_) return run_score<T, D_, HKV_, G_>(ctx, a, s);
  TS_SCORE_GEOMETRIES(X)
#undef X
  return TS_ERR_UNSUPPORTED;
}

}  // namespace ts
