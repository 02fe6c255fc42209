// Token selection over the head soft vote: top-k (TokenSelect deep notes,
// "Head soft vote": TopK of the summed vote) or the top-p mass variant
// (SequenceO1 blog, section 3.2), united with the sink tokens and the local
// window (TokenSelect review, section 4.2, "2K selected + 512 local"), plus
// the Selection Cache refresh of Algorithm 1 (deep notes, Appendix).
//
// Votes are non-negative, so their fp32 bit patterns order like the values.
// The threshold is found by a three-pass radix select over the bit pattern
// (11, 11, 10 bits). Each pass builds integer histograms per CTA, adds them
// into one per-sequence histogram with integer atomics (order-free, hence
// deterministic), and the last CTA picks the digit holding the crossing.
// For top-p the histogram also carries the vote mass in 2^-40 fixed point,
// so the mass sums are exact integers too. Equal votes at the threshold are
// taken in index order by a final count + write pass.
#include <algorithm>

#include "ts_common.cuh"

namespace ts {
namespace {

constexpr int kBins = 2048;
constexpr float kFx = 1099511627776.0f;  // 2^40

__device__ __forceinline__ unsigned long long to_fx(float v) { return __float2ull_rz(v * kFx); }

struct SelKArgs {
  const float* vote;
  int64_t vote_stride;
  const int32_t* seq_lens;
  int max_tokens;
  const uint8_t* hit;
  int mode, k, n_sink, n_local;
  unsigned long long target_fx;  // top-p: p * H in fixed point
  int take_all_topp;             // top-p with p >= 1
  SelState* state;
  unsigned* hist;
  unsigned long long* mass_hist;
  unsigned* counters;
  ChunkCount* chunk_counts;
  int max_chunks;
  int32_t* idx;
  int64_t idx_stride;
  int32_t* count;
  // Selection Cache entry of this layer (null when no cache)
  float* cq;
  int32_t* ct;
  int32_t* ct_count;
  uint8_t* filled;
  int cap;
  const float* q;
  int HD;
  int* status;
  int signed_keys;     // scores of either sign (the logit-sum selection function): ordered keys
};

// The radix key of a score: its bit pattern for non-negative votes (the order of the values),
// the order-preserving key of either sign otherwise.
__device__ __forceinline__ uint32_t sel_key(float v, int signed_keys) {
  return signed_keys ? ordered_key(v) : __float_as_uint(v);
}

// Length of sequence b, or -1 (recorded as an error) when out of range.
__device__ __forceinline__ int seq_len(const SelKArgs& a, int b) {
  const int n = a.seq_lens[b];
  if (n < 0 || n > a.max_tokens) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_error(a.status, TS_ERR_SEQ_LEN);
    return -1;
  }
  return n;
}

__device__ __forceinline__ void sel_domain(const SelKArgs& a, int n, int& lo, int& hi, int& s_end, int& ls) {
  budget_segments(n, a.n_sink, a.n_local, s_end, ls);
  if (a.mode == TS_SELECT_TOPK) {
    lo = s_end;
    hi = ls;
  } else {
    lo = 0;
    hi = n;
  }
}

// Block-wide exclusive scan of one int per thread (blockDim.x == kSelThreads).
__device__ __forceinline__ int block_excl_scan(int x, int* warp_tot, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = x;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(kFull, inc, d);
    if (lane >= d) inc += o;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int nw = kSelThreads / 32;
    int w = lane < nw ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(kFull, wi, d);
      if (lane >= d) wi += o;
    }
    if (lane < nw) warp_tot[lane] = wi - w;
    if (lane == nw - 1) warp_tot[32] = wi;
  }
  __syncthreads();
  const int r = warp_tot[warp] + inc - x;
  total = warp_tot[32];
  __syncthreads();
  return r;
}

template <int MODE>
__global__ void __launch_bounds__(kSelThreads) sel_pass_kernel(SelKArgs a, int pass) {
  const int b = blockIdx.y;
  if (a.hit && a.hit[b]) return;
  const int n = seq_len(a, b);
  if (n < 0) return;
  int lo, hi, s_end, ls;
  sel_domain(a, n, lo, hi, s_end, ls);
  const int len = hi - lo;
  const int nchunks = (len + kSelChunk - 1) / kSelChunk;
  SelState st;
  if (pass == 0) {
    st.prefix = 0u;
    st.mask = 0u;
    st.k_rem = a.k;
    st.n_gt = 0;
    st.mass_rem = a.target_fx;
    st.ties = 0;
    st.all = (MODE == TS_SELECT_TOPK) ? (len <= a.k) : (a.take_all_topp != 0);
    if (MODE == TS_SELECT_TOPK && a.k <= 0 && len > 0) {
      // nothing to take: a threshold above every finite vote
      if (blockIdx.x == 0 && threadIdx.x == 0) {
        st.prefix = 0xffffffffu;
        st.mask = 0xffffffffu;
        a.state[b] = st;
      }
      return;
    }
    if (st.all || len == 0) {
      if (blockIdx.x == 0 && threadIdx.x == 0) {
        st.all = 1;
        a.state[b] = st;
      }
      return;
    }
  } else {
    st = a.state[b];
    if (st.all || st.mask == 0xffffffffu) return;
  }
  if ((int)blockIdx.x >= nchunks) return;
  const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
  const int nbins = pass == 2 ? 1024 : kBins;
  __shared__ unsigned sh[kBins];
  __shared__ unsigned long long smh[MODE == TS_SELECT_TOPP ? kBins : 1];
  __shared__ int s_last;
  const int tid = threadIdx.x;
  for (int i = tid; i < nbins; i += kSelThreads) {
    sh[i] = 0u;
    if (MODE == TS_SELECT_TOPP) smh[i] = 0ull;
  }
  __syncthreads();
  const float* vb = a.vote + (size_t)b * a.vote_stride;
  const int c0 = lo + blockIdx.x * kSelChunk, c1 = min(hi, c0 + kSelChunk);
  for (int t = c0 + tid; t < c1; t += kSelThreads) {
    const float v = vb[t];
    const uint32_t key = sel_key(v, a.signed_keys);
    if ((key & st.mask) == st.prefix) {
      const int bin = (key >> shift) & (nbins - 1);
      atomicAdd(&sh[bin], 1u);
      if (MODE == TS_SELECT_TOPP) atomicAdd(&smh[bin], to_fx(v));
    }
  }
  __syncthreads();
  unsigned* gh = a.hist + (size_t)b * kBins;
  unsigned long long* gm = a.mass_hist + (size_t)b * kBins;
  for (int i = tid; i < nbins; i += kSelThreads) {
    if (sh[i]) {
      atomicAdd(&gh[i], sh[i]);
      if (MODE == TS_SELECT_TOPP) atomicAdd(&gm[i], smh[i]);
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&a.counters[(size_t)b * kCounterSlots + 1], 1u) == (unsigned)(nchunks - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid < 32) {
    // lane l covers bins [nbins-(l+1)*per, nbins-l*per), lane 0 the top range
    const int lane = tid;
    const int per = nbins / 32;
    unsigned cnt = 0;
    unsigned long long ms = 0;
    for (int j = 0; j < per; ++j) {
      const int bin = nbins - 1 - (lane * per + j);
      cnt += __ldcg(&gh[bin]);
      if (MODE == TS_SELECT_TOPP) ms += __ldcg(&gm[bin]);
    }
    unsigned ic = cnt;
    unsigned long long im = ms;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const unsigned oc = __shfl_up_sync(kFull, ic, d);
      const unsigned long long om = __shfl_up_sync(kFull, im, d);
      if (lane >= d) {
        ic += oc;
        im += om;
      }
    }
    const unsigned ec = ic - cnt;
    const unsigned long long em = im - ms;
    const unsigned need_c = (unsigned)st.k_rem;
    const unsigned long long need_m = st.mass_rem;
    const bool crosses = (MODE == TS_SELECT_TOPK) ? (ec < need_c && ic >= need_c) : (em < need_m && im >= need_m);
    const unsigned ballot = __ballot_sync(kFull, crosses);
    if (ballot == 0u) {
      // only possible for top-p when the fixed-point total falls short: keep everything
      if (lane == 0) {
        st.all = 1;
        a.state[b] = st;
      }
    } else if (lane == __ffs(ballot) - 1) {
      unsigned cb = ec;
      unsigned long long mb = em;
      for (int j = 0; j < per; ++j) {
        const int bin = nbins - 1 - (lane * per + j);
        const unsigned hc = __ldcg(&gh[bin]);
        const unsigned long long hm = (MODE == TS_SELECT_TOPP) ? __ldcg(&gm[bin]) : 0ull;
        const bool here = (MODE == TS_SELECT_TOPK) ? (cb + hc >= need_c) : (mb + hm >= need_m);
        if (here) {
          st.prefix |= (uint32_t)bin << shift;
          st.mask |= (uint32_t)(nbins - 1) << shift;
          st.n_gt += (int)cb;
          if (MODE == TS_SELECT_TOPK) {
            st.k_rem = (int)(need_c - cb);
            if (pass == 2) st.ties = st.k_rem;
          } else {
            st.mass_rem = need_m - mb;
            if (pass == 2) {
              const unsigned long long tfx = to_fx(__uint_as_float(st.prefix));
              const unsigned long long t = tfx ? (st.mass_rem + tfx - 1) / tfx : (unsigned long long)hc;
              st.ties = (int)(t < hc ? t : hc);
            }
          }
          break;
        }
        cb += hc;
        mb += hm;
      }
      a.state[b] = st;
    }
  }
  __syncthreads();
  for (int i = tid; i < kBins; i += kSelThreads) {
    gh[i] = 0u;
    if (MODE == TS_SELECT_TOPP) gm[i] = 0ull;
  }
  if (tid == 0) a.counters[(size_t)b * kCounterSlots + 1] = 0u;
}

__global__ void __launch_bounds__(kSelThreads) sel_count_kernel(SelKArgs a) {
  const int b = blockIdx.y;
  if (a.hit && a.hit[b]) return;
  const int n = seq_len(a, b);
  if (n < 0) return;
  int lo, hi, s_end, ls;
  sel_domain(a, n, lo, hi, s_end, ls);
  const int nchunks = (hi - lo + kSelChunk - 1) / kSelChunk;
  if ((int)blockIdx.x >= nchunks) return;
  const SelState st = a.state[b];
  const int c0 = lo + blockIdx.x * kSelChunk, c1 = min(hi, c0 + kSelChunk);
  int gt_all = 0, eq_all = 0, gt_cand = 0, eq_cand = 0, eq_pre = 0;
  const float* vb = a.vote + (size_t)b * a.vote_stride;
  for (int t = c0 + threadIdx.x; t < c1; t += kSelThreads) {
    const uint32_t key = sel_key(vb[t], a.signed_keys);
    const bool gt = st.all || key > st.prefix;
    const bool eq = !st.all && key == st.prefix;
    const bool cand = t >= s_end && t < ls;
    gt_all += gt;
    eq_all += eq;
    gt_cand += gt && cand;
    eq_cand += eq && cand;
    eq_pre += eq && t < s_end;
  }
  __shared__ int red[5][kSelThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  gt_all = warp_sum_i(gt_all);
  eq_all = warp_sum_i(eq_all);
  gt_cand = warp_sum_i(gt_cand);
  eq_cand = warp_sum_i(eq_cand);
  eq_pre = warp_sum_i(eq_pre);
  if (lane == 0) {
    red[0][warp] = gt_all;
    red[1][warp] = eq_all;
    red[2][warp] = gt_cand;
    red[3][warp] = eq_cand;
    red[4][warp] = eq_pre;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    ChunkCount cc{0, 0, 0, 0, 0};
    for (int w = 0; w < kSelThreads / 32; ++w) {
      cc.gt_all += red[0][w];
      cc.eq_all += red[1][w];
      cc.gt_cand += red[2][w];
      cc.eq_cand += red[3][w];
      cc.eq_pre += red[4][w];
    }
    a.chunk_counts[(size_t)b * a.max_chunks + blockIdx.x] = cc;
  }
}

__device__ __forceinline__ int clampi(int x, int lo, int hi) { return x < lo ? lo : (x > hi ? hi : x); }

__global__ void __launch_bounds__(kSelThreads) sel_write_kernel(SelKArgs a) {
  const int b = blockIdx.y;
  if (a.hit && a.hit[b]) return;
  const int n = seq_len(a, b);
  if (n < 0) return;
  int lo, hi, s_end, ls;
  sel_domain(a, n, lo, hi, s_end, ls);
  const int nchunks = (hi - lo + kSelChunk - 1) / kSelChunk;
  const int c = blockIdx.x;
  if (c >= max(nchunks, 1)) return;
  const SelState st = a.state[b];
  __shared__ int warp_tot[33];
  __shared__ int s_pref[4];  // eq before, sel_all before, sel_cand before (this chunk), totals below
  __shared__ int s_tot[2];
  const int tid = threadIdx.x;

  // ---- prefix over the chunks before this one, and the totals
  int eq_run = 0, all_run = 0, cand_run = 0;
  if (tid == 0) {
    s_pref[0] = s_pref[1] = s_pref[2] = 0;
  }
  for (int base = 0; base < nchunks; base += kSelThreads) {
    const int cc_i = base + tid;
    ChunkCount cc{0, 0, 0, 0, 0};
    if (cc_i < nchunks) cc = a.chunk_counts[(size_t)b * a.max_chunks + cc_i];
    int tot;
    const int eqb = eq_run + block_excl_scan(cc.eq_all, warp_tot, tot);
    eq_run += tot;
    const int sel_all = cc.gt_all + clampi(st.ties - eqb, 0, cc.eq_all);
    const int sel_cand = cc.gt_cand + clampi(st.ties - eqb - cc.eq_pre, 0, cc.eq_cand);
    int tot_a, tot_c;
    const int ab = all_run + block_excl_scan(sel_all, warp_tot, tot_a);
    const int cb = cand_run + block_excl_scan(sel_cand, warp_tot, tot_c);
    all_run += tot_a;
    cand_run += tot_c;
    if (cc_i == c) {
      s_pref[0] = eqb;
      s_pref[1] = ab;
      s_pref[2] = cb;
    }
  }
  if (tid == 0) {
    s_tot[0] = all_run;
    s_tot[1] = cand_run;
  }
  __syncthreads();
  const int tot_all = s_tot[0], tot_cand = s_tot[1];
  const int total = s_end + tot_cand + (n - ls);
  const bool fits = total <= a.idx_stride;
  const bool cache_fits = a.ct != nullptr && tot_all <= a.cap;
  int32_t* ib = a.idx + (size_t)b * a.idx_stride;
  int32_t* ctb = a.ct ? a.ct + (size_t)b * a.cap : nullptr;

  if (c == 0 && tid == 0) {
    if (!fits) set_error(a.status, TS_ERR_CAPACITY);
    a.count[b] = fits ? total : 0;
    if (a.ct) {
      if (!cache_fits) set_error(a.status, TS_ERR_CAPACITY);
      a.ct_count[b] = cache_fits ? tot_all : 0;
      a.filled[b] = cache_fits ? 1 : 0;
    }
  }
  if (c == 0) {
    if (fits) {
      for (int j = tid; j < s_end; j += kSelThreads) ib[j] = j;
      for (int j = tid; j < n - ls; j += kSelThreads) ib[s_end + tot_cand + j] = ls + j;
    }
    if (a.cq) {
      const float* qb = a.q + (size_t)b * a.HD;
      float* cqb = a.cq + (size_t)b * a.HD;
      for (int j = tid; j < a.HD; j += kSelThreads) cqb[j] = qb[j];
    }
  }
  if (nchunks == 0) return;

  // ---- this chunk: thread t owns kSelPerThread consecutive tokens
  const float* vb = a.vote + (size_t)b * a.vote_stride;
  const int c0 = lo + c * kSelChunk, c1 = min(hi, c0 + kSelChunk);
  const int t0 = c0 + tid * kSelPerThread;
  uint32_t keys[kSelPerThread];
  int n_eq = 0;
#pragma unroll
  for (int i = 0; i < kSelPerThread; ++i) {
    const int t = t0 + i;
    keys[i] = t < c1 ? sel_key(vb[t], a.signed_keys) : 0u;
    n_eq += (t < c1 && !st.all && keys[i] == st.prefix);
  }
  int dummy;
  int eq_rank = s_pref[0] + block_excl_scan(n_eq, warp_tot, dummy);
  bool sel[kSelPerThread];
  int n_all = 0, n_cand = 0;
#pragma unroll
  for (int i = 0; i < kSelPerThread; ++i) {
    const int t = t0 + i;
    bool s = false;
    if (t < c1) {
      if (st.all || keys[i] > st.prefix) {
        s = true;
      } else if (keys[i] == st.prefix) {
        s = eq_rank < st.ties;
        ++eq_rank;
      }
    }
    sel[i] = s;
    n_all += s;
    n_cand += s && t >= s_end && t < ls;
  }
  int pa = s_pref[1] + block_excl_scan(n_all, warp_tot, dummy);
  int pc = s_pref[2] + block_excl_scan(n_cand, warp_tot, dummy);
#pragma unroll
  for (int i = 0; i < kSelPerThread; ++i) {
    if (!sel[i]) continue;
    const int t = t0 + i;
    if (cache_fits) ctb[pa] = t;
    ++pa;
    if (t >= s_end && t < ls) {
      if (fits) ib[s_end + pc] = t;
      ++pc;
    }
  }
}

// Cache hit: index set = sinks + cached part inside [s_end, local_start) + window.
__global__ void sel_refresh_kernel(SelKArgs a) {
  const int b = blockIdx.x;
  if (!a.hit || !a.hit[b]) return;
  const int n = seq_len(a, b);
  if (n < 0) return;
  int s_end, ls;
  budget_segments(n, a.n_sink, a.n_local, s_end, ls);
  const int32_t* ctb = a.ct + (size_t)b * a.cap;
  __shared__ int s_lo, s_hi;
  if (threadIdx.x == 0) {
    const int cnt = a.filled[b] ? a.ct_count[b] : 0;
    int l = 0, r = cnt;  // first entry >= s_end
    while (l < r) {
      const int m = (l + r) >> 1;
      if (ctb[m] < s_end) l = m + 1; else r = m;
    }
    s_lo = l;
    r = cnt;  // first entry >= ls
    while (l < r) {
      const int m = (l + r) >> 1;
      if (ctb[m] < ls) l = m + 1; else r = m;
    }
    s_hi = l;
  }
  __syncthreads();
  const int m = s_hi - s_lo;
  const int total = s_end + m + (n - ls);
  int32_t* ib = a.idx + (size_t)b * a.idx_stride;
  if (total > a.idx_stride) {
    if (threadIdx.x == 0) {
      set_error(a.status, TS_ERR_CAPACITY);
      a.count[b] = 0;
    }
    return;
  }
  for (int j = threadIdx.x; j < s_end; j += blockDim.x) ib[j] = j;
  for (int j = threadIdx.x; j < m; j += blockDim.x) ib[s_end + j] = ctb[s_lo + j];
  for (int j = threadIdx.x; j < n - ls; j += blockDim.x) ib[s_end + m + j] = ls + j;
  if (threadIdx.x == 0) a.count[b] = total;
}

}  // namespace

ts_status launch_select(ts_ctx* ctx, const SelectCall& c, cudaStream_t s) {
  const ts_config& cfg = ctx->cfg;
  SelKArgs a;
  a.vote = c.vote;
  a.vote_stride = c.vote_stride;
  a.seq_lens = c.seq_lens;
  a.max_tokens = ctx->max_tokens;
  a.hit = c.hit;
  a.mode = c.params.mode;
  a.k = c.params.k;
  a.n_sink = c.params.n_sink;
  a.n_local = c.params.n_local;
  const double target = (double)c.params.top_p * (double)cfg.n_q_heads * 1099511627776.0;
  a.target_fx = (unsigned long long)ceil(target);
  if (a.target_fx == 0ull) a.target_fx = 1ull;
  a.take_all_topp = c.params.top_p >= 1.0f;
  a.state = ctx->sel_state;
  a.hist = ctx->hist;
  a.mass_hist = ctx->mass_hist;
  a.counters = ctx->counters;
  a.chunk_counts = ctx->chunk_counts;
  a.max_chunks = ctx->sel_max_chunks;
  a.idx = c.idx;
  a.idx_stride = c.idx_stride;
  a.count = c.count;
  a.HD = cfg.n_q_heads * cfg.head_dim;
  a.q = c.q;
  a.status = ctx->status;
  a.signed_keys = c.params.score_fn == TS_SCORE_LOGIT_SUM ? 1 : 0;
  if (c.cache) {
    const size_t mb = (size_t)cfg.max_batch;
    a.cq = c.cache->cq + (size_t)c.layer * mb * a.HD;
    a.ct = c.cache->ct + (size_t)c.layer * mb * c.cache->capacity;
    a.ct_count = c.cache->ct_count + (size_t)c.layer * mb;
    a.filled = c.cache->filled + (size_t)c.layer * mb;
    a.cap = c.cache->capacity;
  } else {
    a.cq = nullptr;
    a.ct = nullptr;
    a.ct_count = nullptr;
    a.filled = nullptr;
    a.cap = 0;
  }
  ProfScope ps(ctx, TS_PROF_SELECT, s);
  ctx->kernels += 5 + (c.hit ? 1 : 0);
  if (c.hit) sel_refresh_kernel<<<c.B, 256, 0, s>>>(a);
  const dim3 grid(ctx->sel_max_chunks, c.B);
  for (int pass = 0; pass < 3; ++pass) {
    if (a.mode == TS_SELECT_TOPK)
      sel_pass_kernel<TS_SELECT_TOPK><<<grid, kSelThreads, 0, s>>>(a, pass);
    else
      sel_pass_kernel<TS_SELECT_TOPP><<<grid, kSelThreads, 0, s>>>(a, pass);
  }
  sel_count_kernel<<<grid, kSelThreads, 0, s>>>(a);
  sel_write_kernel<<<grid, kSelThreads, 0, s>>>(a);
  return cuda_status(cudaGetLastError());
}

}  // namespace ts

// ------------------------------------------------ block-level selection contrast
//
// The selection granularity the method argues against (TokenSelect review,
// figure 2(b), observation 1: block-level methods such as InfLLM keep or drop
// whole blocks of consecutive tokens): blocks of `block` tokens are scored by
// their largest vote, the budget / block best blocks are taken (ties to the
// lower block) by the same radix top-k, and every token of them is selected.

namespace ts {
namespace {

// bscore[b][j] = max of the votes of block j of sequence b; nblk[b] = its block count
__global__ void block_max_kernel(const float* vote, int64_t vote_stride, const int32_t* seq_lens, int max_tokens,
                                 int block, float* bscore, int64_t bs_stride, int32_t* nblk, int* status) {
  const int b = blockIdx.y;
  int n = seq_lens[b];
  if (n < 0 || n > max_tokens) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_error(status, TS_ERR_SEQ_LEN);
    n = 0;
  }
  const int nb = (n + block - 1) / block;
  if (blockIdx.x == 0 && threadIdx.x == 0) nblk[b] = nb;
  const float* vb = vote + (size_t)b * vote_stride;
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < nb; j += gridDim.x * blockDim.x) {
    float m = 0.f;                       // votes are >= 0
    const int t1 = min(n, (j + 1) * block);
    for (int t = j * block; t < t1; ++t) m = fmaxf(m, vb[t]);
    bscore[(size_t)b * bs_stride + j] = m;
  }
}

// the tokens of the selected blocks (ascending block indices) as an ascending token list
__global__ void block_expand_kernel(const int32_t* bidx, int64_t bidx_stride, const int32_t* bcount,
                                    const int32_t* seq_lens, int max_tokens, int block, int32_t* idx,
                                    int64_t idx_stride, int32_t* count, int* status) {
  const int b = blockIdx.x;
  int n = seq_lens[b];
  if (n < 0 || n > max_tokens) n = 0;
  const int nsel = max(0, bcount[b]);
  const int32_t* bl = bidx + (size_t)b * bidx_stride;
  int total = 0;
  if (nsel > 0) {
    const int last = bl[nsel - 1];
    total = (nsel - 1) * block + (min(n, (last + 1) * block) - last * block);
  }
  if (total > idx_stride) {
    if (threadIdx.x == 0) {
      set_error(status, TS_ERR_CAPACITY);
      count[b] = 0;
    }
    return;
  }
  for (int i = threadIdx.x; i < total; i += blockDim.x) {
    const int j = i / block;                     // only the last selected block can be ragged
    idx[(size_t)b * idx_stride + i] = bl[j] * block + (i % block);
  }
  if (threadIdx.x == 0) count[b] = total;
}

}  // namespace

ts_status launch_select_blocks(ts_ctx* ctx, const float* vote, int64_t vote_stride, const int32_t* seq_lens, int B,
                               int block, int budget, int32_t* idx, int64_t idx_stride, int32_t* count,
                               cudaStream_t s) {
  const int mt = ctx->max_tokens;
  // block scores in the logit scratch, block counts and the selected blocks in the selection scratch
  float* bscore = ctx->logits;
  int32_t* nblk = ctx->blk_len;
  int32_t* bidx = ctx->blk_idx;
  ctx->kernels += 2;
  block_max_kernel<<<dim3(std::min(1024, (mt / block + 255) / 256 + 1), B), 256, 0, s>>>(
      vote, vote_stride, seq_lens, mt, block, bscore, mt, nblk, ctx->status);
  if (cudaGetLastError() != cudaSuccess) return TS_ERR_CUDA;
  SelectCall sel{};
  sel.cache = nullptr;
  sel.layer = 0;
  sel.q = nullptr;
  sel.vote = bscore;
  sel.vote_stride = mt;
  sel.seq_lens = nblk;
  sel.B = B;
  sel.hit = nullptr;
  sel.params.mode = TS_SELECT_TOPK;
  sel.params.k = budget / block;
  sel.params.n_sink = 0;
  sel.params.n_local = 0;
  sel.params.top_p = 1.f;
  sel.params.theta = 2.f;
  sel.params.softmax_scale = 0.f;
  sel.params.score_fn = TS_SCORE_HEAD_SOFT_VOTE;
  sel.idx = bidx;
  sel.idx_stride = mt;
  sel.count = bidx + (size_t)ctx->cfg.max_batch * mt;   // counts after the lists
  ts_status st = launch_select(ctx, sel, s);
  if (st != TS_OK) return st;
  block_expand_kernel<<<B, 256, 0, s>>>(bidx, mt, sel.count, seq_lens, mt, block, idx, idx_stride, count,
                                        ctx->status);
  return cuda_status(cudaGetLastError());
}

}  // namespace ts
