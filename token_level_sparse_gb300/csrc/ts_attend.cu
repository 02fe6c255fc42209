// Selective sparse attention over the selected tokens.
//
// TokenSelect deep notes, "Formalising selective sparse attention", equation
// for O-hat: per head, softmax(q K_sel^T / sqrt(d)) V_sel over the selected
// tokens (which include the current one). Only indices cross from the
// selection (deep notes, "Paged Dot Product Kernel design": O(k) index I/O
// instead of moving 2kd values); the rows are gathered here through the page
// table.
//
// Grid: (split, KV head, sequence). A CTA takes a contiguous slice of the
// index list, stages the K and V rows of 64 tokens at a time into shared
// memory with one 1-D bulk copy per row (all in flight at once, one mbarrier),
// and runs an online softmax for the G query heads of its KV head. The splits
// are merged by log-sum-exp in split order by the last CTA of each
// (sequence, KV head).
#include "ts_common.cuh"

namespace ts {
namespace {

constexpr int cpow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

template <typename KT, int D, int G>
struct AttShape {
  static constexpr int EPC = KV<KT>::kPerChunk;  // elements per 16-byte chunk
  static constexpr int LPT = D / EPC;            // lanes per token row
  static constexpr int TPW = 32 / LPT;           // tokens per warp step
  static constexpr int GP = cpow2(G);
  static constexpr int WARPS = 4;
  static constexpr int THREADS = WARPS * 32;
  static constexpr int GROUPS = WARPS * TPW;     // independent softmax states per CTA
  static constexpr int SUB = 64;                 // tokens staged per round
  static constexpr int ROW_BYTES = D * (int)sizeof(KT);
  static_assert(32 % LPT == 0 && LPT <= 32 && GP <= LPT, "lane split");
  static_assert(ROW_BYTES % 16 == 0, "row copies");
  static constexpr size_t smem_bytes() {
    return 2ull * SUB * ROW_BYTES + (size_t)GROUPS * G * (D + 2) * sizeof(float) + SUB * sizeof(int) + 16;
  }
};

struct AttKArgs {
  const float* q;
  const unsigned char* k_pool;
  const unsigned char* v_pool;
  const int32_t* page_table;
  int pt_stride;
  int page_shift;  // log2 of the page size: 4 (16 tokens) or 0 (one token per page)
  int64_t num_pages;
  int max_tokens;
  const int32_t* idx;
  int64_t idx_stride;
  const int32_t* count;
  int H, HKV;
  float scale;
  float* out;
  float* lse;
  float* part;  // [B][HKV][nsplit][G*(D+2)]
  unsigned* counters;
  int* status;
};

template <typename KT, int D, int G>
__global__ void __launch_bounds__(AttShape<KT, D, G>::THREADS) attend_kernel(AttKArgs a) {
  using S = AttShape<KT, D, G>;
  extern __shared__ __align__(128) unsigned char smem[];
  KT* Ks = reinterpret_cast<KT*>(smem);
  KT* Vs = Ks + S::SUB * D;
  float* mg = reinterpret_cast<float*>(Vs + S::SUB * D);  // [GROUPS][G][D] then m, l
  float* mm = mg + (size_t)S::GROUPS * G * D;             // [GROUPS][G]
  float* ml = mm + S::GROUPS * G;                          // [GROUPS][G]
  int* tokflag = reinterpret_cast<int*>(ml + S::GROUPS * G);
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_last;

  const int split = blockIdx.x, nsplit = gridDim.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cnt = (int)min((int64_t)max(a.count[b], 0), a.idx_stride);  // never read past the index row
  const int per = (cnt + nsplit - 1) / nsplit;
  const int t_begin = min(cnt, split * per), t_end = min(cnt, t_begin + per);
  const int lt = lane % S::LPT;                       // chunk of the row this lane reads
  const int slot = warp * S::TPW + lane / S::LPT;     // token group of this lane

  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  float qr[S::GP][S::EPC];
#pragma unroll
  for (int j = 0; j < S::GP; ++j)
#pragma unroll
    for (int e = 0; e < S::EPC; ++e)
      qr[j][e] = (j < G) ? a.q[((size_t)b * a.H + g * G + j) * D + lt * S::EPC + e] : 0.f;
  float m[G], l[G], o[G][S::EPC];
#pragma unroll
  for (int j = 0; j < G; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int e = 0; e < S::EPC; ++e) o[j][e] = 0.f;
  }
  __syncthreads();

  const int32_t* ib = a.idx + (size_t)b * a.idx_stride;
  const int32_t* pt = a.page_table + (size_t)b * a.pt_stride;
  uint32_t phase = 0;
  bool ok = true;
  for (int s0 = t_begin; s0 < t_end && ok; s0 += S::SUB) {
    const int ns = min(S::SUB, t_end - s0);
    __syncthreads();  // the previous round is fully consumed
    if (tid == 0) mbar_arrive_expect_tx(&bar, 2u * ns * S::ROW_BYTES);
    __syncthreads();
    for (int i = tid; i < 2 * ns; i += S::THREADS) {
      const int j = i >> 1;
      const int t = ib[s0 + j];
      int page = -1;
      if (t >= 0 && t < a.max_tokens) page = pt[t >> a.page_shift];
      const bool valid = page >= 0 && (int64_t)page < a.num_pages;
      const int slot = t & ((1 << a.page_shift) - 1);
      const size_t off = valid ? ((((size_t)page * a.HKV + g) << a.page_shift) + slot) * S::ROW_BYTES : 0;
      if (i & 1) {
        bulk_g2s(Vs + (size_t)j * D, a.v_pool + off, S::ROW_BYTES, &bar);
      } else {
        bulk_g2s(Ks + (size_t)j * D, a.k_pool + off, S::ROW_BYTES, &bar);
        tokflag[j] = valid;
        if (!valid) set_error(a.status, TS_ERR_PAGE_OOB);
      }
    }
    const bool landed = mbar_wait(&bar, phase);
    phase ^= 1u;
    ok = __syncthreads_and(landed) != 0;  // block-uniform
    if (!ok) {
      if (tid == 0) set_error(a.status, TS_ERR_TIMEOUT);
      break;
    }
    for (int j0 = 0; j0 < ns; j0 += S::GROUPS) {
      const int j = j0 + slot;
      const bool act = j < ns;
      const int jj = act ? j : 0;
      float kf[S::EPC], vf[S::EPC];
      KV<KT>::unpack(lds128(Ks + (size_t)jj * D + lt * S::EPC), kf);
      KV<KT>::unpack(lds128(Vs + (size_t)jj * D + lt * S::EPC), vf);
      float acc[S::GP];
#pragma unroll
      for (int h = 0; h < S::GP; ++h) {
        float x = 0.f;
#pragma unroll
        for (int e = 0; e < S::EPC; ++e) x = fmaf(qr[h][e], kf[e], x);
        acc[h] = x;
      }
      int which;
      const float red = transpose_reduce<S::GP, S::LPT>(acc, lane, which);
      const bool live = act && tokflag[jj] != 0;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float dot = __shfl_sync(kFull, red, (lane & ~(S::LPT - 1)) + h * (S::LPT / S::GP));
        if (live) {
          const float s = dot * a.scale;
          const float mn = fmaxf(m[h], s);
          const float corr = expf(m[h] - mn);
          const float p = expf(s - mn);
          l[h] = l[h] * corr + p;
#pragma unroll
          for (int e = 0; e < S::EPC; ++e) o[h][e] = fmaf(p, vf[e], o[h][e] * corr);
          m[h] = mn;
        }
      }
    }
  }
  // In-flight copies must land before shared memory is reused or released.
  if (!ok && tid == 0) mbar_wait(&bar, phase ^ 1u);
  __syncthreads();

  // ---- merge the token groups of this CTA
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int e = 0; e < S::EPC; ++e) mg[((size_t)slot * G + h) * D + lt * S::EPC + e] = o[h][e];
    if (lt == 0) {
      mm[slot * G + h] = m[h];
      ml[slot * G + h] = l[h];
    }
  }
  __syncthreads();
  const int W = G * (D + 2);
  float* pb = a.part + (((size_t)b * a.HKV + g) * nsplit + split) * W;
  for (int i = tid; i < G * D; i += S::THREADS) {
    const int h = i / D;
    float M = -INFINITY;
    for (int r = 0; r < S::GROUPS; ++r) M = fmaxf(M, mm[r * G + h]);
    float num = 0.f, den = 0.f;
    if (M > -INFINITY) {
      for (int r = 0; r < S::GROUPS; ++r) {
        const float w = expf(mm[r * G + h] - M);
        num = fmaf(w, mg[(size_t)r * G * D + i], num);
        den = fmaf(w, ml[r * G + h], den);
      }
    }
    pb[i] = num;
    if ((i % D) == 0) {
      pb[G * D + h] = M;
      pb[G * D + G + h] = den;
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&a.counters[(size_t)b * kCounterSlots + 2 + g], 1u) == (unsigned)(nsplit - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- the last CTA merges the splits in split order
  const float* pg = a.part + ((size_t)b * a.HKV + g) * nsplit * W;
  for (int i = tid; i < G * D; i += S::THREADS) {
    const int h = i / D;
    float M = -INFINITY;
    for (int r = 0; r < nsplit; ++r) M = fmaxf(M, __ldcg(pg + (size_t)r * W + G * D + h));
    float num = 0.f, den = 0.f;
    if (M > -INFINITY) {
      for (int r = 0; r < nsplit; ++r) {
        const float* pr = pg + (size_t)r * W;
        const float w = expf(__ldcg(pr + G * D + h) - M);
        num = fmaf(w, __ldcg(pr + i), num);
        den = fmaf(w, __ldcg(pr + G * D + G + h), den);
      }
    }
    const int qh = g * G + h;
    a.out[((size_t)b * a.H + qh) * D + (i % D)] = den > 0.f ? num / den : 0.f;
    if (a.lse && (i % D) == 0) a.lse[(size_t)b * a.H + qh] = den > 0.f ? M + logf(den) : -INFINITY;
  }
  if (tid == 0) a.counters[(size_t)b * kCounterSlots + 2 + g] = 0u;
}

template <typename KT, int D, int G>
ts_status run_attend(ts_ctx* ctx, const AttendCall& c, cudaStream_t s) {
  using S = AttShape<KT, D, G>;
  const ts_config& cfg = ctx->cfg;
  auto kern = attend_kernel<KT, D, G>;
  const size_t smem = S::smem_bytes();
  if (!ensure_smem<attend_kernel<KT, D, G>>(smem, ctx->device)) return TS_ERR_CUDA;
  AttKArgs a;
  a.q = c.q;
  a.k_pool = static_cast<const unsigned char*>(c.k_pool);
  a.v_pool = static_cast<const unsigned char*>(c.v_pool);
  a.page_table = c.page_table;
  a.pt_stride = cfg.max_pages_per_seq;
  a.page_shift = ctx->page_shift;
  a.num_pages = cfg.num_pages;
  a.max_tokens = ctx->max_tokens;
  a.idx = c.idx;
  a.idx_stride = c.idx_stride;
  a.count = c.count;
  a.H = cfg.n_q_heads;
  a.HKV = cfg.n_kv_heads;
  a.scale = c.scale;
  a.out = c.out;
  a.lse = c.lse;
  a.part = ctx->attn_part;
  a.counters = ctx->counters;
  a.status = ctx->status;
  int nsplit = (2 * ctx->num_sms + cfg.n_kv_heads * c.B - 1) / (cfg.n_kv_heads * c.B);
  nsplit = nsplit < 1 ? 1 : (nsplit > kAttnMaxSplits ? kAttnMaxSplits : nsplit);
  ProfScope ps(ctx, TS_PROF_ATTEND, s);
  ctx->kernels += 1;
  kern<<<dim3(nsplit, cfg.n_kv_heads, c.B), S::THREADS, smem, s>>>(a);
  return cuda_status(cudaGetLastError());
}

}  // namespace

#define TS_ATTEND_GEOMETRIES(X)        \
  X(TS_KV_F32, float, 64, 1)           \
  X(TS_KV_F32, float, 64, 4)           \
  X(TS_KV_F32, float, 128, 4)          \
  X(TS_KV_BF16, __nv_bfloat16, 128, 4) \
  X(TS_KV_BF16, __nv_bfloat16, 128, 7) \
  X(TS_KV_BF16, __nv_bfloat16, 128, 1) \
  X(TS_KV_BF16, __nv_bfloat16, 64, 2)  \
  X(TS_KV_BF16, __nv_bfloat16, 128, 8)

ts_status launch_attend(ts_ctx* ctx, const AttendCall& a, cudaStream_t s) {
  const ts_config& c = ctx->cfg;
  const int G = c.n_q_heads / c.n_kv_heads;
#define X(DT, T, D_, G_) \
  if (c.kv_dtype == DT && c.head_dim == D_ && G == G_) return run_attend<T, D_, G_>(ctx, a, s);
  TS_ATTEND_GEOMETRIES(X)
#undef X
  return TS_ERR_UNSUPPORTED;
}

}  // namespace ts

// ---------------------------------------------------------------------------
// The no-alloc variant of the sparse attention (ts_sparse_attend_noalloc).
// For callers that may not call cudaMalloc: the scratch lives in one fixed
// static device array instead of a context. Layout: [0, 16 KiB) merge
// counters (kCounterSlots per sequence) and a fallback status slot,
// [16 KiB, end) split partials.

namespace ts {
namespace {

// The new token of each sequence (its last cached position, seq_lens[b] - 1) into the paged
// pools: rows k_new / v_new [B][H_kv][d] (element bytes es) to pool[page][g][slot][:], one
// 16-byte chunk per thread.
__global__ void append_kv_kernel(const unsigned char* k_new, const unsigned char* v_new, const int32_t* page_table,
                                 int pt_stride, int page_shift, const int32_t* seq_lens, int max_tokens,
                                 int64_t num_pages, int HKV,
                                 int row_bytes, unsigned char* k_pool, unsigned char* v_pool, int* status) {
  const int b = blockIdx.x;
  const int n = seq_lens[b];
  if (n < 1 || n > max_tokens) {
    if (threadIdx.x == 0) set_error(status, TS_ERR_SEQ_LEN);
    return;
  }
  const int t = n - 1;
  const int page = page_table[(size_t)b * pt_stride + (t >> page_shift)];
  if (page < 0 || (int64_t)page >= num_pages) {
    if (threadIdx.x == 0) set_error(status, TS_ERR_PAGE_OOB);
    return;
  }
  const int cpr = row_bytes / 16;
  for (int i = threadIdx.x; i < 2 * HKV * cpr; i += blockDim.x) {
    const int isv = i / (HKV * cpr), rem = i % (HKV * cpr), g = rem / cpr, ch = rem % cpr;
    const unsigned char* src = (isv ? v_new : k_new) + ((size_t)b * HKV + g) * row_bytes + ch * 16;
    unsigned char* dst = (isv ? v_pool : k_pool) +
                         ((((size_t)page * HKV + g) << page_shift) + (t & ((1 << page_shift) - 1))) * row_bytes + ch * 16;
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  }
}

}  // namespace

ts_status launch_append_kv(ts_ctx* ctx, const void* k_new, const void* v_new, const int32_t* page_table,
                           const int32_t* seq_lens, int B, void* k_pool, void* v_pool, cudaStream_t s) {
  const ts_config& c = ctx->cfg;
  const int row_bytes = c.head_dim * (c.kv_dtype == TS_KV_BF16 ? 2 : 4);
  ctx->kernels += 1;
  append_kv_kernel<<<B, 128, 0, s>>>(static_cast<const unsigned char*>(k_new), static_cast<const unsigned char*>(v_new),
                                     page_table, c.max_pages_per_seq, ctx->page_shift, seq_lens, ctx->max_tokens,
                                     c.num_pages,
                                     c.n_kv_heads, row_bytes, static_cast<unsigned char*>(k_pool),
                                     static_cast<unsigned char*>(v_pool), ctx->status);
  return cuda_status(cudaGetLastError());
}

}  // namespace ts

#include <cmath>
#include <mutex>

namespace ts {
namespace {

constexpr int kNoAllocMaxBatch = 48;
constexpr size_t kNoAllocHeadBytes = 16384;
constexpr size_t kNoAllocPartFloats = size_t(1) << 20;
constexpr size_t kNoAllocBytes = kNoAllocHeadBytes + kNoAllocPartFloats * sizeof(float);
static_assert(kNoAllocMaxBatch * kCounterSlots * sizeof(unsigned) + sizeof(int) <= kNoAllocHeadBytes,
              "counters must fit the head of the array");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

struct NoAllocDevice {
  unsigned char* base = nullptr;  // device address of g_noalloc_scratch
  int num_sms = 0;
};
constexpr int kNoAllocMaxDevices = 64;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];
std::mutex g_noalloc_mu;

// Device address of the array on the current device (looked up once per device).
ts_status noalloc_setup(int device, NoAllocDevice& out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc_dev[device];
  if (!d.base) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return TS_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return TS_ERR_CUDA;
    d.num_sms = sms;
    d.base = static_cast<unsigned char*>(p);
  }
  out = d;
  return TS_OK;
}

template <typename KT, int D, int G>
ts_status run_attend_noalloc(const AttKArgs& proto, int B, int HKV, int device, const NoAllocDevice& dev,
                             cudaStream_t s) {
  using S = AttShape<KT, D, G>;
  const size_t per_split = (size_t)B * HKV * G * (D + 2);
  if (per_split > kNoAllocPartFloats) return TS_ERR_SCRATCH_LIMIT;
  int nsplit = (2 * dev.num_sms + HKV * B - 1) / (HKV * B);
  nsplit = nsplit < 1 ? 1 : (nsplit > kAttnMaxSplits ? kAttnMaxSplits : nsplit);
  const int fit = (int)(kNoAllocPartFloats / per_split);
  if (nsplit > fit) nsplit = fit;
  if (!ensure_smem<attend_kernel<KT, D, G>>(S::smem_bytes(), device)) return TS_ERR_CUDA;
  AttKArgs a = proto;
  a.counters = reinterpret_cast<unsigned*>(dev.base);
  a.part = reinterpret_cast<float*>(dev.base + kNoAllocHeadBytes);
  if (!a.status) a.status = reinterpret_cast<int*>(dev.base + kNoAllocMaxBatch * kCounterSlots * sizeof(unsigned));
  // the merge counters must start at zero
  if (cudaMemsetAsync(dev.base, 0, (size_t)B * kCounterSlots * sizeof(unsigned), s) != cudaSuccess)
    return TS_ERR_CUDA;
  attend_kernel<KT, D, G><<<dim3(nsplit, HKV, B), S::THREADS, S::smem_bytes(), s>>>(a);
  return cuda_status(cudaGetLastError());
}

}  // namespace
}  // namespace ts

extern "C" ts_status ts_sparse_attend_noalloc(int n_q_heads, int n_kv_heads, int head_dim, int kv_dtype,
                                              const float* q, const void* k_pool, const void* v_pool,
                                              int64_t num_pages, const int32_t* page_table,
                                              int max_pages_per_seq, const int32_t* idx, int64_t idx_stride,
                                              const int32_t* count, int B, float scale, float* out,
                                              float* lse, int32_t* status, void* stream) {
  using namespace ts;
  if (!q || !k_pool || !v_pool || !page_table || !idx || !count || !out) return TS_ERR_INVALID_ARG;
  if (n_q_heads < 1 || n_kv_heads < 1 || n_q_heads % n_kv_heads != 0 || num_pages < 1 ||
      max_pages_per_seq < 1 || idx_stride < 1 || B < 1)
    return TS_ERR_INVALID_ARG;
  if (kv_dtype != TS_KV_F32 && kv_dtype != TS_KV_BF16) return TS_ERR_INVALID_ARG;
  if (std::isnan(scale)) return TS_ERR_INVALID_ARG;   // the same argument check as ts_sparse_attend
  if (reinterpret_cast<uintptr_t>(k_pool) % 16 != 0 || reinterpret_cast<uintptr_t>(v_pool) % 16 != 0)
    return TS_ERR_INVALID_ARG;
  if (B > kNoAllocMaxBatch || n_kv_heads > kCounterSlots - 2) return TS_ERR_SCRATCH_LIMIT;
  if ((int64_t)max_pages_per_seq * kPage > ((int64_t)1 << 30)) return TS_ERR_SHAPE;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kNoAllocMaxDevices) return TS_ERR_CUDA;
  NoAllocDevice dev;
  ts_status st = noalloc_setup(device, dev);
  if (st != TS_OK) return st;
  AttKArgs a;
  a.q = q;
  a.k_pool = static_cast<const unsigned char*>(k_pool);
  a.v_pool = static_cast<const unsigned char*>(v_pool);
  a.page_table = page_table;
  a.pt_stride = max_pages_per_seq;
  a.page_shift = 4;
  a.num_pages = num_pages;
  a.max_tokens = max_pages_per_seq * kPage;
  a.idx = idx;
  a.idx_stride = idx_stride;
  a.count = count;
  a.H = n_q_heads;
  a.HKV = n_kv_heads;
  a.scale = scale == 0.f ? 1.f / sqrtf((float)head_dim) : scale;
  a.out = out;
  a.lse = lse;
  a.part = nullptr;
  a.counters = nullptr;
  a.status = status;
  const int G = n_q_heads / n_kv_heads;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
#define X(DT, T, D_, G_) \
  if (kv_dtype == DT && head_dim == D_ && G == G_) return run_attend_noalloc<T, D_, G_>(a, B, n_kv_heads, device, dev, s);
  TS_ATTEND_GEOMETRIES(X)
#undef X
  return TS_ERR_UNSUPPORTED;
}
