// Chunk-wise prefill selection (TokenSelect deep notes, "Optimising the selection
// frequency of the prefill stage"; review, section 3.2, closing paragraph): the c
// queries of a prefill chunk are averaged, (1/c) sum_i (Q_C)_i, that mean query
// selects once (head soft vote, top-k over the candidates, united with sinks and
// window; no Selection Cache in prefill), and every query of the chunk attends to
// the shared selection. The chunk's own tokens are the last c cached positions,
// so query i attends causally: to the selected tokens at positions <= n - c + i.
//
// The attention of a chunk is a dense contraction (c x G query rows of one KV head
// against its selected keys), so it runs on the tcgen05 tensor cores:
//  * one CTA per (tile of 128 query rows, KV head, sequence); rows are
//    (chunk query i, head j of the group) pairs, row = i * G + j;
//  * the fp32 queries enter as three bf16 terms (hi, mid, lo; products exact,
//    sum within 2^-27 of the query) accumulated into one TMEM accumulator, so
//    the scores carry fp32 accuracy;
//  * two passes over the selected keys in tiles of 128 tokens gathered with
//    cp.async into the 128-byte-swizzled K-major layout: the first pass takes
//    every row's max and sum of exponentials (the scores come back from TMEM),
//    the second recomputes the scores, forms the normalised weights P (two bf16
//    terms, sum within 2^-17 of P), and accumulates O += P V^T in TMEM with V
//    transposed into a K-major tile. No rescaling of O is ever needed, and
//    every sum has a fixed order: the result is deterministic.
#include <cmath>

#include "ts_common.cuh"
#include "ts_tc.cuh"

namespace ts {
namespace {

constexpr int kCaThreads = 256;   // 8 warps: warp w reads TMEM lanes 32 (w % 4).., columns half w / 4
constexpr int kCaRows = 128;      // query rows of a CTA (the MMA's M)
constexpr int kCaTok = 128;       // tokens of a key tile (the score MMA's N, the output MMA's K)

// mean query of every chunk: qm[b][e] = (1/c) sum_i q[b][i][e] over the H*d
// elements e, summed in query order with compensation
__global__ void chunk_mean_kernel(const float* q, int c, int HD, int B, float* qm) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= B * HD) return;
  const int b = idx / HD, e = idx % HD;
  KahanF acc;
  for (int i = 0; i < c; ++i) acc.add(q[((size_t)b * c + i) * HD + e]);
  qm[idx] = (acc.s - acc.c) / (float)c;
}

struct CaArgs {
  const float* q;              // [B][c][H][D] chunk queries
  int c, H, HKV, G;
  const unsigned char* k_pool; // [num_pages][H_kv][page size][D] bf16
  const unsigned char* v_pool;
  int64_t num_pages;
  const int32_t* page_table;
  int pt_stride;
  int page_shift;              // log2 of the page size: 4 (16 tokens) or 0 (one token per page)
  const int32_t* seq_lens;
  int max_tokens;
  const int32_t* idx;          // [B][idx_stride] ascending
  int64_t idx_stride;
  const int32_t* count;
  float scale;
  float* out;                  // [B][c][H][D]
  float* lse;                  // [B][c][H] or null
  int* status;
  uint64_t wait_ns;
};

template <int D>
struct CaShape {
  static constexpr int HALVES = D / 64;                    // 128-byte swizzle rows per operand row
  static constexpr int ROW_BYTES = D * 2;                  // one bf16 K or V row
  static constexpr int QT = kCaRows * D * 2;               // one query term tile
  static constexpr int KT = kCaTok * D * 2;                // one K tile (also P term 0)
  static constexpr int VT = D * kCaTok * 2;                // V^T tile: D rows of 128 tokens
  static constexpr int PT = kCaRows * kCaTok * 2;          // one P term tile
  static constexpr int KP = KT > PT ? KT : PT;             // the K tile, later P term 0
  static constexpr int SMEM = 3 * QT + KP + VT + PT + 1024;  // + alignment slack
  static_assert(D == 64 || D == 128, "head dim");
};

// Byte offset of element (row, k) of a K-major operand with K = 64 * halves elements per
// row: half h = k / 64 is a separate [rows][128 B] swizzled block.
__device__ __forceinline__ uint32_t opnd_offset(int row, int k, int rows) {
  return (uint32_t)(k >> 6) * (uint32_t)(rows * 128) + sw128_offset(row, k & 63);
}

template <int D>
__global__ void __launch_bounds__(kCaThreads, 1) chunk_attend_kernel(const __grid_constant__ CaArgs a) {
  using S = CaShape<D>;
  extern __shared__ unsigned char dsm_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char* sQ = base;                 // 3 query terms
  unsigned char* sK = sQ + 3 * S::QT;       // K tile, then P term 0 of the same tile
  unsigned char* sV = sK + S::KP;           // V^T tile
  unsigned char* sP1 = sV + S::VT;          // P term 1
  __shared__ int s_tok[2][kCaTok], s_page[2][kCaTok];   // token lists of two key tiles
  __shared__ float s_m[2][kCaRows], s_l[2][kCaRows];
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t mbar;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int rows = a.c * a.G, r0 = mt * kCaRows;
  int n = a.seq_lens[b];
  if (n < 0 || n > a.max_tokens) {
    if (tid == 0) set_error(a.status, TS_ERR_SEQ_LEN);
    n = 0;
  }
  const int cnt = max(0, min(a.count[b], (int)a.idx_stride));
  const int ntiles = (cnt + kCaTok - 1) / kCaTok;

  // ---- the query rows of this tile as three bf16 terms, K-major and swizzled; when every query
  // element is a bf16 value (its mid and lo terms are zero) only the first term is multiplied
  constexpr int CPR = D / 8;                            // 8-element chunks of a query row
  int extra = 0;
  for (int i = tid; i < 3 * kCaRows * CPR; i += kCaThreads) {
    const int term = i / (kCaRows * CPR), rem = i % (kCaRows * CPR), r = rem / CPR, ch = rem % CPR;
    const int rg = r0 + r;
    float e8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (rg < rows) {
      const int qi = rg / a.G, head = g * a.G + rg % a.G;
      const float4* src = reinterpret_cast<const float4*>(a.q + (((size_t)b * a.c + qi) * a.H + head) * D + ch * 8);
      const float4 x0 = src[0], x1 = src[1];
      e8[0] = x0.x; e8[1] = x0.y; e8[2] = x0.z; e8[3] = x0.w;
      e8[4] = x1.x; e8[5] = x1.y; e8[6] = x1.z; e8[7] = x1.w;
    }
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = (uint32_t)__bfloat16_as_ushort(bf16_split_term(e8[2 * e], term)) |
             ((uint32_t)__bfloat16_as_ushort(bf16_split_term(e8[2 * e + 1], term)) << 16);
    if (term > 0) extra |= (w[0] | w[1] | w[2] | w[3]) & 0x7fff7fffu;   // a non-zero mid or lo term
    *reinterpret_cast<uint4*>(sQ + term * S::QT + opnd_offset(r, ch * 8, kCaRows)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  const int nterms = __syncthreads_or(extra) ? 3 : 1;
  fence_proxy_async();
  if (warp == 0) {
    tmem_alloc(&s_tmem, 256);                           // S: columns 0..127, O: 128..255
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&mbar, 1);
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tS = s_tmem, tO = s_tmem + 128;
  const int row = 32 * (warp & 3) + lane, chalf = warp >> 2;  // my TMEM lane and column half
  const int rg = r0 + row;
  const int qpos = rg < rows ? n - a.c + rg / a.G : -1;      // last position my query may see
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
  constexpr uint32_t idesc = idesc_bf16_f32(kCaRows, kCaTok);
  constexpr uint32_t idesc_o = idesc_bf16_f32(kCaRows, D);
  float m = -INFINITY, l = 0.f;                             // my row over my column half
  uint32_t phase = 0;
  bool ok = true;

  // waits for the MMAs committed last; false (recorded) once the bound runs out
  auto wait_mma = [&]() -> bool {
    const bool landed = mbar_wait(&mbar, phase, a.wait_ns);
    phase ^= 1u;
    if (!__syncthreads_and(landed)) {
      if (tid == 0) set_error(a.status, TS_ERR_TIMEOUT);
      return false;
    }
    tc_fence_after();
    return true;
  };

  // row of (page, KV head g, token t) in the pool [page][H_kv][page size][D]
  auto pool_row = [&](int page, int g, int t) -> size_t {
    return (((size_t)page * a.HKV + g) << a.page_shift) + (t & ((1 << a.page_shift) - 1));
  };
  // the tokens and pages of key tile kt into list buffer lb (threads below 128)
  auto list_tile = [&](int kt, int lb) {
    if (tid < kCaTok) {
      const int j = kt * kCaTok + tid;
      int t = -1, page = -1;
      if (j < cnt) {
        t = a.idx[(size_t)b * a.idx_stride + j];
        if (t >= 0 && t < a.max_tokens) page = a.page_table[(size_t)b * a.pt_stride + (t >> a.page_shift)];
        if (page < 0 || (int64_t)page >= a.num_pages) {
          set_error(a.status, TS_ERR_PAGE_OOB);
          page = -1;
        }
      }
      s_tok[lb][tid] = page >= 0 ? t : -1;
      s_page[lb][tid] = page;
    }
  };
  // the K rows of list lb into the swizzled tile at dst by cp.async, one commit group (missing
  // tokens read row 0 of the pool: masked when the scores are read)
  auto gather_k = [&](int lb, unsigned char* dst) {
    for (int i = tid; i < kCaTok * CPR; i += kCaThreads) {
      const int r = i / CPR, ch = i % CPR, page = s_page[lb][r];
      const size_t off = page >= 0 ? pool_row(page, g, s_tok[lb][r]) * S::ROW_BYTES : 0;
      cp_async16(dst + opnd_offset(r, ch * 8, kCaTok), a.k_pool + off + ch * 16);
    }
    cp_async_commit();
  };
  // S = Q K^T of the K tile at kbuf: the query terms into one accumulator
  auto issue_scores = [&](const unsigned char* kbuf) {
    if (tid == 0) {
      tc_fence_after();
      const uint32_t q0 = smem_addr(sQ), k0 = smem_addr(kbuf);
#pragma unroll 1
      for (int term = 0; term < nterms; ++term)
#pragma unroll
        for (int h = 0; h < S::HALVES; ++h)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_bf16(tS, sdesc_sw128(q0 + term * S::QT + h * (kCaRows * 128) + ks * 32),
                      sdesc_sw128(k0 + h * (kCaTok * 128) + ks * 32), idesc, (term | h | ks) != 0);
      umma_commit(&mbar);
    }
  };
  // my 64 score columns, masked (causal, missing tokens) and scaled
  float x[64];
  auto read_scores = [&](int lb) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      tmem_ld_x8(tS + lane_off + chalf * 64 + 8 * i, *reinterpret_cast<float(*)[8]>(x + 8 * i));
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      const int t = s_tok[lb][chalf * 64 + j];
      x[j] = (t >= 0 && t <= qpos) ? x[j] * a.scale : -INFINITY;
    }
  };

  // ---- pass 1: every row's max and sum of exponentials. K tiles alternate between the K
  // buffer and the (not yet needed) V buffer, so the next tile's rows land during this one's scores
  if (ntiles > 0) {
    list_tile(0, 0);
    __syncthreads();
    gather_k(0, sK);
  }
  for (int kt = 0; kt < ntiles; ++kt) {
    const int lb = kt & 1;
    unsigned char* kb = lb ? sV : sK;
    if (kt + 1 < ntiles) {
      list_tile(kt + 1, lb ^ 1);
      __syncthreads();
      gather_k(lb ^ 1, lb ? sK : sV);
      cp_async_wait_but_one();
    } else {
      cp_async_wait_all();
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    issue_scores(kb);
    if (!wait_mma()) {
      ok = false;
      break;
    }
    read_scores(lb);
    float tm = -INFINITY;
#pragma unroll
    for (int j = 0; j < 64; ++j) tm = fmaxf(tm, x[j]);
    if (tm > -INFINITY) {
      const float mn = fmaxf(m, tm);
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < 64; ++j) sum += x[j] > -INFINITY ? expf(x[j] - mn) : 0.f;
      l = (m > -INFINITY ? l * expf(m - mn) : 0.f) + sum;
      m = mn;
    }
    tc_fence_before();
    __syncthreads();                            // scores read and list buffer free before they are reused
  }
  cp_async_wait_all();                          // nothing left in flight (a time-out leaves the loop early)
  if (ok) {
    // the row's max and sum over both column halves
    s_m[chalf][row] = m;
    s_l[chalf][row] = l;
    __syncthreads();
    const float m0 = s_m[0][row], m1 = s_m[1][row], M = fmaxf(m0, m1);
    l = M > -INFINITY ? (m0 > -INFINITY ? s_l[0][row] * expf(m0 - M) : 0.f) +
                            (m1 > -INFINITY ? s_l[1][row] * expf(m1 - M) : 0.f)
                      : 0.f;
    m = M;
  }

  // ---- pass 2: the scores again, normalised weights P, O += P V^T
  for (int kt = 0; kt < ntiles && ok; ++kt) {
    list_tile(kt, 0);
    __syncthreads();
    gather_k(0, sK);
    // V rows transposed into V^T [d][token] (K-major over the tokens): lane = token, so the
    // 2-byte stores of a warp fill consecutive columns of one row
    for (int i = tid; i < kCaTok * CPR; i += kCaThreads) {
      const int r = i % kCaTok, ch = i / kCaTok, page = s_page[0][r];
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (page >= 0)
        v = *reinterpret_cast<const uint4*>(a.v_pool + pool_row(page, g, s_tok[0][r]) * S::ROW_BYTES + ch * 16);
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 8; ++e)
        *reinterpret_cast<uint16_t*>(sV + opnd_offset(ch * 8 + e, r, D)) =
            (uint16_t)((w4[e >> 1] >> (16 * (e & 1))) & 0xffffu);
    }
    cp_async_wait_all();
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    issue_scores(sK);
    if (!wait_mma()) {
      ok = false;
      break;
    }
    read_scores(0);
    // normalised weights as two bf16 terms: P0 into the spent K tile, P1 into its own
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      uint32_t w0[4], w1[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float p2[2];
#pragma unroll
        for (int z = 0; z < 2; ++z) {
          const float xx = x[8 * u + 2 * e + z];
          p2[z] = (xx > -INFINITY && l > 0.f) ? expf(xx - m) * inv : 0.f;
        }
        const __nv_bfloat16 h0 = __float2bfloat16_rn(p2[0]), h1 = __float2bfloat16_rn(p2[1]);
        const __nv_bfloat16 l0 = __float2bfloat16_rn(p2[0] - __bfloat162float(h0));
        const __nv_bfloat16 l1 = __float2bfloat16_rn(p2[1] - __bfloat162float(h1));
        w0[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
        w1[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
      }
      const uint32_t off = opnd_offset(row, chalf * 64 + 8 * u, kCaRows);
      *reinterpret_cast<uint4*>(sK + off) = make_uint4(w0[0], w0[1], w0[2], w0[3]);
      *reinterpret_cast<uint4*>(sP1 + off) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    // ---- O += P V^T: two weight terms
    if (tid == 0) {
      tc_fence_after();
      const uint32_t v0 = smem_addr(sV);
#pragma unroll 1
      for (int term = 0; term < 2; ++term) {
        const uint32_t p0 = smem_addr(term == 0 ? sK : sP1);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_bf16(tO, sdesc_sw128(p0 + h * (kCaRows * 128) + ks * 32),
                      sdesc_sw128(v0 + h * (D * 128) + ks * 32), idesc_o, (kt | term | h | ks) != 0);
      }
      umma_commit(&mbar);
    }
    if (!wait_mma()) {
      ok = false;
      break;
    }
  }

  // ---- outputs: my row's half of the output columns, and the row's lse. The TMEM loads are
  // warp-collective (.sync.aligned): every lane of the warp issues them whatever its row, and
  // only the stores depend on the row being real
  if (ok) {
    const bool valid = rg < rows;
    const int qi = valid ? rg / a.G : 0, head = valid ? g * a.G + rg % a.G : 0;
    float* dst = a.out + (((size_t)b * a.c + qi) * a.H + head) * D + chalf * (D / 2);
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      float o8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (ntiles > 0) {                                      // uniform over the CTA
        tmem_ld_x8(tO + lane_off + chalf * (D / 2) + 8 * i, o8);
        tmem_wait_ld();
      }
      if (valid) {
#pragma unroll
        for (int e = 0; e < 8; ++e) dst[8 * i + e] = l > 0.f ? o8[e] : 0.f;
      }
    }
    if (valid && a.lse && chalf == 0) a.lse[((size_t)b * a.c + qi) * a.H + head] = l > 0.f ? m + logf(l) : -INFINITY;
  }
  if (!ok && tid == 0) mbar_wait(&mbar, phase, a.wait_ns);   // a late commit lands before TMEM is freed
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(s_tmem, 256);
  }
}

}  // namespace

bool chunk_attend_supported(const ts_config& c) {
  return c.kv_dtype == TS_KV_BF16 && (c.head_dim == 128 || c.head_dim == 64) && c.n_q_heads % c.n_kv_heads == 0;
}

ts_status launch_chunk_mean(ts_ctx* ctx, const float* q, int c, int B, float* qm, cudaStream_t s) {
  const int HD = ctx->cfg.n_q_heads * ctx->cfg.head_dim;
  ctx->kernels += 1;
  chunk_mean_kernel<<<(B * HD + 255) / 256, 256, 0, s>>>(q, c, HD, B, qm);
  return cuda_status(cudaGetLastError());
}

template <int D>
ts_status run_chunk_attend(ts_ctx* ctx, const CaArgs& a, int B, cudaStream_t s) {
  using S = CaShape<D>;
  if (!ensure_smem<chunk_attend_kernel<D>>((size_t)S::SMEM, ctx->device)) return TS_ERR_CUDA;
  const int mtiles = (a.c * a.G + kCaRows - 1) / kCaRows;
  ctx->kernels += 1;
  chunk_attend_kernel<D><<<dim3(mtiles, a.HKV, B), kCaThreads, S::SMEM, s>>>(a);
  return cuda_status(cudaGetLastError());
}

ts_status launch_chunk_attend(ts_ctx* ctx, const ChunkAttendCall& c, cudaStream_t s) {
  const ts_config& cfg = ctx->cfg;
  if (!chunk_attend_supported(cfg)) return TS_ERR_UNSUPPORTED;
  CaArgs a;
  a.q = c.q;
  a.c = c.c;
  a.H = cfg.n_q_heads;
  a.HKV = cfg.n_kv_heads;
  a.G = cfg.n_q_heads / cfg.n_kv_heads;
  a.k_pool = static_cast<const unsigned char*>(c.k_pool);
  a.v_pool = static_cast<const unsigned char*>(c.v_pool);
  a.num_pages = cfg.num_pages;
  a.page_table = c.page_table;
  a.pt_stride = cfg.max_pages_per_seq;
  a.page_shift = ctx->page_shift;
  a.seq_lens = c.seq_lens;
  a.max_tokens = ctx->max_tokens;
  a.idx = c.idx;
  a.idx_stride = c.idx_stride;
  a.count = c.count;
  a.scale = c.scale;
  a.out = c.out;
  a.lse = c.lse;
  a.status = ctx->status;
  a.wait_ns = ctx->wait_ns;
  ProfScope ps(ctx, TS_PROF_ATTEND, s);
  return cfg.head_dim == 128 ? run_chunk_attend<128>(ctx, a, c.B, s) : run_chunk_attend<64>(ctx, a, c.B, s);
}

}  // namespace ts
