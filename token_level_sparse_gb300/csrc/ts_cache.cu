// Selection Cache test of Algorithm 1 (TokenSelect deep notes, Appendix
// Algorithm 1; review, section 3.2): a (sequence, layer) entry hits when it
// holds a previous selection and cos(Q, C_Q) >= theta over the H*d query.
// C_Q is the query of the last miss (it is only written by the selection).
#include <cmath>

#include "ts_common.cuh"

namespace ts {
namespace {

constexpr int kCheckThreads = 256;

__global__ void __launch_bounds__(kCheckThreads)
    cache_check_kernel(const float* q, const float* cq, const uint8_t* filled, int HD, float theta,
                       uint8_t* hit, float* cos_out) {
  const int b = blockIdx.x;
  if (!filled[b]) {
    if (threadIdx.x == 0) {
      hit[b] = 0;
      if (cos_out) cos_out[b] = __int_as_float(0x7fc00000);
    }
    return;
  }
  const float* x = q + (size_t)b * HD;
  const float* y = cq + (size_t)b * HD;
  float xy = 0.f, xx = 0.f, yy = 0.f;
  for (int i = threadIdx.x; i < HD; i += kCheckThreads) {
    const float u = x[i], v = y[i];
    xy = fmaf(u, v, xy);
    xx = fmaf(u, u, xx);
    yy = fmaf(v, v, yy);
  }
  xy = warp_sum(xy);
  xx = warp_sum(xx);
  yy = warp_sum(yy);
  __shared__ float red[3][kCheckThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    red[0][warp] = xy;
    red[1][warp] = xx;
    red[2][warp] = yy;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    KahanF sxy, sxx, syy;   // fp32: FP64 is a slow pipe here
    for (int w = 0; w < kCheckThreads / 32; ++w) {
      sxy.add(red[0][w]);
      sxx.add(red[1][w]);
      syy.add(red[2][w]);
    }
    const float den = sqrtf(sxx.s - sxx.c) * sqrtf(syy.s - syy.c);
    const float c = den > 0.f ? (sxy.s - sxy.c) / den : __int_as_float(0x7fc00000);
    hit[b] = (c >= theta) ? 1 : 0;  // NaN compares false: a miss
    if (cos_out) cos_out[b] = c;
  }
}

}  // namespace

ts_status launch_cache_check(ts_ctx* ctx, ts_cache* cache, int layer, const float* q, int B,
                             float theta, uint8_t* hit, float* cos_out, cudaStream_t s) {
  const ts_config& cfg = ctx->cfg;
  const int HD = cfg.n_q_heads * cfg.head_dim;
  const size_t mb = (size_t)cfg.max_batch;
  ProfScope ps(ctx, TS_PROF_CHECK, s);
  ctx->kernels += 1;
  cache_check_kernel<<<B, kCheckThreads, 0, s>>>(q, cache->cq + (size_t)layer * mb * HD,
                                                  cache->filled + (size_t)layer * mb, HD, theta, hit,
                                                  cos_out);
  return cuda_status(cudaGetLastError());
}

ts_status launch_cache_reset(ts_cache* cache, cudaStream_t s) {
  const size_t n = (size_t)cache->n_layers * cache->ctx->cfg.max_batch;
  cudaError_t e = cudaMemsetAsync(cache->filled, 0, n, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(cache->ct_count, 0, n * sizeof(int32_t), s);
  return cuda_status(e);
}

}  // namespace ts
