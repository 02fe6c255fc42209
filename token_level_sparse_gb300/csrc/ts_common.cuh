// Device helpers shared by the token-selection kernels (sm_103a).
//
// Bulk copies (cp.async.bulk, the 1-D form of TMA) complete on shared-memory
// mbarriers. Every wait here is bounded by %globaltimer: when it runs out the
// kernel records TS_ERR_TIMEOUT in the status word and returns instead of
// spinning forever.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ts_internal.h"

namespace ts {

constexpr unsigned kFull = 0xffffffffu;
// Default upper bound on any single wait inside a kernel (nanoseconds); the persistent
// decode-step kernel takes its bound from the context (ts_set_wait_limit).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ void set_error(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Ends the use of a barrier object, so that its shared memory may serve something else.
__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Adds bytes to the current phase's expected transaction count without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete; false once limit_ns have passed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// 1-D bulk copy global -> shared, completing `bytes` of transaction on `bar`.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 16 bytes global -> shared without passing through registers (cp.async, cached in L2
// only). For gathers of many short rows: every thread keeps several in flight, where one
// bulk copy per row would queue the rows one after another in the copy engine. Completed by
// cp_async_commit + cp_async_wait_all (an ordinary memory access, like a load).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// all but the most recent commit group of this thread have landed
__device__ __forceinline__ void cp_async_wait_but_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Order-preserving unsigned key of a float (both signs): larger values give larger keys;
// -0 and +0 map to the key of +0, so they tie as the values do.
__device__ __forceinline__ uint32_t ordered_key(float v) {
  const uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);
  return u ^ ((u >> 31) ? 0xffffffffu : 0x80000000u);
}

// An L2 policy that evicts first: for data streamed once (the K scan) so it does
// not push out what is read again soon (the logits).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// bulk_g2s with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// ----------------------------------------------------------- value access

template <typename T>
struct KV;

// 16 bytes of fp32 = 4 elements.
template <>
struct KV<float> {
  static constexpr int kPerChunk = 4;
  __device__ __forceinline__ static void unpack(const uint4& c, float* o) {
    o[0] = __uint_as_float(c.x);
    o[1] = __uint_as_float(c.y);
    o[2] = __uint_as_float(c.z);
    o[3] = __uint_as_float(c.w);
  }
};

// 16 bytes of bf16 = 8 elements; a bf16 is the top half of the fp32 with the same bits.
template <>
struct KV<__nv_bfloat16> {
  static constexpr int kPerChunk = 8;
  __device__ __forceinline__ static void unpack(const uint4& c, float* o) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};

__device__ __forceinline__ uint4 lds128(const void* p) { return *reinterpret_cast<const uint4*>(p); }

__device__ __forceinline__ uint4 ldg_nc128(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ------------------------------------------------------------- reductions

// Sums NV per-lane values over groups of LPR consecutive lanes (both powers of
// two, NV <= LPR). Each butterfly level keeps half of the values and ships the
// other half to the partner, so after log2(NV) levels a lane holds one value;
// the remaining levels add plainly. Returns the full sum of value `which`.
template <int NV, int LPR>
__device__ __forceinline__ float transpose_reduce(float (&v)[NV], int lane, int& which) {
  static_assert(NV >= 1 && LPR >= 1 && NV <= LPR, "bad transpose_reduce shape");
  int base = 0;
  int n = NV;
#pragma unroll
  for (int d = LPR / 2; d >= 1; d >>= 1) {
    const bool upper = (lane & d) != 0;
    if (n > 1) {
      const int half = n / 2;
#pragma unroll
      for (int i = 0; i < NV / 2; ++i) {
        if (i < half) {
          const float send = upper ? v[i] : v[i + half];
          const float keep = upper ? v[i + half] : v[i];
          v[i] = keep + __shfl_xor_sync(kFull, send, d);
        }
      }
      if (upper) base += half;
      n = half;
    } else {
      v[0] += __shfl_xor_sync(kFull, v[0], d);
    }
  }
  which = base;
  return v[0];
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, d));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) x += __shfl_xor_sync(kFull, x, d);
  return x;
}

__device__ __forceinline__ int warp_sum_i(int x) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) x += __shfl_xor_sync(kFull, x, d);
  return x;
}

// Error-free transformation of a sum (Knuth's TwoSum): s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// Sum over the warp of the float pairs hi + lo, every level exact up to the low
// parts (TwoSum on the high parts). Partners combine the same two values, so
// every lane returns the same bits. FP64 is a slow pipe on this part; this keeps
// near-double accuracy on the fp32 pipe.
__device__ __forceinline__ float warp_sum_comp(float hi, float lo = 0.f) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) {
    const float oh = __shfl_xor_sync(kFull, hi, d), ol = __shfl_xor_sync(kFull, lo, d);
    float s, e;
    two_sum(hi, oh, s, e);
    hi = s;
    lo = (lo + ol) + e;
  }
  return hi + lo;
}

// Packed pairs of fp32 (Blackwell's two-lane fp32 arithmetic): each lane rounds like the scalar op.
__device__ __forceinline__ uint64_t pack_f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack_f2(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t fma_f2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Compensated (Kahan) accumulation in fp32.
struct KahanF {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float y = x - c;
    const float t = s + y;
    c = (t - s) - y;
    s = t;
  }
};

// Token segments of a sequence of n tokens: sinks [0, s_end), candidates
// [s_end, local_start), window [local_start, n).
__device__ __forceinline__ void budget_segments(int n, int n_sink, int n_local, int& s_end,
                                                int& local_start) {
  s_end = min(n_sink, n);
  local_start = max(s_end, n - n_local);
}

}  // namespace ts
