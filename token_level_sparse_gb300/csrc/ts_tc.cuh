// Blackwell (sm_103a) tensor-core and tensor-memory primitives used by the
// paged score scan: tiled TMA loads with 128-byte swizzle, tcgen05.mma with
// shared-memory descriptors, TMEM allocation and tcgen05.ld of accumulators.
//
// Layout conventions (PTX ISA, "Tensor Memory" and "Matrix Descriptors" for
// tcgen05):
//  * A and B operands are K-major bf16 tiles in shared memory in the 128-byte
//    swizzle layout: rows of 128 bytes (64 bf16 of the K dimension), the
//    16-byte chunk c of row r stored at chunk c ^ (r % 8), groups of 8 rows
//    1024 bytes apart. A tiled TMA load with CU_TENSOR_MAP_SWIZZLE_128B into a
//    1024-byte aligned buffer writes exactly this layout.
//  * A K-step of 16 elements is 32 bytes inside the 128-byte row: the
//    descriptor's start address moves by 32 bytes per step (the hardware
//    applies the swizzle to the final address).
//  * With M = 128 and cta_group::1, accumulator row i lives in TMEM lane i and
//    column j in TMEM column base + j; warp w of the CTA may read lanes
//    32 * (w % 4) .. + 31.
#pragma once

#include <cstdint>

#include "ts_common.cuh"

namespace ts {

// -------------------------------------------------------------- tiled TMA

// 2-D tiled load of one box at (x, y) (x = innermost, in elements) into dst,
// completing its bytes on bar; x * element size must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA, tensor core) accesses.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders generic-proxy global writes (made visible by a barrier) before this
// thread's later async-proxy reads of them (bulk copies), and vice versa.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ------------------------------------------------------------------- TMEM

// One full warp: allocates ncols columns (a power of two >= 32) and writes
// the TMEM address to *dst (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// One full warp (the allocating one).
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 8 consecutive 32-bit columns of this warp's 32 lanes: lane i of the warp
// receives row (taddr lane + i), columns col .. col + 7.
__device__ __forceinline__ void tmem_ld_x8(uint32_t taddr, float (&r)[8]) {
  uint32_t u[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7])
               : "r"(taddr)
               : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) r[i] = __uint_as_float(u[i]);
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 8 consecutive 32-bit columns of this warp's 32 lanes from registers: lane i of the warp writes
// row (taddr lane + i), columns col .. col + 7.
__device__ __forceinline__ void tmem_st_x8(uint32_t taddr, const float (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(__float_as_uint(r[0])), "r"(__float_as_uint(r[1])), "r"(__float_as_uint(r[2])),
               "r"(__float_as_uint(r[3])), "r"(__float_as_uint(r[4])), "r"(__float_as_uint(r[5])),
               "r"(__float_as_uint(r[6])), "r"(__float_as_uint(r[7]))
               : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------- MMA

// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled operand
// starting at addr: stride between 8-row groups 1024 bytes, descriptor
// version 1, swizzle mode 2 (128 bytes).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);          // start address
  d |= (uint64_t)1 << 16;                            // leading byte offset (unused when swizzled)
  d |= (uint64_t)(1024u >> 4) << 32;                 // stride byte offset
  d |= (uint64_t)1 << 46;                            // version
  d |= (uint64_t)2 << 61;                            // 128-byte swizzle
  return d;
}

// Shared-memory matrix descriptor of a K-major operand without swizzle starting at addr (16-byte
// aligned): core matrices of 8 rows x 16 bytes (8 elements of K) stored as 128 contiguous bytes,
// the next 8 elements of K `lbo` bytes on, the next 8 rows `sbo` bytes on.
__device__ __forceinline__ uint64_t sdesc_kmajor_none(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);          // start address
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;       // leading byte offset: the next 8 of K
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;       // stride byte offset: the next 8 rows
  d |= (uint64_t)1 << 46;                            // version (swizzle mode 0: none)
  return d;
}

// Shared-memory matrix descriptor of an MN-major, 128-byte-swizzled operand starting at addr:
// rows of 128 bytes hold 64 consecutive elements of the M (or N) dimension, one row per element of
// K; groups of 8 K-rows are `sbo` bytes apart and the next 64 elements of M are `lbo` bytes on. A
// tiled TMA load with CU_TENSOR_MAP_SWIZZLE_128B whose rows run along K writes this layout.
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);          // start address
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;       // leading byte offset: the next 64 of M
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;       // stride byte offset: the next 8 of K
  d |= (uint64_t)1 << 46;                            // version
  d |= (uint64_t)2 << 61;                            // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: bf16 A and B (both K-major), fp32 D,
// M x N tile.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4)                       // D: f32
         | (1u << 7)                     // A: bf16
         | (1u << 10)                    // B: bf16
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// The same with A MN-major (transposed: M contiguous in shared memory).
__host__ __device__ constexpr uint32_t idesc_bf16_f32_amn(int M, int N) { return idesc_bf16_f32(M, N) | (1u << 15); }

// D[tmem] (+)= A[smem] x B[smem]^T over one K-step of 16, issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// Arrives once on bar when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

// Byte offset of bf16 element (row, k) inside a K-major 128-byte-swizzled
// tile whose rows hold 64 elements (k < 64); the tile base is 1024-aligned.
__host__ __device__ __forceinline__ uint32_t sw128_offset(int row, int k) {
  return (uint32_t)row * 128u + (uint32_t)((((k >> 3) ^ (row & 7)) << 4) + ((k & 7) << 1));
}

// Term `term` (0, 1, 2) of the three-term bf16 split of x: hi = bf16(x),
// mid = bf16(x - hi), lo = bf16(x - hi - mid); hi + mid + lo equals x to
// within 2^-27 relative, and each product with a bf16 value is exact in fp32.
__device__ __forceinline__ __nv_bfloat16 bf16_split_term(float x, int term) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(hi);
  const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(mid);
  const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
  return term == 0 ? hi : (term == 1 ? mid : lo);
}

}  // namespace ts
