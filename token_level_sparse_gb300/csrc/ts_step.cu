// One persistent, cooperative kernel for a whole decode step (or any of its
// parts): Selection Cache test, paged score + head soft vote, top-k / top-p
// selection united with sinks and window, and sparse attention.
//
// The method is TokenSelect's (deep notes: Appendix Algorithm 1 and 2, "Head
// soft vote", "Formalising selective sparse attention"; review: section 4.2).
// The GB300 mapping, one CTA per SM and grid barriers between phases:
//  * score: each CTA scans a contiguous range of the concatenated (missing)
//    sequences' pages. Warp 0 feeds a ring of tiled TMA loads (one page of all
//    KV heads = 128 rows); one thread of warp 1 issues tcgen05 MMAs of each
//    page against the query heads (each fp32 query split into three bf16
//    terms) into double-buffered TMEM accumulators; warps 4..7 read them out,
//    write the logits (base-2 units) to scratch and keep per-row running
//    (max, sum), reduced into per-CTA partials. Geometries without the tensor
//    core scan use a CUDA-core scan (cuda_scan_wave) in waves of KV heads;
//  * vote: after the barrier every CTA forms the per-head normalisers from the
//    CTA partials and the votes of its own tokens from its logits, which come
//    back into shared memory by bulk copy;
//  * selection: radix histograms of the vote bit pattern, aggregated in shared
//    memory and added with integer atomics (order-free, hence deterministic);
//    once the crossing bin holds at most 2048 tokens they are gathered and
//    ranked exactly (ties go to the lower index; top-p mass in 2^-40 fixed
//    point). Each CTA then writes its selected tokens as an ascending list into
//    a buffer of its own (its logits stay in its scratch);
//  * attention: every CTA attends its own selected tokens (with top-p an equal
//    share of every CTA's lists; a batch of top-k sequences: an equal share
//    over the sequence's group of CTAs) plus a round-robin share of the sinks,
//    window and cached indices, gathering K/V rows by cp.async. Dense top-p
//    selections instead attend each CTA's own range of pages (range_attend):
//    misses from the scan's logits and streamed V pages, cache hits from
//    streamed K and V pages. Per-CTA (max, sum, o) partials are merged after one
//    more barrier, and the index lists and the Selection Cache entries are
//    written from the per-CTA lists.
// Grid barriers and mbarrier waits are bounded by %globaltimer; on time-out
// the kernel records TS_ERR_TIMEOUT and returns. The last CTA to leave zeroes
// the barrier words for the next launch.
#include <algorithm>
#include <cfloat>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <type_traits>

#include "ts_common.cuh"
#include "ts_tc.cuh"

namespace ts {
namespace {

constexpr int kMaxB = 64;          // sequences per call (= most segments one CTA can touch)
constexpr int kCandCap = 2048;     // candidates gathered per sequence
constexpr int kMaxRound = 128;     // attention tokens per gather round
constexpr int kMaxWaveHeads = 32;  // query heads of one scan wave
constexpr int kMaxG = kMaxScanG;   // query heads per KV head
constexpr int kMaxAttH = 64;       // query heads of the attention phase
constexpr int kPreFix = 512;       // fixed attention tokens of a CTA resolved at set-up
constexpr int kOwnBatch = 1024;    // attention: selected tokens (and pages) looked up from other CTAs' lists at once
constexpr int kRangeSlots = 4;     // range attention: ring slots of one V page and its logit rows
constexpr int kRangeSlotsTC = 6;   // the same on the tensor cores (a slot is free only once its MMAs are)
constexpr float kRescaleGap = 8.f; // range attention: a logit this far (base 2) above the running max rescales
constexpr int kStageMin = 160 * 1024;  // attention staging bytes every launch has (checked at launch)
constexpr int kMaxPagesCta = 1024; // page ids of a CTA's range kept in shared memory
constexpr int kScanClaim = 2;      // pages per claim of a shared tensor-core scan
constexpr int kVoteBufs = 2;       // shared-memory buffers of logit chunks for the votes
constexpr int kMaxGrid = 256;      // CTAs of the persistent launch (one per SM)
static_assert(2 * kMaxGrid + 1 <= kMaxPagesCta, "balanced-attention offsets share the page-id array");
constexpr int kMaxSlots = 12;      // ring slots (runtime count per launch)
constexpr int kNoPage = -2147483647 - 1;  // a tile's second page is absent (not an invalid page id)
constexpr int kAbsentRows = -2;           // valid-row count of an absent page of a tile: nothing is stored
constexpr int64_t kLogitL2Budget = 48ll << 20;  // default bytes of logits one scan wave keeps in L2
// radix levels over the vote bits (votes are >= +0, bit 31 is always 0): bits 30..17, 16..6,
// 5..0. The first level is fine enough that its crossing bin usually holds few enough tokens
// to gather them as candidates at once (the votes of long sequences lie close together).
__host__ __device__ constexpr int lvl_shift(int l) { return l == 0 ? 17 : (l == 1 ? 6 : 0); }
__host__ __device__ constexpr int lvl_bins(int l) { return l == 0 ? 16384 : (l == 1 ? 2048 : 64); }
// per sequence: level 0 fine [16384], its coarse sums [128] (fine bins 128 c .. 128 c + 127),
// level 1 [2048], level 2 [64]
constexpr int kCoarseOff = 16384;
__host__ __device__ constexpr int lvl_off(int l) { return l == 0 ? 0 : (l == 1 ? 16384 + 128 : 16384 + 128 + 2048); }
constexpr int kHistPerSeq = kStepHistPerSeq;            // 16384 + 128 + 2048 + 64
static_assert(lvl_off(2) + lvl_bins(2) == kHistPerSeq, "histogram layout");
constexpr float kFx = 1099511627776.0f;  // 2^40
constexpr int kPhCheck = 1, kPhScore = 2, kPhSelect = 4, kPhAttend = 8;
constexpr int kSmemLimit = 232448;  // bytes of shared memory per CTA on sm_103a

constexpr int cpow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}
constexpr int cmin(int a, int b) { return a < b ? a : b; }

__device__ __forceinline__ unsigned long long to_fx(float v) { return __float2ull_rz(v * kFx); }

// N consecutive K or V elements (fp32 or bf16) from shared memory as floats; the address is
// aligned to N elements.
template <typename KT, int N>
__device__ __forceinline__ void load_elems(const KT* p, float (&f)[N]) {
  if constexpr (sizeof(KT) == 4 && N == 4) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  } else if constexpr (sizeof(KT) == 4 && N == 2) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    f[0] = v.x; f[1] = v.y;
  } else if constexpr (sizeof(KT) == 2 && N == 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xffff0000u);
    f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xffff0000u);
  } else if constexpr (sizeof(KT) == 2 && N == 2) {
    const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
    f[0] = __uint_as_float(v << 16); f[1] = __uint_as_float(v & 0xffff0000u);
  } else {
    static_assert(N == 4 || N == 2, "load_elems width");
  }
}

// ------------------------------------------------------------------ shapes

template <typename KT, int D, int HKV, int G>
struct StepShape {
  static constexpr int P = kPage;
  static constexpr int EPC = KV<KT>::kPerChunk;          // elements per 16-byte chunk
  static constexpr int GP = cpow2(G);
  static constexpr int CPL = (GP * 2 * EPC <= 64) ? 2 : 1;  // chunks per lane in the scan
  static constexpr int DPL = EPC * CPL;
  static constexpr int LPR = D / DPL;                     // lanes per K row in the scan
  static constexpr int RPW = 32 / LPR;                    // rows per warp step
  static constexpr int NCW = cmin(16, HKV * P / RPW);     // warps (all consume; the last to finish a
  static constexpr int NW = NCW;                          // stage refills it: no producer warp)
  static constexpr int THREADS = NW * 32;
  static constexpr int ROWS = P * HKV / NCW;              // rows of a stage per consumer warp
  static constexpr int ITERS = ROWS / RPW;
  static constexpr int ROW_BYTES = D * (int)sizeof(KT);
  static constexpr int STAGE_BYTES = HKV * P * ROW_BYTES; // H_kv (page, head) slabs of 16 rows
  static constexpr int MIN_SLOTS = 2;
  static constexpr int TOKEN_BYTES = 2 * HKV * ROW_BYTES; // K and V rows of every KV head
  static_assert(D % DPL == 0 && 32 % LPR == 0 && GP <= LPR, "scan lane split");
  static_assert(NCW >= 1 && (P * HKV) % NCW == 0 && ROWS % RPW == 0 && ITERS >= 1, "scan warp split");
  static_assert(NCW % HKV == 0 && P % ROWS == 0 || ROWS % P == 0, "rows of a warp stay in one page");
  static_assert(NW % HKV == 0, "attention scores: whole warps per KV head");
  static_assert(GP <= 32, "attention reduction");
  static_assert((HKV * G) % 2 == 0, "rows of H (max, sum) pairs are whole 16-byte blocks");
  // tensor-core scan (bf16 pages of 128 rows = H_kv x 16 tokens): one M = 128 tcgen05.mma
  // tile per page against all query heads, each split into three bf16 terms
  // a page of every KV head is HKV x 16 rows: 128 rows fill one M = 128 tile, 64 rows (4 KV heads)
  // take two pages of the same sequence per tile
  static constexpr int TC_ROWS = HKV * P;
  static constexpr int TC_PAGES = TC_ROWS == 64 ? 2 : 1;
  static constexpr bool TC = std::is_same<KT, __nv_bfloat16>::value && (TC_ROWS == 128 || TC_ROWS == 64) &&
                             (D == 128 || D == 64) && 3 * HKV * G <= 256 && G <= 8;
  static constexpr int TC_N = (3 * HKV * G + 15) / 16 * 16;           // B rows (q terms), multiple of 16
  static constexpr int TC_HALVES = D / 64;                             // 128-byte swizzle rows per K row
  static constexpr int TC_TILE = 128 * D * 2;                          // one M = 128 tile of K (1 or 2 pages)
  static constexpr int TC_PAGE_BYTES = TC_ROWS * D * 2;                // one page of K
  static constexpr int PV = TC_PAGES;                                  // partial rows per CTA (one per tile half)
  static_assert(TC_PAGE_BYTES * TC_PAGES <= TC_TILE, "the pages of a tile fit its slot");
  static constexpr int TC_BIMG = TC_N * D * 2;                         // one sequence's query terms
  static constexpr int TC_COLS = TC_N <= 32 ? 32 : (TC_N <= 64 ? 64 : (TC_N <= 128 ? 128 : 256));
  static constexpr int TC_NLD = (6 * G + 7) / 8;                       // 8-column loads per epilogue warp
  static_assert(!TC || (2 * TC_COLS <= 512 && 6 * G * (HKV / 2 - 1) + 8 * TC_NLD <= TC_COLS && NW >= 8 && TC_HALVES >= 1 &&
                        TC_BIMG % 1024 == 0 && TC_TILE % 1024 == 0), "tensor-core scan");
  static_assert(G <= kMaxG, "heads per KV head");
  static_assert(NCW <= kMaxScanWarps && NCW % HKV == 0, "scan warps split evenly over the KV heads");
};

struct GridSync {
  unsigned count;   // barrier arrivals since the launch
  unsigned abort;
  unsigned claim;   // next page chunk of a shared tensor-core scan
  unsigned exits;   // CTAs that have left; the last one zeroes all four for the next launch
};

struct StepKArgs {
  CUtensorMap tmap_k;          // K pool as [num_pages * H_kv * 16][d] bf16, box 64 x (H_kv * 16), 128-byte swizzle
  CUtensorMap tmap_v;          // V pool, the same view (the tensor-core range attention)
  int tc;                      // the tensor-core scan may run (map encoded, geometry supported)
  int nslot_tc;                // its ring slots
  int scan_dyn;                // it may share pages out by claims when at most two sequences scan
  int phases;
  int B, H, max_tokens, pt_stride;
  int64_t num_pages;
  const float* q;
  const unsigned char* k_pool;
  const unsigned char* v_pool;
  const int32_t* page_table;
  const int32_t* seq_lens;
  float scale;
  float scale_l2;              // scale x log2(e): the scan keeps its logits in base-2 units (exp2)
  float scale_l2_lo;           // scale x log2(e) - scale_l2 (the constant to about 2^-48 relative)
  float theta;
  const uint8_t* hit_in;
  uint8_t* hit_out;
  // Selection Cache entries of this layer (null without a cache)
  float* cq;
  int32_t* ct;
  int32_t* ct_count;
  uint8_t* filled;
  int cap;
  // selection
  int mode, k, n_sink, n_local;
  unsigned long long target_fx;
  int take_all_topp;
  // outputs
  float* vote;
  int64_t vote_stride;
  int32_t* idx;
  int64_t idx_stride;
  int32_t* count;
  float* out;
  float* lse;
  // scratch
  float2* partials;            // [B][nCTA][H]
  unsigned* hist;              // [B][kHistPerSeq]: level l at lvl_off(l)
  unsigned long long* mass;    // [B][kHistPerSeq]
  unsigned* cand_n;            // [B]
  unsigned long long* cands;   // [B][kCandCap]  (key << 32 | ~index)
  int* cta_cnt;                // [B][nCTA][4]  cand-range selected, all selected, ties, selected below s_end
  float* apart;                // o [B][H][parts][nCTA][D / parts], then (max, sum) [B][H][nCTA even]
  float* spill;                // per CTA: logits [tok][wave head]
  float2* wpart;               // per CTA: [segment][scan warp][head] (max, sum exp) of a wave
  int64_t spill_floats;
  int64_t l2_budget;           // bytes of logits one scan wave may keep in L2
  GridSync* gsync;
  int* status;
  uint64_t wait_ns;            // bound on every wait of the launch
  int skip_cta, skip_barrier;  // injected fault: CTA skip_cta leaves at its barrier skip_barrier (-1: none)
  unsigned long long* phase_ns;  // CTA 0's %globaltimer at phase boundaries (debug)
  int dyn_bytes;               // dynamic shared memory of the launch
  int nslot;                   // ring slots of STAGE_BYTES each
  int flag_cap;                // bytes reserved at the tail for selection flags (one per token)
  int* sel_rows;               // per CTA [flag_cap]: its selected tokens, ascending per segment
  int range_attend;            // top-p attention over each CTA's own range: 0 never, 1 when dense, 2 always
  int tcv;                     // tmap_v is encoded: the range attention may run on the tensor cores
};

// -------------------------------------------------------------- grid barrier

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// All CTAs of the cooperative grid meet here. The arrival counter only grows
// (zeroed before each launch): barrier e of the launch is passed once it
// reaches (e + 1) x grid size, so the last CTA to arrive releases the others
// with its own increment. *epoch (shared memory, thread 0 only) counts this
// CTA's barriers. Every wait is bounded by limit_ns. False after a time-out or
// an abort raised by another CTA; the caller then returns. A host-injected
// fault (skip_cta, skip_barrier >= 0, one launch only) makes CTA skip_cta leave
// at its barrier skip_barrier without arriving, so that the others' bounded
// wait runs out: the time-out path can be tested without hanging anything.
__device__ __noinline__ bool grid_sync(GridSync* gs, int* status, unsigned* epoch, uint64_t limit_ns,
                                       int skip_cta, int skip_barrier) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const unsigned target = (*epoch + 1u) * gridDim.x;
    if ((int)blockIdx.x == skip_cta && (int)*epoch == skip_barrier) {
      ok = 0;
    } else {
      *epoch += 1u;
      fence_acq_rel_gpu();                      // the CTA's writes (ordered by the CTA barrier) first
      if (atomicAdd(&gs->count, 1u) + 1u < target) {
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire(&gs->count) < target) {
          if (ld_acquire(&gs->abort)) {
            ok = 0;
            break;
          }
          if (globaltimer_ns() - t0 > limit_ns) {
            set_error(status, TS_ERR_TIMEOUT);
            atomicExch(&gs->abort, 1u);
            ok = 0;
            break;
          }
          __nanosleep(32);
        }
      }
      fence_acq_rel_gpu();                      // then everything the others wrote before arriving
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// The value index that transpose_reduce<NV, LPR> leaves in `lane`.
template <int NV, int LPR>
__device__ __forceinline__ int reduce_slot(int lane) {
  int base = 0, n = NV;
#pragma unroll
  for (int d = LPR / 2; d >= 1; d >>= 1) {
    if (n > 1) {
      n /= 2;
      if (lane & d) base += n;
    }
  }
  return base;
}

// Block-wide exclusive scan of one int per thread; total in *total.
__device__ __noinline__ int block_scan(int x, int* wsum, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int inc = x;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(kFull, inc, d);
    if (lane >= d) inc += o;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < nw ? wsum[lane] : 0;
    int wi = w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(kFull, wi, d);
      if (lane >= d) wi += o;
    }
    if (lane < nw) wsum[lane] = wi - w;
    if (lane == 31) wsum[32] = wi;
  }
  __syncthreads();
  const int r = wsum[warp] + inc - x;
  total = wsum[32];
  __syncthreads();
  return r;
}

// The number of entries below x1 and below x2 in the ascending list a[0, n) (global or shared
// memory: generic loads), by one warp (32-ary narrowing with ballots; four rounds for a quarter
// of a million entries), so that several lists are searched at once by different warps.
__device__ __noinline__ void warp_lower_bound2(const int32_t* a, int n, int x1, int x2, int& r1, int& r2) {
  const int lane = threadIdx.x & 31;
  int lo1 = 0, hi1 = n, lo2 = 0, hi2 = n;
  while (hi1 - lo1 > 32 || hi2 - lo2 > 32) {   // warp-uniform
    const int st1 = (hi1 - lo1 + 31) / 32, st2 = (hi2 - lo2 + 31) / 32;
    const int p1 = lo1 + lane * st1, p2 = lo2 + lane * st2;
    const int c1 = __popc(__ballot_sync(kFull, p1 < hi1 && a[p1] < x1));
    const int c2 = __popc(__ballot_sync(kFull, p2 < hi2 && a[p2] < x2));
    if (c1 > 0) lo1 = lo1 + (c1 - 1) * st1 + 1;
    hi1 = min(hi1, lo1 + st1);
    if (c2 > 0) lo2 = lo2 + (c2 - 1) * st2 + 1;
    hi2 = min(hi2, lo2 + st2);
  }
  r1 = lo1 + __popc(__ballot_sync(kFull, lo1 + lane < hi1 && a[lo1 + lane] < x1));
  r2 = lo2 + __popc(__ballot_sync(kFull, lo2 + lane < hi2 && a[lo2 + lane] < x2));
}

// The crossing bin of a histogram scan.
struct Cross {
  int bin;                       // bin index, -1 when the total falls short
  unsigned before_c;             // count of everything above it (including the start count)
  unsigned long long before_m;   // fixed-point mass of everything above it
  unsigned hc;                   // its own count
};

// One warp scans a histogram in shared memory from its highest bin down, starting from the
// count c0 and mass m0 of everything above the histogram's range, and returns the first bin
// where the cumulative count reaches need_c (top-k) or the cumulative mass reaches need_m
// (top-p). nbins is a power of two >= 32. Every lane returns the same result.
__device__ __noinline__ Cross find_crossing(const unsigned* hc_, const unsigned long long* hm_, int nbins, bool topp,
                                            unsigned c0, unsigned long long m0, unsigned need_c,
                                            unsigned long long need_m) {
  const int lane = threadIdx.x & 31;
  // lane L sums the bins nbins-1-(L*per + j), j < per (descending vote); the start is rotated
  // by the lane so that the lanes hit different banks
  const int per = nbins / 32;
  unsigned cnt = 0;
  unsigned long long ms = 0;
  for (int jj = 0; jj < per; ++jj) {
    const int j = (jj + lane) & (per - 1);
    const int bin = nbins - 1 - (lane * per + j);
    cnt += hc_[bin];
    if (topp) ms += hm_[bin];
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
  const bool crosses = topp ? (m0 + im - ms < need_m && m0 + im >= need_m) : (c0 + ic - cnt < need_c && c0 + ic >= need_c);
  const unsigned ballot = __ballot_sync(kFull, crosses);
  Cross r{-1, 0u, 0ull, 0u};
  if (ballot == 0u) return r;
  const int L = __ffs(ballot) - 1;
  unsigned cb = c0 + __shfl_sync(kFull, ic - cnt, L);
  unsigned long long mb = m0 + __shfl_sync(kFull, im - ms, L);
  // the crossing lane's bins, 32 at a time, by the whole warp
  for (int j0 = 0; j0 < per; j0 += 32) {
    const int j = j0 + lane;
    const int bin = nbins - 1 - (L * per + j);
    const bool in = j < per;
    const unsigned hc = in ? hc_[bin] : 0u;
    const unsigned long long hm = (in && topp) ? hm_[bin] : 0ull;
    unsigned xc = hc;
    unsigned long long xm = hm;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const unsigned oc = __shfl_up_sync(kFull, xc, d);
      const unsigned long long om = __shfl_up_sync(kFull, xm, d);
      if (lane >= d) {
        xc += oc;
        xm += om;
      }
    }
    const bool here = in && (topp ? (mb + xm >= need_m) : (cb + xc >= need_c));
    const unsigned hb = __ballot_sync(kFull, here);
    if (hb) {
      const int f = __ffs(hb) - 1;
      r.bin = __shfl_sync(kFull, bin, f);
      r.before_c = __shfl_sync(kFull, cb + xc - hc, f);
      r.before_m = __shfl_sync(kFull, mb + xm - hm, f);
      r.hc = __shfl_sync(kFull, hc, f);
      return r;
    }
    cb += __shfl_sync(kFull, xc, 31);
    mb += __shfl_sync(kFull, xm, 31);
  }
  return r;
}

// ------------------------------------------------------------- shared state

struct SeqState {        // per sequence, identical in every CTA
  int n, hit, s_end, ls, lo, hi;   // length, cache hit, segments, selection domain
  int all;                         // every domain token selected
  int done;                        // threshold resolved
  int cand;                        // candidates gathered at the last level
  int tie_mode;                    // resolve exact ties by per-CTA counts
  uint32_t prefix, mask;
  int k_rem, n_gt;
  unsigned long long mass_rem;
  int ties;                        // ties to take in tie mode
  int first_cta, last_cta;         // CTAs whose page range covers the sequence
  int fx_base, fx_stride;          // CTAs fx_base .. + fx_stride - 1 share its fixed attention tokens
  int pg0, pg1;                    // its pages in the concatenated scan space
};

struct Smem {
  SeqState seq[kMaxB];
  int nseg;
  int seg_b[kMaxB], seg_lp0[kMaxB], seg_t0[kMaxB], seg_ntok[kMaxB], seg_pend[kMaxB];
  int p0, p1, ppc, tok_stride, hpw, nwaves, spill_ok, ptot, region;
  int stage_tok[kMaxSlots][16];  // per ring slot: CTA-local first token of each page (-1: unused)
  int stage_nv[kMaxSlots][16];   // valid slots of each page
  int stage_b[kMaxSlots][16];    // its sequence
  int stage_done[kMaxSlots];     // warps finished with the current use of each ring slot
  int slot_last[kMaxSlots];      // the last ring use issued into each slot (-1: none)
  int ct_lo[kMaxB], ct_hi[kMaxB];  // hit: the cached part inside [s_end, ls)
  int pre_c[kMaxB], pre_a[kMaxB];  // selected tokens of the CTAs before mine (candidates, all)
  int tot_c[kMaxB], tot_a[kMaxB];  // and of all CTAs
  int tie_base[kMaxB];             // exact ties in the CTAs before mine, per segment
  int filled[kMaxB], ctc[kMaxB];   // cache entry filled, its cached index count
  int qst[kMaxB];                  // byte offset of sequence b's query staged in dynamic shared memory, or -1
  int ctst[kMaxB];                 // byte offset of its first staged cached index, or -1
  int pf_ok, pf_off[kMaxB + 1];    // attention: my fixed tokens of every sequence prefetched at set-up
  int pf_t[kPreFix], pf_p[kPreFix];  // their indices and page ids
  int x_bin[kMaxB];                // selection: crossing coarse bin of level 0, and the
  unsigned x_c[kMaxB];             // count and mass above it
  unsigned long long x_m[kMaxB];
  float att_m[kMaxAttH], att_l[kMaxAttH], att_c[kMaxAttH];  // attention: running max, sum, round correction
  int use_tc;                      // this launch scans with the tensor cores
  int scan_dyn;                    // its pages are claimed from a shared counter, not partitioned
  int tc_nimg, tc_seq[2];          // query images of the scan and the sequence of each
  int tc_img_of[kMaxB];            // image of sequence b, or -1
  uint32_t tmem;                   // TMEM base address of the accumulators
  int acc_tl[2][2], acc_nv[2][2], acc_sg[2];  // per accumulator buffer: first token and valid rows of each
                                              // page of the tile, segment
  union {
    int my_pages[kMaxPagesCta];  // physical page ids of my range (first kMaxPagesCta pages)
    struct {                     // balanced attention (my_pages unused then): a sequence's per-CTA
      int pref[kMaxGrid + 1];    // offsets in its concatenated lists, and each CTA's count below s_end
      int nlo[kMaxGrid];
      int range_b[kMaxB];        // sequence b attended over each CTA's own range (range_attend)
    } bal;
  };
  int timed_out;
  unsigned gepoch;                 // grid barriers passed (thread 0)
  int wsum[33];
  int flag;
  float red_f[3][32];
  int red_i[3][32];
  int sel_a[kMaxB], sel_c[kMaxB], sel_lo[kMaxB];  // per segment: my selected tokens, those in [s_end, ls),
                                                  // those below s_end (list in the scratch, ascending)
  int toks[kMaxRound];
  int tval[kMaxRound];
  int my_seg_of[kMaxB];    // segment of sequence b in this CTA, or -1
};

// --------------------------------------------------------------- the kernel

// CTA 0 records the time it reaches phase boundary i (0..63), for diagnosis: 0 start, 5 lengths
// read, 6 cache test, 7 partition, 1 set-up done; scan wave w: 2 + 3 w scanned, 3 + 3 w
// statistics, 4 + 3 w barrier passed; 13 / 14 vote partials / normalisers, 20 votes done;
// 28 + l histogram level l built, 21 levels, 22 candidates, 23 flags; 10 last gather landed,
// 9 last round list built, 11 attended, 24 partials written, 25 last barrier, 26 merged, 27
// end. Finer points: 32 vote chunk landed; 33 + 4 l / 34 + 4 l / 35 + 4 l / 36 + 4 l level l
// histogram started / zeroed / counted (added: 28 + l) / barrier passed; 45 / 46 coarse / fine bins
// fetched; 47 classified, 48 candidate barrier passed, 49 candidates fetched, 50 ranked; 51
// attention queries loaded, 52 fixed rows requested, 53 own rows requested; 54 first merge
// item fetched, 55 counts read; the first attention round's 9, 10, 16 and its end again in 8, 12,
// 19 and 31. Over all CTAs, the latest to finish the tensor-core scan (56), the
// votes (57), the classification (58) and the selection flags (59); 61..63: which CTA that was
// for 57..59. (The marks of waves past the first share slots 5..19 with the
// others; slots 17 and 18 also take the latest start and end over all CTAs.)
#define TS_MARK(i)                                                     \
  do {                                                                 \
    if (c == 0 && tid == 0 && a.phase_ns) a.phase_ns[i] = globaltimer_ns(); \
  } while (0)
// the latest time over all CTAs at which one reaches phase boundary i (the clock only grows, so
// the slot needs no reset between launches)
#define TS_LAST(i)                                                                  \
  do {                                                                              \
    if (tid == 0 && a.phase_ns) atomicMax(&a.phase_ns[i], (unsigned long long)globaltimer_ns()); \
  } while (0)
// and which CTA it was: the low 48 bits of the clock above the CTA index (slot i + 4)
#define TS_LAST_CTA(i)                                                                         \
  do {                                                                                         \
    if (tid == 0 && a.phase_ns)                                                                \
      atomicMax(&a.phase_ns[(i) + 4], ((globaltimer_ns() & ((1ull << 48) - 1)) << 8) | (unsigned)c); \
  } while (0)

// One wave of the CUDA-core scan (geometries and launches without the tensor-core scan): the
// wave's KV heads of my pages stream through the ring of 1-D bulk copies, every warp holds the
// G queries of one KV head in registers, writes logits and keeps per-warp (max, sum exp);
// then the per (segment, head) partials. Out of line so that its register pressure stays
// here. False after a time-out (the abort word is raised).
template <typename KT, int D, int HKV, int G>
__device__ __noinline__ bool cuda_scan_wave(const StepKArgs& a, Smem& sm, unsigned char* ring, uint64_t* full, int wv,
                                             int& stage_seq) {
  using S = StepShape<KT, D, HKV, G>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, nCTA = gridDim.x;
  const int B = a.B, H = a.H;
  const int nslot = a.nslot;
  const int hpw = sm.hpw, HW = hpw * G;
  const int pps = HKV / hpw;                       // pages per stage
  const int np = sm.p1 - sm.p0;
  const int nstages = (np + pps - 1) / pps;
  const int slab = hpw * S::P * S::ROW_BYTES;      // bytes of one page's heads of the wave
  float* eb = a.spill + (size_t)c * sm.region;     // my logits, token-major [tstride][HW]
  float2* wp = a.wpart + (size_t)c * B * S::NCW * G;  // [segment][warp][head of the warp] (max, sum exp)
  const uint64_t pol = l2_evict_first_policy();
  // Issues ring use u (pages si*pps.. of my range, the wave's heads of each) into slot
  // u % nslot: metadata first, then arrive.expect_tx, then the copies.
  auto issue = [&](int u, int si, int g0) {
    const int s = u % nslot;
    sm.slot_last[s] = u;
    uint32_t bytes = 0;
    int pages[16];
    for (int j = 0; j < pps; ++j) {
      const int gp = sm.p0 + si * pps + j;
      sm.stage_tok[s][j] = -1;
      sm.stage_nv[s][j] = 0;
      sm.stage_b[s][j] = 0;
      pages[j] = -1;
      if (gp >= sm.p1) continue;
      int seg = 0;
      while (seg + 1 < sm.nseg && gp >= sm.seg_pend[seg]) ++seg;
      const int b = sm.seg_b[seg];
      const int lp = gp - sm.seq[b].pg0;
      const int page = (gp - sm.p0 < kMaxPagesCta) ? sm.my_pages[gp - sm.p0]
                                                    : a.page_table[(size_t)b * a.pt_stride + lp];
      sm.stage_tok[s][j] = (gp - sm.p0) * S::P;
      sm.stage_b[s][j] = b;
      if (page < 0 || (int64_t)page >= a.num_pages) {
        set_error(a.status, TS_ERR_PAGE_OOB);
        continue;
      }
      sm.stage_nv[s][j] = min(S::P, sm.seq[b].n - lp * S::P);
      pages[j] = page;
      bytes += (uint32_t)slab;
    }
    mbar_arrive_expect_tx(&full[s], bytes);
    for (int j = 0; j < pps; ++j) {
      if (pages[j] < 0) continue;
      bulk_g2s_hint(ring + (size_t)s * S::STAGE_BYTES + (size_t)j * slab,
                    a.k_pool + ((size_t)pages[j] * HKV + g0) * S::P * S::ROW_BYTES, (uint32_t)slab, &full[s], pol);
    }
  };
  const int g0 = wv * hpw;
  if (tid == 0)  // the ring is idle between waves: fill it
    for (int si = 0; si < min(nslot, nstages); ++si) issue(stage_seq + si, si, g0);
  {
    // ---- warp -> KV head g0 + gi, ROWS rows of that head in each stage
    const int wph = S::NCW / hpw;
    const int gi = warp / wph;
    const int row0 = (warp % wph) * S::ROWS;     // ROWS divides P or P divides ROWS
    const int lrow = lane / S::LPR, lin = lane % S::LPR;
    float qr[S::GP][S::DPL];
#pragma unroll
    for (int j = 0; j < S::GP; ++j)
#pragma unroll
      for (int e = 0; e < S::DPL; ++e) qr[j][e] = 0.f;
    int qb = -1;                                 // sequence whose queries sit in qr
    const bool writer = (lin & (S::LPR / S::GP - 1)) == 0;
    const int mywhich = reduce_slot<S::GP, S::LPR>(lane);   // the head this lane's sums belong to
    // (max, sum exp) of this warp's rows of each of my segments, this wave's heads
    int cur_sg = -1;
    float run_m = -INFINITY;
    KahanF run_z;
    for (int i = lane; i < sm.nseg * G; i += 32)
      wp[((size_t)(i / G) * S::NCW + warp) * G + (i % G)] = make_float2(-INFINITY, 0.f);
    __syncwarp();
    auto flush = [&](int sg) {
      if (sg >= 0 && lrow == 0 && writer && mywhich < G)
        wp[((size_t)sg * S::NCW + warp) * G + mywhich] = make_float2(run_m, run_z.s - run_z.c);
    };
    for (int si = 0; si < nstages; ++si) {
      const int u = stage_seq + si;
      const int s = u % nslot;
      if (!mbar_wait(&full[s], (u / nslot) & 1, a.wait_ns)) {
        set_error(a.status, TS_ERR_TIMEOUT);
        sm.timed_out = 1;
        break;
      }
      const KT* st = reinterpret_cast<const KT*>(ring + (size_t)s * S::STAGE_BYTES);
#pragma unroll
      for (int it = 0; it < S::ITERS; ++it) {
        const int r = row0 + it * S::RPW + lrow;   // row among this head's pps*16 rows
        const int j = r / S::P, slot = r % S::P;   // all lanes of a step share the page j
        const int tl = sm.stage_tok[s][j];
        if (tl < 0) continue;                    // past my range (uniform in the warp)
        const int nv = sm.stage_nv[s][j];
        const int bq = sm.stage_b[s][j];
        if (bq != qb) {                          // new sequence: its queries of this KV head
#pragma unroll
          for (int jj = 0; jj < S::GP; ++jj) {
            const float* qh = a.q + ((size_t)bq * H + (g0 + gi) * G + jj) * D;
#pragma unroll
            for (int cc = 0; cc < S::CPL; ++cc)
#pragma unroll
              for (int e = 0; e < S::EPC; ++e)
                qr[jj][cc * S::EPC + e] = (jj < G) ? qh[(lin + cc * S::LPR) * S::EPC + e] : 0.f;
          }
          qb = bq;
        }
        const int sg = sm.my_seg_of[bq];
        if (sg != cur_sg) {                      // new segment: its running statistics
          flush(cur_sg);
          cur_sg = sg;
          run_m = -INFINITY;
          run_z = KahanF();
        }
        const KT* rp = st + ((size_t)(j * hpw + gi) * S::P + slot) * D;
        float acc0[S::GP], acc1[S::GP];
#pragma unroll
        for (int jj = 0; jj < S::GP; ++jj) acc0[jj] = acc1[jj] = 0.f;
#pragma unroll
        for (int cc = 0; cc < S::CPL; ++cc) {
          float kf[S::EPC];
          KV<KT>::unpack(lds128(rp + (lin + cc * S::LPR) * S::EPC), kf);
#pragma unroll
          for (int jj = 0; jj < S::GP; ++jj)
#pragma unroll
            for (int e = 0; e < S::EPC; ++e) {
              if ((S::CPL == 2 ? cc : (e & 1)) == 0)
                acc0[jj] = fmaf(qr[jj][cc * S::EPC + e], kf[e], acc0[jj]);
              else
                acc1[jj] = fmaf(qr[jj][cc * S::EPC + e], kf[e], acc1[jj]);
            }
        }
        float v[S::GP];
#pragma unroll
        for (int jj = 0; jj < S::GP; ++jj) v[jj] = acc0[jj] + acc1[jj];
        int which;
        const float dot = transpose_reduce<S::GP, S::LPR>(v, lane, which);
        const float x = slot < nv ? fmaf(dot, a.scale_l2, dot * a.scale_l2_lo) : -INFINITY;
        if (writer && which < G) eb[(size_t)(tl + slot) * HW + gi * G + which] = x;
        // running max and compensated sum of exp over the rows of this step (lanes of equal `which`)
        float mi = x;
#pragma unroll
        for (int d = S::LPR; d < 32; d <<= 1) mi = fmaxf(mi, __shfl_xor_sync(kFull, mi, d));
        const float mn = fmaxf(run_m, mi);
        float ex = mn > -INFINITY ? exp2f(x - mn) : 0.f;
#pragma unroll
        for (int d = S::LPR; d < 32; d <<= 1) ex += __shfl_xor_sync(kFull, ex, d);
        if (mn > run_m && run_m > -INFINITY) {
          const float f = exp2f(run_m - mn);
          run_z.s *= f;
          run_z.c *= f;
        }
        run_z.add(ex);
        run_m = mn;
      }
      // the last warp done with this use of the slot refills it
      __syncwarp();
      if (lane == 0) {
        if (atomicAdd(&sm.stage_done[s], 1) == S::NCW - 1) {
          sm.stage_done[s] = 0;
          if (si + nslot < nstages) issue(u + nslot, si + nslot, g0);
        }
      }
    }
    flush(cur_sg);
  }
  stage_seq += nstages;
  __syncthreads();
  if (sm.timed_out) {
    if (tid == 0) {
      // copies issued but never consumed land before the CTA leaves
      for (int ss = 0; ss < nslot; ++ss)
        if (sm.slot_last[ss] >= 0) mbar_wait(&full[ss], (sm.slot_last[ss] / nslot) & 1, a.wait_ns);
      atomicExch(&a.gsync->abort, 1u);   // the others leave at their next barrier
    }
    return false;
  }
  TS_MARK(2 + 3 * min(wv, 5));

  // ---- per (segment, wave head): combine the warps' (max, sum exp) -> partials
  {
    const int wph = S::NCW / hpw;
    for (int item = warp; item < sm.nseg * HW; item += S::NW) {
      const int sg = item / HW, hl = item % HW;
      const int gi = hl / G, w = hl % G;
      float2 mz = make_float2(-INFINITY, 0.f);
      if (lane < wph) mz = wp[((size_t)sg * S::NCW + gi * wph + lane) * G + w];
      const float m = warp_max(mz.x);
      const float z = warp_sum_comp((m > -INFINITY && mz.y > 0.f) ? mz.y * exp2f(mz.x - m) : 0.f);
      if (lane == 0) {
        float2* pr = a.partials + (((size_t)sm.seg_b[sg] * nCTA + c) * S::PV) * H + g0 * G + hl;
        pr[0] = make_float2(m, z);
        if (S::PV == 2) pr[H] = make_float2(-INFINITY, 0.f);
      }
    }
  }
  return true;
}


// Ring slots of the range attention (hit: pages of K too) that fit `stage_bytes`, or 0 below two.
template <typename KT, int D, int HKV, int G, bool HIT>
__host__ __device__ constexpr int range_slots(int stage_bytes, int flag_cap) {
  constexpr int VPAGE = HKV * kPage * D * (int)sizeof(KT), LROWS = kPage * HKV * G * 4;
  constexpr int SLOT = (HIT ? 2 : 1) * VPAGE + 2 * LROWS;
  const int n = (stage_bytes - kRangeSlots * 8 - (3 * (flag_cap / kPage) + kRangeSlots) * 4) / SLOT;
  return n < 2 ? 0 : (n > kRangeSlots ? kRangeSlots : n);
}

// Range attention, for dense selections (top-p keeping a large share of a sequence): I attend the
// tokens of a range of pages of sequence b that are selected, sinks or in the window.
//  * A miss (HIT false): the range is my own scanned segment sgi, the tokens are those flagged
//    selected, and their logits are the scan's (base 2, still in my scratch region), so K is not
//    read again; each page with an attended token brings its V rows of every KV head and its 16
//    logit rows into a ring by bulk copy.
//  * A hit of the Selection Cache (HIT true): nothing was scanned; the sequence's pages are split
//    evenly over the CTAs, the tokens are the cached part (an ascending list) with the sinks and
//    the window, and each page brings its K and V rows; the warps of a KV head compute its 16
//    tokens' logits for the G heads (as the scan does: base 2, fp32).
// Weights are 2^(l - m) against a running max m per head, which moves only when a logit passes it
// by more than kRescaleGap (then sums and outputs are rescaled once). A thread owns (KV head, 8
// columns) for the G query heads of that KV head over a share of each page's tokens, in packed
// fp32 pairs. The CTA's partial (o, max in natural units, sum) goes where the gathered attention
// puts it. False after a time-out (recorded, the abort word raised, the copies in flight waited
// for).
template <typename KT, int D, int HKV, int G, bool HIT>
__device__ __noinline__ bool range_attend(const StepKArgs& a, Smem& sm, unsigned char* stage, int stage_bytes,
                                          const uint8_t* selflag, int b, int sgi, float* ao, float2* aml,
                                          int nCTAp, int dq) {
  using S = StepShape<KT, D, HKV, G>;
  constexpr int HQ = HKV * G, D4 = D / 4, D8 = D / 8, PVT = HKV * D8, NSPL = S::THREADS / PVT;
  constexpr int EPC = KV<KT>::kPerChunk;             // elements of a 16-byte chunk of V
  constexpr int EPL = D / 32;                        // hit scores: dimensions per lane
  constexpr int NWG = S::NW / HKV;                   // hit scores: warps per KV head
  constexpr int VPAGE = S::STAGE_BYTES;              // one V (or K) page of every KV head, [g][16][D]
  constexpr int LROWS = S::P * HQ * 4;               // its 16 logit rows [16][H]
  constexpr int SLOT = (HIT ? 2 : 1) * VPAGE + 2 * LROWS;   // [V][K (hit)][logits][weights]
  static_assert(S::THREADS % PVT == 0 && S::P * HQ <= S::THREADS && SLOT % 16 == 0 && D % 8 == 0 && 8 % EPC == 0,
                "range attention layout");
  constexpr float kLn2 = 0.693147180559945309f;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, c = blockIdx.x, nCTA = gridDim.x;
  const SeqState& st = sm.seq[b];
  int lp0, ntok;
  const uint8_t* fl = nullptr;
  const float* eb = nullptr;
  if constexpr (HIT) {
    const int npg_seq = (st.n + S::P - 1) / S::P;
    const int pa = (int)((int64_t)c * npg_seq / nCTA), pb = (int)((int64_t)(c + 1) * npg_seq / nCTA);
    lp0 = pa;
    ntok = max(0, min((pb - pa) * S::P, st.n - pa * S::P));
  } else {
    const int t0l = sm.seg_t0[sgi];
    lp0 = sm.seg_lp0[sgi];
    ntok = sm.seg_ntok[sgi];
    fl = selflag + t0l;                                                // my flags of the segment
    eb = a.spill + (size_t)c * sm.region + (size_t)t0l * HQ;           // its logit rows
  }
  const int npg = (ntok + S::P - 1) / S::P;
  const int nslot = range_slots<KT, D, HKV, G, HIT>(stage_bytes, a.flag_cap);   // >= 2: checked by the caller
  uint64_t* bars = reinterpret_cast<uint64_t*>(stage + (size_t)nslot * SLOT);
  int* plist = reinterpret_cast<int*>(bars + kRangeSlots);            // my pages with an attended token
  int* ppage = plist + a.flag_cap / S::P;                              // and their page ids
  int* pv_ok = ppage + a.flag_cap / S::P;                              // per slot: its pages are valid
  uint32_t* pmask = reinterpret_cast<uint32_t*>(pv_ok + kRangeSlots);  // hit: attended tokens per page
  auto attended = [&](int i) -> bool {                                 // token lp0 * 16 + i of the sequence
    if constexpr (HIT) {
      return i < ntok && ((pmask[i >> 4] >> (i & 15)) & 1u);
    } else {
      const int t = lp0 * S::P + i;
      return i < ntok && (t < st.s_end || t >= st.ls || fl[i] == 1);
    }
  };
  if constexpr (HIT) {
    // the attended tokens of my pages: sinks, window and the cached part inside my range
    const int tb = lp0 * S::P;
    #pragma unroll 1
    for (int j = tid; j < npg; j += S::THREADS) pmask[j] = 0u;
    __syncthreads();
    #pragma unroll 1
    for (int i = tid; i < ntok; i += S::THREADS)
      if (tb + i < st.s_end || tb + i >= st.ls) atomicOr(&pmask[i >> 4], 1u << (i & 15));
    const int32_t* ctb = a.ct + (size_t)b * a.cap + sm.ct_lo[b];
    const int nct = sm.ct_hi[b] - sm.ct_lo[b];
    if (warp == 0) {
      int r1, r2;
      warp_lower_bound2(ctb, nct, tb, tb + ntok, r1, r2);
      if (lane == 0) {
        sm.red_i[0][0] = r1;
        sm.red_i[0][1] = r2;
      }
    }
    __syncthreads();
    #pragma unroll 1
    for (int j = sm.red_i[0][0] + tid; j < sm.red_i[0][1]; j += S::THREADS) {
      const int i = ctb[j] - tb;
      atomicOr(&pmask[i >> 4], 1u << (i & 15));
    }
    __syncthreads();
  }

  // ---- the pages of my segment with at least one attended token, ascending
  int nlist = 0;
  #pragma unroll 1
  for (int j0 = 0; j0 < npg; j0 += S::THREADS) {
    const int j = j0 + tid;
    int any = 0;
    if (j < npg) {
      if constexpr (HIT) {
        any = pmask[j] != 0u;
      } else {
        #pragma unroll 1
        for (int r = 0; r < S::P && !any; ++r) any = attended(j * S::P + r);
      }
    }
    int tot;
    const int pos = block_scan(any, sm.wsum, tot);
    if (any) {
      plist[nlist + pos] = j;
      ppage[nlist + pos] = a.page_table[(size_t)b * a.pt_stride + lp0 + j];
    }
    nlist += tot;
  }
  if (nlist == 0) {
    if (tid < HQ) aml[((size_t)b * HQ + tid) * nCTAp + c] = make_float2(-INFINITY, 0.f);
    fence_proxy_async_global();
    __syncthreads();
    return true;
  }
  if (tid == 0) {
    #pragma unroll 1
    for (int s = 0; s < nslot; ++s) mbar_init(&bars[s], 1);
    mbar_fence_init();
  }
  if (tid < HQ) sm.att_m[tid] = -INFINITY;
  __syncthreads();
  // page k of the list into slot k % nslot (thread 0)
  auto issue = [&](int k) {
    const int s = k % nslot, j = plist[k], page = ppage[k];
    const bool ok = page >= 0 && (int64_t)page < a.num_pages;
    pv_ok[s] = ok;
    unsigned char* dst = stage + (size_t)s * SLOT;
    if constexpr (HIT) {
      mbar_arrive_expect_tx(&bars[s], ok ? 2 * VPAGE : 0);
      if (ok) {
        bulk_g2s(dst, a.v_pool + (size_t)page * VPAGE, VPAGE, &bars[s]);
        bulk_g2s(dst + VPAGE, a.k_pool + (size_t)page * VPAGE, VPAGE, &bars[s]);
      }
    } else {
      mbar_arrive_expect_tx(&bars[s], (ok ? VPAGE : 0) + LROWS);
      if (ok) bulk_g2s(dst, a.v_pool + (size_t)page * VPAGE, VPAGE, &bars[s]);
      bulk_g2s(dst + VPAGE, eb + (size_t)j * S::P * HQ, LROWS, &bars[s]);
    }
    if (!ok) set_error(a.status, TS_ERR_PAGE_OOB);
  };
  // hit scores: warp -> (KV head gw, tokens wsl, wsl + NWG, ...), its G queries in registers
  const int gw = warp % HKV, wsl = warp / HKV;
  float qreg[S::GP][EPL];
  if constexpr (HIT) {
#pragma unroll
    for (int h = 0; h < S::GP; ++h)
#pragma unroll
      for (int e = 0; e < EPL; ++e)
        qreg[h][e] = h < G ? a.q[((size_t)b * HQ + gw * G + h) * D + lane * EPL + e] : 0.f;
  }
  if (tid == 0) {
    fence_proxy_async_global();
    #pragma unroll 1
    for (int k = 0; k < min(nslot, nlist); ++k) issue(k);
  }
  // weights: thread (row r, head h); outputs: thread (split sp, KV head g, columns 8 d8 .. 8 d8 + 7)
  const bool wt = tid < S::P * HQ;
  const int wr = tid / HQ, wh = tid % HQ;
  const int sp = tid / PVT, gd = tid % PVT, g = gd / D8, d8 = gd % D8;
  KahanF lsum;
  uint64_t acc[G][4];   // head jj, columns (8 d8 + 2 e, 8 d8 + 2 e + 1)
#pragma unroll
  for (int jj = 0; jj < G; ++jj) acc[jj][0] = acc[jj][1] = acc[jj][2] = acc[jj][3] = 0ull;   // (+0, +0)
  #pragma unroll 1
  for (int k = 0; k < nlist; ++k) {
    const int s = k % nslot, j = plist[k];
    const bool landed = mbar_wait(&bars[s], (k / nslot) & 1, a.wait_ns);
    unsigned char* slot = stage + (size_t)s * SLOT;
    const KT* Vp = reinterpret_cast<const KT*>(slot);
    float* Lp = reinterpret_cast<float*>(slot + (HIT ? 2 : 1) * VPAGE);
    float* Wp = Lp + S::P * HQ;
    if constexpr (HIT) {
      // the page's logits for every query head (rows past the sequence or of a page outside the
      // pool are computed but never attended)
      const KT* Kp = reinterpret_cast<const KT*>(slot + VPAGE);
      #pragma unroll 1
      for (int r = wsl; r < S::P; r += NWG) {
        float kf[EPL];
        load_elems<KT, EPL>(Kp + ((size_t)gw * S::P + r) * D + lane * EPL, kf);
        float accq[S::GP];
#pragma unroll
        for (int h = 0; h < S::GP; ++h) {
          float x = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) x = fmaf(qreg[h][e], kf[e], x);
          accq[h] = x;
        }
        int which;
        const float dot = transpose_reduce<S::GP, 32>(accq, lane, which);
        if ((lane & (32 / S::GP - 1)) == 0 && which < G)
          Lp[r * HQ + gw * G + which] = fmaf(dot, a.scale_l2, dot * a.scale_l2_lo);
      }
      __syncthreads();
    }
    float xl = -INFINITY;
    bool att = false;
    if (wt && landed) {
      att = attended(j * S::P + wr) && pv_ok[s];
      if (att) xl = Lp[wr * HQ + wh];
    }
    const bool need = att && xl - sm.att_m[wh] > kRescaleGap;   // (a max of -inf always rescales)
    if (__syncthreads_or(!landed || need)) {
      if (__syncthreads_or(!landed)) {
        if (tid == 0) {
          set_error(a.status, TS_ERR_TIMEOUT);
          atomicExch(&a.gsync->abort, 1u);
          const int issued = min(nlist, k == 0 ? nslot : k - 1 + nslot);
          #pragma unroll 1
          for (int kk = k; kk < issued; ++kk)                    // copies in flight land first
            mbar_wait(&bars[kk % nslot], (kk / nslot) & 1, a.wait_ns);
        }
        return false;
      }
      // a new running max for the heads that passed it: the page's max, then the corrections
      if (wt) Wp[tid] = xl;
      __syncthreads();
      if (tid < HQ) {
        float pm = -INFINITY;
        #pragma unroll 1
        for (int r = 0; r < S::P; ++r) pm = fmaxf(pm, Wp[r * HQ + tid]);
        const float m0 = sm.att_m[tid];
        const float mn = fmaxf(m0, pm);
        sm.att_c[tid] = m0 == -INFINITY ? 0.f : exp2f(m0 - mn);
        sm.att_m[tid] = mn;
      }
      __syncthreads();
      if (wt) {
        lsum.s *= sm.att_c[wh];
        lsum.c *= sm.att_c[wh];
      }
#pragma unroll
      for (int jj = 0; jj < G; ++jj) {
        const float f = sm.att_c[g * G + jj];
        const uint64_t ff = pack_f2(f, f);
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[jj][e] = fma_f2(acc[jj][e], ff, 0ull);
      }
    }
    // the slot of page k - 1 is free (every thread has passed its outputs): refill it
    if (tid == 0 && k >= 1 && k - 1 + nslot < nlist) issue(k - 1 + nslot);
    if (wt) {
      const float w = att ? exp2f(xl - sm.att_m[wh]) : 0.f;
      Wp[tid] = w;
      lsum.add(w);
    }
    __syncthreads();
    // only the page's rows of the sequence (past its end a row may hold anything, and a zero weight
    // times a NaN is a NaN), none of a page outside the pool
    const int nvr = pv_ok[s] ? min(S::P, ntok - j * S::P) : 0;
    #pragma unroll 2
    for (int r = sp; r < nvr; r += NSPL) {
      float v[8];
#pragma unroll
      for (int ch = 0; ch < 8 / EPC; ++ch)
        KV<KT>::unpack(lds128(Vp + ((size_t)g * S::P + r) * D + d8 * 8 + ch * EPC), v + ch * EPC);
      uint64_t vp[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) vp[e] = pack_f2(v[2 * e], v[2 * e + 1]);
      float wv[G];
      if constexpr (G % 4 == 0) {                       // 16-byte aligned: rows of H floats, G | H
#pragma unroll
        for (int jj = 0; jj < G; jj += 4) {
          const float4 w4 = *reinterpret_cast<const float4*>(Wp + r * HQ + g * G + jj);
          wv[jj] = w4.x;
          wv[jj + 1] = w4.y;
          wv[jj + 2] = w4.z;
          wv[jj + 3] = w4.w;
        }
      } else {
#pragma unroll
        for (int jj = 0; jj < G; ++jj) wv[jj] = Wp[r * HQ + g * G + jj];
      }
#pragma unroll
      for (int jj = 0; jj < G; ++jj) {
        const uint64_t wb = pack_f2(wv[jj], wv[jj]);
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[jj][e] = fma_f2(vp[e], wb, acc[jj][e]);
      }
    }
  }
  // ---- every copy has landed and been read: the splits' outputs and the rows' sums, reduced in a
  // fixed order into the CTA's partial
  __syncthreads();
  if (tid == 0)
    #pragma unroll 1
    for (int s = 0; s < nslot; ++s) mbar_inval(&bars[s]);
  float* red = reinterpret_cast<float*>(stage);                  // [HQ][D]: the splits added in order
  float* lred = red + (size_t)HQ * D;                            // [16][HQ]
  if (wt) lred[tid] = lsum.s - lsum.c;
  #pragma unroll 1
  for (int x = 0; x < NSPL; ++x) {
    if (sp == x)
#pragma unroll
      for (int jj = 0; jj < G; ++jj) {
        float4* dst = reinterpret_cast<float4*>(red + (size_t)(g * G + jj) * D + d8 * 8);
        float o[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) unpack_f2(acc[jj][e], o[2 * e], o[2 * e + 1]);
        float4 p0 = make_float4(o[0], o[1], o[2], o[3]), p1 = make_float4(o[4], o[5], o[6], o[7]);
        if (x > 0) {
          const float4 q0 = dst[0], q1 = dst[1];
          p0 = make_float4(q0.x + p0.x, q0.y + p0.y, q0.z + p0.z, q0.w + p0.w);
          p1 = make_float4(q1.x + p1.x, q1.y + p1.y, q1.z + p1.z, q1.w + p1.w);
        }
        dst[0] = p0;
        dst[1] = p1;
      }
    __syncthreads();
  }
  const int Dq = D / dq;
  #pragma unroll 1
  for (int it = tid; it < HQ * D4; it += S::THREADS) {
    const int h = it / D4, e4 = it % D4, qq = e4 / (Dq / 4);
    reinterpret_cast<float4*>(ao + ((((size_t)b * HQ + h) * dq + qq) * nCTA + c) * Dq)[e4 % (Dq / 4)] =
        reinterpret_cast<const float4*>(red + (size_t)h * D)[e4];
  }
  if (tid < HQ) {
    KahanF z;
    #pragma unroll 1
    for (int r = 0; r < S::P; ++r) z.add(lred[r * HQ + tid]);
    const float m2 = sm.att_m[tid], l = z.s - z.c;
    aml[((size_t)b * HQ + tid) * nCTAp + c] =
        (m2 > -INFINITY && l > 0.f) ? make_float2(m2 * kLn2, l) : make_float2(-INFINITY, 0.f);
  }
  fence_proxy_async_global();
  __syncthreads();
  return true;
}

// Ring slots of the tensor-core range attention that fit `stage_bytes` of shared memory (its
// base aligned up to 1024 bytes at most 1023 bytes on), or 0 when fewer than two fit.
template <int D, int HKV, int G>
__host__ __device__ constexpr int range_tc_slots(int stage_bytes, int flag_cap) {
  constexpr int VPAGE = HKV * kPage * D * 2, LROWS = kPage * HKV * G * 4, BBUF = HKV * 16 * 32;
  const int fixed = 1023 + 2 * BBUF + (kRangeSlotsTC + 2) * 8 + (2 * (flag_cap / kPage) + kRangeSlotsTC) * 4;
  const int n = (stage_bytes - fixed) / (VPAGE + LROWS);
  return n < 2 ? 0 : (n > kRangeSlotsTC ? kRangeSlotsTC : n);
}

// Range attention on the tensor cores (bf16 pools, d = 128): range_attend with O^T = V^T W per page
// and KV head on tcgen05. The V page arrives by tiled TMA in the scan's 128-byte-swizzled layout
// (rows (KV head g, token), 64 columns per half); read MN-major it is A, with M the 128 columns of
// d and K the page's 16 tokens. B holds the KV head's weights as two bf16 terms per query head,
// hi in row j and lo in row G + j, so that every product is exact in fp32: 16 rows of 16 tokens,
// K-major without swizzle (core matrices of 8 rows x 8 tokens; the second 8 tokens 128 bytes on,
// the second 8 rows 256 bytes on). The accumulator of KV head g is TMEM columns [16 g, 16 g + 16)
// over lanes d; query head g G + j is the sum of its two columns. A move of the running max
// rescales the accumulators in TMEM once the MMAs issued so far have completed. False after a
// time-out (recorded, the abort word raised, the copies and MMAs in flight waited for, TMEM freed).
template <typename KT, int D, int HKV, int G>
__device__ __noinline__ bool range_attend_tc(const StepKArgs& a, Smem& sm, unsigned char* stage_raw, int stage_bytes,
                                             const uint8_t* selflag, int b, int sgi, float* ao, float2* aml,
                                             int nCTAp, int dq) {
  using S = StepShape<KT, D, HKV, G>;
  constexpr int HQ = HKV * G, D4 = D / 4;
  constexpr int ROWS = HKV * S::P;                 // rows (g, token) of a V page
  constexpr int VHALF = ROWS * 128;                // its 64-column half
  constexpr int VPAGE = 2 * VHALF;
  constexpr int LROWS = S::P * HQ * 4;             // the page's logit rows [16][H]
  constexpr int BTILE = 16 * 32;                   // one KV head's weight rows (16 tokens each)
  constexpr int BBUF = HKV * BTILE;
  constexpr int NCOL = HKV * 16;
  constexpr int TCOLS = NCOL <= 32 ? 32 : (NCOL <= 64 ? 64 : (NCOL <= 128 ? 128 : 256));
  static_assert(D == 128 && 2 * G <= 16 && S::P * HQ <= S::THREADS && S::NW >= 4 && NCOL <= 256,
                "tensor-core range attention");
  constexpr float kLn2 = 0.693147180559945309f;
  constexpr uint32_t idesc = idesc_bf16_f32_amn(128, 16);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, c = blockIdx.x, nCTA = gridDim.x;
  const SeqState& st = sm.seq[b];
  const int t0l = sm.seg_t0[sgi], lp0 = sm.seg_lp0[sgi], ntok = sm.seg_ntok[sgi];
  const int npg = (ntok + S::P - 1) / S::P;
  const uint8_t* fl = selflag + t0l;
  const float* eb = a.spill + (size_t)c * sm.region + (size_t)t0l * HQ;
  const int nslot = range_tc_slots<D, HKV, G>(stage_bytes, a.flag_cap);   // >= 2: checked by the caller
  unsigned char* vslots =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(stage_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char* bbuf = vslots + (size_t)nslot * VPAGE;                  // two buffers of weights
  float* lslots = reinterpret_cast<float*>(bbuf + 2 * BBUF);
  uint64_t* full = reinterpret_cast<uint64_t*>(lslots + (size_t)nslot * (LROWS / 4));
  uint64_t* mmad = full + kRangeSlotsTC;                                 // [2]: MMAs of a weight buffer done
  int* plist = reinterpret_cast<int*>(mmad + 2);
  int* ppage = plist + a.flag_cap / S::P;
  int* pv_ok = ppage + a.flag_cap / S::P;
  auto attended = [&](int i) -> bool {
    const int t = lp0 * S::P + i;
    return i < ntok && (t < st.s_end || t >= st.ls || fl[i] == 1);
  };
  auto b_off = [](int n, int k) -> int {          // byte of B element (row n, token k)
    return (n >> 3) * 256 + (k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2;
  };

  // ---- the pages of my segment with at least one attended token, ascending, and their ids
  int nlist = 0;
  #pragma unroll 1
  for (int j0 = 0; j0 < npg; j0 += S::THREADS) {
    const int j = j0 + tid;
    int any = 0;
    if (j < npg)
      #pragma unroll 1
      for (int r = 0; r < S::P && !any; ++r) any = attended(j * S::P + r);
    int tot;
    const int pos = block_scan(any, sm.wsum, tot);
    if (any) {
      plist[nlist + pos] = j;
      ppage[nlist + pos] = a.page_table[(size_t)b * a.pt_stride + lp0 + j];
    }
    nlist += tot;
  }
  if (nlist == 0) {
    if (tid < HQ) aml[((size_t)b * HQ + tid) * nCTAp + c] = make_float2(-INFINITY, 0.f);
    fence_proxy_async_global();
    __syncthreads();
    return true;
  }
  if (warp == 0) tmem_alloc(&sm.tmem, TCOLS);   // (no relinquish: another sequence may allocate again)
  if (tid == 0) {
    #pragma unroll 1
    for (int s = 0; s < nslot; ++s) mbar_init(&full[s], 1);
    mbar_init(&mmad[0], 1);
    mbar_init(&mmad[1], 1);
    mbar_fence_init();
  }
  if (tid < HQ) sm.att_m[tid] = -INFINITY;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;
  int issued = 0;   // pages whose copies were issued (thread 0)
  auto issue = [&](int k) {
    const int s = k % nslot, j = plist[k], page = ppage[k];
    const bool ok = page >= 0 && (int64_t)page < a.num_pages;
    pv_ok[s] = ok;
    mbar_arrive_expect_tx(&full[s], (ok ? VPAGE : 0) + LROWS);
    if (ok) {
      const uint64_t pol = l2_evict_first_policy();     // each V row is read once
      tma_load_2d(vslots + (size_t)s * VPAGE, &a.tmap_v, 0, page * ROWS, &full[s], pol);
      tma_load_2d(vslots + (size_t)s * VPAGE + VHALF, &a.tmap_v, 64, page * ROWS, &full[s], pol);
    } else {
      set_error(a.status, TS_ERR_PAGE_OOB);
    }
    bulk_g2s(lslots + (size_t)s * (LROWS / 4), eb + (size_t)j * S::P * HQ, LROWS, &full[s]);
    ++issued;
  };
  if (tid == 0) {
    fence_proxy_async_global();
    #pragma unroll 1
    for (int k = 0; k < min(nslot, nlist); ++k) issue(k);
  }
  // a time-out: the copies issued and the MMAs committed land first, then TMEM is freed
  auto bail = [&](int kdone) -> bool {
    if (tid == 0) {
      set_error(a.status, TS_ERR_TIMEOUT);
      atomicExch(&a.gsync->abort, 1u);
      #pragma unroll 1
      for (int kk = kdone; kk < issued; ++kk) mbar_wait(&full[kk % nslot], (kk / nslot) & 1, a.wait_ns);
      if (kdone > 0) mbar_wait(&mmad[(kdone - 1) & 1], ((kdone - 1) >> 1) & 1, a.wait_ns);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
      tc_fence_after();
      tmem_dealloc(tmem, TCOLS);
    }
    return false;
  };
  const bool wt = tid < S::P * HQ;
  const int wr = tid / HQ, wh = tid % HQ;
  KahanF lsum;
  bool started = false;   // the accumulators hold a page (uniform)
  #pragma unroll 1
  for (int k = 0; k < nlist; ++k) {
    const int s = k % nslot, kb = k & 1, j = plist[k];
    // the weight buffer and the V slot of page k - 2 are free once its MMAs have completed: the
    // slot takes page k - 2 + nslot
    bool landed = true;
    if (tid == 0 && k >= 2) {
      landed = mbar_wait(&mmad[kb], ((k - 2) >> 1) & 1, a.wait_ns);
      if (landed && k - 2 + nslot < nlist) issue(k - 2 + nslot);
    }
    landed = mbar_wait(&full[s], (k / nslot) & 1, a.wait_ns) && landed;
    const float* Lp = lslots + (size_t)s * (LROWS / 4);
    const int nv = min(S::P, ntok - j * S::P);
    float xl = -INFINITY;
    bool att = false;
    if (wt && landed) {
      att = wr < nv && pv_ok[s] && attended(j * S::P + wr);
      if (att) xl = Lp[wr * HQ + wh];
    }
    const bool need = att && xl - sm.att_m[wh] > kRescaleGap;
    if (__syncthreads_or(!landed || need)) {
      if (__syncthreads_or(!landed)) return bail(k);
      float* Wm = reinterpret_cast<float*>(bbuf + (size_t)kb * BBUF);   // scratch: the page's masked logits
      if (wt) Wm[tid] = xl;
      __syncthreads();
      if (tid < HQ) {
        float pm = -INFINITY;
        #pragma unroll 1
        for (int r = 0; r < S::P; ++r) pm = fmaxf(pm, Wm[r * HQ + tid]);
        const float m0 = sm.att_m[tid];
        const float mn = fmaxf(m0, pm);
        sm.att_c[tid] = m0 == -INFINITY ? 0.f : exp2f(m0 - mn);
        sm.att_m[tid] = mn;
      }
      bool mma_ok = true;
      if (started && tid == 0) mma_ok = mbar_wait(&mmad[(k - 1) & 1], ((k - 1) >> 1) & 1, a.wait_ns);
      if (!__syncthreads_and(mma_ok)) return bail(k);
      if (wt) {
        lsum.s *= sm.att_c[wh];
        lsum.c *= sm.att_c[wh];
      }
      if (started) {
        // the accumulators of every query head, scaled by its correction (lanes = columns of d)
        tc_fence_after();
        if (warp < 4) {
          #pragma unroll 1
          for (int g = 0; g < HKV; ++g)
#pragma unroll
            for (int c0 = 0; c0 < 16; c0 += 8) {
              const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(g * 16 + c0);
              float r[8];
              tmem_ld_x8(ta, r);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int col = c0 + i, jj = col < G ? col : col - G;
                r[i] *= col < 2 * G ? sm.att_c[g * G + jj] : 1.f;
              }
              tmem_st_x8(ta, r);
            }
          tmem_wait_st();
        }
        tc_fence_before();
      }
      __syncthreads();
    }
    // ---- the weights into buffer kb as two bf16 terms, rows j (hi) and G + j (lo) of the KV head
    unsigned char* bk = bbuf + (size_t)kb * BBUF;
    if (wt) {
      const float w = att ? exp2f(xl - sm.att_m[wh]) : 0.f;
      lsum.add(w);
      const int g = wh / G, jj = wh % G;
      const __nv_bfloat16 hi = __float2bfloat16_rn(w);
      const __nv_bfloat16 lo = __float2bfloat16_rn(w - __bfloat162float(hi));
      *reinterpret_cast<__nv_bfloat16*>(bk + g * BTILE + b_off(jj, wr)) = hi;
      *reinterpret_cast<__nv_bfloat16*>(bk + g * BTILE + b_off(G + jj, wr)) = lo;
    }
    // the weight rows past 2 G and a partial page's V rows past the sequence are zero (a zero
    // weight times a NaN is a NaN)
    for (int i = tid; i < HKV * (16 - 2 * G) * 2; i += S::THREADS) {
      const int g = i / ((16 - 2 * G) * 2), rr = 2 * G + (i / 2) % (16 - 2 * G), kg = i & 1;
      *reinterpret_cast<uint4*>(bk + g * BTILE + b_off(rr, kg * 8)) = make_uint4(0u, 0u, 0u, 0u);
    }
    const bool vok = pv_ok[s] != 0;
    if (vok && nv < S::P) {
      unsigned char* vp = vslots + (size_t)s * VPAGE;
      const int nz = HKV * (S::P - nv);                  // rows (g, token >= nv), both halves, 8 chunks each
      for (int i = tid; i < nz * 16; i += S::THREADS) {
        const int row = i / 16, ch = i % 16, g = row / (S::P - nv), t = nv + row % (S::P - nv);
        *reinterpret_cast<uint4*>(vp + (ch >> 3) * VHALF + (g * S::P + t) * 128 + (ch & 7) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      if (vok) {
        const uint32_t va = smem_addr(vslots + (size_t)s * VPAGE), ba = smem_addr(bk);
        #pragma unroll 1
        for (int g = 0; g < HKV; ++g)
          umma_bf16(tmem + (uint32_t)(g * 16), sdesc_sw128_mn(va + g * S::P * 128, VHALF, 1024),
                    sdesc_kmajor_none(ba + g * BTILE, 128, 256), idesc, started);
      }
      umma_commit(&mmad[kb]);     // (with no MMA it arrives at once: the phases stay in step)
    }
    started = started || vok;
  }
  // ---- every MMA done: outputs from TMEM (warps 0..3: lane = column of d), sums, the CTA's partial
  bool done = true;
  if (tid == 0) done = mbar_wait(&mmad[(nlist - 1) & 1], ((nlist - 1) >> 1) & 1, a.wait_ns);
  if (!__syncthreads_and(done)) return bail(nlist);
  tc_fence_after();
  float* red = reinterpret_cast<float*>(vslots);                 // [HQ][D] (the slots are spent)
  float* lred = red + (size_t)HQ * D;                            // [16][HQ]
  if (warp < 4) {
    #pragma unroll 1
    for (int g = 0; g < HKV; ++g) {
      float r[16];
      const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(g * 16);
      tmem_ld_x8(ta, *reinterpret_cast<float(*)[8]>(r));
      tmem_ld_x8(ta + 8, *reinterpret_cast<float(*)[8]>(r + 8));
      tmem_wait_ld();
#pragma unroll
      for (int jj = 0; jj < G; ++jj)
        red[(size_t)(g * G + jj) * D + warp * 32 + lane] = started ? r[jj] + r[G + jj] : 0.f;
    }
  }
  if (wt) lred[tid] = lsum.s - lsum.c;
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TCOLS);
  }
  if (tid == 0) {
    #pragma unroll 1
    for (int s = 0; s < nslot; ++s) mbar_inval(&full[s]);
    mbar_inval(&mmad[0]);
    mbar_inval(&mmad[1]);
  }
  const int Dq = D / dq;
  #pragma unroll 1
  for (int it = tid; it < HQ * D4; it += S::THREADS) {
    const int h = it / D4, e4 = it % D4, qq = e4 / (Dq / 4);
    reinterpret_cast<float4*>(ao + ((((size_t)b * HQ + h) * dq + qq) * nCTA + c) * Dq)[e4 % (Dq / 4)] =
        reinterpret_cast<const float4*>(red + (size_t)h * D)[e4];
  }
  if (tid < HQ) {
    KahanF z;
    #pragma unroll 1
    for (int r = 0; r < S::P; ++r) z.add(lred[r * HQ + tid]);
    const float m2 = sm.att_m[tid], l = z.s - z.c;
    aml[((size_t)b * HQ + tid) * nCTAp + c] =
        (m2 > -INFINITY && l > 0.f) ? make_float2(m2 * kLn2, l) : make_float2(-INFINITY, 0.f);
  }
  fence_proxy_async_global();
  __syncthreads();
  return true;
}

template <typename KT, int D, int HKV, int G>
__device__ __forceinline__ void step_body(const StepKArgs& a) {
  using S = StepShape<KT, D, HKV, G>;
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ Smem sm;
  __shared__ __align__(8) uint64_t full[kMaxSlots];
  __shared__ __align__(8) uint64_t empty[kMaxSlots];  // tensor-core scan: ring slot read by its MMAs
  __shared__ __align__(8) uint64_t accf[2], acce[2];   // accumulator buffer written / read out
  __shared__ __align__(8) uint64_t drainb;            // every MMA issued has completed
  __shared__ __align__(8) uint64_t xbar;              // bulk copies of partials (vote, merge)
  __shared__ __align__(8) uint64_t vbar[kVoteBufs];  // chunks of my logits for the votes

  unsigned char* ring = dsm;                                               // a.nslot x STAGE_BYTES of K
  uint8_t* selflag = dsm + a.dyn_bytes - a.flag_cap;                       // selection flags of my tokens
  // tensor-core scan: 1024-aligned ring of pages, then the query-term images of two sequences
  unsigned char* tcr = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~(uintptr_t)1023);
  unsigned char* tcb = tcr + (size_t)a.nslot_tc * S::TC_TILE;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, nCTA = gridDim.x;
  const int B = a.B, H = a.H;
  // Whole-CTA fetch of up to two contiguous global blocks (written by other CTAs before a grid
  // barrier) into shared memory by bulk copy; false (and a recorded time-out) if they do not land.
  uint32_t xph = 0;
  auto bulk_fetch = [&](void* d0, const void* s0, uint32_t n0, void* d1, const void* s1, uint32_t n1) -> bool {
    if (tid == 0) {
      fence_proxy_async_global();
      mbar_arrive_expect_tx(&xbar, n0 + n1);
      bulk_g2s(d0, s0, n0, &xbar);
      if (n1) bulk_g2s(d1, s1, n1, &xbar);
    }
    const bool landed = mbar_wait(&xbar, xph, a.wait_ns);
    xph ^= 1u;
    const bool ok = __syncthreads_and(landed) != 0;
    if (!ok && tid == 0) set_error(a.status, TS_ERR_TIMEOUT);
    return ok;
  };

  TS_MARK(0);
  if (tid == 0) {
    #pragma unroll 1
    for (int s = 0; s < kMaxSlots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      sm.stage_done[s] = 0;
      sm.slot_last[s] = -1;
    }
    #pragma unroll 1
    for (int i = 0; i < 2; ++i) {
      mbar_init(&accf[i], 2);     // the MMAs' commit and the issuer's own arrive (metadata)
      mbar_init(&acce[i], 128);   // every epilogue thread
    }
    mbar_init(&drainb, 1);
    mbar_init(&xbar, 1);
    for (int i = 0; i < kVoteBufs; ++i) mbar_init(&vbar[i], 1);
    mbar_fence_init();
    sm.timed_out = 0;
    sm.gepoch = 0u;
  }

  // ------------------------------------------------ setup: lengths, cache test, partition
  // one round of independent loads per sequence: length, cache entry state
  // (a cache entry matters only when a hit is possible: a cache test, or hits given by the caller)
  const bool have_cache = a.ct != nullptr && a.filled != nullptr && ((a.phases & kPhCheck) || a.hit_in != nullptr);
  #pragma unroll 1
  for (int b = tid; b < B; b += blockDim.x) {
    int n = a.seq_lens[b];
    if (n < 0 || n > a.max_tokens) {
      if (c == 0) set_error(a.status, TS_ERR_SEQ_LEN);
      n = 0;
    }
    SeqState& st = sm.seq[b];
    st.n = n;
    budget_segments(n, a.n_sink, a.n_local, st.s_end, st.ls);
    if (a.mode == TS_SELECT_TOPK) {
      st.lo = st.s_end;
      st.hi = st.ls;
    } else {
      st.lo = 0;
      st.hi = n;
    }
    st.hit = (!(a.phases & kPhCheck) && a.hit_in) ? (a.hit_in[b] != 0) : 0;
    sm.my_seg_of[b] = -1;
    sm.tc_img_of[b] = -1;
    sm.ct_lo[b] = 0;
    sm.ct_hi[b] = 0;
    sm.filled[b] = have_cache ? a.filled[b] : 0;
    sm.qst[b] = -1;
    sm.ctst[b] = -1;
    sm.ctc[b] = have_cache ? max(0, min(a.ct_count[b], a.cap)) : 0;
  }
  __syncthreads();
  TS_MARK(5);
  // every filled entry in one pass without barriers: cos(q, C_Q) (Algorithm 1: hit iff
  // cos >= theta) and, for the reuse on a hit, how many cached indices lie below s_end and
  // below ls; per-warp partials in shared memory, summed in a fixed order below
  {
    float* cr = reinterpret_cast<float*>(dsm);                       // [B][3][NW]
    int* cn = reinterpret_cast<int*>(cr + (size_t)B * 3 * S::NW);     // [B][2][NW]
    const bool check = (a.phases & kPhCheck) != 0;
    const int HD = H * D;
    // few sequences: q, C_Q and the used part of C_T of every filled entry arrive in shared
    // memory in one bulk-copy transaction (one round trip instead of one per operand)
    const int cap16 = (a.cap + 8 + 3) & ~3;   // ints per staged C_T: the entries plus alignment slack, 16-byte rows
    unsigned char* stg = dsm + (((size_t)B * 5 * S::NW * 4 + 15) & ~(size_t)15);
    const size_t room_b = (size_t)(a.dyn_bytes - a.flag_cap) - (size_t)(stg - dsm);
    const bool stage_ct = (size_t)B * (2 * HD + cap16) * 4 <= room_b;     // C_T too (top-k sizes)
    const size_t per_b = (size_t)(2 * HD + (stage_ct ? cap16 : 0)) * 4;
    const bool staged = have_cache && B * per_b <= room_b && (reinterpret_cast<uintptr_t>(a.q) & 15) == 0 &&
                        (HD * 4) % 16 == 0;
    if (staged) {
      if (tid == 0) {
        uint32_t bytes = 0;
        #pragma unroll 1
        for (int b = 0; b < B; ++b) {
          if (!sm.filled[b]) continue;
          const uintptr_t c0 = reinterpret_cast<uintptr_t>(a.ct + (size_t)b * a.cap);
          const uintptr_t c1 = reinterpret_cast<uintptr_t>(a.ct + (size_t)b * a.cap + sm.ctc[b]);
          const uint32_t ctbytes = stage_ct ? (uint32_t)(((c1 + 15) & ~(uintptr_t)15) - (c0 & ~(uintptr_t)15)) : 0u;
          bytes += (check ? 2u * HD * 4u : 0u) + ctbytes;
        }
        fence_proxy_async_global();
        mbar_arrive_expect_tx(&xbar, bytes);
        #pragma unroll 1
        for (int b = 0; b < B; ++b) {
          if (!sm.filled[b]) continue;
          unsigned char* d = stg + b * per_b;
          if (check) {
            sm.qst[b] = (int)(d - dsm);
            bulk_g2s(d, a.q + (size_t)b * HD, (uint32_t)HD * 4u, &xbar);
            bulk_g2s(d + HD * 4, a.cq + (size_t)b * HD, (uint32_t)HD * 4u, &xbar);
          }
          if (stage_ct) {
            const uintptr_t c0 = reinterpret_cast<uintptr_t>(a.ct + (size_t)b * a.cap);
            const uintptr_t c1 = reinterpret_cast<uintptr_t>(a.ct + (size_t)b * a.cap + sm.ctc[b]);
            const uint32_t ctbytes = (uint32_t)(((c1 + 15) & ~(uintptr_t)15) - (c0 & ~(uintptr_t)15));
            if (ctbytes) bulk_g2s(d + 2 * HD * 4, reinterpret_cast<const void*>(c0 & ~(uintptr_t)15), ctbytes, &xbar);
            sm.ctst[b] = (int)(d + 2 * HD * 4 - dsm) + (int)(c0 & 15);
          }
        }
      }
      const bool landed = mbar_wait(&xbar, xph, a.wait_ns);
      xph ^= 1u;
      if (!__syncthreads_and(landed)) {
        if (tid == 0) {
          set_error(a.status, TS_ERR_TIMEOUT);
          atomicExch(&a.gsync->abort, 1u);   // the others leave at their first barrier
        }
        return;
      }
    }
    #pragma unroll 1
    for (int b = 0; b < B; ++b) {
      if (!sm.filled[b]) continue;
      const unsigned char* sb = stg + b * per_b;
      if (check) {
        const float* x = staged ? reinterpret_cast<const float*>(sb) : a.q + (size_t)b * HD;
        const float* y = staged ? reinterpret_cast<const float*>(sb + HD * 4) : a.cq + (size_t)b * HD;
        float xy = 0.f, xx = 0.f, yy = 0.f;
#pragma unroll 2
        for (int i = tid; i < HD; i += blockDim.x) {
          const float u = x[i], v = y[i];
          xy = fmaf(u, v, xy);
          xx = fmaf(u, u, xx);
          yy = fmaf(v, v, yy);
        }
        xy = warp_sum(xy);
        xx = warp_sum(xx);
        yy = warp_sum(yy);
        if (lane == 0) {
          cr[(b * 3 + 0) * S::NW + warp] = xy;
          cr[(b * 3 + 1) * S::NW + warp] = xx;
          cr[(b * 3 + 2) * S::NW + warp] = yy;
        }
      }
      const int32_t* ctb = sm.ctst[b] >= 0 ? reinterpret_cast<const int32_t*>(dsm + sm.ctst[b])
                                           : a.ct + (size_t)b * a.cap;
      const int se = sm.seq[b].s_end, ls = sm.seq[b].ls;
      int below_s = 0, below_l = 0;
      if (sm.ctc[b] > 4096) {
        // long lists (top-p selections) are searched below, one warp per sequence
      } else {
#pragma unroll 1
        for (int j = tid; j < sm.ctc[b]; j += blockDim.x) {
          const int v = ctb[j];
          below_s += v < se;
          below_l += v < ls;
        }
        below_s = warp_sum_i(below_s);
        below_l = warp_sum_i(below_l);
        if (lane == 0) {
          cn[(b * 2 + 0) * S::NW + warp] = below_s;
          cn[(b * 2 + 1) * S::NW + warp] = below_l;
        }
      }
    }
    // long cached lists: entries below s_end and ls by a 32-ary search, one warp per sequence
    #pragma unroll 1
    for (int b = warp; b < B; b += S::NW) {
      if (!sm.filled[b] || sm.ctc[b] <= 4096) continue;
      const int32_t* ctb = sm.ctst[b] >= 0 ? reinterpret_cast<const int32_t*>(dsm + sm.ctst[b])
                                           : a.ct + (size_t)b * a.cap;
      int r1, r2;
      warp_lower_bound2(ctb, sm.ctc[b], sm.seq[b].s_end, sm.seq[b].ls, r1, r2);
      if (lane == 0) {
        #pragma unroll 1
        for (int w = 0; w < S::NW; ++w) {
          cn[(b * 2 + 0) * S::NW + w] = w == 0 ? r1 : 0;
          cn[(b * 2 + 1) * S::NW + w] = w == 0 ? r2 : 0;
        }
      }
    }
    __syncthreads();
    #pragma unroll 1
    for (int b = tid; b < B; b += blockDim.x) {
      if (!sm.filled[b]) continue;
      if (check) {
        KahanF sxy, sxx, syy;                                         // fp32: FP64 is a slow pipe here
        #pragma unroll 1
        for (int w = 0; w < S::NW; ++w) {
          sxy.add(cr[(b * 3 + 0) * S::NW + w]);
          sxx.add(cr[(b * 3 + 1) * S::NW + w]);
          syy.add(cr[(b * 3 + 2) * S::NW + w]);
        }
        const float den = sqrtf(sxx.s - sxx.c) * sqrtf(syy.s - syy.c);
        const float cs = den > 0.f ? (sxy.s - sxy.c) / den : __int_as_float(0x7fc00000);
        sm.seq[b].hit = (cs >= a.theta) ? 1 : 0;
      }
      int lo = 0, hi = 0;
      #pragma unroll 1
      for (int w = 0; w < S::NW; ++w) {
        lo += cn[(b * 2 + 0) * S::NW + w];
        hi += cn[(b * 2 + 1) * S::NW + w];
      }
      sm.ct_lo[b] = lo;
      sm.ct_hi[b] = hi;
    }
    __syncthreads();
  }
  TS_MARK(6);
  if (tid == 0) {
    int pg = 0;
    #pragma unroll 1
    for (int b = 0; b < B; ++b) {
      SeqState& st = sm.seq[b];
      st.pg0 = pg;
      if (!st.hit && (a.phases & (kPhScore | kPhSelect))) pg += (st.n + S::P - 1) / S::P;
      st.pg1 = pg;
      st.all = 0;
      st.done = 0;
      st.cand = 0;
      st.tie_mode = 0;
      st.prefix = 0u;
      st.mask = 0u;
      st.k_rem = a.k;
      st.n_gt = 0;
      st.mass_rem = a.target_fx;
      st.ties = 0;
    }
    const int ptot = pg;
    sm.ptot = ptot;
    const int ppc = (ptot + nCTA - 1) / nCTA;
    sm.ppc = ppc;
    sm.p0 = min(ptot, c * ppc);
    sm.p1 = min(ptot, sm.p0 + ppc);
    sm.tok_stride = ppc * S::P;
    #pragma unroll 1
    for (int b = 0; b < B; ++b) {
      SeqState& st = sm.seq[b];
      if (st.pg1 > st.pg0) {
        st.first_cta = st.pg0 / ppc;
        st.last_cta = (st.pg1 - 1) / ppc;
      } else {
        st.first_cta = 0;
        st.last_cta = -1;
      }
    }
    int ns = 0;
    #pragma unroll 1
    for (int b = 0; b < B; ++b) {
      const SeqState& st = sm.seq[b];
      const int lo = max(st.pg0, sm.p0), hi = min(st.pg1, sm.p1);
      if (hi <= lo) continue;
      sm.seg_b[ns] = b;
      sm.seg_lp0[ns] = lo - st.pg0;
      sm.seg_t0[ns] = (lo - sm.p0) * S::P;
      sm.seg_ntok[ns] = min((hi - lo) * S::P, st.n - (lo - st.pg0) * S::P);
      sm.seg_pend[ns] = hi;
      sm.my_seg_of[b] = ns;
      ++ns;
    }
    sm.nseg = ns;
    // the tensor-core scan holds the query terms of two sequences: it runs when no CTA's page
    // range meets three (a middle sequence inside one CTA whose neighbours both reach it)
    int use_tc = 0;
    if constexpr (S::TC) {
      use_tc = a.tc && (a.phases & kPhScore) && H <= kMaxWaveHeads;
      int prev = -1, prev2 = -1;
      #pragma unroll 1
      for (int b = 0; b < B && use_tc; ++b) {
        const SeqState& st = sm.seq[b];
        if (st.pg1 <= st.pg0) continue;
        if (prev2 >= 0) {
          const SeqState& m = sm.seq[prev];
          if (m.first_cta == m.last_cta && sm.seq[prev2].last_cta == m.first_cta && st.first_cta == m.last_cta)
            use_tc = 0;
        }
        prev2 = prev;
        prev = b;
      }
    }
    sm.use_tc = use_tc;
    // with at most two sequences to scan every CTA holds both query images, and the pages are
    // claimed in chunks from a counter so that CTAs with more bandwidth take more of them;
    // otherwise each CTA scans its own range with the images of its segments
    int nsc = 0;
    #pragma unroll 1
    for (int b = 0; b < B; ++b) nsc += sm.seq[b].pg1 > sm.seq[b].pg0;
    sm.scan_dyn = use_tc && a.scan_dyn && nsc <= 2;
    sm.tc_nimg = 0;
    if (use_tc) {
      #pragma unroll 1
      for (int b = 0; b < B; ++b) {
        const bool mine = sm.scan_dyn ? sm.seq[b].pg1 > sm.seq[b].pg0 : sm.my_seg_of[b] >= 0;
        if (!mine) continue;
        sm.tc_img_of[b] = sm.tc_nimg;
        sm.tc_seq[sm.tc_nimg++] = b;
      }
    }
    // scan waves: the most KV heads per wave (a power-of-two divisor of H_kv) whose
    // logits stay within the L2 budget (the tensor-core scan takes every head at once)
    int hpw = HKV;
    while (!use_tc && hpw > 1 && ((int64_t)ptot * S::P * hpw * G * 4 > a.l2_budget || hpw * G > kMaxWaveHeads))
      hpw >>= 1;
    sm.hpw = hpw;
    sm.nwaves = HKV / hpw;
    // my logits [tok_stride][hpw*G] in scratch
    sm.region = ppc * hpw * G * S::P;
    sm.spill_ok = (int64_t)nCTA * sm.region <= a.spill_floats && sm.tok_stride <= a.flag_cap &&
                  hpw * G <= kMaxWaveHeads;
    sm.flag = 0;
    // attention: how many fixed tokens of every sequence are mine. A scanned sequence's fixed
    // tokens go round-robin over the CTAs that hold its pages (they attend its selected tokens
    // anyway), so a CTA attends only the sequences of its own range; hits, and top-p (whose
    // selected tokens are shared out over every CTA), use every CTA
    // (a batch of top-k sequences instead gives every sequence its own group of CTAs, which
    // shares out its fixed and selected tokens evenly: attend_grouped below)
    const bool sel_att = (a.phases & kPhSelect) && (a.phases & kPhAttend);
    const bool bal_mode = a.mode == TS_SELECT_TOPP && sel_att;
    const bool grp_mode = a.mode == TS_SELECT_TOPK && sel_att && B > 1 && ptot > 0;
    int tot = 0;
    #pragma unroll 1
    for (int b = 0; b < B; ++b) {
      SeqState& st = sm.seq[b];
      int nfix = st.s_end + (st.n - st.ls);
      if (st.hit && a.ct) nfix += sm.ct_hi[b] - sm.ct_lo[b];
      const bool ranged = !bal_mode && st.pg1 > st.pg0;
      st.fx_base = ranged ? st.first_cta : 0;
      st.fx_stride = ranged ? st.last_cta - st.first_cta + 1 : nCTA;
      if (grp_mode) {
        st.fx_base = (int)((int64_t)b * nCTA / B);
        st.fx_stride = (int)((int64_t)(b + 1) * nCTA / B) - st.fx_base;
      }
      const int rel = c - st.fx_base;
      sm.pf_off[b] = tot;
      tot += (rel >= 0 && rel < st.fx_stride && rel < nfix) ? (nfix - rel + st.fx_stride - 1) / st.fx_stride : 0;
    }
    sm.pf_off[B] = tot;
    sm.pf_ok = (a.phases & kPhAttend) && (a.phases & kPhSelect) && tot <= kPreFix;
  }
  __syncthreads();
  if (!sm.spill_ok) {
    if (c == 0 && tid == 0) set_error(a.status, TS_ERR_SHAPE);
    return;  // the same decision in every CTA, before any grid barrier
  }
  // my selected tokens, ascending: the list of segment sg from row seg_t0[sg] (my logits stay in
  // my scratch region for the attention)
  int* const sel_list = a.sel_rows + (size_t)c * a.flag_cap;
  TS_MARK(7);
  // the tensor-core scan runs this launch: warps 8.. finish the set-up while the pages stream
  const bool tc_scan = S::TC && sm.use_tc && (a.phases & kPhScore) && sm.ptot > 0;
  // set-up needed only after the scan
  auto late_setup = [&](int ltid, int lth) {
    // page ids of my range, read once (ring refills and attention gathers need no global load),
    // and in the same pass my share of every sequence's fixed attention tokens -- sinks and
    // window, plus the cached indices on a hit -- with their page ids
    #pragma unroll 1
    for (int i = ltid; i < min(sm.p1 - sm.p0, kMaxPagesCta); i += lth) {
      const int gp = sm.p0 + i;
      int sg = 0;
      while (sg + 1 < sm.nseg && gp >= sm.seg_pend[sg]) ++sg;
      const int b = sm.seg_b[sg];
      sm.my_pages[i] = a.page_table[(size_t)b * a.pt_stride + (gp - sm.seq[b].pg0)];
    }
    if (sm.pf_ok) {
      #pragma unroll 1
      for (int i = ltid; i < sm.pf_off[B]; i += lth) {
        int b = 0;
        while (b + 1 < B && sm.pf_off[b + 1] <= i) ++b;
        const SeqState& st = sm.seq[b];
        const int f = (c - st.fx_base) + (i - sm.pf_off[b]) * st.fx_stride;
        const int nmid = (st.hit && a.ct) ? sm.ct_hi[b] - sm.ct_lo[b] : 0;
        int t;
        if (f < st.s_end) {
          t = f;
        } else if (f < st.s_end + nmid) {
          const int j = sm.ct_lo[b] + (f - st.s_end);
          // (the staged copy lies in the ring, which the producer may be filling)
          t = (!tc_scan && sm.ctst[b] >= 0) ? reinterpret_cast<const int32_t*>(dsm + sm.ctst[b])[j]
                                            : a.ct[(size_t)b * a.cap + j];
        } else {
          t = st.ls + (f - st.s_end - nmid);
        }
        sm.pf_t[i] = t;
        sm.pf_p[i] = (t >= 0 && t < a.max_tokens) ? a.page_table[(size_t)b * a.pt_stride + t / S::P] : -1;
      }
    }
    if (a.phases & kPhSelect) {
      // zero the selection histograms (first touched after a barrier)
      const size_t nh = (size_t)B * kHistPerSeq;
      #pragma unroll 1
      for (size_t i = (size_t)c * lth + ltid; i < nh; i += (size_t)nCTA * lth) {
        a.hist[i] = 0u;
        if (a.mode == TS_SELECT_TOPP) a.mass[i] = 0ull;
      }
      if (c == 0 && ltid < B) a.cand_n[ltid] = 0u;
    }
  };
  if (c == 0 && tid < B && (a.phases & kPhCheck) && a.hit_out) a.hit_out[tid] = (uint8_t)sm.seq[tid].hit;
  // (with 16 warps the tensor-core scan leaves warps 8.. free to do it while the pages stream; a
  // block of 8 warps has none, so it is done here first)
  const bool late_in_scan = tc_scan && S::NW > 8;
  if (!late_in_scan) late_setup(tid, (int)blockDim.x);
  if constexpr (S::TC) {
    if (sm.use_tc) {
      // B operand of each of my (at most two) sequences: row n = 3 h + term holds that term of
      // query head h, K-major in the 128-byte swizzle layout; rows past 3 H are zero
      constexpr int CH = D / 8;                        // 16-byte chunks of a row
      const int total = sm.tc_nimg * S::TC_N * CH;
      #pragma unroll 1
      for (int i0 = tid; i0 < total; i0 += 2 * blockDim.x) {   // two chunks' loads in flight
        float4 qv[2][2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int i = i0 + k * blockDim.x;
          const int sg = i / (S::TC_N * CH), rem = i % (S::TC_N * CH);
          const int n = rem / CH, ch = rem % CH, h = n / 3;
          qv[k][0] = qv[k][1] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (i < total && h < H) {
            const int b = sm.tc_seq[sg], off = sm.qst[b];
            // the query staged by the cache test, when it lies below the image region
            const float* qb = (off >= 0 && off + H * D * 4 <= (int)(tcb - dsm))
                                  ? reinterpret_cast<const float*>(dsm + off)
                                  : a.q + (size_t)b * H * D;
            const float4* qh = reinterpret_cast<const float4*>(qb + (size_t)h * D + ch * 8);
            qv[k][0] = qh[0];
            qv[k][1] = qh[1];
          }
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int i = i0 + k * blockDim.x;
          if (i >= total) continue;
          const int sg = i / (S::TC_N * CH), rem = i % (S::TC_N * CH);
          const int n = rem / CH, ch = rem % CH, term = n % 3;
          const float e8[8] = {qv[k][0].x, qv[k][0].y, qv[k][0].z, qv[k][0].w,
                               qv[k][1].x, qv[k][1].y, qv[k][1].z, qv[k][1].w};
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = (uint32_t)__bfloat16_as_ushort(bf16_split_term(e8[2 * e], term)) |
                   ((uint32_t)__bfloat16_as_ushort(bf16_split_term(e8[2 * e + 1], term)) << 16);
          *reinterpret_cast<uint4*>(tcb + (size_t)sg * S::TC_BIMG + (ch / 8) * (S::TC_N * 128) +
                                    sw128_offset(n, (ch % 8) * 8)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async();
    }
  }
  __syncthreads();
  TS_MARK(1);

  // which sequences need no selection (hits, empty domains, k <= 0, everything fits, top-p 1):
  // decided before the scan so that the vote pass can build the first histogram level
  if (a.phases & kPhSelect) {
    if (tid == 0) {
      #pragma unroll 1
      for (int b = 0; b < B; ++b) {
        SeqState& st = sm.seq[b];
        const int len = st.hi - st.lo;
        if (st.hit || len <= 0) {
          st.done = 1;
          st.all = !st.hit && len > 0;
        } else if (a.mode == TS_SELECT_TOPK) {
          if (a.k <= 0) {
            st.done = 1;
            st.prefix = 0xffffffffu;     // above every finite vote: nothing selected
            st.mask = 0xffffffffu;
          } else if (len <= a.k) {
            st.done = 1;
            st.all = 1;
          }
        } else if (a.take_all_topp) {
          st.done = 1;
          st.all = 1;
        }
      }
    }
    __syncthreads();
  }
  // ========================================================================= SCORE
  if ((a.phases & kPhScore) && sm.ptot > 0) {   // nothing to scan when every sequence hits
    // my logits [row = token of my range][HW] pass through shared memory past the vote scratch
    // in chunks of whole rows by bulk copy: at once when the range fits, else through
    // kVoteBufs buffers with all but one in flight
    const size_t vsb = ((size_t)kMaxB * kMaxWaveHeads * 8 + (size_t)nCTA * S::PV * H * 8 + S::NW * 32 * 8 + 15) &
                       ~(size_t)15;
    float* vbuf = reinterpret_cast<float*>(ring + vsb);
    const int vrows = (sm.p1 - sm.p0) * S::P;
    uint32_t vph = 0u;                                             // phase bit of each chunk buffer
    auto chunk_rows = [&](int HW) -> int {
      const int fit = (int)(((size_t)(a.dyn_bytes - a.flag_cap) - vsb) / ((size_t)HW * 4));
      return vrows <= fit ? vrows : max(16, (fit / kVoteBufs) & ~15);
    };
    auto issue_chunk = [&](const float* eb, int k, int HW, int crow) {   // thread 0
      const uint32_t bytes = (uint32_t)min(crow, vrows - k * crow) * (uint32_t)HW * 4u;
      const unsigned char* src = reinterpret_cast<const unsigned char*>(eb + (size_t)k * crow * HW);
      unsigned char* dst = reinterpret_cast<unsigned char*>(vbuf + (size_t)(k % kVoteBufs) * crow * HW);
      fence_proxy_async_global();
      mbar_arrive_expect_tx(&vbar[k % kVoteBufs], bytes);
      #pragma unroll 1
      for (uint32_t o = 0; o < bytes; o += 32768u)
        bulk_g2s(dst + o, src + o, min(32768u, bytes - o), &vbar[k % kVoteBufs]);
    };
    // each head's normaliser over the CTAs of the sequence, then the votes of my tokens for
    // heads [g0 G, g0 G + HW); eb holds my logits [row][HW], of which the first `pre` chunks
    // are already on their way
    auto vote_pass = [&](const float* eb, int g0, int HW, int wv, int pre) -> bool {
      float2* wz = reinterpret_cast<float2*>(ring);                // [segment][kMaxWaveHeads]: (max, 1 / sum)
      float2* pcs = wz + kMaxB * kMaxWaveHeads;                    // one segment's partials [cta][H]
      #pragma unroll 1
      for (int sg = 0; sg < sm.nseg; ++sg) {
        const SeqState& st = sm.seq[sm.seg_b[sg]];
        // a shared scan leaves partials of every sequence in every CTA
        const int fc = sm.scan_dyn ? 0 : st.first_cta, ncta = sm.scan_dyn ? nCTA : st.last_cta - st.first_cta + 1;
        const int nrow = ncta * S::PV;                                    // partial rows: PV per CTA
        float* rmx = reinterpret_cast<float*>(pcs + (size_t)nrow * H);   // [NW][32] per-slice maxima
        float* rz = rmx + S::NW * 32;                                    // [NW][32] per-slice sums
        if (!bulk_fetch(pcs, a.partials + ((size_t)sm.seg_b[sg] * nCTA + fc) * S::PV * H,
                        (uint32_t)(nrow * H * sizeof(float2)), nullptr, nullptr, 0u)) {
          if (tid == 0) atomicExch(&a.gsync->abort, 1u);
          return false;
        }
        TS_MARK(13);
        // lane = head of the wave, warp = a slice of the CTAs: conflict-free rows of H pairs
        const int per = (nrow + S::NW - 1) / S::NW;
        const int c0 = min(nrow, warp * per), c1 = min(nrow, c0 + per);
        const bool lh = lane < HW;
        float m = -INFINITY;
        if (lh)
          #pragma unroll 1
          for (int cc = c0; cc < c1; ++cc) m = fmaxf(m, pcs[cc * H + g0 * G + lane].x);
        rmx[warp * 32 + lane] = m;
        __syncthreads();
        float M = -INFINITY;
        #pragma unroll 1
        for (int w = 0; w < S::NW; ++w) M = fmaxf(M, rmx[w * 32 + lane]);
        KahanF kz;
        if (lh && M > -INFINITY)
          #pragma unroll 1
          for (int cc = c0; cc < c1; ++cc) {
            const float2 mz = pcs[cc * H + g0 * G + lane];
            if (mz.y > 0.f) kz.add(mz.y * exp2f(mz.x - M));
          }
        rz[warp * 32 + lane] = kz.s - kz.c;
        __syncthreads();
        if (warp == 0 && lh) {
          KahanF z;
          #pragma unroll 1
          for (int w = 0; w < S::NW; ++w) z.add(rz[w * 32 + lane]);
          const float Z = z.s - z.c;
          wz[sg * kMaxWaveHeads + lane] = (M > -INFINITY && Z > 0.f) ? make_float2(M, 1.f / Z)
                                                                     : make_float2(INFINITY, 0.f);
        }
        __syncthreads();
        TS_MARK(14);
      }
      // v_i (+)= sum over the wave's heads of 2^(l - M) / Z (base-2 logits: exp(l - M) in natural
      // units), chunk by chunk
      const int crow = chunk_rows(HW), nch = (vrows + crow - 1) / crow;
      if (tid == 0)
        #pragma unroll 1
        for (int k = pre; k < min(nch, kVoteBufs); ++k) issue_chunk(eb, k, HW, crow);
      const int q4 = HW >> 2;
      int lpt = 1;                                  // lanes per row, one float4 (4 heads) each
      while (lpt < q4) lpt <<= 1;
      const bool coop = (HW & 3) == 0 && lpt <= 32;
      const int tpi = 32 / lpt, rl = lane / lpt, qd = lane % lpt;
      #pragma unroll 1
      for (int k = 0; k < nch; ++k) {
        const int kb = k % kVoteBufs;
        const bool landed = mbar_wait(&vbar[kb], (vph >> kb) & 1u, a.wait_ns);
        vph ^= 1u << kb;
        TS_MARK(32);
        if (!__syncthreads_and(landed)) {
          if (tid == 0) {
            set_error(a.status, TS_ERR_TIMEOUT);
            atomicExch(&a.gsync->abort, 1u);
            #pragma unroll 1
            for (int j = k + 1; j < min(nch, k + kVoteBufs); ++j)   // copies in flight land first
              mbar_wait(&vbar[j % kVoteBufs], (vph >> (j % kVoteBufs)) & 1u, a.wait_ns);
          }
          return false;
        }
        const int r0 = k * crow, r1 = min(vrows, r0 + crow);
        const float* cb = vbuf + (size_t)kb * crow * HW;   // row r at cb + (r - r0) HW
        #pragma unroll 1
        for (int sg = 0; sg < sm.nseg; ++sg) {
          const int b = sm.seg_b[sg], t0 = sm.seg_t0[sg];
          const int lo = max(t0, r0), hi = min(t0 + sm.seg_ntok[sg], r1);   // rows of the segment here
          if (hi <= lo) continue;
          float* vb = a.vote + (size_t)b * a.vote_stride + (size_t)sm.seg_lp0[sg] * S::P;   // row t0 + i -> i
          const float2* w = wz + sg * kMaxWaveHeads;
          if (coop) {
            // warp-cooperative: a load instruction covers 32 / lpt whole rows; each lane forms its 4
            // terms, then the lpt lanes of a row add theirs (xor tree)
            float2 wl[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) wl[i] = qd < q4 ? w[4 * qd + i] : make_float2(INFINITY, 0.f);
            #pragma unroll 1
            for (int rw = lo + warp * 2 * tpi; rw < hi; rw += S::NW * 2 * tpi) {
              float part[2];
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int r = rw + u * tpi + rl;
                float4 xv = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                if (r < hi && qd < q4) xv = reinterpret_cast<const float4*>(cb + (size_t)(r - r0) * HW)[qd];
                part[u] = (exp2f(xv.x - wl[0].x) * wl[0].y + exp2f(xv.y - wl[1].x) * wl[1].y) +
                          (exp2f(xv.z - wl[2].x) * wl[2].y + exp2f(xv.w - wl[3].x) * wl[3].y);
              }
              #pragma unroll 1
              for (int d = lpt / 2; d >= 1; d >>= 1) {
                part[0] += __shfl_xor_sync(kFull, part[0], d);
                part[1] += __shfl_xor_sync(kFull, part[1], d);
              }
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int r = rw + u * tpi + rl;
                if (qd == 0 && r < hi) vb[r - t0] = (wv == 0) ? part[u] : vb[r - t0] + part[u];
              }
            }
          } else {
            #pragma unroll 1
            for (int r = lo + tid; r < hi; r += blockDim.x) {
              const float* row = cb + (size_t)(r - r0) * HW;
              KahanF acc;
              #pragma unroll 1
              for (int hl = 0; hl < HW; ++hl) acc.add(exp2f(row[hl] - w[hl].x) * w[hl].y);
              const float v = acc.s - acc.c;
              vb[r - t0] = (wv == 0) ? v : vb[r - t0] + v;
            }
          }
        }
        __syncthreads();                            // buffer kb is free again
        if (tid == 0 && k + kVoteBufs < nch) issue_chunk(eb, k + kVoteBufs, HW, crow);
      }
      __syncthreads();
      return true;
    };
    bool scanned = false;
    if constexpr (S::TC) {
      if (sm.use_tc) {
        scanned = true;
        // ---- pages of my range (or claimed ones) through a ring of TMA tiles fed by warp 0; one
        // elected thread of warp 1 multiplies each page (128 rows = H_kv heads x 16 tokens) by the
        // query terms of its sequence into a TMEM accumulator (two buffers); warps 4..7 read the
        // accumulators out: logits to the scratch, running (max, sum 2^x) per row and head in
        // registers, reduced into the CTA's partials at the end; warps 8.. finish the set-up
        const int nsl = a.nslot_tc;
        float* eb = a.spill + (size_t)c * sm.region;             // [tok_stride][H]
        if (warp == 2) tmem_alloc(&sm.tmem, 2 * S::TC_COLS);   // (the permit is kept: the range
                                                                // attention allocates again later)
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        const uint32_t tmem = sm.tmem;
        if (warp == 0) {
          if (lane == 0) {                                       // producer
            const uint64_t pol = l2_evict_first_policy();
            int u = 0;                                           // ring uses so far
            // pages gp (and gp + 1 when a tile takes two: page2 != kNoPage) of sequence b, physical
            // ids page / page2, into the next ring slot, page i at row i * TC_ROWS of the tile;
            // false after a time-out
            auto put = [&](int gp, int b, int page, int page2) -> bool {
              const int s = u % nsl;
              if (u >= nsl && !mbar_wait(&empty[s], ((u / nsl) - 1) & 1, a.wait_ns)) return false;
              uint32_t bytes = 0;
              bool valid[S::TC_PAGES];
#pragma unroll
              for (int pi = 0; pi < S::TC_PAGES; ++pi) {
                const int pg = pi == 0 ? page : page2, lp = gp + pi - sm.seq[b].pg0;
                const bool present = pi == 0 || page2 != kNoPage;
                valid[pi] = present && pg >= 0 && (int64_t)pg < a.num_pages;
                if (present && !valid[pi]) set_error(a.status, TS_ERR_PAGE_OOB);
                sm.stage_tok[s][pi] = (gp + pi) * S::P;
                sm.stage_b[s][pi] = b;
                sm.stage_nv[s][pi] = !present ? kAbsentRows : (valid[pi] ? min(S::P, sm.seq[b].n - lp * S::P) : 0);
                bytes += valid[pi] ? (uint32_t)S::TC_PAGE_BYTES : 0u;
              }
              sm.slot_last[s] = u;
              if (bytes) {
                mbar_arrive_expect_tx(&full[s], bytes);
#pragma unroll
                for (int pi = 0; pi < S::TC_PAGES; ++pi)
                  if (valid[pi])
#pragma unroll
                    for (int h = 0; h < S::TC_HALVES; ++h)
                      tma_load_2d(tcr + (size_t)s * S::TC_TILE + h * (S::TC_TILE / S::TC_HALVES) + pi * (S::TC_ROWS * 128),
                                  &a.tmap_k, h * 64, (pi == 0 ? page : page2) * S::TC_ROWS, &full[s], pol);
              } else {
                mbar_arrive(&full[s]);
              }
              ++u;
              return true;
            };
            bool ok = true;
            if (sm.scan_dyn) {
              // chunks of kScanClaim pages, claimed two ahead; the page ids of the next chunk load
              // while the ring takes the current one
              const int b0 = sm.tc_seq[0], b1 = sm.tc_nimg > 1 ? sm.tc_seq[1] : b0;
              const int split = sm.tc_nimg > 1 ? sm.seq[b1].pg0 : sm.ptot;
              auto load_ids = [&](int g0, int (&pid)[kScanClaim]) {
#pragma unroll
                for (int j = 0; j < kScanClaim; ++j) {
                  const int gp = g0 + j, b = gp >= split ? b1 : b0;
                  pid[j] = gp < sm.ptot ? a.page_table[(size_t)b * a.pt_stride + (gp - sm.seq[b].pg0)] : -1;
                }
              };
              int c1 = (int)atomicAdd(&a.gsync->claim, 1u) * kScanClaim, p1[kScanClaim];
              load_ids(c1, p1);
              int c2 = (int)atomicAdd(&a.gsync->claim, 1u) * kScanClaim;
              #pragma unroll 1
              while (ok && c1 < sm.ptot) {
                const int cur = c1;
                int pid[kScanClaim];
#pragma unroll
                for (int j = 0; j < kScanClaim; ++j) pid[j] = p1[j];
                c1 = c2;
                load_ids(c1, p1);
                c2 = (int)atomicAdd(&a.gsync->claim, 1u) * kScanClaim;
                #pragma unroll 1   // one copy of put; pid (loaded a chunk ago) picked by selects
                for (int j = 0; j < kScanClaim; ++j) {
                  int pj = pid[0];
#pragma unroll
                  for (int k = 1; k < kScanClaim; ++k)
                    if (j == k) pj = pid[k];
                  if (ok && cur + j < sm.ptot) ok = put(cur + j, cur + j >= split ? b1 : b0, pj, kNoPage);
                }
              }
            } else if constexpr (S::TC_PAGES == 2) {
              // my range in tiles of two pages of the same sequence (one where a sequence ends); the
              // next tile's page ids load while the current one is put
              int sg = 0;
              auto ids = [&](int g0, int& b, int& i0, int& i1) {
                while (sg + 1 < sm.nseg && g0 >= sm.seg_pend[sg]) ++sg;
                b = sm.seg_b[sg];
                i0 = a.page_table[(size_t)b * a.pt_stride + (g0 - sm.seq[b].pg0)];
                i1 = (g0 + 1 < sm.p1 && g0 + 1 < sm.seg_pend[sg])
                         ? a.page_table[(size_t)b * a.pt_stride + (g0 + 1 - sm.seq[b].pg0)]
                         : kNoPage;
              };
              int gp = sm.p0, nb = 0, n0 = 0, n1 = kNoPage;
              if (gp < sm.p1) ids(gp, nb, n0, n1);
              #pragma unroll 1
              while (ok && gp < sm.p1) {
                const int cg = gp, cb = nb, c0 = n0, c1 = n1;
                gp += c1 != kNoPage ? 2 : 1;
                if (gp < sm.p1) ids(gp, nb, n0, n1);
                ok = put(cg, cb, c0, c1);
              }
            } else {
              // my range, eight pages at a time; the next eight page ids load while the ring takes
              // the current ones (warps 8.. fill my_pages meanwhile)
              int sg = 0;
              auto load_ids = [&](int g0, int (&pid)[8], int (&pb)[8]) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const int gp = g0 + j;
                  while (sg + 1 < sm.nseg && gp >= sm.seg_pend[sg]) ++sg;
                  pb[j] = sm.seg_b[sg];
                  pid[j] = gp < sm.p1 ? a.page_table[(size_t)pb[j] * a.pt_stride + (gp - sm.seq[pb[j]].pg0)] : -1;
                }
              };
              int np_[8], nb_[8];
              load_ids(sm.p0, np_, nb_);
              #pragma unroll 1
              for (int gp0 = sm.p0; ok && gp0 < sm.p1; gp0 += 8) {
                int pid[8], pb[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  pid[j] = np_[j];
                  pb[j] = nb_[j];
                }
                if (gp0 + 8 < sm.p1) load_ids(gp0 + 8, np_, nb_);
                #pragma unroll 1   // one copy of put; pid (loaded eight pages ago) picked by selects
                for (int j = 0; j < 8; ++j) {
                  int pj = pid[0], bj = pb[0];
#pragma unroll
                  for (int k = 1; k < 8; ++k)
                    if (j == k) {
                      pj = pid[k];
                      bj = pb[k];
                    }
                  if (ok && gp0 + j < sm.p1) ok = put(gp0 + j, bj, pj, kNoPage);
                }
              }
            }
            if (ok) {                                            // end of the stream: a slot with no page
              const int s = u % nsl;
              if (u >= nsl && !mbar_wait(&empty[s], ((u / nsl) - 1) & 1, a.wait_ns)) {
                ok = false;
              } else {
                sm.stage_nv[s][0] = -1;
                mbar_arrive(&full[s]);
              }
            }
            if (!ok) {
              set_error(a.status, TS_ERR_TIMEOUT);
              sm.timed_out = 1;
            }
          }
        } else if (warp >= 8) {
          late_setup(tid - 256, (int)blockDim.x - 256);
        } else if (warp == 1) {
          if (lane == 0) {                                       // MMA issuer
            constexpr uint32_t idesc = idesc_bf16_f32(128, S::TC_N);
            #pragma unroll 1
            for (int u = 0;; ++u) {
              const int s = u % nsl, buf = u & 1;
              if (!mbar_wait(&full[s], (u / nsl) & 1, a.wait_ns) || (u >= 2 && !mbar_wait(&acce[buf], ((u >> 1) - 1) & 1, a.wait_ns))) {
                set_error(a.status, TS_ERR_TIMEOUT);
                sm.timed_out = 1;
                break;
              }
              tc_fence_after();
              const int nv = sm.stage_nv[s][0];
              const int nv2 = S::TC_PAGES == 2 ? sm.stage_nv[s][1] : 0;
              sm.acc_nv[buf][0] = nv;
              sm.acc_nv[buf][1] = nv2;
              if (nv < 0) {                // end of the stream, forwarded to the epilogue
                umma_commit(&accf[buf]);
                mbar_arrive(&accf[buf]);
                break;
              }
              const int sgi = sm.tc_img_of[sm.stage_b[s][0]];
              sm.acc_tl[buf][0] = sm.stage_tok[s][0];
              sm.acc_tl[buf][1] = sm.stage_tok[s][1];
              sm.acc_sg[buf] = sgi;
              if (nv > 0 || nv2 > 0) {
                const uint32_t a0 = smem_addr(tcr + (size_t)s * S::TC_TILE);
                const uint32_t b0 = smem_addr(tcb + (size_t)sgi * S::TC_BIMG);
#pragma unroll
                for (int h = 0; h < S::TC_HALVES; ++h)
#pragma unroll
                  for (int ks = 0; ks < 4; ++ks)
                    umma_bf16(tmem + buf * S::TC_COLS, sdesc_sw128(a0 + h * (S::TC_TILE / S::TC_HALVES) + ks * 32),
                              sdesc_sw128(b0 + h * (S::TC_N * 128) + ks * 32), idesc, (h | ks) != 0);
              }
              umma_commit(&empty[s]);      // the slot is free once its MMAs have read it
              umma_commit(&accf[buf]);     // the accumulator is complete
              mbar_arrive(&accf[buf]);     // and its metadata above is published
            }
            umma_commit(&drainb);
          }
        } else if (warp >= 4 && warp < 8) {                      // epilogue: thread = row (page, head g, slot t)
          const int q4 = warp & 3, row = q4 * 32 + lane;
          const int half = S::TC_PAGES == 2 ? (q4 >> 1) : 0;    // the page of the tile
          const int prow = row - half * S::TC_ROWS, g = prow >> 4, t = prow & 15;
          const bool odd = (g & 1) != 0;                         // second KV head of the warp's columns
          const int cb = q4 % (HKV / 2);                         // the warp's pair of KV heads
          const uint32_t tq = tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(6 * G * cb);
          float run_m[G];
          KahanF run_z[G];
          int cur = -1;
          // the partials of (image, head): the 16 rows of KV head g are 16 lanes of this warp; images
          // this CTA never meets stay (-inf, 0)
          // (each tile half has its own partial row: the vote pass merges the PV rows of every CTA)
          float2* pt = a.partials + ((size_t)c * S::PV + half) * H + g * G;   // + sequence * nCTA * PV * H + j
          if (t == 0)
            #pragma unroll 1
            for (int im = 0; im < sm.tc_nimg; ++im)
#pragma unroll
              for (int j = 0; j < G; ++j)
                pt[(size_t)sm.tc_seq[im] * nCTA * S::PV * H + j] = make_float2(-INFINITY, 0.f);
          auto flush = [&]() {                                   // whole warp (cur is uniform)
            if (cur < 0) return;
#pragma unroll
            for (int j = 0; j < G; ++j) {
              float m = run_m[j];
#pragma unroll
              for (int d = 8; d >= 1; d >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, d));
              const float rz = run_z[j].s - run_z[j].c;
              float z = (m > -INFINITY && rz > 0.f) ? rz * exp2f(run_m[j] - m) : 0.f, zl = 0.f;
#pragma unroll
              for (int d = 8; d >= 1; d >>= 1) {                // compensated sum over the 16 lanes
                const float oh = __shfl_xor_sync(kFull, z, d), ol = __shfl_xor_sync(kFull, zl, d);
                float sum, err;
                two_sum(z, oh, sum, err);
                z = sum;
                zl = (zl + ol) + err;
              }
              if (t == 0) pt[(size_t)sm.tc_seq[cur] * nCTA * S::PV * H + j] = make_float2(m, z + zl);
            }
          };
          #pragma unroll 1
          for (int u = 0;; ++u) {
            const int buf = u & 1;
            if (!__all_sync(kFull, mbar_wait(&accf[buf], (u >> 1) & 1, a.wait_ns))) {
              if (lane == 0) {
                set_error(a.status, TS_ERR_TIMEOUT);
                sm.timed_out = 1;
              }
              break;
            }
            tc_fence_after();
            if (sm.acc_nv[buf][0] < 0) break;
            const int tl = sm.acc_tl[buf][half], sgi = sm.acc_sg[buf], nvh = sm.acc_nv[buf][half];
            float r[8 * S::TC_NLD];
#pragma unroll
            for (int i = 0; i < S::TC_NLD; ++i)
              tmem_ld_x8(tq + buf * S::TC_COLS + 8 * i, *reinterpret_cast<float(*)[8]>(r + 8 * i));
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&acce[buf]);
            if (sgi != cur) {
              flush();
              cur = sgi;
#pragma unroll
              for (int j = 0; j < G; ++j) {
                run_m[j] = -INFINITY;
                run_z[j] = KahanF();
              }
            }
            float x[G];
#pragma unroll
            for (int j = 0; j < G; ++j) {
              const float hi = odd ? r[3 * G + 3 * j] : r[3 * j];
              const float mid = odd ? r[3 * G + 3 * j + 1] : r[3 * j + 1];
              const float lo = odd ? r[3 * G + 3 * j + 2] : r[3 * j + 2];
              // one rounding of the scaled dot product, with the scale constant in two parts
              const float acc = (lo + mid) + hi;
              x[j] = t < nvh ? fmaf(acc, a.scale_l2, acc * a.scale_l2_lo) : -INFINITY;
            }
            // (the rows of an absent second page belong to no token of this tile: nothing to store)
            float* dst = a.spill + (size_t)(tl + t) * H + g * G;
            if (nvh != kAbsentRows) {
              if constexpr (G == 4) {
                *reinterpret_cast<float4*>(dst) = make_float4(x[0], x[1], x[2], x[3]);
              } else {
#pragma unroll
                for (int j = 0; j < G; ++j) dst[j] = x[j];
              }
            }
#pragma unroll
            for (int j = 0; j < G; ++j) {
              if (x[j] > run_m[j]) {
                if (run_m[j] > -INFINITY) {
                  const float f = exp2f(run_m[j] - x[j]);
                  run_z[j].s *= f;
                  run_z[j].c *= f;
                }
                run_z[j].add(1.f);
                run_m[j] = x[j];
              } else if (x[j] > -INFINITY) {
                run_z[j].add(exp2f(x[j] - run_m[j]));
              }
            }
          }
          flush();
        }
        tc_fence_before();
        __syncthreads();
        if (tid == 32 && !mbar_wait(&drainb, 0, a.wait_ns)) {               // every MMA issued has completed
          set_error(a.status, TS_ERR_TIMEOUT);
          sm.timed_out = 1;
        }
        __syncthreads();
        if (tid == 0 && sm.timed_out) {
          // copies issued but never consumed land before the CTA leaves
          #pragma unroll 1
          for (int ss = 0; ss < nsl; ++ss)
            if (sm.slot_last[ss] >= 0) mbar_wait(&full[ss], (sm.slot_last[ss] / nsl) & 1, a.wait_ns);
        }
        __syncthreads();
        if (warp == 2) {
          tc_fence_after();
          tmem_dealloc(tmem, 2 * S::TC_COLS);
        }
        if (sm.timed_out) {
          if (tid == 0) atomicExch(&a.gsync->abort, 1u);   // the others leave at their next barrier
          return;
        }
        TS_MARK(2);
        TS_LAST(56);
        fence_proxy_async_global();
        // the first chunk of my logits (all written by this CTA) comes back into shared memory
        // while the other CTAs finish their scans
        const int pre = (!sm.scan_dyn && vrows > 0) ? 1 : 0;
        if (pre) {
          __syncthreads();                                       // after every writer's proxy fence
          if (tid == 0) issue_chunk(eb, 0, H, chunk_rows(H));
        }
        TS_MARK(3);
        if (!grid_sync(a.gsync, a.status, &sm.gepoch, a.wait_ns, a.skip_cta, a.skip_barrier)) {
          if (tid == 0 && pre) mbar_wait(&vbar[0], 0u, a.wait_ns);         // lands before the CTA leaves
          return;
        }
        TS_MARK(4);
        if (!vote_pass(eb, 0, H, 0, pre)) return;
      }
    }
    if (!scanned) {
      const int hpw = sm.hpw, HW = hpw * G, nwaves = sm.nwaves;
      float* eb = a.spill + (size_t)c * sm.region;   // my logits, token-major [tstride][HW]
      int stage_seq = 0;                             // ring use counter across waves
      #pragma unroll 1
      for (int wv = 0; wv < nwaves; ++wv) {
        const int g0 = wv * hpw;
        if (!cuda_scan_wave<KT, D, HKV, G>(a, sm, ring, full, wv, stage_seq)) return;
        fence_proxy_async_global();
        TS_MARK(3 + 3 * min(wv, 5));
        if (!grid_sync(a.gsync, a.status, &sm.gepoch, a.wait_ns, a.skip_cta, a.skip_barrier)) return;
        TS_MARK(4 + 3 * min(wv, 5));
        if (!vote_pass(eb, g0, HW, wv, 0)) return;
      }
    }
  }

  TS_MARK(20);
  TS_LAST(57);
  TS_LAST_CTA(57);
  // ======================================================================== SELECT
  // (nothing to select when every sequence hits or is empty: no pages were partitioned)
  if ((a.phases & kPhSelect) && sm.ptot > 0) {
    if (!(a.phases & kPhScore)) {
      if (!grid_sync(a.gsync, a.status, &sm.gepoch, a.wait_ns, a.skip_cta, a.skip_barrier)) return;   // the histograms are zero everywhere
    }
    // shared memory while selecting, one use after another: this CTA's histogram (counts,
    // then masses at a fixed offset); after the barrier, the global histograms of a batch of
    // sequences; later the gathered candidates
    unsigned* sh = reinterpret_cast<unsigned*>(ring);
    unsigned long long* smh = reinterpret_cast<unsigned long long*>(ring + lvl_bins(0) * sizeof(unsigned));
    unsigned long long* scand = reinterpret_cast<unsigned long long*>(ring);
    unsigned char* bat = ring;
    const bool topp = a.mode == TS_SELECT_TOPP;
    __syncthreads();
#pragma unroll 1   // one copy of the level code: it runs once per level and is fetched cold
    for (int level = 0; level < 3; ++level) {
      if (tid == 0) {
        int any = 0;
        #pragma unroll 1
        for (int b = 0; b < B; ++b) any |= !sm.seq[b].done;
        sm.flag = any;
      }
      __syncthreads();
      if (!sm.flag) break;                     // identical in every CTA
      const int shift = lvl_shift(level), nbins = lvl_bins(level);
      unsigned* gh = a.hist + lvl_off(level);                  // + b * kHistPerSeq
      unsigned long long* gm = a.mass + lvl_off(level);
      const int room = max(1, (a.dyn_bytes - a.flag_cap) / (nbins * (topp ? 12 : 4)));
      #pragma unroll 1
      for (int sg = 0; sg < sm.nseg; ++sg) {
        const int b = sm.seg_b[sg];
        const SeqState& st = sm.seq[b];
        if (st.done) continue;
        TS_MARK(33 + 4 * level);
        #pragma unroll 1
        for (int i = tid; i < nbins / 4; i += blockDim.x) {
          reinterpret_cast<uint4*>(sh)[i] = make_uint4(0u, 0u, 0u, 0u);
          if (topp) {
            reinterpret_cast<uint4*>(smh)[2 * i] = make_uint4(0u, 0u, 0u, 0u);
            reinterpret_cast<uint4*>(smh)[2 * i + 1] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        __syncthreads();
        TS_MARK(34 + 4 * level);
        const int tl0 = sm.seg_lp0[sg] * S::P;
        const int lo = max(st.lo, tl0), hi = min(st.hi, tl0 + sm.seg_ntok[sg]);
        const float* vb = a.vote + (size_t)b * a.vote_stride;
        #pragma unroll 2
        for (int t = lo + tid; t < hi; t += blockDim.x) {
          const float v = __ldcg(vb + t);
          const uint32_t key = __float_as_uint(v);
          const bool in = (key & st.mask) == st.prefix;
          const int bin = in ? (int)((key >> shift) & (nbins - 1)) : -1;
          // lanes with the same bin add once (the votes of a sequence crowd into few bins): the
          // count by the group's size, the top-p mass by the leader's sum of the group's masses
          // (staged in the selection-flag area, not yet in use)
          const unsigned am = __activemask();
          const unsigned peers = __match_any_sync(am, bin);
          const int leader = __ffs(peers) - 1;
          if (in && lane == leader) atomicAdd(&sh[bin], (unsigned)__popc(peers));
          if (topp) {
            unsigned long long* ms = reinterpret_cast<unsigned long long*>(selflag) + warp * 32;
            ms[lane] = in ? to_fx(v) : 0ull;
            __syncwarp(am);
            if (in && lane == leader) {
              unsigned long long sum = 0ull;
              for (unsigned pm = peers; pm; pm &= pm - 1u) sum += ms[__ffs(pm) - 1];
              atomicAdd(&smh[bin], sum);
            }
            __syncwarp(am);
          }
        }
        __syncthreads();
        TS_MARK(35 + 4 * level);
        #pragma unroll 1
        for (int i4 = tid; i4 < nbins / 4; i4 += blockDim.x) {
          const uint4 cv = reinterpret_cast<const uint4*>(sh)[i4];
          if (cv.x | cv.y | cv.z | cv.w) {
            const unsigned c4[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (c4[j]) {
                atomicAdd(&gh[(size_t)b * kHistPerSeq + 4 * i4 + j], c4[j]);
                if (topp) atomicAdd(&gm[(size_t)b * kHistPerSeq + 4 * i4 + j], smh[4 * i4 + j]);
              }
            }
          }
        }
        if (level == 0) {
          // coarse sums of 128 fine bins, one warp each, added once per CTA
          #pragma unroll 1
          for (int cbn = warp; cbn < 128; cbn += S::NW) {
            const uint4 v = reinterpret_cast<const uint4*>(sh + cbn * 128)[lane];
            const unsigned scn = __reduce_add_sync(kFull, v.x + v.y + v.z + v.w);
            unsigned long long smm = 0ull;
            if (topp) {
#pragma unroll
              for (int j = 0; j < 4; ++j) smm += smh[cbn * 128 + lane * 4 + j];
#pragma unroll
              for (int d = 16; d >= 1; d >>= 1) smm += __shfl_xor_sync(kFull, smm, d);
            }
            if (lane == 0 && scn) {
              atomicAdd(&a.hist[(size_t)b * kHistPerSeq + kCoarseOff + cbn], scn);
              if (topp) atomicAdd(&a.mass[(size_t)b * kHistPerSeq + kCoarseOff + cbn], smm);
            }
          }
        }
        __syncthreads();
      }
      fence_proxy_async_global();   // the histograms are read back by bulk copy
      TS_MARK(28 + level);
      if (!grid_sync(a.gsync, a.status, &sm.gepoch, a.wait_ns, a.skip_cta, a.skip_barrier)) return;
      TS_MARK(36 + 4 * level);
      // every CTA finds the crossing bin of every unresolved sequence from shared copies of
      // the global histograms (bulk copies); level 0 in two steps: its 128 coarse bins, then
      // the 128 fine bins of the crossing coarse bin
      auto apply = [&](SeqState& st, int bin, const Cross& r) {   // lane 0 of the scanning warp
        st.prefix |= (uint32_t)bin << shift;
        st.mask |= (uint32_t)(nbins - 1) << shift;
        st.n_gt += (int)r.before_c;
        if (topp)
          st.mass_rem = st.mass_rem - r.before_m;
        else
          st.k_rem = st.k_rem - (int)r.before_c;
        if (r.hc <= (unsigned)kCandCap) {
          st.cand = 1;
          st.done = 1;
        } else if (level == 2) {
          st.tie_mode = 1;
          st.done = 1;
          if (!topp) {
            st.ties = st.k_rem;
          } else {
            const unsigned long long tfx = to_fx(__uint_as_float(st.prefix));
            const unsigned long long t = tfx ? (st.mass_rem + tfx - 1) / tfx : (unsigned long long)r.hc;
            st.ties = (int)(t < r.hc ? t : r.hc);
          }
        }
      };
      // whole CTA: one bulk-copy transaction of a 128-bin block (counts, masses) per unresolved
      // sequence, at block offset off(b) of its histogram
      auto fetch128 = [&](unsigned* dc, unsigned long long* dm, auto off) -> bool {
        if (tid == 0) {
          uint32_t bytes = 0;
          #pragma unroll 1
          for (int b = 0; b < B; ++b)
            if (!sm.seq[b].done) bytes += topp ? 128u * 12u : 128u * 4u;
          fence_proxy_async_global();
          mbar_arrive_expect_tx(&xbar, bytes);
          #pragma unroll 1
          for (int b = 0; b < B; ++b) {
            if (sm.seq[b].done) continue;
            bulk_g2s(dc + b * 128, a.hist + (size_t)b * kHistPerSeq + off(b), 512u, &xbar);
            if (topp) bulk_g2s(dm + b * 128, a.mass + (size_t)b * kHistPerSeq + off(b), 1024u, &xbar);
          }
        }
        const bool landed = mbar_wait(&xbar, xph, a.wait_ns);
        xph ^= 1u;
        if (__syncthreads_and(landed)) return true;
        if (tid == 0) {
          set_error(a.status, TS_ERR_TIMEOUT);
          atomicExch(&a.gsync->abort, 1u);
        }
        return false;
      };
      if (level == 0) {
        unsigned* cc_ = reinterpret_cast<unsigned*>(bat);                                   // [B][128]
        unsigned long long* cm_ = reinterpret_cast<unsigned long long*>(bat + (size_t)B * 512);
        if (!fetch128(cc_, cm_, [](int) { return kCoarseOff; })) return;
        TS_MARK(45);
        #pragma unroll 1
        for (int b = warp; b < B; b += S::NW) {
          SeqState& st = sm.seq[b];
          if (st.done) continue;
          const Cross r = find_crossing(cc_ + b * 128, cm_ + b * 128, 128, topp, 0u, 0ull, (unsigned)st.k_rem,
                                        st.mass_rem);
          if (lane == 0) {
            if (r.bin < 0) {        // top-p whose fixed-point total falls short: the whole domain
              st.all = 1;
              st.done = 1;
            } else {
              sm.x_bin[b] = r.bin;
              sm.x_c[b] = r.before_c;
              sm.x_m[b] = r.before_m;
            }
          }
        }
        __syncthreads();
        if (!fetch128(cc_, cm_, [&](int b) { return sm.x_bin[b] * 128; })) return;
        TS_MARK(46);
        #pragma unroll 1
        for (int b = warp; b < B; b += S::NW) {
          SeqState& st = sm.seq[b];
          if (st.done) continue;
          const Cross r = find_crossing(cc_ + b * 128, cm_ + b * 128, 128, topp, sm.x_c[b], sm.x_m[b],
                                        (unsigned)st.k_rem, st.mass_rem);
          if (lane == 0 && r.bin >= 0) apply(st, sm.x_bin[b] * 128 + r.bin, r);
        }
        __syncthreads();
      } else {
        const int room = max(1, (a.dyn_bytes - a.flag_cap) / (nbins * (topp ? 12 : 4)));
        #pragma unroll 1
        for (int b0 = 0; b0 < B; b0 += room) {
          const int nb = min(room, B - b0);
          unsigned* bc = reinterpret_cast<unsigned*>(bat);                                  // [nb][nbins]
          unsigned long long* bm = reinterpret_cast<unsigned long long*>(bat + (size_t)room * nbins * 4);
          if (tid == 0) {
            uint32_t bytes = 0;
            #pragma unroll 1
            for (int bi = 0; bi < nb; ++bi)
              if (!sm.seq[b0 + bi].done) bytes += (uint32_t)nbins * (topp ? 12u : 4u);
            fence_proxy_async_global();
            mbar_arrive_expect_tx(&xbar, bytes);
            #pragma unroll 1
            for (int bi = 0; bi < nb; ++bi) {
              if (sm.seq[b0 + bi].done) continue;
              bulk_g2s(bc + (size_t)bi * nbins, gh + (size_t)(b0 + bi) * kHistPerSeq, (uint32_t)nbins * 4u, &xbar);
              if (topp)
                bulk_g2s(bm + (size_t)bi * nbins, gm + (size_t)(b0 + bi) * kHistPerSeq, (uint32_t)nbins * 8u, &xbar);
            }
          }
          {
            const bool landed = mbar_wait(&xbar, xph, a.wait_ns);
            xph ^= 1u;
            if (!__syncthreads_and(landed)) {
              if (tid == 0) {
                set_error(a.status, TS_ERR_TIMEOUT);
                atomicExch(&a.gsync->abort, 1u);
              }
              return;
            }
          }
          #pragma unroll 1
          for (int bi = warp; bi < nb; bi += S::NW) {
            SeqState& st = sm.seq[b0 + bi];
            if (st.done) continue;
            const Cross r = find_crossing(bc + (size_t)bi * nbins, bm + (size_t)bi * nbins, nbins, topp, 0u, 0ull,
                                          (unsigned)st.k_rem, st.mass_rem);
            if (lane == 0) {
              if (r.bin < 0) {
                st.all = 1;
                st.done = 1;
              } else {
                apply(st, r.bin, r);
              }
            }
          }
          __syncthreads();
        }
      }
    }

    TS_MARK(21);
    // ---- (1) the class of each of my tokens, a byte in the flags: 0 out, 1 selected, 2 in the
    // crossing bin (ranked below against every CTA's), 3 an exact tie of the crossing value. Warp
    // w takes a contiguous run of the segment's tokens, so per-warp counts give positions in token
    // order. Crossing-bin tokens are appended to the sequence's candidate list; exact ties are
    // counted per CTA.
    int need_cand = 0, need_tie = 0;
    #pragma unroll 1
    for (int b = 0; b < B; ++b) {
      need_cand |= sm.seq[b].cand;
      need_tie |= sm.seq[b].tie_mode;
    }
    auto warp_run = [&](int nt, int& w0, int& w1) {
      const int per = ((nt + S::NW * 32 - 1) / (S::NW * 32)) * 32;   // tokens per warp, whole 32s
      w0 = min(nt, warp * per);
      w1 = min(nt, w0 + per);
    };
    #pragma unroll 1
    for (int sg = 0; sg < sm.nseg; ++sg) {
      const int b = sm.seg_b[sg];
      const SeqState& st = sm.seq[b];
      const int tl0 = sm.seg_lp0[sg] * S::P, nt = sm.seg_ntok[sg];
      const float* vb = a.vote + (size_t)b * a.vote_stride;
      uint8_t* fl = selflag + sm.seg_t0[sg];
      int w0, w1;
      warp_run(nt, w0, w1);
      int nties = 0;
      #pragma unroll 1
      for (int i0 = w0; i0 < w1; i0 += 4 * 32) {   // four loads in flight per lane
        uint32_t key[4];
        uint8_t cls[4];
        unsigned cm = 0;                              // bit u: token u of this lane is in the crossing bin
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * 32 + lane;
          key[u] = i < w1 ? __float_as_uint(__ldcg(vb + tl0 + i)) : 0u;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * 32 + lane, t = tl0 + i;
          cls[u] = 0;
          if (i < w1 && t >= st.lo && t < st.hi) {
            const uint32_t km = key[u] & st.mask;
            if (st.all || km > st.prefix) cls[u] = 1;
            else if (km == st.prefix) cls[u] = st.cand ? 2 : (st.tie_mode ? 3 : 0);
          }
          if (i < w1) fl[i] = cls[u];
          nties += cls[u] == 3;
          cm |= (unsigned)(cls[u] == 2) << u;
        }
        if (__any_sync(kFull, cm != 0)) {
          #pragma unroll 1
          for (int u = 0; u < 4; ++u) {
            const bool is = (cm >> u) & 1u;
            const unsigned bal = __ballot_sync(kFull, is);
            if (!bal) continue;
            unsigned base = 0;
            if (lane == 0) base = atomicAdd(&a.cand_n[b], (unsigned)__popc(bal));
            base = __shfl_sync(kFull, base, 0);
            const unsigned pos = base + __popc(bal & ((1u << lane) - 1u));
            uint32_t kk = key[0];
#pragma unroll
            for (int v = 1; v < 4; ++v)
              if (u == v) kk = key[v];
            if (is && pos < (unsigned)kCandCap)
              a.cands[(size_t)b * kCandCap + pos] =
                  ((unsigned long long)kk << 32) | (0xffffffffu - (uint32_t)(tl0 + i0 + u * 32 + lane));
          }
        }
      }
      if (st.tie_mode) {
        nties = warp_sum_i(nties);
        if (lane == 0) sm.red_i[0][warp] = nties;
        __syncthreads();
        if (tid == 0) {
          int tot = 0;
          #pragma unroll 1
          for (int w = 0; w < S::NW; ++w) tot += sm.red_i[0][w];
          a.cta_cnt[((size_t)b * nCTA + c) * 4 + 2] = tot;
        }
        __syncthreads();
      }
    }
    TS_MARK(47);
    TS_LAST(58);
    TS_LAST_CTA(58);
    if (need_cand || need_tie) {
      if (!grid_sync(a.gsync, a.status, &sm.gepoch, a.wait_ns, a.skip_cta, a.skip_barrier)) return;
    }
    TS_MARK(48);
    if (need_tie) {
      // exact ties before mine, per segment, one warp each
      #pragma unroll 1
      for (int sg = warp; sg < sm.nseg; sg += S::NW) {
        const int b = sm.seg_b[sg];
        const SeqState& st = sm.seq[b];
        int s = 0;
        if (st.tie_mode)
          #pragma unroll 1
          for (int cc = st.first_cta + lane; cc < c; cc += 32) s += __ldcg(&a.cta_cnt[((size_t)b * nCTA + cc) * 4 + 2]);
        s = warp_sum_i(s);
        if (lane == 0) sm.tie_base[sg] = s;
      }
      __syncthreads();
    }

    TS_MARK(22);
    // ---- (2) exact ties and crossing-bin tokens decided, then my selected tokens as an ascending
    // list and the counts for the output positions
    #pragma unroll 1
    for (int sg = 0; sg < sm.nseg; ++sg) {
      const int b = sm.seg_b[sg];
      const SeqState& st = sm.seq[b];
      const int tl0 = sm.seg_lp0[sg] * S::P, t0l = sm.seg_t0[sg], nt = sm.seg_ntok[sg];
      const float* vb = a.vote + (size_t)b * a.vote_stride;
      uint8_t* fl = selflag + t0l;
      int w0, w1;
      warp_run(nt, w0, w1);
      const int m_cand = st.cand ? (int)min(__ldcg(&a.cand_n[b]), (unsigned)kCandCap) : 0;
      #pragma unroll 4
      for (int j = tid; j < m_cand; j += blockDim.x) scand[j] = __ldcg(&a.cands[(size_t)b * kCandCap + j]);
      __syncthreads();
      TS_MARK(49);
      // exact ties in token order: the first st.ties of them over the sequence are taken
      if (st.tie_mode) {
        int nties = 0;
        #pragma unroll 1
        for (int i0 = w0; i0 < w1; i0 += 32) nties += __popc(__ballot_sync(kFull, i0 + lane < w1 && fl[i0 + lane] == 3));
        if (lane == 0) sm.red_i[0][warp] = nties;
        __syncthreads();
        int off = sm.tie_base[sg];
        #pragma unroll 1
        for (int w = 0; w < warp; ++w) off += sm.red_i[0][w];
        #pragma unroll 1
        for (int i0 = w0; i0 < w1; i0 += 32) {
          const int i = i0 + lane;
          const bool tie = i < w1 && fl[i] == 3;
          const unsigned bal = __ballot_sync(kFull, tie);
          if (tie) fl[i] = (off + __popc(bal & ((1u << lane) - 1u))) < st.ties ? 1 : 0;
          off += __popc(bal);
        }
        __syncthreads();                                  // red_i is reused below
      }
      // tokens of the crossing bin: the warp ranks those of its own range against the gathered
      // candidates (a chunk's crossing tokens have their votes loaded at once, one per lane)
      if (st.cand) {
        int ncross = 0;
        #pragma unroll 1
        for (int i0 = w0; i0 < w1; i0 += 32) {
          const bool cr = i0 + lane < w1 && fl[i0 + lane] == 2;
          const uint32_t mykey = cr ? __float_as_uint(__ldcg(vb + tl0 + i0 + lane)) : 0u;
          unsigned bal = __ballot_sync(kFull, cr);
          ncross += __popc(bal);
          while (bal) {
            const int src = __ffs(bal) - 1, ii = i0 + src;
            bal &= bal - 1u;
            const uint32_t kk = __shfl_sync(kFull, mykey, src);
            const unsigned long long me = ((unsigned long long)kk << 32) | (0xffffffffu - (uint32_t)(tl0 + ii));
            unsigned above = 0;
            unsigned long long cum = 0;
            #pragma unroll 8   // independent loads in flight together (a warp may rank dozens of tokens)
            for (int j = lane; j < m_cand; j += 32) {
              const unsigned long long y = scand[j];
              if (y > me) {
                ++above;
                if (topp) cum += to_fx(__uint_as_float((uint32_t)(y >> 32)));
              }
            }
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) {
              above += __shfl_xor_sync(kFull, above, d);
              cum += __shfl_xor_sync(kFull, cum, d);
            }
            if (lane == 0) fl[ii] = (topp ? (cum < st.mass_rem) : (above < (unsigned)st.k_rem)) ? 1 : 0;
            __syncwarp();
          }
        }
        // diagnosis (slot 60): the most crossing tokens one warp ranked, above the candidate count
        // and the CTA
        if (lane == 0 && a.phase_ns)
          atomicMax(&a.phase_ns[60], ((unsigned long long)ncross << 32) | ((unsigned long long)m_cand << 8) | (unsigned)c);
      }
      TS_MARK(50);
      // counts per warp (all, in [s_end, ls), below s_end), then the list in token order, the list
      // of this segment from its row t0l
      int na = 0, nc = 0, nlo = 0;
      #pragma unroll 1
      for (int i0 = w0; i0 < w1; i0 += 32) {
        const int i = i0 + lane, t = tl0 + i;
        const bool f = i < w1 && fl[i] == 1;
        na += __popc(__ballot_sync(kFull, f));
        nc += __popc(__ballot_sync(kFull, f && t >= st.s_end && t < st.ls));
        nlo += __popc(__ballot_sync(kFull, f && t < st.s_end));
      }
      if (lane == 0) {
        sm.red_i[0][warp] = na;
        sm.red_i[1][warp] = nc;
        sm.red_i[2][warp] = nlo;
      }
      __syncthreads();
      int off = 0;
      #pragma unroll 1
      for (int w = 0; w < warp; ++w) off += sm.red_i[0][w];
      #pragma unroll 1
      for (int i0 = w0; i0 < w1; i0 += 32) {
        const int i = i0 + lane;
        const bool f = i < w1 && fl[i] == 1;
        const unsigned bal = __ballot_sync(kFull, f);
        if (f) sel_list[t0l + off + __popc(bal & ((1u << lane) - 1u))] = tl0 + i;
        off += __popc(bal);
      }
      if (tid == 0) {
        int ta = 0, tc = 0, tlo = 0;
        #pragma unroll 1
        for (int w = 0; w < S::NW; ++w) {
          ta += sm.red_i[0][w];
          tc += sm.red_i[1][w];
          tlo += sm.red_i[2][w];
        }
        a.cta_cnt[((size_t)b * nCTA + c) * 4 + 0] = tc;
        a.cta_cnt[((size_t)b * nCTA + c) * 4 + 1] = ta;
        a.cta_cnt[((size_t)b * nCTA + c) * 4 + 3] = tlo;
        sm.sel_a[sg] = ta;
        sm.sel_c[sg] = tc;
        sm.sel_lo[sg] = tlo;
      }
      __syncthreads();
    }
  }

  TS_MARK(23);
  TS_LAST(59);
  TS_LAST_CTA(59);
  // With top-p the selected tokens can crowd into a few CTAs' ranges: after one more barrier
  // every CTA takes an equal share of each sequence's selected tokens (the CTAs' lists in
  // order, a fixed assignment) instead of its own
  const bool bal = a.mode == TS_SELECT_TOPP && (a.phases & kPhSelect) && (a.phases & kPhAttend) && sm.ptot > 0;
  // A batch of top-k sequences: sequence b's fixed and selected tokens are shared out evenly over
  // its group of CTAs [fx_base, fx_base + fx_stride), so that short sequences (few CTAs hold their
  // pages) do not load a few CTAs with every one of their tokens
  const bool attend_grouped = a.mode == TS_SELECT_TOPK && (a.phases & kPhSelect) && (a.phases & kPhAttend) &&
                              B > 1 && sm.ptot > 0;
  if ((bal || attend_grouped) && !grid_sync(a.gsync, a.status, &sm.gepoch, a.wait_ns, a.skip_cta, a.skip_barrier))
    return;
  const bool shared_lists = bal || attend_grouped;   // selected tokens read from every CTA's list
  // ======================================================================== ATTEND
  // My tokens per sequence: a round-robin share of the fixed ones (sinks and
  // window, the cached part of a hit, or the caller's index list) and my own
  // selected candidates; gathered by bulk copy; one partial per CTA and head.
  // attention partials, each (sequence, head, part of the d columns) contiguous for one bulk copy
  // in the merge: o [B][H][dq][nCTA][D / dq], then (max, sum) [B][H][nCTAp] (nCTAp even: 16-byte
  // blocks); the columns split into dq parts (a power of two, D / dq >= 32) so that the merge
  // has about one item per CTA
  const int nCTAp = (nCTA + 1) & ~1;
  int dq = 1;
  while (2 * dq * 32 <= D && B * H * 2 * dq <= nCTA) dq *= 2;
  const int Dq = D / dq;
  float* ao = a.apart;
  float2* aml = reinterpret_cast<float2*>(a.apart + (size_t)B * H * nCTA * D);
  if (a.phases & kPhAttend) {
    // Per gather round: (1) one warp per (token, KV head) pair writes the G scores to shared
    // memory, (2) one warp per query head takes the round's max, turns scores into weights
    // against a running (max, sum) and keeps the correction of earlier rounds, (3) each thread
    // owns float4 slices of the output and adds the weighted V rows. The CTA's partial per
    // head (o, max, sum) goes to scratch for the merge after the last barrier.
    constexpr int HQ = HKV * G, EPL = D / 32, D4 = D / 4, NGRP = HQ * D4;
    constexpr int NG = (NGRP + S::THREADS - 1) / S::THREADS;
    static_assert(HQ <= kMaxAttH && D % 32 == 0, "attention layout");
    const bool given = !(a.phases & kPhSelect);
    // the staging area ends with the batch of looked-up selected tokens and their pages
    const int stage_bytes = a.dyn_bytes - a.flag_cap - 2 * kOwnBatch * (int)sizeof(int);
    int* const ob_t = reinterpret_cast<int*>(dsm + stage_bytes);
    int* const ob_p = ob_t + kOwnBatch;
    const int around = min(kMaxRound, (stage_bytes - HQ * 4) / (S::TOKEN_BYTES + HQ * 4));
    KT* Ks = reinterpret_cast<KT*>(dsm);
    KT* Vs = Ks + (size_t)around * HKV * D;
    float* Ps = reinterpret_cast<float*>(Vs + (size_t)around * HKV * D);   // [HQ][ldp] scores, weights
    const int ldp = around | 1;                        // odd row stride: a warp's column reads hit distinct banks
    // scores: warp -> one KV head (NW is a multiple of H_kv), its G queries in registers
    constexpr int NWG = S::NW / HKV;
    const int gw = warp % HKV, wsl = warp / HKV;
    constexpr bool kRangeGeom = D % 8 == 0 && S::THREADS % (HKV * (D / 8)) == 0 && S::P * HQ <= S::THREADS;
    // the tensor-core variant: bf16 pools, d = 128 (M = the columns of d), the two weight terms of
    // the G heads in 16 columns, and its ring (at least two slots) with the outputs' reduction
    // inside the V slots
    constexpr bool kRangeTC = S::TC && D == 128 && 2 * G <= 16 && HKV * 16 <= 256 &&
                              range_tc_slots<D, HKV, G>(kStageMin, kStepFlagCap) >= 2 &&
                              (HQ * D + S::P * HQ) * 4 <= 2 * HKV * S::P * D * 2;
    const bool topp_att = a.mode == TS_SELECT_TOPP && (a.phases & kPhSelect) && (a.phases & kPhAttend);
    if (topp_att) {
      // top-p sequences that take the range attention (1: a miss over each CTA's scanned range; 2:
      // a hit over an even split of its pages) when the selection is dense enough that streaming
      // pages beats sharing the tokens out, in the ratio of their measured costs: for a miss the
      // pages of the busiest range against the even share of tokens, for a hit all its pages
      // (K and V) against all its attended tokens. The same decision in every CTA, from the
      // per-CTA counts published before the barrier and the cache state read at set-up.
      constexpr int RSLOT = S::STAGE_BYTES + 2 * S::P * HQ * 4;
      const int rslots = range_slots<KT, D, HKV, G, false>(stage_bytes, a.flag_cap);
      const bool range_ok = kRangeGeom && bal && a.range_attend > 0 && sm.hpw == HKV && !sm.scan_dyn &&
                            ((kRangeTC && a.tcv) || (rslots >= 2 && HQ * D * 4 + S::P * HQ * 4 <= rslots * RSLOT));
      const bool hit_ok = kRangeGeom && a.range_attend > 0 && a.ct != nullptr &&
                          range_slots<KT, D, HKV, G, true>(stage_bytes, a.flag_cap) >= 2 &&
                          HQ * D * 4 + S::P * HQ * 4 <= 2 * (2 * S::STAGE_BYTES + 2 * S::P * HQ * 4);
      #pragma unroll 1
      for (int b = 0; b < B; ++b) {
        const SeqState& st = sm.seq[b];
        int take = 0;
        if (range_ok && !st.hit && st.pg1 > st.pg0) {
          const int nfix = st.s_end + (st.n - st.ls);
          int umax = 0, tot = 0;
          #pragma unroll 1
          for (int cc = st.first_cta + tid; cc <= st.last_cta; cc += blockDim.x) {
            const int pages = min(st.pg1, (cc + 1) * sm.ppc) - max(st.pg0, cc * sm.ppc);
            umax = max(umax, min(pages, __ldcg(&a.cta_cnt[((size_t)b * nCTA + cc) * 4 + 1]) + nfix));
            tot += __ldcg(&a.cta_cnt[((size_t)b * nCTA + cc) * 4 + 0]);
          }
          umax = __reduce_max_sync(kFull, umax);
          tot = __reduce_add_sync(kFull, tot);
          if (lane == 0) {
            sm.red_i[0][warp] = umax;
            sm.red_i[1][warp] = tot;
          }
          __syncthreads();
          if (tid == 0) {
            #pragma unroll 1
            for (int w = 1; w < S::NW; ++w) {
              umax = max(umax, sm.red_i[0][w]);
              tot += sm.red_i[1][w];
            }
            take = a.range_attend == 2 || (int64_t)umax * 4 * nCTA <= (int64_t)(tot + nfix) * 3;
          }
          __syncthreads();
        } else if (hit_ok && st.hit && st.n > 0) {
          const int npg_seq = (st.n + S::P - 1) / S::P;
          const int nfix = st.s_end + (st.n - st.ls) + (sm.ct_hi[b] - sm.ct_lo[b]);
          if ((npg_seq + nCTA - 1) / nCTA <= a.flag_cap / S::P &&
              (a.range_attend == 2 || (int64_t)npg_seq * 5 <= (int64_t)nfix))
            take = 2;
        }
        if (tid == 0) sm.bal.range_b[b] = take;
      }
      __syncthreads();
    }
    #pragma unroll 1
    for (int b = 0; b < B; ++b) {
      const SeqState& st = sm.seq[b];
      if (topp_att && sm.bal.range_b[b]) {
        if (sm.bal.range_b[b] == 2) {          // a hit: every CTA takes its share of the pages
          if constexpr (kRangeGeom)
            if (!range_attend<KT, D, HKV, G, true>(a, sm, dsm, stage_bytes, selflag, b, -1, ao, aml, nCTAp, dq))
              return;
          continue;
        }
        const int sgr = sm.my_seg_of[b];
        if (sgr >= 0) {
          if constexpr (kRangeTC) {
            if (a.tcv) {
              if (!range_attend_tc<KT, D, HKV, G>(a, sm, dsm, stage_bytes, selflag, b, sgr, ao, aml, nCTAp, dq))
                return;
              continue;
            }
          }
          if constexpr (kRangeGeom)
            if (!range_attend<KT, D, HKV, G, false>(a, sm, dsm, stage_bytes, selflag, b, sgr, ao, aml, nCTAp, dq))
              return;
        } else {
          if (tid < HQ) aml[((size_t)b * H + tid) * nCTAp + c] = make_float2(-INFINITY, 0.f);
          fence_proxy_async_global();
        }
        continue;
      }
      const int32_t* gib = a.idx + (size_t)b * a.idx_stride;
      const int32_t* ctb = nullptr;
      int nfix, ct_lo = 0, ct_hi = 0;
      if (given) {
        nfix = max(0, min(a.count[b], (int)a.idx_stride));
      } else {
        nfix = st.s_end + (st.n - st.ls);
        if (st.hit && a.ct) {
          ctb = a.ct + (size_t)b * a.cap;
          ct_lo = sm.ct_lo[b];
          ct_hi = sm.ct_hi[b];
          nfix += ct_hi - ct_lo;
        }
      }
      const int nmid = ct_hi - ct_lo;
      const int sgi = sm.my_seg_of[b];
      const bool in_group = c >= st.fx_base && c < st.fx_base + st.fx_stride;
      const bool own = !given && !st.hit &&
                       (bal ? st.pg1 > st.pg0 : (attend_grouped ? (st.pg1 > st.pg0 && in_group) : sgi >= 0));
      int own_nc = own && !shared_lists ? sm.sel_c[sgi] : 0, own_s0 = 0;
      const int* own_lst = own && !shared_lists ? sel_list + sm.seg_t0[sgi] + sm.sel_lo[sgi] : nullptr;
      if (own && shared_lists) {
        // the sequence's CTAs' counts of selected tokens in [s_end, ls): prefix offsets, and my share
        int tot = 0;
        #pragma unroll 1
        for (int c0 = 0; c0 < nCTA; c0 += blockDim.x) {
          const int cc = c0 + tid;
          const bool mine = cc >= st.first_cta && cc <= st.last_cta;
          const int x = mine ? __ldcg(&a.cta_cnt[((size_t)b * nCTA + cc) * 4 + 0]) : 0;
          const int xlo = mine ? __ldcg(&a.cta_cnt[((size_t)b * nCTA + cc) * 4 + 3]) : 0;
          int t_;
          const int r = block_scan(x, sm.wsum, t_);
          if (cc < nCTA) {
            sm.bal.pref[cc] = tot + r;
            sm.bal.nlo[cc] = xlo;
          }
          tot += t_;
        }
        if (tid == 0) sm.bal.pref[nCTA] = tot;
        // my equal share: of every CTA (top-p), or of the sequence's group
        const int sh0 = bal ? 0 : st.fx_base, shn = bal ? nCTA : st.fx_stride;
        own_s0 = (int)((int64_t)(c - sh0) * tot / shn);
        own_nc = (int)((int64_t)(c - sh0 + 1) * tot / shn) - own_s0;
        __syncthreads();
      }
      const int own_lp0 = own ? sm.seg_lp0[sgi] : 0, own_t0 = own ? sm.seg_t0[sgi] : 0;
      const int fstride = given ? nCTA : st.fx_stride;
      const int fbase = given ? 0 : st.fx_base;
      const int nfix_mine = (c - fbase >= 0 && c - fbase < fstride && c - fbase < nfix)
                                ? (nfix - (c - fbase) + fstride - 1) / fstride
                                : 0;
      if (!own && nfix_mine == 0) {
        // nothing of this sequence here: an empty partial (the merge gives it weight 0)
        if (tid < HQ) aml[((size_t)b * H + tid) * nCTAp + c] = make_float2(-INFINITY, 0.f);
        fence_proxy_async_global();
        continue;
      }
      float qreg[S::GP][EPL];
#pragma unroll
      for (int h = 0; h < S::GP; ++h)
#pragma unroll
        for (int e = 0; e < EPL; ++e)
          qreg[h][e] = h < G ? a.q[((size_t)b * HQ + gw * G + h) * D + lane * EPL + e] : 0.f;
      if (tid < HQ) {
        sm.att_m[tid] = -INFINITY;
        sm.att_l[tid] = 0.f;
      }
      TS_MARK(51);
      float4 o[NG];
#pragma unroll
      for (int k = 0; k < NG; ++k) o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      int fdone = 0;     // fixed tokens of mine already taken
      int opos = 0;      // next own token (position in my list)
      bool first_round = true;   // (diagnosis: the first round's marks go to slots 8, 12, 19 and 31)
      int ob0 = 0, ob_end = 0;   // my share's positions [ob0, ob_end) looked up in ob_t / ob_p
      // the K and V rows of every KV head of list entries [j0, j1), 16 bytes per thread and copy
      // (all of them in flight at once), as one commit group
      auto gather_rows = [&](int j0, int j1) {
        constexpr int CPR = S::ROW_BYTES / 16;         // 16-byte chunks of a row
        static_assert(S::ROW_BYTES % 16 == 0, "rows of whole 16-byte chunks");
        #pragma unroll 2
        for (int i = tid; i < 2 * (j1 - j0) * HKV * CPR; i += blockDim.x) {
          const int rr = i / CPR, ch = i % CPR;
          const int ti = j0 + rr / (2 * HKV), rem = rr % (2 * HKV), g = rem >> 1, isv = rem & 1;
          const int t = sm.toks[ti];
          const int page = sm.tval[ti];
          size_t off = 0;
          if (page >= 0 && (int64_t)page < a.num_pages) {
            off = (((size_t)page * HKV + g) * S::P + (t % S::P)) * S::ROW_BYTES;
          } else if (rem == 0 && ch == 0) {
            set_error(a.status, TS_ERR_PAGE_OOB);
          }
          cp_async16(reinterpret_cast<unsigned char*>((isv ? Vs : Ks) + ((size_t)ti * HKV + g) * D) + ch * 16,
                     (isv ? a.v_pool : a.k_pool) + off + ch * 16);
        }
        cp_async_commit();
      };
      __syncthreads();
      while (true) {
        // ---- this round's tokens: fixed share first, then own selected ones
        int cnt = 0;
        const int nf = min(around, nfix_mine - fdone);
        const bool pf = !given && sm.pf_ok;
        #pragma unroll 1
        for (int i = tid; i < nf; i += blockDim.x) {
          int t, page = -1;
          if (pf) {
            t = sm.pf_t[sm.pf_off[b] + fdone + i];
            page = sm.pf_p[sm.pf_off[b] + fdone + i];
          } else {
            const int f = (c - fbase) + (fdone + i) * fstride;
            if (given) t = gib[f];
            else if (f < st.s_end) t = f;
            else if (f < st.s_end + nmid) t = __ldcg(ctb + ct_lo + (f - st.s_end));
            else t = st.ls + (f - st.s_end - nmid);
            if (t >= 0 && t < a.max_tokens) page = a.page_table[(size_t)b * a.pt_stride + t / S::P];
          }
          sm.toks[i] = t;
          sm.tval[i] = page;
        }
        fdone += nf;
        cnt = nf;
        // the fixed tokens' rows start moving now; the own selected ones are listed meanwhile
        if (nf > 0) {
          __syncthreads();
          gather_rows(0, nf);
        }
        TS_MARK(52);
        if (own && opos < own_nc && cnt < around) {
          // my selected tokens in [s_end, ls), in list order, as many as fit
          const int take = min(around - cnt, own_nc - opos);
          if (shared_lists && opos + take > ob_end) {
            // the next batch of my share: every entry looked up at once (position in the sequence's
            // concatenated lists -> the CTA whose list holds it -> the token -> its page)
            ob0 = opos;
            ob_end = min(own_nc, opos + kOwnBatch);
            #pragma unroll 1
            for (int r = tid; r < ob_end - ob0; r += blockDim.x) {
              const int p = own_s0 + ob0 + r;
              int lo = st.first_cta, hi = st.last_cta;
              while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (sm.bal.pref[mid] <= p) lo = mid;
                else hi = mid - 1;
              }
              const int* lst = a.sel_rows + (size_t)lo * a.flag_cap +
                               (max(st.pg0, lo * sm.ppc) - lo * sm.ppc) * S::P + sm.bal.nlo[lo];
              const int t = __ldcg(lst + (p - sm.bal.pref[lo]));
              ob_t[r] = t;
              ob_p[r] = a.page_table[(size_t)b * a.pt_stride + t / S::P];
            }
            __syncthreads();
          }
          #pragma unroll 1
          for (int r = tid; r < take; r += blockDim.x) {
            int t, page;
            if (shared_lists) {
              t = ob_t[opos - ob0 + r];
              page = ob_p[opos - ob0 + r];
            } else {
              t = own_lst[opos + r];
              const int lpg = (own_t0 + (t - own_lp0 * S::P)) / S::P;   // my page of the token
              page = lpg < kMaxPagesCta ? sm.my_pages[lpg] : a.page_table[(size_t)b * a.pt_stride + t / S::P];
            }
            sm.toks[cnt + r] = t;
            sm.tval[cnt + r] = page;
          }
          opos += take;
          cnt += take;
          __syncthreads();
        }
        TS_MARK(9);
        if (first_round) TS_MARK(8);
        if (cnt == 0) break;                          // uniform: same counters in every thread
        // ---- the own tokens' rows, then every row of the round has landed
        __syncthreads();
        gather_rows(nf, cnt);
        TS_MARK(53);
        cp_async_wait_all();
        __syncthreads();
        TS_MARK(10);
        if (first_round) TS_MARK(12);
        // ---- (1) scores: warp -> (its KV head, tokens wsl, wsl + NWG, ...); lane holds EPL dims,
        // the G dot products are reduced across the warp so that lane `which` ends with head `which`
#pragma unroll 4   // independent tokens: their loads and shuffle trees overlap
        for (int j = wsl; j < cnt; j += NWG) {
          float kf[EPL];
          load_elems<KT, EPL>(Ks + ((size_t)j * HKV + gw) * D + lane * EPL, kf);
          float acc[S::GP];
#pragma unroll
          for (int h = 0; h < S::GP; ++h) {
            float x = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) x = fmaf(qreg[h][e], kf[e], x);
            acc[h] = x;
          }
          int which;
          const float dot = transpose_reduce<S::GP, 32>(acc, lane, which);
          const bool live = sm.tval[j] >= 0 && (int64_t)sm.tval[j] < a.num_pages;
          if ((lane & (32 / S::GP - 1)) == 0 && which < G) Ps[(gw * G + which) * ldp + j] = live ? dot * a.scale : -INFINITY;
        }
        __syncthreads();
        TS_MARK(15);
        // ---- (2) weights: warp per query head
        #pragma unroll 1
        for (int h = warp; h < HQ; h += S::NW) {
          float mr = -INFINITY;
          #pragma unroll 1
          for (int t = lane; t < cnt; t += 32) mr = fmaxf(mr, Ps[h * ldp + t]);
          mr = warp_max(mr);
          const float mo = sm.att_m[h], mn = fmaxf(mo, mr);
          float sum = 0.f;
          #pragma unroll 1
          for (int t = lane; t < cnt; t += 32) {
            const float w = mn > -INFINITY ? expf(Ps[h * ldp + t] - mn) : 0.f;
            Ps[h * ldp + t] = w;
            sum += w;
          }
          sum = warp_sum_comp(sum);
          if (lane == 0) {
            const float corr = mo > -INFINITY ? expf(mo - mn) : 0.f;
            sm.att_c[h] = corr;
            sm.att_l[h] = fmaf(sm.att_l[h], corr, sum);
            sm.att_m[h] = mn;
          }
        }
        __syncthreads();
        TS_MARK(16);
        if (first_round) TS_MARK(19);
        // ---- (3) outputs: thread -> float4 slices (head, 4 dims)
#pragma unroll
        for (int k = 0; k < NG; ++k) {
          const int qd = tid + k * S::THREADS;
          if (qd < NGRP) {
            const int h = qd / D4, d4 = qd % D4, g = h / G;
            const float corr = sm.att_c[h];
            // four tokens per step into two accumulators: the loads of a step are in flight together
            float4 acc = make_float4(o[k].x * corr, o[k].y * corr, o[k].z * corr, o[k].w * corr);
            float4 acc2 = make_float4(0.f, 0.f, 0.f, 0.f);
            int t = 0;
            #pragma unroll 1
            for (; t + 4 <= cnt; t += 4) {
              float w[4], vf[4][4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                w[u] = Ps[h * ldp + t + u];
                load_elems<KT, 4>(Vs + ((size_t)(t + u) * HKV + g) * D + d4 * 4, vf[u]);
              }
#pragma unroll
              for (int u = 0; u < 4; u += 2) {
                acc.x = fmaf(w[u], vf[u][0], acc.x);
                acc.y = fmaf(w[u], vf[u][1], acc.y);
                acc.z = fmaf(w[u], vf[u][2], acc.z);
                acc.w = fmaf(w[u], vf[u][3], acc.w);
                acc2.x = fmaf(w[u + 1], vf[u + 1][0], acc2.x);
                acc2.y = fmaf(w[u + 1], vf[u + 1][1], acc2.y);
                acc2.z = fmaf(w[u + 1], vf[u + 1][2], acc2.z);
                acc2.w = fmaf(w[u + 1], vf[u + 1][3], acc2.w);
              }
            }
            #pragma unroll 1
            for (; t < cnt; ++t) {
              const float w = Ps[h * ldp + t];
              float vf[4];
              load_elems<KT, 4>(Vs + ((size_t)t * HKV + g) * D + d4 * 4, vf);
              acc.x = fmaf(w, vf[0], acc.x);
              acc.y = fmaf(w, vf[1], acc.y);
              acc.z = fmaf(w, vf[2], acc.z);
              acc.w = fmaf(w, vf[3], acc.w);
            }
            o[k] = make_float4(acc.x + acc2.x, acc.y + acc2.y, acc.z + acc2.z, acc.w + acc2.w);
          }
        }
        __syncthreads();
        if (first_round) TS_MARK(31);
        first_round = false;
      }
      TS_MARK(11);
      // ---- this CTA's partial of every query head (read back by bulk copy after the barrier)
#pragma unroll
      for (int k = 0; k < NG; ++k) {
        const int qd = tid + k * S::THREADS;
        if (qd < NGRP) {
          const int h = qd / D4, d4 = qd % D4, qq = d4 / (Dq / 4);
          reinterpret_cast<float4*>(ao + ((((size_t)b * H + h) * dq + qq) * nCTA + c) * Dq)[d4 % (Dq / 4)] = o[k];
        }
      }
      if (tid < HQ) aml[((size_t)b * H + tid) * nCTAp + c] = make_float2(sm.att_m[tid], sm.att_l[tid]);
      fence_proxy_async_global();
      __syncthreads();
    }
  }

  TS_MARK(24);
  // ============================================== outputs, after one more barrier
  if (!(a.phases & (kPhSelect | kPhAttend))) return;
  if (!grid_sync(a.gsync, a.status, &sm.gepoch, a.wait_ns, a.skip_cta, a.skip_barrier)) return;
  TS_MARK(25);
  if (a.phases & kPhAttend) {
    // merge the CTA partials of one (sequence, query head, column part) per CTA pass: the item's
    // rows and (max, sum) pairs arrive by bulk copy, then weights, then the weighted rows reduced
    // in a fixed order
    float* po = reinterpret_cast<float*>(dsm);                          // [nCTA][Dq]
    float2* pml = reinterpret_cast<float2*>(po + (size_t)nCTA * Dq);    // [nCTAp]
    float* pw = reinterpret_cast<float*>(pml + nCTAp);                  // [nCTA] weights
    float4* racc = reinterpret_cast<float4*>(dsm + (((size_t)nCTA * Dq * 4 + (size_t)nCTAp * 8 + (size_t)nCTA * 4 + 15) &
                                                     ~(size_t)15));     // [ngrp][Dq/4]
    const int ncol = Dq / 4;
    const int ngrp = min((int)blockDim.x / ncol, 16);
    const int col = tid % ncol, grp = tid / ncol;
    #pragma unroll 1
    for (int item = c; item < B * H * dq; item += nCTA) {
      const int bh = item / dq, qq = item % dq, b = bh / H, h = bh % H;
      if (!bulk_fetch(po, ao + ((size_t)bh * dq + qq) * nCTA * Dq, (uint32_t)(nCTA * Dq * 4), pml,
                      aml + (size_t)bh * nCTAp, (uint32_t)(nCTAp * 8))) {
        if (tid == 0) atomicExch(&a.gsync->abort, 1u);
        return;
      }
      TS_MARK(54);
      float M = -INFINITY;
      #pragma unroll 1
      for (int cc = lane; cc < nCTA; cc += 32) M = fmaxf(M, pml[cc].x);
      M = warp_max(M);                                       // every warp computes the same M
      #pragma unroll 1
      for (int cc = tid; cc < nCTA; cc += blockDim.x)
        pw[cc] = (M > -INFINITY && pml[cc].x > -INFINITY) ? expf(pml[cc].x - M) : 0.f;
      __syncthreads();
      if (warp == 0) {
        float den = 0.f;
        #pragma unroll 1
        for (int cc = lane; cc < nCTA; cc += 32) den = fmaf(pw[cc], pml[cc].y, den);
        den = warp_sum(den);
        if (lane == 0) sm.red_f[0][0] = den;
      }
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (grp < ngrp) {
        #pragma unroll 1
        for (int cc = grp; cc < nCTA; cc += ngrp) {
          const float w = pw[cc];
          if (w != 0.f) {
            const float4 v = reinterpret_cast<const float4*>(po + (size_t)cc * Dq)[col];
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
          }
        }
        racc[grp * ncol + col] = acc;
      }
      __syncthreads();
      const float den = sm.red_f[0][0];
      if (tid < ncol) {
        float4 s4 = racc[tid];
        #pragma unroll 1
        for (int g = 1; g < ngrp; ++g) {
          const float4 v = racc[g * ncol + tid];
          s4.x += v.x;
          s4.y += v.y;
          s4.z += v.z;
          s4.w += v.w;
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
        float* o = a.out + ((size_t)b * H + h) * D + qq * Dq + 4 * tid;   // the caller's buffer: 4-byte aligned only
        o[0] = s4.x * inv;
        o[1] = s4.y * inv;
        o[2] = s4.z * inv;
        o[3] = s4.w * inv;
      }
      if (a.lse && tid == 0 && qq == 0) a.lse[(size_t)b * H + h] = den > 0.f ? M + logf(den) : -INFINITY;
      __syncthreads();
    }
  }
  TS_MARK(26);
  if (a.phases & kPhSelect) {
    // counts of the CTAs before mine and of all CTAs, every sequence at once (warp per sequence)
    #pragma unroll 1
    for (int b = warp; b < B; b += S::NW) {
      const SeqState& st = sm.seq[b];
      int pc = 0, pa = 0, tc = 0, ta = 0;
      if (!st.hit)
        #pragma unroll 8
        for (int cc = st.first_cta + lane; cc <= st.last_cta; cc += 32) {
          const int xc = __ldcg(&a.cta_cnt[((size_t)b * nCTA + cc) * 4 + 0]);
          const int xa = __ldcg(&a.cta_cnt[((size_t)b * nCTA + cc) * 4 + 1]);
          if (cc < c) {
            pc += xc;
            pa += xa;
          }
          tc += xc;
          ta += xa;
        }
      pc = warp_sum_i(pc);
      pa = warp_sum_i(pa);
      tc = warp_sum_i(tc);
      ta = warp_sum_i(ta);
      if (lane == 0) {
        sm.pre_c[b] = pc;
        sm.pre_a[b] = pa;
        sm.tot_c[b] = tc;
        sm.tot_a[b] = ta;
      }
    }
    __syncthreads();
    TS_MARK(55);
    // ascending index lists and Selection Cache entries
    #pragma unroll 1
    for (int b = 0; b < B; ++b) {
      const SeqState& st = sm.seq[b];
      int32_t* ib = a.idx + (size_t)b * a.idx_stride;
      if (st.hit) {
        const int32_t* ctb = a.ct ? a.ct + (size_t)b * a.cap : nullptr;
        const int lo = sm.ct_lo[b];
        const int mcount = sm.ct_hi[b] - lo;
        const int total = st.s_end + mcount + (st.n - st.ls);
        if (total > a.idx_stride) {
          if (c == 0 && tid == 0) {
            set_error(a.status, TS_ERR_CAPACITY);
            a.count[b] = 0;
          }
          continue;
        }
        const int per = (total + nCTA - 1) / nCTA;
        #pragma unroll 1
        for (int j = c * per + tid; j < min(total, (c + 1) * per); j += blockDim.x) {
          int v;
          if (j < st.s_end) v = j;
          else if (j < st.s_end + mcount) v = __ldcg(ctb + lo + j - st.s_end);
          else v = st.ls + (j - st.s_end - mcount);
          ib[j] = v;
        }
        if (c == 0 && tid == 0) a.count[b] = total;
        continue;
      }
      const int tot_c = sm.tot_c[b], tot_a = sm.tot_a[b];
      const int pre_c = sm.pre_c[b], pre_a = sm.pre_a[b];
      const int total = st.s_end + tot_c + (st.n - st.ls);
      const bool fits = total <= a.idx_stride;
      const bool cfits = a.ct != nullptr && tot_a <= a.cap;
      if (c == 0 && tid == 0) {
        if (!fits) set_error(a.status, TS_ERR_CAPACITY);
        a.count[b] = fits ? total : 0;
        if (a.ct) {
          if (!cfits) set_error(a.status, TS_ERR_CAPACITY);
          a.ct_count[b] = cfits ? tot_a : 0;
          a.filled[b] = cfits ? 1 : 0;
        }
      }
      {
        // sinks and window, and the new C_Q, spread over every CTA (grid-stride)
        const int gs = nCTA * blockDim.x, gi = c * blockDim.x + tid;
        if (fits) {
          #pragma unroll 1
          for (int j = gi; j < st.s_end; j += gs) ib[j] = j;
          #pragma unroll 1
          for (int j = gi; j < st.n - st.ls; j += gs) ib[st.s_end + tot_c + j] = st.ls + j;
        }
        if (a.cq) {
          const float* qb = a.q + (size_t)b * H * D;
          float* cqb = a.cq + (size_t)b * H * D;
          #pragma unroll 1
          for (int j = gi; j < H * D; j += gs) cqb[j] = qb[j];
        }
      }
      const int sgi = sm.my_seg_of[b];
      if (sgi < 0) continue;
      // my selected tokens from the ascending list: all of them into C_T, those in [s_end, ls)
      // into the index list after the sinks
      const int* lst = sel_list + sm.seg_t0[sgi];
      const int na = sm.sel_a[sgi], nlo = sm.sel_lo[sgi], nc = sm.sel_c[sgi];
      int32_t* ctb = cfits ? a.ct + (size_t)b * a.cap : nullptr;
      #pragma unroll 1
      for (int j = tid; j < na; j += blockDim.x) {
        const int t = lst[j];
        if (ctb) ctb[pre_a + j] = t;
        if (fits && j >= nlo && j < nlo + nc) ib[st.s_end + pre_c + (j - nlo)] = t;
      }
    }
  }
  TS_MARK(27);
}

template <typename KT, int D, int HKV, int G>
__global__ void __launch_bounds__(StepShape<KT, D, HKV, G>::THREADS, 1) step_kernel(const __grid_constant__ StepKArgs a) {
  // diagnosis: the latest CTA start (slot 17) and the latest CTA end (slot 18) of the launch
  if (threadIdx.x == 0 && a.phase_ns) atomicMax(&a.phase_ns[17], globaltimer_ns());
  step_body<KT, D, HKV, G>(a);
  if (threadIdx.x == 0 && a.phase_ns) atomicMax(&a.phase_ns[18], globaltimer_ns());
  // Every CTA leaves through here, whichever way the body ended; thread 0 is the only one that
  // touches the barrier words, so once every CTA's thread 0 has counted itself out the last one
  // zeroes them for the next launch (no memset between launches).
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&a.gsync->exits, 1u) + 1u == gridDim.x) {
      a.gsync->count = 0u;
      a.gsync->abort = 0u;
      a.gsync->claim = 0u;
      a.gsync->exits = 0u;
      __threadfence();
    }
  }
}

// ------------------------------------------------------------------- launch

// Tensor map of a bf16 K pool seen as [num_pages * rows][d], rows = H_kv x 16 (one page of every
// KV head): boxes of 64 elements x `rows` rows (one page), 128-byte swizzle. The encoder comes from the driver through the runtime, so the
// library needs no link against the driver library. False when it cannot be encoded.
bool encode_kmap(CUtensorMap* map, const void* k_pool, int64_t num_pages, int d, int rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static bool looked = false;
  if (!looked) {
    looked = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if (!encode || (reinterpret_cast<uintptr_t>(k_pool) & 15) != 0 || num_pages <= 0 ||
      num_pages * rows > (int64_t)0x7fffffff)
    return false;
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)num_pages * rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)rows};
  const cuuint32_t estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(k_pool), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename KT, int D, int HKV, int G>
ts_status run_step(ts_ctx* ctx, const StepCall& c, cudaStream_t s) {
  using S = StepShape<KT, D, HKV, G>;
  auto kern = step_kernel<KT, D, HKV, G>;
  static int static_bytes = -1;   // per instantiation: the kernel's static shared memory
  if (static_bytes < 0) {
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return TS_ERR_CUDA;
    static_bytes = (int)fa.sharedSizeBytes;
  }
  static int smem_avail = -1;      // shared memory one CTA of the SM may use in all
  if (smem_avail < 0) {
    int optin = 0, per_sm = 0, reserved = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, ctx->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, ctx->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, ctx->device) != cudaSuccess)
      return TS_ERR_CUDA;
    smem_avail = min(min(optin, per_sm - reserved), kSmemLimit);
    if (ctx->debug)
      std::fprintf(stderr, "ts step: smem optin %d, per SM %d, reserved/block %d\n", optin, per_sm, reserved);
    // the whole unified L1/shared array as shared memory for this kernel
    if (cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
      return TS_ERR_CUDA;
  }
  const int dyn = (smem_avail - static_bytes - 1024) / 128 * 128;
  const int flag_cap = kStepFlagCap;   // one byte per token of a CTA's range
  // ring slots of one stage of K each; the selection scratch and one
  // sequence's global histograms (with masses) alias the same space later
  const int nslot = std::min(kMaxSlots, (dyn - flag_cap) / S::STAGE_BYTES);
  // (the vote pass keeps (max, 1/sum) per segment and head, one segment's CTA partials and
  // per-warp reductions; the merge one (sequence, head)'s CTA rows)
  if (nslot < S::MIN_SLOTS || dyn - flag_cap < lvl_bins(0) * 12 || dyn - flag_cap < kCandCap * 8 ||
      dyn - flag_cap < kMaxB * 128 * 12 ||
      dyn - flag_cap < kMaxB * kMaxWaveHeads * 8 + ctx->num_sms * S::PV * ctx->cfg.n_q_heads * 8 + 2 * 16 * 32 * 4 + 16 +
                           kVoteBufs * 16 * kMaxWaveHeads * 4 ||   // vote scratch, then the chunks of 16 logit rows
      dyn < ctx->num_sms * (D * 4 + 8 + 4) + 8 + 16 + S::THREADS * 16)   // the merge's rows, pairs, weights
    return TS_ERR_UNSUPPORTED;
  if (!ensure_smem<step_kernel<KT, D, HKV, G>>((size_t)dyn, ctx->device)) {
    if (ctx->debug) std::fprintf(stderr, "ts step: smem attribute %d B refused\n", dyn);
    return TS_ERR_CUDA;
  }
  const bool debug = ctx->debug;
  if (ctx->step_grid <= 0) {
    int per_sm = 0;
    const cudaError_t oe = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, S::THREADS, (size_t)dyn);
    if (debug)
      std::fprintf(stderr, "ts step: static %d B, dynamic %d B, threads %d, ring slots %d, blocks/SM %d (%s)\n",
                   static_bytes, dyn, S::THREADS, nslot, per_sm, cudaGetErrorString(oe));
    if (oe != cudaSuccess || per_sm < 1) return TS_ERR_COOP_UNAVAILABLE;
    ctx->step_grid = ctx->num_sms;
  }
  if (ctx->step_grid > kMaxGrid) return TS_ERR_UNSUPPORTED;
  const ts_config& cfg = ctx->cfg;
  StepKArgs a{};
  a.phases = c.phases;
  a.B = c.B;
  a.H = cfg.n_q_heads;
  a.max_tokens = ctx->max_tokens;
  a.pt_stride = cfg.max_pages_per_seq;
  a.num_pages = cfg.num_pages;
  a.q = c.q;
  a.k_pool = static_cast<const unsigned char*>(c.k_pool);
  a.v_pool = static_cast<const unsigned char*>(c.v_pool);
  a.page_table = c.page_table;
  a.seq_lens = c.seq_lens;
  a.scale = c.scale;
  {
    const double sl2 = (double)c.scale * 1.4426950408889634;
    a.scale_l2 = (float)sl2;
    a.scale_l2_lo = (float)(sl2 - (double)a.scale_l2);
  }
  a.theta = c.theta;
  a.hit_in = c.hit_in;
  a.hit_out = c.hit_out;
  if (c.cache) {
    const size_t mb = (size_t)cfg.max_batch, HD = (size_t)cfg.n_q_heads * cfg.head_dim;
    a.cq = c.cache->cq + (size_t)c.layer * mb * HD;
    a.ct = c.cache->ct + (size_t)c.layer * mb * c.cache->capacity;
    a.ct_count = c.cache->ct_count + (size_t)c.layer * mb;
    a.filled = c.cache->filled + (size_t)c.layer * mb;
    a.cap = c.cache->capacity;
  }
  a.mode = c.params.mode;
  a.k = c.params.k;
  a.n_sink = c.params.n_sink;
  a.n_local = c.params.n_local;
  const double target = (double)c.params.top_p * (double)cfg.n_q_heads * 1099511627776.0;
  a.target_fx = (unsigned long long)ceil(target);
  if (a.target_fx == 0ull) a.target_fx = 1ull;
  a.take_all_topp = c.params.top_p >= 1.0f;
  a.vote = c.vote;
  a.vote_stride = c.vote_stride;
  a.idx = c.idx;
  a.idx_stride = c.idx_stride;
  a.count = c.count;
  a.out = c.out;
  a.lse = c.lse;
  a.partials = ctx->step_partials;
  a.hist = ctx->step_hist;
  a.mass = ctx->step_mass;
  a.cand_n = ctx->cand_n;
  a.cands = ctx->cands;
  a.cta_cnt = ctx->cta_cnt;
  a.apart = ctx->apart;
  a.spill = ctx->logits;
  a.spill_floats = ctx->logits_floats;
  a.wpart = reinterpret_cast<float2*>(ctx->step_wpart);
  a.l2_budget = ctx->l2_budget > 0 ? ctx->l2_budget : kLogitL2Budget;
  a.gsync = reinterpret_cast<GridSync*>(ctx->gsync);
  a.status = ctx->status;
  a.wait_ns = ctx->wait_ns;
  a.skip_cta = ctx->inject_skip_cta;       // an injected fault applies to this launch only
  a.skip_barrier = ctx->inject_skip_barrier;
  ctx->inject_skip_cta = ctx->inject_skip_barrier = -1;
  a.phase_ns = ctx->phase_ns;
  a.dyn_bytes = dyn;
  a.nslot = nslot;
  a.tc = 0;
  a.nslot_tc = 0;
  a.scan_dyn = 0;
  a.tcv = 0;
  if constexpr (S::TC) {
    // tensor-core scan: 1024-aligned ring of page tiles plus two query-term images
    const int nslot_tc = std::min(kMaxSlots, (dyn - flag_cap - 1024 - 2 * S::TC_BIMG) / S::TC_TILE);
    // the tensor map of a pool, from a cache of recent ones (one per layer and pool in a decode
    // loop), or null when it cannot be encoded
    auto pool_map = [&](const void* pool) -> const void* {
      auto& cache = ctx->kmaps;
      constexpr int n = (int)(sizeof(cache) / sizeof(cache[0]));
      int hitc = -1;
      for (int i = 0; i < n; ++i)
        if (cache[i].pool == pool && cache[i].num_pages == cfg.num_pages) hitc = i;
      if (hitc < 0) {
        hitc = ctx->kmap_next;
        ctx->kmap_next = (ctx->kmap_next + 1) % n;
        cache[hitc].pool = nullptr;
        if (encode_kmap(reinterpret_cast<CUtensorMap*>(cache[hitc].map), pool, cfg.num_pages, D, S::TC_ROWS)) {
          cache[hitc].pool = pool;
          cache[hitc].num_pages = cfg.num_pages;
        }
      }
      return cache[hitc].pool == pool ? cache[hitc].map : nullptr;
    };
    if (!ctx->no_tc && nslot_tc >= 2 && (c.phases & kPhScore) && c.k_pool && (reinterpret_cast<uintptr_t>(c.q) & 15) == 0) {
      if (const void* m = pool_map(c.k_pool)) {
        std::memcpy(&a.tmap_k, m, sizeof(CUtensorMap));
        a.tc = 1;
        a.nslot_tc = nslot_tc;
        // CTAs may claim pages of one or two scanned sequences from a shared counter instead of
        // each scanning its own range (TOKENSELECT_SCAN_CLAIM=1 at context creation). Faster where
        // bandwidth differs between SMs, but which CTA sums which pages then varies, so repeated
        // runs may differ in the last bits.
        a.scan_dyn = (ctx->scan_claim && S::TC_PAGES == 1) ? 1 : 0;   // tiles of one page only
      }
    }
    // the V map for the tensor-core range attention of top-p (d = 128, enough staging memory; on
    // request only: eight MMAs of N = 16 per page measured slower than P.V on the CUDA cores)
    if (D == 128 && a.tc && c.params.mode == TS_SELECT_TOPP && ctx->range_tc && c.v_pool &&
        dyn - flag_cap - 2 * kOwnBatch * (int)sizeof(int) >= kStageMin) {
      if (const void* m = pool_map(c.v_pool)) {
        std::memcpy(&a.tmap_v, m, sizeof(CUtensorMap));
        a.tcv = 1;
      }
    }
  }
  a.flag_cap = flag_cap;
  a.sel_rows = ctx->sel_rows;
  a.range_attend = ctx->range_attend;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(ctx->step_grid);
  lc.blockDim = dim3(S::THREADS);
  lc.dynamicSmemBytes = (size_t)dyn;
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  ctx->kernels += 1;
  ProfScope ps(ctx, TS_PROF_STEP, s);
  const cudaError_t e = cudaLaunchKernelEx(&lc, kern, a);
  if (debug && e != cudaSuccess) std::fprintf(stderr, "ts step launch: %s\n", cudaGetErrorString(e));
  if (e == cudaErrorCooperativeLaunchTooLarge) return TS_ERR_COOP_UNAVAILABLE;
  return cuda_status(e);
}

}  // namespace

bool step_supported(const ts_config& c) {
  const int G = c.n_kv_heads > 0 ? c.n_q_heads / c.n_kv_heads : 0;
#define X(DT, T, D_, HKV_, G_) \
  if (c.kv_dtype == DT && c.head_dim == D_ && c.n_kv_heads == HKV_ && G == G_) return true;
  TS_STEP_GEOMETRIES(X)
#undef X
  return false;
}

ts_status launch_step(ts_ctx* ctx, const StepCall& a, cudaStream_t s) {
  const ts_config& c = ctx->cfg;
  const int G = c.n_q_heads / c.n_kv_heads;
  if (a.B > kMaxB) return TS_ERR_UNSUPPORTED;
#define X(DT, T, D_, HKV_, G_) \
  if (c.kv_dtype == DT && c.head_dim == D_ && c.n_kv_heads == HKV_ && G == G_) return run_step<T, D_, HKV_, G_>(ctx, a, s);
  TS_STEP_GEOMETRIES(X)
#undef X
  return TS_ERR_UNSUPPORTED;
}

}  // namespace ts
