// One persistent, cooperative kernel for a whole decode step (or any of its
// parts): Selection Cache test, paged score + head soft vote, top-k / top-p
// selection united with sinks and window, and sparse attention.
//
// The method is TokenSelect's (deep notes: Appendix Algorithm 1 and 2, "Head
// soft vote", "Formalising selective sparse attention"; review: section 4.2).
// The GB300 mapping:
//  * one CTA per SM: one producer warp streams the KV pages of a contiguous
//    range of the concatenated (missing) sequences into a shared-memory ring
//    with 1-D bulk copies (TMA); up to 16 consumer warps hold the G queries of
//    a KV head in registers and read every K element once;
//  * each head's logits stay in shared memory as exp(l - m_cta); per-CTA
//    (max, sum) partials cross CTAs through a grid barrier, after which every
//    CTA forms its tokens' votes with one FMA per (token, head). When the
//    logits of all heads do not fit, the heads are scanned in waves (one
//    barrier per wave) and the votes accumulate in global memory;
//  * selection: radix histograms of the vote bit pattern, aggregated in
//    shared memory and added with integer atomics (order-free, hence
//    deterministic); as soon as the crossing bin holds at most 2048 tokens
//    they are gathered and each CTA ranks its own candidates exactly (ties
//    go to the lower index; top-p mass in 2^-40 fixed point);
//  * attention: every CTA attends its own selected tokens plus a round-robin
//    share of the sinks, window and cached indices, gathering K/V rows by
//    bulk copy; per-CTA (max, sum, o) partials are merged after one barrier.
// Grid barriers and mbarrier waits are bounded by %globaltimer; on time-out
// the kernel records TS_ERR_TIMEOUT and returns.
#include <cfloat>
#include <cmath>
#include <cstdio>
#include <cstdlib>

#include "ts_common.cuh"

namespace ts {
namespace {

constexpr int kMaxB = 64;          // sequences per call (= most segments one CTA can touch)
constexpr int kCandCap = 2048;     // candidates gathered per sequence
constexpr int kBins = 2048;
constexpr int kMaxRound = 128;     // attention tokens per gather round
constexpr int kMaxWaveHeads = 32;  // query heads of one scan wave
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
  static constexpr int NST = STAGE_BYTES <= 8192 ? 6 : (STAGE_BYTES <= 16384 ? 4 : (STAGE_BYTES <= 32768 ? 3 : 2));
  static constexpr int RING_BYTES = NST * STAGE_BYTES;
  // attention: a lane reads ACB bytes of a row; ALPT lanes per row
  // (8-byte lane chunks keep the per-lane softmax state small: 17 warps leave 96 registers)
  static constexpr int ACB = (D * (int)sizeof(KT) / 8 <= 32) ? 8 : 16;
  static constexpr int ALPT = D * (int)sizeof(KT) / ACB;
  static constexpr int AEPC = ACB / (int)sizeof(KT);
  static constexpr int ATPW = 32 / ALPT;                  // tokens per warp step
  static constexpr int TOKEN_BYTES = 2 * HKV * ROW_BYTES; // K and V rows of every KV head
  static_assert(D % DPL == 0 && 32 % LPR == 0 && GP <= LPR, "scan lane split");
  static_assert(NCW >= 1 && (P * HKV) % NCW == 0 && ROWS % RPW == 0 && ITERS >= 1, "scan warp split");
  static_assert(NCW % HKV == 0 && P % ROWS == 0 || ROWS % P == 0, "rows of a warp stay in one page");
  static_assert(32 % ALPT == 0 && GP <= ALPT, "attention lane split");
  static_assert(RING_BYTES >= kBins * 12 + kCandCap * 8, "histograms and candidates alias the ring");
  static_assert(G <= kMaxWaveHeads, "heads per KV head");
};

struct GridSync {
  unsigned count, gen, abort, pad;
};

struct StepKArgs {
  int phases;
  int B, H, max_tokens, pt_stride;
  int64_t num_pages;
  const float* q;
  const unsigned char* k_pool;
  const unsigned char* v_pool;
  const int32_t* page_table;
  const int32_t* seq_lens;
  float scale;
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
  unsigned* hist;              // [3][B][kBins]
  unsigned long long* mass;    // [3][B][kBins]
  unsigned* cand_n;            // [B]
  unsigned long long* cands;   // [B][kCandCap]  (key << 32 | ~index)
  int* cta_cnt;                // [B][nCTA][3]  cand-range selected, all selected, ties
  float* apart;                // [B][nCTA][H][D + 2]
  float* spill;                // e-values past the shared-memory capacity
  int64_t spill_floats;
  GridSync* gsync;
  int* status;
  int dyn_bytes;               // dynamic shared memory of the launch
  int e_cap;                   // floats of the shared e-buffer
  int flag_cap;                // bytes reserved at the tail for selection flags
};

// -------------------------------------------------------------- grid barrier

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// All CTAs of the cooperative grid meet here. False after a time-out or an
// abort raised by another CTA; the caller then returns.
__device__ bool grid_sync(GridSync* gs, int* status) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const unsigned gen0 = ld_acquire(&gs->gen);
    __threadfence();
    const unsigned arrived = atomicAdd(&gs->count, 1u) + 1u;
    if (arrived == gridDim.x) {
      atomicExch(&gs->count, 0u);
      __threadfence();
      st_release(&gs->gen, gen0 + 1u);
    } else {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire(&gs->gen) == gen0) {
        if (ld_acquire(&gs->abort)) {
          ok = 0;
          break;
        }
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          set_error(status, TS_ERR_TIMEOUT);
          atomicExch(&gs->abort, 1u);
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// Block-wide exclusive scan of one int per thread; total in *total.
__device__ __forceinline__ int block_scan(int x, int* wsum, int& total) {
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

// First index in the ascending list a[0, n) that is >= x.
__device__ __forceinline__ int lower_bound_i(const int32_t* a, int n, int x) {
  int l = 0, r = n;
  while (l < r) {
    const int m = (l + r) >> 1;
    if (a[m] < x) l = m + 1; else r = m;
  }
  return l;
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
  int pg0, pg1;                    // its pages in the concatenated scan space
};

struct Smem {
  SeqState seq[kMaxB];
  int nseg;
  int seg_b[kMaxB], seg_lp0[kMaxB], seg_t0[kMaxB], seg_ntok[kMaxB], seg_pend[kMaxB];
  int p0, p1, ppc, tok_stride, hpw, nwaves, tok_smem, spill_ok, ptot;
  int stage_tok[8][16];    // per ring stage: CTA-local first token of each page (-1: unused)
  int stage_nv[8][16];     // valid slots of each page
  int stage_b[8][16];      // its sequence
  int stage_done[8];       // warps finished with the current use of each ring slot
  int slot_last[8];        // the last ring use issued into each slot (-1: none)
  int timed_out;
  int wsum[33];
  int flag;
  float red_f[3][32];
  int toks[kMaxRound];
  int tval[kMaxRound];
  int my_seg_of[kMaxB];    // segment of sequence b in this CTA, or -1
};

// --------------------------------------------------------------- the kernel

template <typename KT, int D, int HKV, int G>
__global__ void __launch_bounds__(StepShape<KT, D, HKV, G>::THREADS, 1) step_kernel(StepKArgs a) {
  using S = StepShape<KT, D, HKV, G>;
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ Smem sm;
  __shared__ __align__(8) uint64_t full[S::NST];
  __shared__ __align__(8) uint64_t abar;

  unsigned char* ring = dsm;
  float* ebuf = reinterpret_cast<float*>(dsm + S::RING_BYTES);
  uint8_t* selflag = dsm + a.dyn_bytes - a.flag_cap;       // selection flags of my tokens
  float* wts = reinterpret_cast<float*>(selflag);          // vote weights [segment][wave head] while scoring

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, nCTA = gridDim.x;
  const int B = a.B, H = a.H;

  if (tid == 0) {
    for (int s = 0; s < S::NST; ++s) {
      mbar_init(&full[s], 1);
      sm.stage_done[s] = 0;
      sm.slot_last[s] = -1;
    }
    sm.timed_out = 0;
    mbar_init(&abar, 1);
    mbar_fence_init();
  }

  // ------------------------------------------------ setup: lengths, cache test, partition
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
  }
  __syncthreads();
  if (a.phases & kPhCheck) {
    // Algorithm 1: hit iff the entry is filled and cos(q, C_Q) >= theta
    const int HD = H * D;
    for (int b = 0; b < B; ++b) {
      if (!a.filled[b]) continue;
      const float* x = a.q + (size_t)b * HD;
      const float* y = a.cq + (size_t)b * HD;
      float xy = 0.f, xx = 0.f, yy = 0.f;
      for (int i = tid; i < HD; i += blockDim.x) {
        const float u = x[i], v = __ldcg(y + i);
        xy = fmaf(u, v, xy);
        xx = fmaf(u, u, xx);
        yy = fmaf(v, v, yy);
      }
      xy = warp_sum(xy);
      xx = warp_sum(xx);
      yy = warp_sum(yy);
      if (lane == 0) {
        sm.red_f[0][warp] = xy;
        sm.red_f[1][warp] = xx;
        sm.red_f[2][warp] = yy;
      }
      __syncthreads();
      if (tid == 0) {
        double sxy = 0, sxx = 0, syy = 0;
        for (int w = 0; w < S::NW; ++w) {
          sxy += sm.red_f[0][w];
          sxx += sm.red_f[1][w];
          syy += sm.red_f[2][w];
        }
        const double den = sqrt(sxx) * sqrt(syy);
        const float cs = den > 0.0 ? (float)(sxy / den) : __int_as_float(0x7fc00000);
        sm.seq[b].hit = (cs >= a.theta) ? 1 : 0;
      }
      __syncthreads();
    }
  }
  if (tid == 0) {
    int pg = 0;
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
    // scan waves: the largest power-of-two divisor hpw of H_kv whose e-values fit
    int hpw = HKV;
    while (hpw > 1 && ((int64_t)hpw * G * sm.tok_stride > a.e_cap || hpw * G > kMaxWaveHeads)) hpw >>= 1;
    sm.hpw = hpw;
    sm.nwaves = HKV / hpw;
    sm.tok_smem = min(sm.tok_stride, a.e_cap / (hpw * G));
    sm.spill_ok = (int64_t)nCTA * hpw * G * (sm.tok_stride - sm.tok_smem) <= a.spill_floats &&
                  sm.tok_stride <= a.flag_cap;
    sm.flag = 0;
  }
  __syncthreads();
  if (!sm.spill_ok) {
    if (c == 0 && tid == 0) set_error(a.status, TS_ERR_SHAPE);
    return;  // uniform across CTAs: same inputs, same decision, before any barrier
  }
  if (c == 0 && tid < B && (a.phases & kPhCheck) && a.hit_out) a.hit_out[tid] = (uint8_t)sm.seq[tid].hit;
  if (a.phases & kPhSelect) {
    // zero the selection histograms (first touched after a barrier)
    const size_t nh = (size_t)3 * B * kBins;
    for (size_t i = (size_t)c * blockDim.x + tid; i < nh; i += (size_t)nCTA * blockDim.x) {
      a.hist[i] = 0u;
      if (a.mode == TS_SELECT_TOPP) a.mass[i] = 0ull;
    }
    if (c == 0 && tid < B) a.cand_n[tid] = 0u;
  }

  const int tstride = sm.tok_stride;
  const int tsm = sm.tok_smem;
  auto eaddr = [&](int hl, int t) -> float* {
    return t < tsm ? ebuf + (size_t)hl * tsm + t
                   : a.spill + ((size_t)c * (sm.hpw * G) + hl) * (size_t)(tstride - tsm) + (t - tsm);
  };

  // ========================================================================= SCORE
  if ((a.phases & kPhScore) && sm.ptot > 0) {   // nothing to scan when every sequence hits
    const int hpw = sm.hpw, HW = hpw * G, nwaves = sm.nwaves;
    const int pps = HKV / hpw;                       // pages per stage
    const int np = sm.p1 - sm.p0;
    const int nstages = (np + pps - 1) / pps;
    const int slab = hpw * S::P * S::ROW_BYTES;      // bytes of one page's heads of the wave
    int stage_seq = 0;                               // ring use counter across waves
    // Issues ring use u = stage_seq + si (the pps pages si*pps.. of my range, the wave's
    // heads of each) into slot u % NST: metadata first, then arrive.expect_tx, then the copies.
    auto issue = [&](int u, int si, int g0) {
      const int s = u % S::NST;
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
        const int page = a.page_table[(size_t)b * a.pt_stride + lp];
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
        bulk_g2s(ring + (size_t)s * S::STAGE_BYTES + (size_t)j * slab,
                 a.k_pool + ((size_t)pages[j] * HKV + g0) * S::P * S::ROW_BYTES, (uint32_t)slab, &full[s]);
      }
    };
    for (int wv = 0; wv < nwaves; ++wv) {
      const int g0 = wv * hpw;
      // the ring is idle between waves: fill it
      if (tid == 0)
        for (int si = 0; si < min(S::NST, nstages); ++si) issue(stage_seq + si, si, g0);
      __syncthreads();
      {
        // ---- warp -> KV head g0 + gi, ROWS rows of that head in each stage
        const int wph = S::NCW / hpw;
        const int gi = warp / wph;
        const int row0 = (warp % wph) * S::ROWS;     // rows of one page: ROWS divides P or P divides ROWS
        const int lrow = lane / S::LPR, lin = lane % S::LPR;
        float qr[S::GP][S::DPL];
#pragma unroll
        for (int j = 0; j < S::GP; ++j)
#pragma unroll
          for (int e = 0; e < S::DPL; ++e) qr[j][e] = 0.f;
        int qb = -1;                                 // sequence whose queries sit in qr
        const bool writer = (lin & (S::LPR / S::GP - 1)) == 0;
        for (int si = 0; si < nstages; ++si) {
          const int u = stage_seq + si;
          const int s = u % S::NST;
          if (!mbar_wait(&full[s], (u / S::NST) & 1)) {
            set_error(a.status, TS_ERR_TIMEOUT);
            sm.timed_out = 1;
            break;
          }
          const KT* st = reinterpret_cast<const KT*>(ring + (size_t)s * S::STAGE_BYTES);
#pragma unroll
          for (int it = 0; it < S::ITERS; ++it) {
            const int r = row0 + it * S::RPW + lrow;   // row among this head's pps*16 rows
            const int j = r / S::P, slot = r % S::P;   // all lanes of a step share the page j
            const int tloc = sm.stage_tok[s][j];
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
            if (writer && which < G && tloc >= 0)
              *eaddr(gi * G + which, tloc + slot) = slot < nv ? dot * a.scale : -INFINITY;
          }
          __syncwarp();
          if (lane == 0) {
            // the last warp done with this use of the slot refills it with use u + NST
            if (atomicAdd(&sm.stage_done[s], 1) == S::NCW - 1) {
              sm.stage_done[s] = 0;
              if (si + S::NST < nstages) issue(u + S::NST, si + S::NST, g0);
            }
          }
        }
      }
      stage_seq += nstages;
      __syncthreads();
      if (sm.timed_out && tid == 0) {
        // copies issued but never consumed must land before the ring is reused
        for (int ss = 0; ss < S::NST; ++ss)
          if (sm.slot_last[ss] >= 0) mbar_wait(&full[ss], (sm.slot_last[ss] / S::NST) & 1);
      }
      __syncthreads();

      // ---- per (segment, wave head): max, exp in place, compensated sum -> partials
      for (int item = warp; item < sm.nseg * HW; item += S::NW) {
        const int sg = item / HW, hl = item % HW;
        const int t0 = sm.seg_t0[sg], nt = sm.seg_ntok[sg];
        float m = -INFINITY;
        for (int t = lane; t < nt; t += 32) m = fmaxf(m, *eaddr(hl, t0 + t));
        m = warp_max(m);
        KahanF z;
        for (int t = lane; t < nt; t += 32) {
          float* p = eaddr(hl, t0 + t);
          const float e = (m > -INFINITY) ? expf(*p - m) : 0.f;
          *p = e;
          z.add(e);
        }
        const double zs = warp_sum_f64((double)z.s - (double)z.c);
        if (lane == 0) a.partials[((size_t)sm.seg_b[sg] * nCTA + c) * H + g0 * G + hl] = make_float2(m, (float)zs);
      }
      if (!grid_sync(a.gsync, a.status)) return;

      // ---- each head's normaliser over the CTAs of the sequence, then my votes
      for (int item = warp; item < sm.nseg * HW; item += S::NW) {
        const int sg = item / HW, hl = item % HW;
        const SeqState& st = sm.seq[sm.seg_b[sg]];
        const float2* pp = a.partials + (size_t)sm.seg_b[sg] * nCTA * H + g0 * G + hl;
        float M = -INFINITY;
        for (int cc = st.first_cta + lane; cc <= st.last_cta; cc += 32) M = fmaxf(M, __ldcg(pp + (size_t)cc * H).x);
        M = warp_max(M);
        KahanF kz;
        for (int cc = st.first_cta + lane; cc <= st.last_cta; cc += 32) {
          const float2 mz = __ldcg(pp + (size_t)cc * H);
          if (mz.y > 0.f) kz.add(mz.y * expf(mz.x - M));
        }
        const double z = warp_sum_f64((double)kz.s - (double)kz.c);
        if (lane == 0) {
          const float mine = __ldcg(pp + (size_t)c * H).x;
          wts[sg * kMaxWaveHeads + hl] = (mine > -INFINITY && z > 0.0) ? (float)((double)expf(mine - M) / z) : 0.f;
        }
      }
      __syncthreads();
      for (int sg = 0; sg < sm.nseg; ++sg) {
        const int b = sm.seg_b[sg], t0 = sm.seg_t0[sg], nt = sm.seg_ntok[sg];
        float* vb = a.vote + (size_t)b * a.vote_stride + (size_t)sm.seg_lp0[sg] * S::P;
        for (int t = tid; t < nt; t += blockDim.x) {
          KahanF acc;
          for (int hl = 0; hl < HW; ++hl) acc.add(*eaddr(hl, t0 + t) * wts[sg * kMaxWaveHeads + hl]);
          const float v = acc.s - acc.c;
          vb[t] = (wv == 0) ? v : vb[t] + v;
        }
      }
      __syncthreads();
    }
  }

  // ======================================================================== SELECT
  if (a.phases & kPhSelect) {
    if (!(a.phases & kPhScore) && sm.ptot > 0) {
      if (!grid_sync(a.gsync, a.status)) return;   // the histograms are zero everywhere
    }
    unsigned* sh = reinterpret_cast<unsigned*>(ring);
    unsigned long long* smh = reinterpret_cast<unsigned long long*>(ring + kBins * sizeof(unsigned));
    unsigned long long* scand = reinterpret_cast<unsigned long long*>(ring + kBins * 12);
    if (tid == 0) {
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
    for (int level = 0; level < 3; ++level) {
      if (tid == 0) {
        int any = 0;
        for (int b = 0; b < B; ++b) any |= !sm.seq[b].done;
        sm.flag = any;
      }
      __syncthreads();
      if (!sm.flag) break;                     // identical in every CTA
      const int shift = level == 0 ? 21 : (level == 1 ? 10 : 0);
      const int nbins = level == 2 ? 1024 : kBins;
      unsigned* gh = a.hist + (size_t)level * B * kBins;
      unsigned long long* gm = a.mass + (size_t)level * B * kBins;
      for (int sg = 0; sg < sm.nseg; ++sg) {
        const int b = sm.seg_b[sg];
        const SeqState& st = sm.seq[b];
        if (st.done) continue;
        for (int i = tid; i < nbins; i += blockDim.x) {
          sh[i] = 0u;
          if (a.mode == TS_SELECT_TOPP) smh[i] = 0ull;
        }
        __syncthreads();
        const int tl0 = sm.seg_lp0[sg] * S::P;
        const int lo = max(st.lo, tl0), hi = min(st.hi, tl0 + sm.seg_ntok[sg]);
        const float* vb = a.vote + (size_t)b * a.vote_stride;
        for (int t = lo + tid; t < hi; t += blockDim.x) {
          const float v = __ldcg(vb + t);
          const uint32_t key = __float_as_uint(v);
          if ((key & st.mask) == st.prefix) {
            const int bin = (key >> shift) & (nbins - 1);
            atomicAdd(&sh[bin], 1u);
            if (a.mode == TS_SELECT_TOPP) atomicAdd(&smh[bin], to_fx(v));
          }
        }
        __syncthreads();
        for (int i = tid; i < nbins; i += blockDim.x) {
          if (sh[i]) {
            atomicAdd(&gh[(size_t)b * kBins + i], sh[i]);
            if (a.mode == TS_SELECT_TOPP) atomicAdd(&gm[(size_t)b * kBins + i], smh[i]);
          }
        }
        __syncthreads();
      }
      if (!grid_sync(a.gsync, a.status)) return;
      // every CTA: the crossing bin of every unresolved sequence, one warp each
      for (int b = warp; b < B; b += S::NW) {
        SeqState& st = sm.seq[b];
        if (st.done) continue;
        const int per = nbins / 32;
        unsigned cnt = 0;
        unsigned long long ms = 0;
        for (int j = 0; j < per; ++j) {
          const int bin = nbins - 1 - (lane * per + j);
          cnt += __ldcg(&gh[(size_t)b * kBins + bin]);
          if (a.mode == TS_SELECT_TOPP) ms += __ldcg(&gm[(size_t)b * kBins + bin]);
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
        const bool crosses = (a.mode == TS_SELECT_TOPK) ? (ec < need_c && ic >= need_c) : (em < need_m && im >= need_m);
        const unsigned ballot = __ballot_sync(kFull, crosses);
        if (ballot == 0u) {
          if (lane == 0) {  // top-p whose fixed-point total falls short: the whole domain
            st.all = 1;
            st.done = 1;
          }
        } else if (lane == __ffs(ballot) - 1) {
          unsigned cb = ec;
          unsigned long long mb = em;
          for (int j = 0; j < per; ++j) {
            const int bin = nbins - 1 - (lane * per + j);
            const unsigned hc = __ldcg(&gh[(size_t)b * kBins + bin]);
            const unsigned long long hm = (a.mode == TS_SELECT_TOPP) ? __ldcg(&gm[(size_t)b * kBins + bin]) : 0ull;
            const bool here = (a.mode == TS_SELECT_TOPK) ? (cb + hc >= need_c) : (mb + hm >= need_m);
            if (here) {
              st.prefix |= (uint32_t)bin << shift;
              st.mask |= (uint32_t)(nbins - 1) << shift;
              st.n_gt += (int)cb;
              if (a.mode == TS_SELECT_TOPK)
                st.k_rem = (int)(need_c - cb);
              else
                st.mass_rem = need_m - mb;
              if (hc <= (unsigned)kCandCap) {
                st.cand = 1;
                st.done = 1;
              } else if (level == 2) {
                st.tie_mode = 1;
                st.done = 1;
                if (a.mode == TS_SELECT_TOPK) {
                  st.ties = st.k_rem;
                } else {
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
        }
      }
      __syncthreads();
    }

    // ---- gather the crossing-bin tokens (candidates); per-CTA exact-tie counts
    int need_cand = 0, need_tie = 0;
    for (int b = 0; b < B; ++b) {
      need_cand |= sm.seq[b].cand;
      need_tie |= sm.seq[b].tie_mode;
    }
    for (int sg = 0; sg < sm.nseg; ++sg) {
      const int b = sm.seg_b[sg];
      const SeqState& st = sm.seq[b];
      if (!st.cand && !st.tie_mode) continue;
      const int tl0 = sm.seg_lp0[sg] * S::P;
      const int lo = max(st.lo, tl0), hi = min(st.hi, tl0 + sm.seg_ntok[sg]);
      const float* vb = a.vote + (size_t)b * a.vote_stride;
      int n_eq = 0;
      for (int t0 = lo; t0 < hi; t0 += blockDim.x) {
        const int t = t0 + tid;
        bool is = false;
        uint32_t key = 0;
        if (t < hi) {
          key = __float_as_uint(__ldcg(vb + t));
          is = (key & st.mask) == st.prefix;
        }
        if (st.tie_mode) {
          n_eq += is;
          continue;
        }
        const unsigned bal = __ballot_sync(kFull, is);
        unsigned base = 0;
        if (lane == 0 && bal) base = atomicAdd(&a.cand_n[b], (unsigned)__popc(bal));
        base = __shfl_sync(kFull, base, 0);
        if (is) {
          const unsigned pos = base + __popc(bal & ((1u << lane) - 1u));
          if (pos < (unsigned)kCandCap)
            a.cands[(size_t)b * kCandCap + pos] = ((unsigned long long)key << 32) | (0xffffffffu - (uint32_t)t);
        }
      }
      if (st.tie_mode) {
        int tot;
        block_scan(n_eq, sm.wsum, tot);
        if (tid == 0) a.cta_cnt[((size_t)b * nCTA + c) * 3 + 2] = tot;
      }
    }
    if (need_cand || need_tie) {
      if (!grid_sync(a.gsync, a.status)) return;
    }

    // ---- the selection flag of each of my tokens, and the counts for output positions
    for (int sg = 0; sg < sm.nseg; ++sg) {
      const int b = sm.seg_b[sg];
      const SeqState& st = sm.seq[b];
      const int tl0 = sm.seg_lp0[sg] * S::P, t0l = sm.seg_t0[sg], nt = sm.seg_ntok[sg];
      const float* vb = a.vote + (size_t)b * a.vote_stride;
      int tie_base = 0;
      if (st.tie_mode)
        for (int cc = st.first_cta; cc < c; ++cc) tie_base += __ldcg(&a.cta_cnt[((size_t)b * nCTA + cc) * 3 + 2]);
      const int m_cand = st.cand ? (int)min(__ldcg(&a.cand_n[b]), (unsigned)kCandCap) : 0;
      for (int j = tid; j < m_cand; j += blockDim.x) scand[j] = __ldcg(&a.cands[(size_t)b * kCandCap + j]);
      __syncthreads();
      int n_sel_cand = 0, n_sel_all = 0;
      for (int base = 0; base < nt; base += blockDim.x) {
        const int i = base + tid;
        const int t = tl0 + i;
        int f = 0;
        bool tie = false, rank_me = false;
        uint32_t key = 0;
        if (i < nt && t >= st.lo && t < st.hi) {
          key = __float_as_uint(__ldcg(vb + t));
          if (st.all) {
            f = 1;
          } else if ((key & st.mask) > st.prefix) {
            f = 1;
          } else if ((key & st.mask) == st.prefix) {
            if (st.cand) rank_me = true;
            else if (st.tie_mode) tie = true;
          }
        }
        int tie_tot;
        const int tr = block_scan(tie ? 1 : 0, sm.wsum, tie_tot);
        if (tie) f = (tie_base + tr) < st.ties;
        tie_base += tie_tot;
        // candidates: one warp ranks one candidate against the gathered list
        if (st.cand) {
          int nr;
          const int rr = block_scan(rank_me ? 1 : 0, sm.wsum, nr);
          if (rank_me && rr < kMaxRound) {
            sm.toks[rr] = i;
            sm.tval[rr] = (int)key;
          }
          __syncthreads();
          for (int r0 = 0; r0 < nr; r0 += kMaxRound) {
            const int nrr = min(kMaxRound, nr - r0);
            if (r0 > 0) {
              // more than kMaxRound candidates in this chunk: refill the list
              const int rrr = rr - r0;
              __syncthreads();
              if (rank_me && rrr >= 0 && rrr < kMaxRound) {
                sm.toks[rrr] = i;
                sm.tval[rrr] = (int)key;
              }
              __syncthreads();
            }
            for (int q = warp; q < nrr; q += S::NW) {
              const int ii = sm.toks[q];
              const uint32_t kk = (uint32_t)sm.tval[q];
              const unsigned long long me = ((unsigned long long)kk << 32) | (0xffffffffu - (uint32_t)(tl0 + ii));
              unsigned above = 0;
              unsigned long long cum = 0;
              for (int j = lane; j < m_cand; j += 32) {
                const unsigned long long y = scand[j];
                if (y > me) {
                  ++above;
                  if (a.mode == TS_SELECT_TOPP) cum += to_fx(__uint_as_float((uint32_t)(y >> 32)));
                }
              }
#pragma unroll
              for (int d = 16; d >= 1; d >>= 1) {
                above += __shfl_xor_sync(kFull, above, d);
                cum += __shfl_xor_sync(kFull, cum, d);
              }
              if (lane == 0) {
                const int sel = (a.mode == TS_SELECT_TOPK) ? (above < (unsigned)st.k_rem) : (cum < st.mass_rem);
                selflag[t0l + ii] = (uint8_t)sel;
              }
            }
            __syncthreads();
          }
          if (rank_me) f = selflag[t0l + i];
        }
        if (i < nt) selflag[t0l + i] = (uint8_t)f;
        n_sel_all += f;
        n_sel_cand += f && t >= st.s_end && t < st.ls;
        __syncthreads();
      }
      int tot_c, tot_a;
      block_scan(n_sel_cand, sm.wsum, tot_c);
      block_scan(n_sel_all, sm.wsum, tot_a);
      if (tid == 0) {
        a.cta_cnt[((size_t)b * nCTA + c) * 3 + 0] = tot_c;
        a.cta_cnt[((size_t)b * nCTA + c) * 3 + 1] = tot_a;
      }
    }
    __syncthreads();
  }

  // ======================================================================== ATTEND
  // My tokens per sequence: a round-robin share of the fixed ones (sinks and
  // window, the cached part of a hit, or the caller's index list) and my own
  // selected candidates; gathered by bulk copy; one partial per CTA and head.
  if (a.phases & kPhAttend) {
    const bool given = !(a.phases & kPhSelect);
    const int stage_bytes = a.dyn_bytes - a.flag_cap;
    const int around = min(kMaxRound, stage_bytes / S::TOKEN_BYTES);
    KT* Ks = reinterpret_cast<KT*>(dsm);
    KT* Vs = Ks + (size_t)around * HKV * D;
    uint32_t aphase = 0;
    const int hw = warp % HKV;                         // warp -> KV head
    const int wslot = warp / HKV;
    const int wph = (S::NW - hw + HKV - 1) / HKV;      // warps on head hw
    const int lt = lane % S::ALPT, tslot = lane / S::ALPT;
    for (int b = 0; b < B; ++b) {
      const SeqState& st = sm.seq[b];
      const int32_t* gib = a.idx + (size_t)b * a.idx_stride;
      const int32_t* ctb = nullptr;
      int nfix, ct_lo = 0, ct_hi = 0;
      if (given) {
        nfix = max(0, min(a.count[b], (int)a.idx_stride));
      } else {
        nfix = st.s_end + (st.n - st.ls);
        if (st.hit && a.ct) {
          ctb = a.ct + (size_t)b * a.cap;
          const int cnt = a.filled[b] ? a.ct_count[b] : 0;
          ct_lo = lower_bound_i(ctb, cnt, st.s_end);
          ct_hi = lower_bound_i(ctb, cnt, st.ls);
          nfix += ct_hi - ct_lo;
        }
      }
      const int nmid = ct_hi - ct_lo;
      const int sgi = sm.my_seg_of[b];
      const bool own = !given && !st.hit && sgi >= 0;
      const int own_n = own ? sm.seg_ntok[sgi] : 0;
      const int nfix_mine = c < nfix ? (nfix - c + nCTA - 1) / nCTA : 0;
      float qr[S::GP][S::AEPC];
      float m_[G], l_[G], o_[G][S::AEPC];
#pragma unroll
      for (int j = 0; j < G; ++j) {
        m_[j] = -INFINITY;
        l_[j] = 0.f;
#pragma unroll
        for (int e = 0; e < S::AEPC; ++e) o_[j][e] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < S::GP; ++j)
#pragma unroll
        for (int e = 0; e < S::AEPC; ++e)
          qr[j][e] = (j < G) ? a.q[((size_t)b * H + hw * G + j) * D + lt * S::AEPC + e] : 0.f;
      int fdone = 0;     // fixed tokens of mine already taken
      int opos = 0;      // next own token (segment-local) to examine
      bool ok = true;
      while (true) {
        // ---- this round's tokens: fixed share first, then own selected ones
        int cnt = 0;
        const int nf = min(around, nfix_mine - fdone);
        for (int i = tid; i < nf; i += blockDim.x) {
          const int f = c + (fdone + i) * nCTA;
          int t;
          if (given) t = gib[f];
          else if (f < st.s_end) t = f;
          else if (f < st.s_end + nmid) t = ctb[ct_lo + (f - st.s_end)];
          else t = st.ls + (f - st.s_end - nmid);
          sm.toks[i] = t;
        }
        fdone += nf;
        cnt = nf;
        while (own && opos < own_n && cnt < around) {
          // one chunk of blockDim own tokens; take as many selected ones as fit
          const int i = opos + tid;
          const int t = sm.seg_lp0[sgi] * S::P + i;
          const bool take = i < own_n && selflag[sm.seg_t0[sgi] + i] && t >= st.s_end && t < st.ls;
          int tot;
          const int r = block_scan(take ? 1 : 0, sm.wsum, tot);
          const int room = around - cnt;
          if (take && r < room) sm.toks[cnt + r] = t;
          if (tot <= room) {
            opos += blockDim.x;
            cnt += tot;
          } else {
            // stop right after the room-th taken token of the chunk
            if (take && r == room - 1) sm.flag = i + 1;
            __syncthreads();
            opos = sm.flag;
            cnt = around;
          }
          __syncthreads();
        }
        if (cnt == 0) break;                          // uniform: same counters in every thread
        // ---- gather K and V rows of every KV head
        if (tid == 0) mbar_arrive_expect_tx(&abar, (uint32_t)(cnt * S::TOKEN_BYTES));
        for (int i = tid; i < cnt; i += blockDim.x) {
          const int t = sm.toks[i];
          int page = -1;
          if (t >= 0 && t < a.max_tokens) page = a.page_table[(size_t)b * a.pt_stride + t / S::P];
          const bool valid = page >= 0 && (int64_t)page < a.num_pages;
          if (!valid) set_error(a.status, TS_ERR_PAGE_OOB);
          sm.tval[i] = valid;
        }
        __syncthreads();
        for (int i = tid; i < 2 * cnt * HKV; i += blockDim.x) {
          const int ti = i / (2 * HKV), rem = i % (2 * HKV), g = rem >> 1, isv = rem & 1;
          const int t = sm.toks[ti];
          size_t off = 0;
          if (sm.tval[ti]) {
            const int page = a.page_table[(size_t)b * a.pt_stride + t / S::P];
            off = (((size_t)page * HKV + g) * S::P + (t % S::P)) * S::ROW_BYTES;
          }
          bulk_g2s((isv ? Vs : Ks) + ((size_t)ti * HKV + g) * D, (isv ? a.v_pool : a.k_pool) + off,
                   S::ROW_BYTES, &abar);
        }
        const bool landed = mbar_wait(&abar, aphase);
        aphase ^= 1u;
        ok = __syncthreads_and(landed) != 0;
        if (!ok) {
          if (tid == 0) {
            set_error(a.status, TS_ERR_TIMEOUT);
            mbar_wait(&abar, aphase ^ 1u);   // copies still in flight land before the CTA leaves
          }
          __syncthreads();
          break;
        }
        // ---- online softmax: warp -> KV head hw, tokens strided over that head's warps
        for (int j0 = wslot * S::ATPW; j0 < cnt; j0 += wph * S::ATPW) {
          const int j = j0 + tslot;
          const bool act = j < cnt;
          const int jj = act ? j : 0;
          const KT* kr = Ks + ((size_t)jj * HKV + hw) * D + lt * S::AEPC;
          const KT* vr = Vs + ((size_t)jj * HKV + hw) * D + lt * S::AEPC;
          float kf[S::AEPC], vf[S::AEPC];
          if constexpr (S::ACB == 16) {
            KV<KT>::unpack(lds128(kr), kf);
            KV<KT>::unpack(lds128(vr), vf);
          } else {
            const uint2 k2 = *reinterpret_cast<const uint2*>(kr);
            const uint2 v2 = *reinterpret_cast<const uint2*>(vr);
            if constexpr (sizeof(KT) == 2) {
              kf[0] = __uint_as_float(k2.x << 16);
              kf[1] = __uint_as_float(k2.x & 0xffff0000u);
              kf[2] = __uint_as_float(k2.y << 16);
              kf[3] = __uint_as_float(k2.y & 0xffff0000u);
              vf[0] = __uint_as_float(v2.x << 16);
              vf[1] = __uint_as_float(v2.x & 0xffff0000u);
              vf[2] = __uint_as_float(v2.y << 16);
              vf[3] = __uint_as_float(v2.y & 0xffff0000u);
            } else {
              kf[0] = __uint_as_float(k2.x);
              kf[1] = __uint_as_float(k2.y);
              vf[0] = __uint_as_float(v2.x);
              vf[1] = __uint_as_float(v2.y);
            }
          }
          float acc[S::GP];
#pragma unroll
          for (int h = 0; h < S::GP; ++h) {
            float x = 0.f;
#pragma unroll
            for (int e = 0; e < S::AEPC; ++e) x = fmaf(qr[h][e], kf[e], x);
            acc[h] = x;
          }
          int which;
          const float red = transpose_reduce<S::GP, S::ALPT>(acc, lane, which);
          const bool live = act && sm.tval[jj] != 0;
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float dot = __shfl_sync(kFull, red, (lane & ~(S::ALPT - 1)) + h * (S::ALPT / S::GP));
            if (live) {
              const float sc = dot * a.scale;
              const float mn = fmaxf(m_[h], sc);
              const float corr = expf(m_[h] - mn);
              const float p = expf(sc - mn);
              l_[h] = l_[h] * corr + p;
#pragma unroll
              for (int e = 0; e < S::AEPC; ++e) o_[h][e] = fmaf(p, vf[e], o_[h][e] * corr);
              m_[h] = mn;
            }
          }
        }
        __syncthreads();
      }
      if (!ok) {
        if (tid == 0) atomicExch(&a.gsync->abort, 1u);   // the others leave the last barrier
        return;
      }
      // ---- this CTA's partial of every query head: merge all warps' token slots
      float* mg = reinterpret_cast<float*>(dsm);      // [NW*ATPW][G][D], then m and l
      const int slots = S::NW * S::ATPW;
      float* mm = mg + (size_t)slots * G * D;
      float* ml = mm + slots * G;
      const int myslot = warp * S::ATPW + tslot;
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int e = 0; e < S::AEPC; ++e) mg[((size_t)myslot * G + h) * D + lt * S::AEPC + e] = o_[h][e];
        if (lt == 0) {
          mm[myslot * G + h] = m_[h];
          ml[myslot * G + h] = l_[h];
        }
      }
      __syncthreads();
      float* pb = a.apart + ((size_t)b * nCTA + c) * H * (D + 2);
      for (int i = tid; i < HKV * G * D; i += blockDim.x) {
        const int hg = i / (G * D), rem = i % (G * D), h = rem / D, d = rem % D;
        float M = -INFINITY;
        for (int w = hg; w < S::NW; w += HKV)
          for (int ts = 0; ts < S::ATPW; ++ts) M = fmaxf(M, mm[(w * S::ATPW + ts) * G + h]);
        float num = 0.f, den = 0.f;
        if (M > -INFINITY) {
          for (int w = hg; w < S::NW; w += HKV)
            for (int ts = 0; ts < S::ATPW; ++ts) {
              const int sl = w * S::ATPW + ts;
              const float wgt = expf(mm[sl * G + h] - M);
              num = fmaf(wgt, mg[((size_t)sl * G + h) * D + d], num);
              den = fmaf(wgt, ml[sl * G + h], den);
            }
        }
        const int qh = hg * G + h;
        pb[(size_t)qh * (D + 2) + d] = num;
        if (d == 0) {
          pb[(size_t)qh * (D + 2) + D] = M;
          pb[(size_t)qh * (D + 2) + D + 1] = den;
        }
      }
      __syncthreads();
    }
  }

  // ============================================== outputs, after one more barrier
  if (!(a.phases & (kPhSelect | kPhAttend))) return;
  if (!grid_sync(a.gsync, a.status)) return;
  if (a.phases & kPhAttend) {
    // merge the CTA partials: item = (sequence, query head, 32-dim slice)
    const int nslice = D / 32;
    for (int item = c * S::NW + warp; item < B * H * nslice; item += nCTA * S::NW) {
      const int b = item / (H * nslice), rem = item % (H * nslice), h = rem / nslice, sl = rem % nslice;
      const float* pp = a.apart + (size_t)b * nCTA * H * (D + 2) + (size_t)h * (D + 2);
      float M = -INFINITY;
      for (int cc = lane; cc < nCTA; cc += 32) M = fmaxf(M, __ldcg(pp + (size_t)cc * H * (D + 2) + D));
      M = warp_max(M);
      float num = 0.f, den = 0.f;
      if (M > -INFINITY) {
        for (int cc = 0; cc < nCTA; ++cc) {
          const float* pc = pp + (size_t)cc * H * (D + 2);
          const float mc = __ldcg(pc + D);
          if (mc == -INFINITY) continue;
          const float wgt = expf(mc - M);
          num = fmaf(wgt, __ldcg(pc + sl * 32 + lane), num);
          den = fmaf(wgt, __ldcg(pc + D + 1), den);
        }
      }
      a.out[((size_t)b * H + h) * D + sl * 32 + lane] = den > 0.f ? num / den : 0.f;
      if (a.lse && sl == 0 && lane == 0) a.lse[(size_t)b * H + h] = den > 0.f ? M + logf(den) : -INFINITY;
    }
  }
  if (a.phases & kPhSelect) {
    // ascending index lists and Selection Cache entries
    for (int b = 0; b < B; ++b) {
      const SeqState& st = sm.seq[b];
      int32_t* ib = a.idx + (size_t)b * a.idx_stride;
      if (st.hit) {
        const int32_t* ctb = a.ct ? a.ct + (size_t)b * a.cap : nullptr;
        const int cnt = (ctb && a.filled[b]) ? a.ct_count[b] : 0;
        const int lo = ctb ? lower_bound_i(ctb, cnt, st.s_end) : 0;
        const int mcount = ctb ? lower_bound_i(ctb, cnt, st.ls) - lo : 0;
        const int total = st.s_end + mcount + (st.n - st.ls);
        if (total > a.idx_stride) {
          if (c == 0 && tid == 0) {
            set_error(a.status, TS_ERR_CAPACITY);
            a.count[b] = 0;
          }
          continue;
        }
        const int per = (total + nCTA - 1) / nCTA;
        for (int j = c * per + tid; j < min(total, (c + 1) * per); j += blockDim.x) {
          int v;
          if (j < st.s_end) v = j;
          else if (j < st.s_end + mcount) v = ctb[lo + j - st.s_end];
          else v = st.ls + (j - st.s_end - mcount);
          ib[j] = v;
        }
        if (c == 0 && tid == 0) a.count[b] = total;
        continue;
      }
      int tot_c = 0, tot_a = 0, pre_c = 0, pre_a = 0;
      for (int cc = st.first_cta; cc <= st.last_cta; ++cc) {
        const int xc = __ldcg(&a.cta_cnt[((size_t)b * nCTA + cc) * 3 + 0]);
        const int xa = __ldcg(&a.cta_cnt[((size_t)b * nCTA + cc) * 3 + 1]);
        if (cc < c) {
          pre_c += xc;
          pre_a += xa;
        }
        tot_c += xc;
        tot_a += xa;
      }
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
      if (c == 0) {
        if (fits) {
          for (int j = tid; j < st.s_end; j += blockDim.x) ib[j] = j;
          for (int j = tid; j < st.n - st.ls; j += blockDim.x) ib[st.s_end + tot_c + j] = st.ls + j;
        }
        if (a.cq) {
          const float* qb = a.q + (size_t)b * H * D;
          float* cqb = a.cq + (size_t)b * H * D;
          for (int j = tid; j < H * D; j += blockDim.x) cqb[j] = qb[j];
        }
      }
      const int sgi = sm.my_seg_of[b];
      if (sgi < 0) continue;
      const int tl0 = sm.seg_lp0[sgi] * S::P, nt = sm.seg_ntok[sgi], t0l = sm.seg_t0[sgi];
      int32_t* ctb = cfits ? a.ct + (size_t)b * a.cap : nullptr;
      for (int base = 0; base < nt; base += blockDim.x) {
        const int i = base + tid;
        const int t = tl0 + i;
        const bool f = i < nt && selflag[t0l + i];
        const bool fc = f && t >= st.s_end && t < st.ls;
        int ta, tc;
        const int ra = block_scan(f ? 1 : 0, sm.wsum, ta);
        const int rc = block_scan(fc ? 1 : 0, sm.wsum, tc);
        if (f && ctb) ctb[pre_a + ra] = t;
        if (fc && fits) ib[st.s_end + pre_c + rc] = t;
        pre_a += ta;
        pre_c += tc;
      }
    }
  }
}

// ------------------------------------------------------------------- launch

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
    if (std::getenv("TS_DEBUG"))
      std::fprintf(stderr, "ts step: smem optin %d, per SM %d, reserved/block %d\n", optin, per_sm, reserved);
    // the whole unified L1/shared array as shared memory for this kernel
    if (cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
      return TS_ERR_CUDA;
  }
  const int dyn = (smem_avail - static_bytes - 1024) / 128 * 128;
  const int flag_cap = 8192;   // >= kMaxB * kMaxWaveHeads * 4 (vote weights alias it)
  static_assert(kMaxB * kMaxWaveHeads * 4 <= 8192, "weights fit the flag area");
  const int e_bytes = dyn - S::RING_BYTES - flag_cap;
  if (e_bytes < 16 * 1024) return TS_ERR_UNSUPPORTED;
  if (!ensure_smem<step_kernel<KT, D, HKV, G>>((size_t)dyn, ctx->device)) {
    if (std::getenv("TS_DEBUG")) std::fprintf(stderr, "ts step: smem attribute %d B refused\n", dyn);
    return TS_ERR_CUDA;
  }
  const bool debug = std::getenv("TS_DEBUG") != nullptr;
  if (ctx->step_grid <= 0) {
    int per_sm = 0;
    const cudaError_t oe = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, S::THREADS, (size_t)dyn);
    if (debug)
      std::fprintf(stderr, "ts step: static %d B, dynamic %d B, threads %d, blocks/SM %d (%s)\n", static_bytes, dyn,
                   S::THREADS, per_sm, cudaGetErrorString(oe));
    if (oe != cudaSuccess || per_sm < 1) return TS_ERR_COOP_UNAVAILABLE;
    ctx->step_grid = ctx->num_sms;
  }
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
  a.gsync = reinterpret_cast<GridSync*>(ctx->gsync);
  a.status = ctx->status;
  a.dyn_bytes = dyn;
  a.e_cap = e_bytes / 4;
  a.flag_cap = flag_cap;
  if (cudaMemsetAsync(ctx->gsync, 0, sizeof(GridSync), s) != cudaSuccess) return TS_ERR_CUDA;
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
