// flat.cu -- the flat O(N^2/C) BSA-style selector used as the comparator.
// agihunt.info summary of "Block Sparse Attention with Log-Linear
// Complexity", model paragraph: BSA is NSA's selected branch with
// mean-pooled block summaries; rcap.io post: standard block-sparse attention
// scores every query against every block summary.  Each query head h' takes
// p_h'(i) = softmax over the complete past blocks i < qb of s q_h'.mu_i, the
// block score is the sum over the GQA group's heads, and the Top-K of E plus
// the forced blocks is returned (same output format as the pyramid path).
//
// Same GB300 machinery as the pyramid leaf stage: a 128-row tile holds
// 128/G consecutive queries x G heads (gathered once per tile with cp.async
// into the 128-byte swizzled K-major layout), the leaf means are rounded to
// bf16 once and streamed as 128-leaf TMA tiles, tcgen05.mma accumulates
// 128 x 128 fp32 scores in TMEM.  Pass 1 keeps a per-row online
// log2-sum-exp2; pass 2 recomputes the scores, forms the probabilities, sums
// the G head rows with shuffles and keeps a sorted Top-K list per query.
#include <algorithm>

#include "pisa_common.cuh"
#include "pisa_internal.h"
#include "tc_ptx.cuh"

namespace pisa {

constexpr int kFRows = 128;
constexpr int kFCols = 128;
constexpr int kFStagesB = 2;
constexpr int kFCap = kMaxK;  // Top-K list per query and column slice
// Epilogue warps: each TMEM lane quadrant (32 rows) is read by S warps, one
// per slice of 128 / S columns; S grows with the group size so the per-slice
// Top-K lists of the 128 / G queries of a tile fit in shared memory.
template <int G>
constexpr int flat_slices() { return G >= 4 ? 4 : G; }
template <int G>
constexpr int flat_threads() { return 32 * (3 + 4 * flat_slices<G>()); }

// Bounded wait for the epilogue warps, which wait for most of a tile: after a
// short spin they sleep between probes so that waiting warps leave issue
// slots to the loader and MMA warps of the SM.
__device__ __forceinline__ bool flat_wait_sleepy(uint32_t bar, uint32_t parity, volatile int32_t* abort,
                                                 uint64_t limit_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  uint32_t ns = 32;
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (it >= 8) {
      __nanosleep(ns);
      if (ns < 256) ns *= 2;
    }
    if ((it & 15u) == 0) {
      if (*abort) return false;
      if (ptx::globaltimer_ns() - t0 > limit_ns) return false;
    }
  }
}

// (score, block) ordering of the Top-K: higher score first, then lower block
// (empty entries, (-inf, -1), last).
__device__ __forceinline__ bool flat_better(float x, int32_t xi, float y, int32_t yi) {
  return x > y || (x == y && (uint32_t)xi < (uint32_t)yi);
}

// Two lanes' sorted best-8 lists (lanes l and l ^ o) merged into the best 8
// of their union, sorted, in both lanes: the element-wise better of one list
// and the other reversed holds the best 8 as a bitonic sequence, which three
// half-cleaner stages sort.
__device__ __forceinline__ void flat_merge8_xor(float (&a)[8], int32_t (&ai)[8], int o) {
  float b[8];
  int32_t bi[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    b[i] = __shfl_xor_sync(0xffffffffu, a[i], o);
    bi[i] = __shfl_xor_sync(0xffffffffu, ai[i], o);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool tb = flat_better(b[7 - i], bi[7 - i], a[i], ai[i]);
    a[i] = tb ? b[7 - i] : a[i];
    ai[i] = tb ? bi[7 - i] : ai[i];
  }
#pragma unroll
  for (int d = 4; d >= 1; d >>= 1)
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((i & d) == 0) {
        const bool sw = flat_better(a[i + d], ai[i + d], a[i], ai[i]);
        const float t = a[i];
        const int32_t ti = ai[i];
        a[i] = sw ? a[i + d] : a[i];
        ai[i] = sw ? ai[i + d] : ai[i];
        a[i + d] = sw ? t : a[i + d];
        ai[i + d] = sw ? ti : ai[i + d];
      }
}

// Eight entries sorted by block index, ascending (empty entries, block -1,
// last): a 19-comparator sorting network.
__device__ __forceinline__ void flat_sort8_by_block(float (&a)[8], int32_t (&ai)[8]) {
  constexpr int kNet[19][2] = {{0, 2}, {1, 3}, {4, 6}, {5, 7}, {0, 4}, {1, 5}, {2, 6}, {3, 7}, {0, 1}, {2, 3},
                               {4, 5}, {6, 7}, {2, 4}, {3, 5}, {1, 4}, {3, 6}, {1, 2}, {3, 4}, {5, 6}};
#pragma unroll
  for (int c = 0; c < 19; ++c) {
    const int i = kNet[c][0], j = kNet[c][1];
    const bool sw = (uint32_t)ai[j] < (uint32_t)ai[i];
    const float t = a[i];
    const int32_t ti = ai[i];
    a[i] = sw ? a[j] : a[i];
    ai[i] = sw ? ai[j] : ai[i];
    a[j] = sw ? t : a[j];
    ai[j] = sw ? ti : ai[j];
  }
}

constexpr int kFAcc = 4;  // TMEM accumulators: the MMA runs up to four tiles ahead of the epilogue
constexpr uint32_t kFTmemCols = kFAcc * kFCols;
constexpr uint64_t kFWaitNs = 4000000000ull;

template <int D, int G>
struct FlatSmem {
  static constexpr int S = flat_slices<G>();
  uint8_t a[2][kFRows * D * 2];
  uint8_t b[kFStagesB][kFCols * D * 2];
  float top_s[S][kFRows / G][kFCap];   // per (slice, query): best K so far, score descending
  int32_t top_i[S][kFRows / G][kFCap];
  int32_t top_n[S][kFRows];            // entries per list, by (slice, row of the list's lane)
  float2 part[S][kFRows];              // per (slice, row): online (max, sum) of pass 0
  float cut[kFRows / G];               // per query: the largest K-th best of its full slice lists (a lower
                                       // bound on its final K-th best); non-negative, so ordered as int bits
  float stash[4 * S][1024 / G];        // per epilogue warp: a chunk's scores awaiting insertion
  uint64_t full_a[2], empty_a[2], full_b[kFStagesB], empty_b[kFStagesB];
  uint64_t tfull[kFAcc], tempty[kFAcc], done;
  uint64_t ep_bar;                     // the epilogue warps' rendezvous (two phases per query tile)
  uint32_t tmem_base;
  int32_t abort, zero;
};

__global__ void means_to_bf16_kernel(int64_t nbh, int64_t P, int64_t nb, int d, const float* __restrict__ pyr,
                                     __nv_bfloat16* __restrict__ mu) {
  pdl_wait();
  const int64_t n = nbh * nb * d;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t c = i % d, row = i / d, leaf = row % nb, bh = row / nb;
    mu[i] = __float2bfloat16_rn(pyr[(bh * P + leaf) * d + c]);
  }
}

struct FlatTiles {
  int64_t nqt;  // query tiles per (sequence, key head)
  int32_t Qt;   // queries per tile
};

// columns (leaf blocks) needed by a query tile: blocks [0, qb_last)
__device__ __forceinline__ int flat_nj(const Prob& pr, int64_t t0, int Qt) {
  int64_t tl = t0 + Qt - 1;
  if (tl >= pr.N) tl = pr.N - 1;
  const int64_t qb_last = tl / pr.C;
  return (int)ceil_div64(qb_last, kFCols);
}

template <int D, int G, int KR>
__global__ void __launch_bounds__(flat_threads<G>(), 1)
    flat_tc_kernel(Prob pr, FlatTiles ft, int64_t nb, const __grid_constant__ CUtensorMap mumap,
                   const uint16_t* __restrict__ q, int32_t* __restrict__ out_idx, float* __restrict__ out_score,
                   int32_t* __restrict__ status) {
  pdl_wait();
  extern __shared__ unsigned char smem_raw[];
  FlatSmem<D, G>& sm = *reinterpret_cast<FlatSmem<D, G>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                    ~static_cast<uintptr_t>(1023));
  constexpr int kHalf = kFRows * 128;
  constexpr uint32_t kBBytes = kFCols * D * 2;
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kFRows, kFCols);
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  volatile int32_t* abort = &sm.abort;
  const int64_t QT = pr.B * pr.Hkv * ft.nqt;
  const int Qt = ft.Qt;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(ptx::smem_u32(&sm.full_a[s]), 32);
      ptx::mbar_init(ptx::smem_u32(&sm.empty_a[s]), 1);
    }
    for (int s = 0; s < kFAcc; ++s) {
      ptx::mbar_init(ptx::smem_u32(&sm.tfull[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&sm.tempty[s]), 4 * FlatSmem<D, G>::S);
    }
    for (int s = 0; s < kFStagesB; ++s) {
      ptx::mbar_init(ptx::smem_u32(&sm.full_b[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&sm.empty_b[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&sm.done), 1);
    ptx::mbar_init(ptx::smem_u32(&sm.ep_bar), 4 * FlatSmem<D, G>::S);
    sm.abort = 0;
    sm.zero = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&sm.tmem_base), kFTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------- query gathers
    constexpr int CPR = D / 8, RPI = 32 / CPR;
    const int ch = lane % CPR;
    int ia = 0;
    bool ok = true;
    for (int64_t qt = blockIdx.x; qt < QT && ok; qt += gridDim.x) {
      const int64_t bh = qt / ft.nqt, t0 = (qt % ft.nqt) * Qt;
      const int64_t b = bh / pr.Hkv, h = bh % pr.Hkv;
      const int nj = flat_nj(pr, t0, Qt);
      if (nj == 0) continue;
      const int sa = ia & 1;
      ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sm.empty_a[sa]), ((ia >> 1) & 1) ^ 1, abort, kFWaitNs);
      if (!ok) break;
      const uint32_t abase = ptx::smem_u32(sm.a[sa]);
      for (int r0 = 0; r0 < kFRows; r0 += RPI) {
        const int r = r0 + lane / CPR;
        const int64_t t = t0 + r / G;
        if (t < pr.N) {
          const uint16_t* src = q + (((b * pr.Hq + h * G + (r % G)) * pr.N + t) * D + ch * 8);
          ptx::cp_async_16(abase + (ch >> 3) * kHalf + r * 128 + (((ch & 7) ^ (r & 7)) << 4), src);
        }
      }
      ptx::cp_async_commit();
      ptx::cp_async_wait<0>();
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(ptx::smem_u32(&sm.full_a[sa]));
      ++ia;
    }
    if (!ok) *abort = 1;
  } else if (warp == 2) {
    // ------------------------------------------------------- key-mean tiles
    if (lane == 0) {
      int ib = 0;
      bool ok = true;
      for (int64_t qt = blockIdx.x; qt < QT && ok; qt += gridDim.x) {
        const int64_t bh = qt / ft.nqt, t0 = (qt % ft.nqt) * Qt;
        const int nj = flat_nj(pr, t0, Qt);
        for (int pass = 0; pass < 2 && ok; ++pass)
          for (int j = 0; j < nj; ++j) {
            const int sb = ib % kFStagesB, ub = ib / kFStagesB;
            ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sm.empty_b[sb]), (ub & 1) ^ 1, abort, kFWaitNs);
            if (!ok) break;
            const uint32_t fb = ptx::smem_u32(&sm.full_b[sb]);
            ptx::mbar_arrive_expect_tx(fb, kBBytes);
            const int32_t y = (int32_t)(bh * nb + (int64_t)j * kFCols);
#pragma unroll
            for (int hh = 0; hh < D / 64; ++hh)
              ptx::tma_load_2d(ptx::smem_u32(sm.b[sb]) + hh * kHalf, &mumap, 64 * hh, y, fb);
            ++ib;
          }
      }
      if (!ok) *abort = 1;
      // every issued load lands before the CTA can exit, whoever gave up
      for (int k = ib > kFStagesB ? ib - kFStagesB : 0; k < ib; ++k)
        ptx::mbar_wait_bounded(ptx::smem_u32(&sm.full_b[k % kFStagesB]), (k / kFStagesB) & 1, &sm.zero,
                               kFWaitNs);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      int ia = 0, ib = 0, it = 0;
      bool ok = true;
      for (int64_t qt = blockIdx.x; qt < QT && ok; qt += gridDim.x) {
        const int64_t t0 = (qt % ft.nqt) * Qt;
        const int nj = flat_nj(pr, t0, Qt);
        if (nj == 0) continue;
        const int sa = ia & 1;
        ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sm.full_a[sa]), (ia >> 1) & 1, abort, kFWaitNs);
        if (!ok) break;
        for (int pass = 0; pass < 2 && ok; ++pass)
          for (int j = 0; j < nj; ++j) {
            const int sb = ib % kFStagesB, acc = it % kFAcc;
            ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sm.full_b[sb]), (ib / kFStagesB) & 1, abort, kFWaitNs) &&
                 ptx::mbar_wait_bounded(ptx::smem_u32(&sm.tempty[acc]), ((it / kFAcc) & 1) ^ 1, abort, kFWaitNs);
            if (!ok) break;
            ptx::tc_fence_after();
            const uint32_t a0 = ptx::smem_u32(sm.a[sa]), b0 = ptx::smem_u32(sm.b[sb]);
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
              const uint32_t off = (k >> 2) * kHalf + (k & 3) * 32;
              ptx::mma_bf16(tmem + acc * kFCols, ptx::desc_sw128(a0 + off), ptx::desc_sw128(b0 + off), kIdesc,
                            k > 0 ? 1u : 0u);
            }
            ptx::mma_commit(ptx::smem_u32(&sm.empty_b[sb]));
            ptx::mma_commit(ptx::smem_u32(&sm.tfull[acc]));
            ++ib;
            ++it;
          }
        if (ok) ptx::mma_commit(ptx::smem_u32(&sm.empty_a[sa]));
        ++ia;
      }
      if (!ok) *abort = 1;
      ptx::mma_commit(ptx::smem_u32(&sm.done));
      ptx::mbar_wait_bounded(ptx::smem_u32(&sm.done), 0, &sm.zero, kFWaitNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // warp (quadrant q4, slice sl): rows q4 * 32 + lane, columns
    // [sl * SW, sl * SW + SW) of every 128-column tile.  A warp can only read
    // the TMEM lane quadrant warp % 4, so q4 = warp & 3; the slices take the
    // epilogue warps in groups of four
    constexpr int S = FlatSmem<D, G>::S;
    constexpr int SW = kFCols / S;  // 32, 64 or 128 columns
    // K <= 8 and G <= 4: a register list per lane (over the lane's columns of
    // each chunk); otherwise one list per query, kept by its g == 0 lane
    constexpr bool kLaneLists = KR <= 8 && G <= 4;
    constexpr int LG = kLaneLists ? G : 1;  // lists per (slice, query)
    const int mth = (pr.K + LG - 1) / LG - 1;  // list entry whose minimum over the query's lanes bounds its K-th best
    const int q4 = warp & 3, sl = (warp - 3) >> 2;
    const int r = q4 * 32 + lane;
    const int g = r % G, qi = r / G;
    const float sc = pr.scale2;
    const int K = pr.K, W = K + 3;
    float* ts = sm.top_s[sl][qi];
    int32_t* tix = sm.top_i[sl][qi];  // used by the g == 0 lane of each query
    int it = 0, eph = 0;
    bool ok = true;
    // the epilogue warps' rendezvous: every warp arrives, then waits (bounded)
    auto rendezvous = [&]() -> bool {
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&sm.ep_bar));
      const bool okw = ptx::mbar_wait_bounded(ptx::smem_u32(&sm.ep_bar), eph & 1, abort, kFWaitNs);
      ++eph;
      return __all_sync(0xffffffffu, okw);
    };
    for (int64_t qt = blockIdx.x; qt < QT && ok; qt += gridDim.x) {
      const int64_t bh = qt / ft.nqt, t0 = (qt % ft.nqt) * Qt;
      const int nj = flat_nj(pr, t0, Qt);
      const int64_t t = t0 + qi;
      const int64_t qb = t < pr.N ? t / pr.C : 0;  // valid columns: [0, qb)
      const int qb32 = (int)qb;
      float m = -INFINITY, ssum = 0.0f, lse = 0.0f;
      int cnt = 0;              // entries in this slice's list of the query (g == 0 lane)
      float theta = -INFINITY;  // its K-th best, once cnt has reached K
      // K <= 8: the list lives in the g == 0 lane's registers, sorted (best
      // first, -inf padded); positions past K may hold stale entries below
      // the K-th best, which the output never reads
      float rl[8];
      int32_t ri[8];
      float pub = 0.0f;  // the largest bound this lane has published to the query's cut
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        rl[i] = -INFINITY;
        ri[i] = -1;
      }
      for (int pass = 0; pass < 2 && ok; ++pass) {
        if (pass == 1) {
          // the row's log2-sum-exp2 from the S slices' partials; the query's
          // shared cut restarts (no slice reads it before this rendezvous,
          // and slice 0 resets it after merging the previous tile's lists)
          sm.part[sl][r] = make_float2(m, ssum);
          if (sl == 0 && g == 0) sm.cut[qi] = 0.0f;
          if (!rendezvous()) { ok = false; *abort = 1; break; }
          float mm = -INFINITY;
#pragma unroll
          for (int u = 0; u < S; ++u) mm = fmaxf(mm, sm.part[u][r].x);
          float ss = 0.0f;
#pragma unroll
          for (int u = 0; u < S; ++u) {
            const float2 pu = sm.part[u][r];
            if (pu.x > -INFINITY) ss += pu.y * ptx::ex2(pu.x - mm);
          }
          lse = mm + ptx::lg2(ss);
          // the lists are rewritten below only after this rendezvous, which
          // the slice-0 warps reach after merging the previous tile's lists
        }
        for (int j = 0; j < nj; ++j) {
          const int acc = it % kFAcc;
          const bool okw = flat_wait_sleepy(ptx::smem_u32(&sm.tfull[acc]), (it / kFAcc) & 1, abort, kFWaitNs);
          if (!__all_sync(0xffffffffu, okw)) { ok = false; *abort = 1; break; }
          ptx::tc_fence_after();
          const uint32_t taddr = tmem + ((uint32_t)(q4 * 32) << 16) + acc * kFCols + sl * SW;
          const int col0 = j * kFCols + sl * SW;  // block indices fit in 32 bits (N <= 2^26)
          if (pass == 0) {
            // raw dots (scale applied in the exponent; s > 0 keeps the order)
            float tm = -INFINITY;
            float x[SW];
#pragma unroll
            for (int c4 = 0; c4 < SW / 32; ++c4) {
              uint32_t v[32];
              ptx::tmem_ld32(taddr + c4 * 32, v);
              ptx::tmem_ld_wait();
              const int nv = qb32 - (col0 + c4 * 32);  // columns c < nv are past blocks
              if (__all_sync(0xffffffffu, nv >= 32)) {
#pragma unroll
                for (int c = 0; c < 32; ++c) x[c4 * 32 + c] = __uint_as_float(v[c]);
              } else {
#pragma unroll
                for (int c = 0; c < 32; ++c) x[c4 * 32 + c] = c < nv ? __uint_as_float(v[c]) : -INFINITY;
              }
#pragma unroll
              for (int c = 0; c < 32; c += 2) tm = fmaxf(tm, fmaxf(x[c4 * 32 + c], x[c4 * 32 + c + 1]));
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&sm.tempty[acc]));
            if (tm > -INFINITY) {
              const float mn = fmaxf(m, tm * sc);
              float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
              for (int c = 0; c < SW; ++c) s4[c & 3] += ptx::ex2(fmaf(x[c], sc, -mn));
              ssum = ssum * ptx::ex2(m - mn) + ((s4[0] + s4[1]) + (s4[2] + s4[3]));
              m = mn;
            }
          } else {
#pragma unroll 1
            for (int c4 = 0; c4 < SW / 32; ++c4) {
              uint32_t v[32];
              ptx::tmem_ld32(taddr + c4 * 32, v);
              ptx::tmem_ld_wait();
              const int cb = col0 + c4 * 32;
              const int nv = qb32 - cb;                  // c < nv: past blocks (in the softmax)
              const int elo = 1 - cb, ehi = qb32 - 2 - cb;  // elo <= c <= ehi: in E (ranked)
              if constexpr (kLaneLists) {
                // every lane keeps a list of its own columns: the G lanes of a
                // query reduce-scatter the head sum, lane g ending with
                // columns [CPL g, CPL g + CPL) of the chunk
                constexpr int CPL = 32 / G;
                const bool inner = __all_sync(0xffffffffu, elo <= 0 && ehi >= 31);
                float e[32];
                if (inner) {
#pragma unroll
                  for (int c = 0; c < 32; ++c) e[c] = ptx::ex2(fmaf(__uint_as_float(v[c]), sc, -lse));
                } else {
#pragma unroll
                  for (int c = 0; c < 32; ++c) e[c] = c < nv ? ptx::ex2(fmaf(__uint_as_float(v[c]), sc, -lse)) : 0.0f;
                }
#pragma unroll
                for (int o = G / 2, n = 32; o >= 1; o >>= 1, n >>= 1) {
                  const bool up = (lane & o) != 0;
#pragma unroll
                  for (int i = 0; i < n / 2; ++i) {
                    const float keep = up ? e[i + n / 2] : e[i];
                    const float send = up ? e[i] : e[i + n / 2];
                    e[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                  }
                }
                const int cg = CPL * g;  // this lane's first column of the chunk
                float bm = -INFINITY;
#pragma unroll
                for (int i = 0; i < CPL; ++i) {
                  if (!inner) e[i] = (cg + i >= elo && cg + i <= ehi) ? e[i] : -INFINITY;  // Top-K over E only
                  bm = fmaxf(bm, e[i]);
                }
                // columns at or above the query's shared cut (the largest K-th
                // best of its full lists, at most its final K-th best) and
                // above the lane's own K-th best, then sorted insertion of each
                // (select-shift over the register list; ties keep the earlier
                // column, and the merge orders ties across lists by index)
                // the lists of the query's G lanes are disjoint, so the
                // smallest of their m-th bests (m = ceil(K / G) - 1) is reached
                // by at least K columns: a lower bound on the final K-th best
                float tm = rl[0];
#pragma unroll
                for (int u = 1; u < 8; ++u) tm = (u == mth) ? rl[u] : tm;
#pragma unroll
                for (int o = 1; o < G; o <<= 1) tm = fminf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
                if (g == 0 && tm > pub) {
                  pub = tm;
                  atomicMax(reinterpret_cast<int*>(&sm.cut[qi]), __float_as_int(tm));
                }
                float cut = fmaxf(fmaxf(theta, tm), sm.cut[qi]);
                if (bm >= cut) {
                  uint32_t msk = 0;
#pragma unroll
                  for (int i = 0; i < CPL; ++i) msk |= (e[i] >= cut && e[i] > theta) ? (1u << i) : 0u;
                  float* st = sm.stash[warp - 3] + lane * CPL;
#pragma unroll
                  for (int i = 0; i < CPL; i += 4)
                    *reinterpret_cast<float4*>(st + i) = make_float4(e[i], e[i + 1], e[i + 2], e[i + 3]);
                  while (msk) {
                    const int i = __ffs(msk) - 1;
                    msk &= msk - 1;
                    const float x = st[i];
                    if (!(x > theta) || x < cut) continue;
                    const int32_t col = cb + cg + i;
                    bool ge[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) ge[u] = rl[u] >= x;
#pragma unroll
                    for (int u = 7; u >= 1; --u) {
                      rl[u] = ge[u] ? rl[u] : (ge[u - 1] ? x : rl[u - 1]);
                      ri[u] = ge[u] ? ri[u] : (ge[u - 1] ? col : ri[u - 1]);
                    }
                    rl[0] = ge[0] ? rl[0] : x;
                    ri[0] = ge[0] ? ri[0] : col;
                    if (cnt < K) ++cnt;
                    if (cnt == K) {
                      float kth = rl[0];
#pragma unroll
                      for (int u = 1; u < 8; ++u) kth = (u == K - 1) ? rl[u] : kth;
                      theta = kth;
                      cut = fmaxf(cut, theta);
                      atomicMax(reinterpret_cast<int*>(&sm.cut[qi]), __float_as_int(theta));
                    }
                  }
                }
              } else {
                float pv[32];
                float bmax = -INFINITY;
                if (__all_sync(0xffffffffu, elo <= 0 && ehi >= 31)) {
#pragma unroll
                  for (int c = 0; c < 32; ++c) {
                    float p = ptx::ex2(fmaf(__uint_as_float(v[c]), sc, -lse));
#pragma unroll
                    for (int o = 1; o < G; o <<= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
                    pv[c] = p;
                  }
                } else {
#pragma unroll
                  for (int c = 0; c < 32; ++c) {
                    float p = c < nv ? ptx::ex2(fmaf(__uint_as_float(v[c]), sc, -lse)) : 0.0f;
#pragma unroll
                    for (int o = 1; o < G; o <<= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
                    pv[c] = (c >= elo && c <= ehi) ? p : -INFINITY;  // Top-K runs over E only
                  }
                }
#pragma unroll
                for (int c = 0; c < 32; c += 2) bmax = fmaxf(bmax, fmaxf(pv[c], pv[c + 1]));
                // the group's first lane keeps this slice's best K of its query
                // sorted (higher score first; a later column never passes an
                // equal score, so ties keep the lower block index).  A column
                // below the query's shared cut -- the largest K-th best of any
                // slice's full list, hence at most the final K-th best -- cannot
                // be kept; equal ones are, and the merge orders ties by index.
                if constexpr (KR <= 8) {
                  // columns above the cut, one bit each; then sorted insertion of
                  // each (select-shift over the register list, ties keeping the
                  // earlier column)
                  if (g == 0) {
                    float cut = fmaxf(theta, sm.cut[qi]);
                    if (bmax >= cut) {
                      uint32_t msk = 0;
#pragma unroll
                      for (int c = 0; c < 32; ++c) msk |= (pv[c] >= cut && pv[c] > theta) ? (1u << c) : 0u;
                      float* st = sm.stash[warp - 3] + (qi % (32 / G)) * 32;
#pragma unroll
                      for (int c = 0; c < 32; c += 4)
                        *reinterpret_cast<float4*>(st + c) = make_float4(pv[c], pv[c + 1], pv[c + 2], pv[c + 3]);
                      while (msk) {
                        const int c = __ffs(msk) - 1;
                        msk &= msk - 1;
                        const float x = st[c];
                        if (!(x > theta) || x < cut) continue;
                        bool ge[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) ge[i] = rl[i] >= x;
#pragma unroll
                        for (int i = 7; i >= 1; --i) {
                          rl[i] = ge[i] ? rl[i] : (ge[i - 1] ? x : rl[i - 1]);
                          ri[i] = ge[i] ? ri[i] : (ge[i - 1] ? cb + c : ri[i - 1]);
                        }
                        rl[0] = ge[0] ? rl[0] : x;
                        ri[0] = ge[0] ? ri[0] : cb + c;
                        if (cnt < K) ++cnt;
                        if (cnt == K) {
                          float kth = rl[0];
#pragma unroll
                          for (int i = 1; i < 8; ++i) kth = (i == K - 1) ? rl[i] : kth;
                          theta = kth;
                          cut = fmaxf(cut, theta);
                          atomicMax(reinterpret_cast<int*>(&sm.cut[qi]), __float_as_int(theta));
                        }
                      }
                    }
                  }
                } else {
                  if (g == 0) {
                    float cut = fmaxf(theta, sm.cut[qi]);
                    if (bmax >= cut) {
                      float* st = sm.stash[warp - 3] + (qi % (32 / G)) * 32;
#pragma unroll
                      for (int c = 0; c < 32; c += 4)
                        *reinterpret_cast<float4*>(st + c) = make_float4(pv[c], pv[c + 1], pv[c + 2], pv[c + 3]);
                      for (int c = 0; c < 32; ++c) {
                        const float pc = st[c];
                        if (pc < cut || (cnt == K && !(pc > theta))) continue;
                        int pos = cnt < K ? cnt : K - 1;
                        while (pos > 0 && ts[pos - 1] < pc) {
                          ts[pos] = ts[pos - 1];
                          tix[pos] = tix[pos - 1];
                          --pos;
                        }
                        ts[pos] = pc;
                        tix[pos] = cb + c;
                        if (cnt < K) ++cnt;
                        if (cnt == K) {
                          theta = ts[K - 1];
                          cut = fmaxf(cut, theta);
                          atomicMax(reinterpret_cast<int*>(&sm.cut[qi]), __float_as_int(theta));
                        }
                      }
                    }
                  }
                }
            
              }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&sm.tempty[acc]));
          }
          ++it;
        }
      }
      if (!ok) break;
      if constexpr (kLaneLists) {
        // the slice's best 8 of the query, from its G lanes' lists
#pragma unroll
        for (int o = 1; o < G; o <<= 1) flat_merge8_xor(rl, ri, o);
        if (g == 0) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            ts[i] = rl[i];
            tix[i] = ri[i];
          }
        }
      } else {
        if constexpr (KR <= 8) {
          if (g == 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              ts[i] = rl[i];
              tix[i] = ri[i];
            }
          }
        }
        if (g == 0) sm.top_n[sl][r] = cnt;
      }
      if (!rendezvous()) { ok = false; *abort = 1; break; }  // every slice's list is complete
      // output (slice-0 warps): the best K of the S sorted lists (ties to the
      // lower block index), ascending, together with F
      if constexpr (kLaneLists) {
        if (sl == 0) {  // warp-uniform
          // lane g takes slice g's list (S == G here); the G lanes merge them
          float ml[8];
          int32_t mi[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            ml[i] = sm.top_s[g][qi][i];
            mi[i] = sm.top_i[g][qi][i];
          }
#pragma unroll
          for (int o = 1; o < G; o <<= 1) flat_merge8_xor(ml, mi, o);
          // the best K (entries past K and empty ones sort last), block order
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (i >= K) {
              ml[i] = -INFINITY;
              mi[i] = -1;
            }
          flat_sort8_by_block(ml, mi);
          if (g == 0 && t < pr.N) {
            const int64_t qrow = bh * pr.N + t;
            int32_t* oi = out_idx + qrow * W;
            float* os = out_score ? out_score + qrow * W : nullptr;
            int pos = 0;
            oi[pos] = 0; if (os) os[pos] = INFINITY; ++pos;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (mi[i] >= 0) { oi[pos] = mi[i]; if (os) os[pos] = ml[i]; ++pos; }
            if (qb - 1 > 0) { oi[pos] = (int32_t)(qb - 1); if (os) os[pos] = INFINITY; ++pos; }
            if (qb > 0) { oi[pos] = (int32_t)qb; if (os) os[pos] = INFINITY; ++pos; }
            for (; pos < W; ++pos) { oi[pos] = -1; if (os) os[pos] = -INFINITY; }
          }
        }
      } else if (sl == 0 && g == 0 && t < pr.N) {
        float bs[kFCap];
        int32_t bi[kFCap];
        // lists (u, l): slice u, lane l of the query (one list per query
        // when LG = 1); entries at top_s[u][qi][8 l ...]
        int head[S * LG];
#pragma unroll
        for (int u = 0; u < S * LG; ++u) head[u] = 0;
        int n = 0;
        for (; n < K; ++n) {
          int bu = -1;
#pragma unroll
          for (int u = 0; u < S * LG; ++u) {
            const int us = u / LG, ul = u % LG;
            if (head[u] < sm.top_n[us][qi * G + ul]) {
              const float su = sm.top_s[us][qi][ul * 8 + head[u]];
              const int32_t iu = sm.top_i[us][qi][ul * 8 + head[u]];
              if (bu < 0 || su > bs[n] || (su == bs[n] && iu < bi[n])) {
                bu = u;
                bs[n] = su;
                bi[n] = iu;
              }
            }
          }
          if (bu < 0) break;
#pragma unroll
          for (int u = 0; u < S * LG; ++u) head[u] += (u == bu) ? 1 : 0;
        }
        // insertion sort of the kept entries by block index
        for (int u = 1; u < n; ++u) {
          const float sv = bs[u];
          const int32_t iv = bi[u];
          int w = u - 1;
          while (w >= 0 && bi[w] > iv) { bs[w + 1] = bs[w]; bi[w + 1] = bi[w]; --w; }
          bs[w + 1] = sv; bi[w + 1] = iv;
        }
        const int64_t qrow = bh * pr.N + t;
        int32_t* oi = out_idx + qrow * W;
        float* os = out_score ? out_score + qrow * W : nullptr;
        int pos = 0;
        oi[pos] = 0; if (os) os[pos] = INFINITY; ++pos;
        for (int u = 0; u < n; ++u) { oi[pos] = bi[u]; if (os) os[pos] = bs[u]; ++pos; }
        if (qb - 1 > 0) { oi[pos] = (int32_t)(qb - 1); if (os) os[pos] = INFINITY; ++pos; }
        if (qb > 0) { oi[pos] = (int32_t)qb; if (os) os[pos] = INFINITY; ++pos; }
        for (; pos < W; ++pos) { oi[pos] = -1; if (os) os[pos] = -INFINITY; }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, kFTmemCols);
  if (threadIdx.x == 0 && sm.abort) set_status(status, PISA_DEV_TIMEOUT);
}

template <int D, int G, int KR>
static cudaError_t launch_flat_t(const Prob& pr, int64_t nb, const void* q, const CUtensorMap& mumap, int32_t* out_idx,
                                 float* out_score, int32_t* status, int grid, cudaStream_t st) {
  const size_t smem = sizeof(FlatSmem<D, G>) + 1024;
  auto kern = flat_tc_kernel<D, G, KR>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  FlatTiles ft;
  ft.Qt = kFRows / G;
  ft.nqt = ceil_div64(pr.N, ft.Qt);
  note_launch();
  return launch_pdl(true, kern, dim3(grid), dim3(flat_threads<G>()), smem, st, pr, ft, nb, mumap, (const uint16_t*)q,
                    out_idx, out_score, status);
}

cudaError_t launch_flat(const Prob& pr, const Pyr& s, const void* q, const float* pyr, char* ws, int32_t* out_idx,
                        float* out_score, int num_sms, cudaStream_t st) {
  if (pr.dtype != PISA_BF16) return cudaErrorNotSupported;  // the comparator runs on bf16 inputs
  int32_t* status = (int32_t*)ws;
  __nv_bfloat16* mu = (__nv_bfloat16*)(ws + 256);
  const int64_t nbh = pr.B * pr.Hkv;
  const int64_t n = nbh * s.nb * pr.d;
  note_launch();
  cudaError_t e = launch_pdl(false, means_to_bf16_kernel, dim3((unsigned)std::min<int64_t>(ceil_div64(n, 256), 4096)),
                             dim3(256), 0, st, nbh, s.P, s.nb, pr.d, pyr, mu);
  if (e != cudaSuccess) return e;
  CUtensorMap mumap;
  if (!make_tmap_rows(&mumap, mu, nbh * s.nb, pr.d, kFCols)) return cudaErrorInvalidValue;
  const int grid = num_sms > 0 ? num_sms : 148;
#define PISA_FLAT_CASE(DD, GG) \
  if (pr.d == DD && pr.G == GG)                                                                           \
    return pr.K <= 8 ? launch_flat_t<DD, GG, 8>(pr, s.nb, q, mumap, out_idx, out_score, status, grid, st)  \
                     : launch_flat_t<DD, GG, kFCap>(pr, s.nb, q, mumap, out_idx, out_score, status, grid, st);
  PISA_FLAT_CASE(128, 1) PISA_FLAT_CASE(128, 2) PISA_FLAT_CASE(128, 4) PISA_FLAT_CASE(128, 8)
  PISA_FLAT_CASE(64, 1) PISA_FLAT_CASE(64, 2) PISA_FLAT_CASE(64, 4) PISA_FLAT_CASE(64, 8)
#undef PISA_FLAT_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pisa
