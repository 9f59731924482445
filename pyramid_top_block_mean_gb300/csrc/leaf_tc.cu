// leaf_tc.cu -- leaf LSE scoring on the tcgen05 tensor cores, and the final
// Top-K.  agihunt.info summary of "Block Sparse Attention with Log-Linear
// Complexity", kernel paragraph: stage 2 of prefill scores the leaves with
// LSE over their raw keys, grouping the queries that need the same leaf so
// each leaf key tile is loaded once (Qtile), without materialising a dense
// score matrix; rcap.io post, kernel paragraph (two-stage prefill).
//
// GB300 design.  A query's leaf candidates come in sibling pairs: the two
// leaves under each kept level-2 node.  Pairs (query, kept level-2 node p)
// are counting-sorted by (sequence, key head, query chunk, p).  One tile is
// 128 rows = 128/G queries x G heads of one bucket against the 128 keys of
// leaves 2p and 2p+1:
//   - a loader warp brings the 128 x d bf16 key tile into shared memory by
//     TMA (128-byte swizzle) once per run of consecutive tiles with the same
//     key tile, up to three key tiles ahead;
//   - eight producer warps gather the 128 query-head rows (16 each) with
//     cp.async into the same swizzled K-major layout (TMA four-row gathers
//     measured 2.3x slower for these 256-byte rows: one TMA operation per
//     512 bytes);
//   - one thread issues tcgen05.mma (M = 128, N = 128, K = d) into a TMEM
//     accumulator (four accumulators rotate);
//   - eight epilogue warps (two per TMEM lane quadrant, one per leaf) read
//     their 32 lanes x 64 columns, take the per-row log2-sum-exp2 over the
//     leaf's keys, sum the G head rows of a query, and write one score per
//     (query, leaf).  No score matrix reaches HBM.
// Persistent CTAs (one per SM) walk the tile list in interleaved groups of
// four consecutive tiles, so all SMs sweep the same query chunk together.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "pisa_common.cuh"
#include "pisa_internal.h"
#include "tc_ptx.cuh"

namespace pisa {

constexpr int kTileRows = 128;  // MMA M: queries x heads
constexpr int kTileKeys = 128;  // MMA N: leaves 2p and 2p+1
constexpr int kStagesA = 4;  // query-row tiles in flight
constexpr int kStagesB = 3;  // key tiles
constexpr int kAcc = 4;      // TMEM accumulators (4 x 128 columns)
static_assert(kAcc == kStagesA, "a query-row stage is released by its tile's accumulator barrier");
constexpr int kGroup = 4;
constexpr int kProdWarps = 8;          // warps 0-7 gather 16 query-head rows each
constexpr int kProdRows = kTileRows / kProdWarps;
constexpr int kLoadWarp = kProdWarps;  // loads the key tiles (TMA)
constexpr int kMmaWarp = kLoadWarp + 1;  // issues the MMAs, owns TMEM
constexpr int kEpiWarps = 8;             // the next 8 warps: (TMEM lane quadrant, leaf)
constexpr int kLeafTcThreads = 32 * (kMmaWarp + 1 + kEpiWarps);
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 4000000000ull;

// Host-side fault injection for tests of the bounded waits
// (pisa_test_inject_leaf_timeout): a shorter wait limit, and whether CTA 0
// announces its first key tile on the stage barrier without issuing the copy,
// so that the first MMA wait can only run out.  Zero means the defaults.
std::atomic<uint64_t> g_test_wait_ns{0};
std::atomic<int32_t> g_test_drop_tile{0};

struct LeafWaits {
  uint64_t limit_ns;
  int32_t drop_first_tile;
};

template <int D>
struct LeafTcSmem {
  uint8_t a[kStagesA][kTileRows * D * 2];
  uint8_t b[kStagesB][kTileKeys * D * 2];
  uint64_t full_a[kStagesA], full_b[kStagesB], empty_b[kStagesB];
  uint64_t tfull[kAcc], tempty[kAcc], done;
  uint32_t tmem_base;
  int32_t abort;
  int32_t zero;  // stays 0: a wait that must not give up early on abort
};

// ---------------------------------------------------------------- bucketing
struct BucketArgs {
  int64_t nq, N, n2, nchunk;
  int32_t K;      // entries per query
  int32_t shift;  // a pair is (t << shift) | slot, read as uint32
  int32_t dedup;  // skip an entry equal to an earlier one of its query
};

// Does entry `slot` of a query's row count: in [0, n2) and, with dedup, not
// equal to an earlier entry of the row?
__device__ __forceinline__ bool entry_counts(const BucketArgs& a, const int32_t* row, int slot, int32_t p) {
  if (p < 0 || p >= a.n2) return false;
  if (a.dedup)
    for (int u = 0; u < slot; ++u)
      if (row[u] == p) return false;
  return true;
}

__device__ __forceinline__ int32_t encode_pair(const BucketArgs& a, int64_t t, int64_t slot) {
  return (int32_t)(((uint32_t)t << a.shift) | (uint32_t)slot);
}

__device__ __forceinline__ int64_t bucket_of(const BucketArgs& a, int64_t qi, int32_t p) {
  const int64_t t = qi % a.N, bh = qi / a.N;
  return ((bh * a.nchunk) + (t >> kChunkShift)) * a.n2 + p;
}

__global__ void count_kernel(BucketArgs a, const int32_t* __restrict__ kept2, int32_t* __restrict__ counts) {
  pdl_wait();
  const int64_t n = a.nq * a.K;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t p = kept2[i];
    const int64_t qi = i / a.K;
    const int slot = (int)(i - qi * a.K);
    if (entry_counts(a, kept2 + qi * a.K, slot, p)) atomicAdd(&counts[bucket_of(a, qi, p)], 1);
  }
}

// Shared-memory histogram versions for n2 <= kSmemBins level-2 nodes: one CTA
// per kQueriesPerCta query positions of one (sequence, key head); the range
// never crosses a query chunk, so a bucket is (CTA's chunk, node p).
constexpr int kQueriesPerCta = 2048;
constexpr int kSmemBins = 16384;
static_assert(((1 << kChunkShift) % kQueriesPerCta) == 0, "a CTA's queries stay in one chunk");

// Histogram pass over a CTA's ne entries (thread t of kBucketThreads takes
// entries t + kBucketThreads j):
// the entries of a chunk are loaded into registers first, so a thread keeps
// 32 loads in flight instead of one per shared-memory atomic.  f(e, p) is
// called for every entry e < ne with its node p.
constexpr int kEntryChunk = 32;
constexpr int kBucketThreads = 512;  // threads of the shared-memory histogram kernels
template <class F>
__device__ __forceinline__ void for_entry_chunks(const int32_t* __restrict__ src, int ne, F&& f) {
  for (int e0 = 0; e0 < ne; e0 += kBucketThreads * kEntryChunk) {
    int32_t pv[kEntryChunk];
#pragma unroll
    for (int j = 0; j < kEntryChunk; ++j) {
      const int e = e0 + (int)threadIdx.x + kBucketThreads * j;
      pv[j] = e < ne ? src[e] : -1;
    }
#pragma unroll
    for (int j = 0; j < kEntryChunk; ++j) {
      const int e = e0 + (int)threadIdx.x + kBucketThreads * j;
      if (e < ne) f(e, pv[j]);
    }
  }
}

__global__ void __launch_bounds__(kBucketThreads) count_smem_kernel(BucketArgs a, const int32_t* __restrict__ kept2,
                                                        int32_t* __restrict__ counts) {
  pdl_wait();
  extern __shared__ int32_t hist[];
  const int n2 = (int)a.n2, K = a.K;
  const int64_t bh = blockIdx.y, t0 = (int64_t)blockIdx.x * kQueriesPerCta;
  const int ne = (int)(a.N - t0 < kQueriesPerCta ? a.N - t0 : kQueriesPerCta) * K;
  for (int i = threadIdx.x; i < n2; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int32_t* src = kept2 + (bh * a.N + t0) * K;
  for_entry_chunks(src, ne, [&](int e, int32_t p) {
    const int qn = e / K;
    if (entry_counts(a, src + qn * K, e - qn * K, p)) atomicAdd(&hist[p], 1);
  });
  __syncthreads();
  int32_t* dst = counts + (bh * a.nchunk + (t0 >> kChunkShift)) * a.n2;
  for (int i = threadIdx.x; i < n2; i += blockDim.x)
    if (hist[i]) atomicAdd(&dst[i], hist[i]);
}

__global__ void __launch_bounds__(kBucketThreads) scatter_smem_kernel(BucketArgs a, const int32_t* __restrict__ kept2,
                                                          const int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ cursor, int32_t* __restrict__ pairs) {
  pdl_wait();
  extern __shared__ int32_t hist[];
  const int n2 = (int)a.n2, K = a.K;
  const int64_t bh = blockIdx.y, t0 = (int64_t)blockIdx.x * kQueriesPerCta;
  const int ne = (int)(a.N - t0 < kQueriesPerCta ? a.N - t0 : kQueriesPerCta) * K;
  for (int i = threadIdx.x; i < n2; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int32_t* src = kept2 + (bh * a.N + t0) * K;
  for_entry_chunks(src, ne, [&](int e, int32_t p) {
    const int qn = e / K;
    if (entry_counts(a, src + qn * K, e - qn * K, p)) atomicAdd(&hist[p], 1);
  });
  __syncthreads();
  // reserve this CTA's range in every bucket it touches
  const int64_t b0 = (bh * a.nchunk + (t0 >> kChunkShift)) * a.n2;
  for (int i = threadIdx.x; i < n2; i += blockDim.x) {
    const int32_t c = hist[i];
    if (c) hist[i] = offsets[b0 + i] + atomicAdd(&cursor[b0 + i], c);
  }
  __syncthreads();
  for_entry_chunks(src, ne, [&](int e, int32_t p) {
    const int qn = e / K;
    if (entry_counts(a, src + qn * K, e - qn * K, p)) pairs[atomicAdd(&hist[p], 1)] = encode_pair(a, t0 + qn, e - qn * K);
  });
}

// Exclusive scans of the pair counts and of the tiles per bucket (one CTA),
// in rounds of 1024 x 32 buckets (one round up to 32768 buckets): each thread
// takes 32 consecutive buckets with 16-byte loads and stores, warp-shuffle
// scans combine the thread sums, and a carry runs between rounds.  Q (rows
// per tile / G) is a power of two.
constexpr int kScanPer = 32;
__global__ void __launch_bounds__(1024) scan_kernel(int64_t nb, int32_t Q, const int32_t* __restrict__ counts,
                                                    int32_t* __restrict__ offsets, int32_t* __restrict__ tile_off) {
  pdl_wait();
  __shared__ int32_t wp[32], wt[32];
  __shared__ int32_t carry[2];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int qs = __ffs(Q) - 1;
  if (tid == 0) { carry[0] = 0; carry[1] = 0; }
  __syncthreads();
  for (int64_t base = 0; base < nb; base += 1024 * kScanPer) {
    const int64_t b0 = base + (int64_t)tid * kScanPer;
    // a whole run in range is 128-byte aligned (the arrays start 256-byte
    // aligned); the counts are read twice (sums, then offsets) rather than
    // held across the block scan
    const bool whole = b0 + kScanPer <= nb;
    int32_t sp = 0, st = 0;
    if (whole) {
#pragma unroll
      for (int j = 0; j < kScanPer / 4; ++j) {
        const int4 v = reinterpret_cast<const int4*>(counts + b0)[j];
        sp += (v.x + v.y) + (v.z + v.w);
        st += (((v.x + Q - 1) >> qs) + ((v.y + Q - 1) >> qs)) + (((v.z + Q - 1) >> qs) + ((v.w + Q - 1) >> qs));
      }
    } else {
      for (int j = 0; j < kScanPer; ++j) {
        const int32_t c = b0 + j < nb ? counts[b0 + j] : 0;
        sp += c;
        st += (c + Q - 1) >> qs;
      }
    }
    // inclusive warp scans of the thread sums, then of the warp totals
    int32_t ip = sp, it = st;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t x = __shfl_up_sync(0xffffffffu, ip, o), y = __shfl_up_sync(0xffffffffu, it, o);
      if (lane >= o) { ip += x; it += y; }
    }
    if (lane == 31) { wp[wid] = ip; wt[wid] = it; }
    __syncthreads();
    if (wid == 0) {
      int32_t x = wp[lane], y = wt[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t xx = __shfl_up_sync(0xffffffffu, x, o), yy = __shfl_up_sync(0xffffffffu, y, o);
        if (lane >= o) { x += xx; y += yy; }
      }
      wp[lane] = x - wp[lane];  // exclusive warp offsets
      wt[lane] = y - wt[lane];
    }
    __syncthreads();
    int32_t op = carry[0] + wp[wid] + (ip - sp), ot = carry[1] + wt[wid] + (it - st);
    if (whole) {
#pragma unroll
      for (int j = 0; j < kScanPer / 4; ++j) {
        const int4 v = reinterpret_cast<const int4*>(counts + b0)[j];
        int4 vo, vt;
        vo.x = op; vt.x = ot; op += v.x; ot += (v.x + Q - 1) >> qs;
        vo.y = op; vt.y = ot; op += v.y; ot += (v.y + Q - 1) >> qs;
        vo.z = op; vt.z = ot; op += v.z; ot += (v.z + Q - 1) >> qs;
        vo.w = op; vt.w = ot; op += v.w; ot += (v.w + Q - 1) >> qs;
        reinterpret_cast<int4*>(offsets + b0)[j] = vo;
        reinterpret_cast<int4*>(tile_off + b0)[j] = vt;
      }
    } else {
      for (int j = 0; j < kScanPer; ++j) {
        const int32_t c = b0 + j < nb ? counts[b0 + j] : 0;
        if (b0 + j < nb) { offsets[b0 + j] = op; tile_off[b0 + j] = ot; }
        op += c;
        ot += (c + Q - 1) >> qs;
      }
    }
    __syncthreads();  // every thread has read carry and the warp offsets
    if (tid == 1023) { carry[0] = op; carry[1] = ot; }
    __syncthreads();
  }
  if (tid == 0) { offsets[nb] = carry[0]; tile_off[nb] = carry[1]; }
}

__global__ void scatter_kernel(BucketArgs a, const int32_t* __restrict__ kept2, const int32_t* __restrict__ offsets,
                               int32_t* __restrict__ cursor, int32_t* __restrict__ pairs) {
  pdl_wait();
  const int64_t n = a.nq * a.K;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t p = kept2[i];
    const int64_t qi = i / a.K;
    if (!entry_counts(a, kept2 + qi * a.K, (int)(i - qi * a.K), p)) continue;
    const int64_t bk = bucket_of(a, qi, p);
    const int32_t pos = offsets[bk] + atomicAdd(&cursor[bk], 1);
    pairs[pos] = encode_pair(a, qi % a.N, i % a.K);
  }
}

// Tile descriptor: {sequence x key head bh, first pair, pair count, level-2 node}.
__global__ void tiles_kernel(int64_t nb, int64_t n2, int64_t nchunk, int32_t Q, const int32_t* __restrict__ counts,
                             const int32_t* __restrict__ offsets, const int32_t* __restrict__ tile_off,
                             int4* __restrict__ tile_info) {
  pdl_wait();
  for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < nb; j += (int64_t)gridDim.x * blockDim.x) {
    const int32_t n = counts[j], t0 = tile_off[j], p0 = offsets[j];
    const int32_t bh = (int32_t)((j / n2) / nchunk), node = (int32_t)(j % n2);
    for (int32_t i = 0; i * Q < n; ++i) tile_info[t0 + i] = make_int4(bh, p0 + i * Q, min(Q, n - i * Q), node);
  }
}

// ------------------------------------------------------------ tile schedule
struct TileIter {
  int T, i, gend, g;
  __device__ TileIter(int total) : T(total), g(blockIdx.x) {
    i = g * kGroup;
    gend = min(T, i + kGroup);
  }
  __device__ bool valid() const { return i < T; }
  __device__ void next() {
    if (++i >= gend) {
      g += gridDim.x;
      i = g * kGroup;
      gend = min(T, i + kGroup);
    }
  }
  __device__ int peek() const {  // the tile after this one, or -1
    if (i + 1 < gend) return i + 1;
    const int j = (g + (int)gridDim.x) * kGroup;
    return j < T ? j : -1;
  }
};

// Every wait of the leaf kernel passes a suspend-time hint (20 us); measured
// with the packed epilogue arithmetic at 262144 tokens: 1.75 against 1.78 ms
// (either change alone was slower).
constexpr uint32_t kLeafWaitHintNs = 20000;
__device__ __forceinline__ bool leaf_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort, uint64_t limit_ns) {
  return ptx::mbar_wait_bounded_hint(bar, parity, abort, limit_ns, kLeafWaitHintNs);
}

template <int D, int G>
__global__ void __launch_bounds__(kLeafTcThreads, 1)
    leaf_tc_kernel(Prob pr, const __grid_constant__ CUtensorMap kmap,
                   const uint16_t* __restrict__ q, const int4* __restrict__ tile_info,
                   const int32_t* __restrict__ tile_total, const int32_t* __restrict__ pairs,
                   float* __restrict__ leaf_score, int32_t* __restrict__ status, LeafWaits waits) {
  pdl_wait();
  const uint64_t kWaitLimitNs = waits.limit_ns;  // shadows the default: every wait below is bounded by it
  extern __shared__ unsigned char smem_raw[];
  LeafTcSmem<D>& sm = *reinterpret_cast<LeafTcSmem<D>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr int kHalf = kTileRows * 128;  // bytes of one 64-element K slice
  constexpr uint32_t kBBytes = kTileKeys * D * 2;
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kTileRows, kTileKeys);
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  volatile int32_t* abort = &sm.abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesA; ++s) {
      ptx::mbar_init(ptx::smem_u32(&sm.full_a[s]), 32 * kProdWarps);
    }
    for (int s = 0; s < kStagesB; ++s) {
      ptx::mbar_init(ptx::smem_u32(&sm.full_b[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&sm.empty_b[s]), 1);
    }
    for (int s = 0; s < kAcc; ++s) {
      ptx::mbar_init(ptx::smem_u32(&sm.tfull[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&sm.tempty[s]), kEpiWarps);
    }
    ptx::mbar_init(ptx::smem_u32(&sm.done), 1);
    sm.abort = 0;
    sm.zero = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(&sm.tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int T = *tile_total;

  if (warp < kProdWarps) {
    // ------------------------------------------------------------ producers
    // warp w gathers rows [16w, 16w + 16) of every tile with cp.async
    constexpr int CPR = D / 8;     // 16-byte chunks per row
    constexpr int RPI = 32 / CPR;  // rows per warp instruction
    constexpr int QPW = kProdRows / G;  // queries per producer warp
    const int4 kNoTile = make_int4(-1, 0, 0, 0);
    const int ch = lane % CPR;
    const int row0 = warp * kProdRows, qbase = row0 / G;
    int it = 0;
    bool ok = true;
    // When G >= RPI, the rows of one copy instruction belong to one query and
    // lane row hi = lane / CPR is head (r0 % G) + hi: every lane keeps the
    // warp's QPW query positions in registers and the row address is a few
    // integer operations (no shuffles).  Otherwise the positions are
    // broadcast from the lane that loaded them.
    constexpr bool kFast = G >= RPI && G % RPI == 0;
    constexpr int NT = kFast ? QPW : 1;  // query positions kept per lane
    const int hi = lane / CPR;
    const int64_t ND = pr.N * D;
    const uint32_t dlane = (ch >> 3) * kHalf + (row0 + hi) * 128;
    const int xl = (ch & 7) ^ hi;  // swizzle term for row r: (ch & 7) ^ (r & 7), r & 7 = (r0 & 7) + hi
    auto positions = [&](const int4& inf, int32_t (&tq)[NT]) {
      if constexpr (kFast) {
#pragma unroll
        for (int j = 0; j < QPW; ++j)
          tq[j] = (inf.x >= 0 && qbase + j < inf.z) ? (pairs[inf.y + qbase + j] >> 5) : 0;
      } else {
        tq[0] = (inf.x >= 0 && lane < QPW && qbase + lane < inf.z) ? (pairs[inf.y + qbase + lane] >> 5) : 0;
      }
    };
    // Descriptors run two tiles ahead and query positions one tile ahead.
    // The loop is unrolled three times over rotating slots, so a prefetched
    // value is never copied between registers (which would wait for it).
    TileIter ti(T), ahead(T);
    if (ahead.valid()) ahead.next();
    int4 d0 = ti.valid() ? tile_info[ti.i] : kNoTile;
    int4 d1 = ahead.valid() ? tile_info[ahead.i] : kNoTile, d2;
    int32_t v0[NT], v1[NT], v2[NT];
    positions(d0, v0);
    auto step = [&](const int4& info, const int4& info1, int4& slot2, const int32_t (&tq)[NT],
                    int32_t (&slot1)[NT]) -> bool {
      if (!ti.valid()) return false;
      if (ahead.valid()) ahead.next();
      slot2 = ahead.valid() ? tile_info[ahead.i] : kNoTile;  // tile it + 2
      const int bh = info.x;
      const int b = bh / (int)pr.Hkv, h = bh - b * (int)pr.Hkv;
      const int sa = it % kStagesA, use = it / kStagesA;
      // the stage is free once the MMAs of its previous tile have completed,
      // which is when that tile's accumulator is announced full (one stage per
      // accumulator)
      ok = leaf_wait(ptx::smem_u32(&sm.tfull[sa]), (use & 1) ^ 1, abort, kWaitLimitNs);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; return false; }
      // gather this warp's query-head rows
      const uint32_t abase = ptx::smem_u32(sm.a[sa]) + dlane;
      const int cnt = info.z;
      if constexpr (kFast) {
        const uint16_t* qh = q + ((int64_t)b * pr.Hq + h * G + hi) * ND + ch * 8;  // head hi of the group
#pragma unroll
        for (int r0 = 0; r0 < kProdRows; r0 += RPI) {
          if (qbase + r0 / G < cnt) {
            const uint16_t* src = qh + (r0 % G) * ND + (int64_t)tq[r0 / G] * D;
            ptx::cp_async_16(abase + r0 * 128 + ((xl ^ (r0 & 7)) << 4), src);
          }
        }
      } else {
#pragma unroll
        for (int r0 = 0; r0 < kProdRows; r0 += RPI) {
          const int rl = r0 + hi;
          const int r = row0 + rl;
          const int64_t t = __shfl_sync(0xffffffffu, tq[0], rl / G);
          if (qbase + rl / G < cnt) {
            const int g = r % G;
            const uint16_t* src = q + ((((int64_t)b * pr.Hq + h * G + g) * pr.N + t) * D + ch * 8);
            ptx::cp_async_16(abase + r0 * 128 + (((ch & 7) ^ (r & 7)) << 4), src);
          }
        }
      }
      // the stage's barrier counts this thread once its copies have landed
      ptx::cp_async_arrive_noinc(ptx::smem_u32(&sm.full_a[sa]));
      // query positions of tile it + 1 (its descriptor arrived a tile ago)
      positions(info1, slot1);
      ++it;
      ti.next();
      return true;
    };
    while (step(d0, d1, d2, v0, v1) && step(d1, d2, d0, v1, v2) && step(d2, d0, d1, v2, v0)) {
    }
    ptx::cp_async_wait_all();  // no copy may still target this CTA's memory when it exits
    if (!ok) *abort = 1;
  } else if (warp == kLoadWarp) {
    // ------------------------------------------------------- key-tile loads
    // one TMA load of the 128 x d keys of leaves 2p, 2p+1 per run of tiles
    // with the same (bh, p); it runs up to kStagesB key tiles ahead
    if (lane == 0) {
      int bcount = 0, last_bh = -1, last_p = -1;
      bool ok = true;
      const int4 kNone = make_int4(-1, 0, 0, 0);
      TileIter ti(T), ahead(T);
      if (ahead.valid()) ahead.next();
      int4 info = ti.valid() ? tile_info[ti.i] : kNone;
      int4 info1 = ahead.valid() ? tile_info[ahead.i] : kNone;
      for (; ti.valid(); ti.next()) {
        if (ahead.valid()) ahead.next();
        const int4 info2 = ahead.valid() ? tile_info[ahead.i] : kNone;
        const int bh = info.x, p = info.w;
        if (bh != last_bh || p != last_p) {
          const int sb = bcount % kStagesB, ub = bcount / kStagesB;
          ok = leaf_wait(ptx::smem_u32(&sm.empty_b[sb]), (ub & 1) ^ 1, abort, kWaitLimitNs);
          if (!ok) break;
          const uint32_t fb = ptx::smem_u32(&sm.full_b[sb]);
          ptx::mbar_arrive_expect_tx(fb, kBBytes);
          const int32_t y = (int32_t)(bh * pr.N + 128 * (int64_t)p);
          // injected fault (tests only): the first tile is announced, never copied
          const bool drop = waits.drop_first_tile && blockIdx.x == 0 && bcount == 0;
          if (!drop)
#pragma unroll
            for (int hh = 0; hh < D / 64; ++hh)
              ptx::tma_load_2d(ptx::smem_u32(sm.b[sb]) + hh * kHalf, &kmap, 64 * hh, y, fb);
          ++bcount;
          last_bh = bh;
          last_p = p;
        }
        info = info1;
        info1 = info2;
      }
      if (!ok) *abort = 1;
      // let every TMA load issued land before the CTA can exit, whoever gave
      // up (the MMA thread may abort while loads it will never consume are in
      // flight); after a normal run these phases have completed already
      for (int k = bcount > kStagesB ? bcount - kStagesB : 0; k < bcount; ++k)
        leaf_wait(ptx::smem_u32(&sm.full_b[k % kStagesB]), (k / kStagesB) & 1, &sm.zero,
                               kWaitLimitNs);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      int it = 0, bcount = 0, last_bh = -1, last_p = -1, sb = 0;
      bool ok = true;
      // descriptors four tiles ahead (five rotating slots: a prefetched value
      // is never copied between registers, which would wait for it)
      const int4 kNoTile = make_int4(-1, 0, 0, 0);
      TileIter ti(T), ahead(T);
      int4 d0 = ti.valid() ? tile_info[ti.i] : kNoTile, d1, d2, d3, d4;
      if (ahead.valid()) ahead.next();
      d1 = ahead.valid() ? tile_info[ahead.i] : kNoTile;
      if (ahead.valid()) ahead.next();
      d2 = ahead.valid() ? tile_info[ahead.i] : kNoTile;
      if (ahead.valid()) ahead.next();
      d3 = ahead.valid() ? tile_info[ahead.i] : kNoTile;
      auto step = [&](const int4& info, const int4& ninfo, int4& slot4) -> bool {
        if (!ti.valid()) return false;
        if (ahead.valid()) ahead.next();
        slot4 = ahead.valid() ? tile_info[ahead.i] : kNoTile;
        const int sa = it % kStagesA, use = it / kStagesA;
        const int acc = it % kAcc, uacc = it / kAcc;
        if (info.x != last_bh || info.w != last_p) {
          sb = bcount % kStagesB;
          ok = leaf_wait(ptx::smem_u32(&sm.full_b[sb]), (bcount / kStagesB) & 1, abort, kWaitLimitNs);
          if (!ok) return false;
          ++bcount;
          last_bh = info.x;
          last_p = info.w;
        }
        ok = leaf_wait(ptx::smem_u32(&sm.full_a[sa]), use & 1, abort, kWaitLimitNs) &&
             leaf_wait(ptx::smem_u32(&sm.tempty[acc]), (uacc & 1) ^ 1, abort, kWaitLimitNs);
        if (!ok) return false;
        // the rows arrived through cp.async (generic proxy); the MMA reads
        // them through the async proxy
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_after();
        const uint32_t d = tmem + acc * kTileKeys;
        const uint32_t a0 = ptx::smem_u32(sm.a[sa]), b0 = ptx::smem_u32(sm.b[sb]);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * kHalf + (k & 3) * 32;
          ptx::mma_bf16(d, ptx::desc_sw128(a0 + off), ptx::desc_sw128(b0 + off), kIdesc, k > 0 ? 1u : 0u);
        }
        ptx::mma_commit(ptx::smem_u32(&sm.tfull[acc]));
        if (ninfo.x != info.x || ninfo.w != info.w) ptx::mma_commit(ptx::smem_u32(&sm.empty_b[sb]));
        ++it;
        ti.next();
        return true;
      };
      while (step(d0, d1, d4) && step(d1, d2, d0) && step(d2, d3, d1) && step(d3, d4, d2) && step(d4, d0, d3)) {
      }
      if (!ok) *abort = 1;
      // every MMA has finished before TMEM is released
      ptx::mma_commit(ptx::smem_u32(&sm.done));
      leaf_wait(ptx::smem_u32(&sm.done), 0, &sm.zero, kWaitLimitNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // warp -> (TMEM lane quadrant warp % 4, leaf): 32 rows x 64 key columns
    const int q4 = warp & 3;
    const int leaf = (warp - (kMmaWarp + 1)) / 4;
    const int r = q4 * 32 + lane;
    const float sc = pr.scale2;
    int it = 0;
    // this tile's descriptor and pair come from the previous iteration
    const int qr = r / G;
    TileIter ti(T);
    int4 info = ti.valid() ? tile_info[ti.i] : make_int4(-1, 0, 0, 0);
    int32_t pe = (ti.valid() && qr < info.z) ? pairs[info.y + qr] : 0;
    for (; ti.valid(); ti.next()) {
      const int nx = ti.peek();
      const int4 ninfo = nx >= 0 ? tile_info[nx] : make_int4(-1, 0, 0, 0);
      const int acc = it % kAcc, use = it / kAcc;
      const bool okw = leaf_wait(ptx::smem_u32(&sm.tfull[acc]), use & 1, abort, kWaitLimitNs);
      if (!__all_sync(0xffffffffu, okw)) { *abort = 1; break; }
      ptx::tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(q4 * 32) << 16) + acc * kTileKeys + leaf * 64;
      uint32_t v0[32], v1[32];
      ptx::tmem_ld32(taddr, v0);
      ptx::tmem_ld32(taddr + 32, v1);
      ptx::tmem_ld_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&sm.tempty[acc]));
      const int32_t npe = (ninfo.x >= 0 && qr < ninfo.z) ? pairs[ninfo.y + qr] : 0;
      // raw dots; the scale (> 0) is applied inside the exponent's FMA
      float x[64];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        x[j] = __uint_as_float(v0[j]);
        x[32 + j] = __uint_as_float(v1[j]);
      }
      float lse;
      if (pr.scorer == PISA_SCORER_LSE) {
        // Three-input maxima (a tree of 32) and packed fp32x2 exponent
        // arguments and sums: 160 instructions a row instead of 256.
        float t[22];
#pragma unroll
        for (int j = 0; j < 21; ++j) t[j] = ptx::max3(x[3 * j], x[3 * j + 1], x[3 * j + 2]);
        t[21] = x[63];
        float u[8];
#pragma unroll
        for (int j = 0; j < 7; ++j) u[j] = ptx::max3(t[3 * j], t[3 * j + 1], t[3 * j + 2]);
        u[7] = t[21];
        const float m = ptx::max3(ptx::max3(u[0], u[1], u[2]), ptx::max3(u[3], u[4], u[5]), fmaxf(u[6], u[7])) * sc;
        const uint64_t sc2 = ptx::pack2(sc, sc), nm2 = ptx::pack2(-m, -m);
        uint64_t ss2[4] = {0ull, 0ull, 0ull, 0ull};  // packed (+0, +0)
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float a0, a1;
          ptx::unpack2(ptx::fma2(ptx::pack2(x[2 * j], x[2 * j + 1]), sc2, nm2), a0, a1);
          ss2[j & 3] = ptx::add2(ss2[j & 3], ptx::pack2(ptx::ex2(a0), ptx::ex2(a1)));
        }
        const uint64_t s2 = ptx::add2(ptx::add2(ss2[0], ss2[1]), ptx::add2(ss2[2], ss2[3]));
        float s0, s1;
        ptx::unpack2(s2, s0, s1);
        lse = m + ptx::lg2(s0 + s1);
      } else {
        // PISA-1 / PISA-2: mean and centred second moment of the 64 dots
        float s1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int j = 0; j < 64; ++j) s1[j & 3] += x[j];
        const float mean = ((s1[0] + s1[1]) + (s1[2] + s1[3])) * (1.0f / 64.0f);
        float s2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int j = 0; j < 64; ++j) s2[j & 3] = fmaf(x[j] - mean, x[j] - mean, s2[j & 3]);
        lse = moment_score(pr.scorer, 64.0f, mean * sc, ((s2[0] + s2[1]) + (s2[2] + s2[3])) * (sc * sc));
      }
#pragma unroll
      for (int o = 1; o < G; o <<= 1) lse += __shfl_xor_sync(0xffffffffu, lse, o);
      if ((r % G) == 0 && qr < info.z) {
        const int64_t bh = info.x;
        const int64_t t = pe >> 5, slot = pe & 31;
        leaf_score[((bh * pr.N + t) * pr.K + slot) * 2 + leaf] = lse;
      }
      info = ninfo;
      pe = npe;
      ++it;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0 && sm.abort) set_status(status, PISA_DEV_TIMEOUT);
}

// -------------------------------------------------------------- finalize
// One warp per query: Top-K of its eligible candidate leaves (group LSE,
// ties to the lower index) together with the forced blocks, ascending.
__global__ void __launch_bounds__(256) finalize_kernel(Prob pr, const int32_t* __restrict__ kept2,
                                                       const float* __restrict__ leaf_score,
                                                       int32_t* __restrict__ out_idx, float* __restrict__ out_score) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t qi = (int64_t)blockIdx.x * 8 + threadIdx.x / 32;
  if (qi >= pr.B * pr.Hkv * pr.N) return;
  const int64_t t = qi % pr.N;
  const int64_t qb = t / pr.C;
  const int K = pr.K, W = K + 3, nc = 2 * K;
  float sc[2];
  int32_t lf[2];
  bool val[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int c = lane + 32 * j;
    val[j] = false; sc[j] = -INFINITY; lf[j] = -1;
    if (c < nc) {
      const int32_t p = kept2[qi * K + (c >> 1)];
      if (p >= 0) {
        lf[j] = 2 * p + (c & 1);
        val[j] = node_eligible(1, lf[j], qb);
        if (val[j]) {
          const float v = leaf_score[(qi * K + (c >> 1)) * 2 + (c & 1)];
          sc[j] = v != v ? -INFINITY : v;  // NaN ranks as -inf
        }
      }
    }
  }
  int rank[2] = {0, 0};
  const int rounds = nc > 32 ? 2 : 1;
  for (int jr = 0; jr < rounds; ++jr) {
    for (int src = 0; src < 32; ++src) {
      const float so = __shfl_sync(0xffffffffu, sc[jr], src);
      const int32_t lo = __shfl_sync(0xffffffffu, lf[jr], src);
      const bool vo = __shfl_sync(0xffffffffu, val[jr] ? 1 : 0, src) != 0;
      if (!vo) continue;
#pragma unroll
      for (int j = 0; j < 2; ++j)
        if (val[j] && beats(so, lo, sc[j], lf[j])) ++rank[j];
    }
  }
  int32_t* oi = out_idx + qi * W;
  float* os = out_score ? out_score + qi * W : nullptr;
  int nkept = 0;
  for (int j = 0; j < rounds; ++j) {
    const bool keep = val[j] && rank[j] < K;
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    const int pos = 1 + nkept + __popc(bal & ((1u << lane) - 1));
    if (keep && pos <= K) {  // the ranking order is total: at most K are kept
      oi[pos] = lf[j];
      if (os) os[pos] = sc[j] * kLn2;
    }
    nkept += __popc(bal);
  }
  if (lane == 0) {
    oi[0] = 0;
    if (os) os[0] = INFINITY;
    int pos = 1 + nkept;
    if (qb - 1 > 0) { oi[pos] = (int32_t)(qb - 1); if (os) os[pos] = INFINITY; ++pos; }
    if (qb > 0) { oi[pos] = (int32_t)qb; if (os) os[pos] = INFINITY; ++pos; }
    for (; pos < W; ++pos) { oi[pos] = -1; if (os) os[pos] = -INFINITY; }
  }
}

// One thread per query for K <= 8: the <= 16 candidates are ranked in
// registers (the loads and stores of consecutive threads are contiguous).
__global__ void __launch_bounds__(256, 1) finalize_small_kernel(Prob pr, const int32_t* __restrict__ kept2,
                                                             const float* __restrict__ leaf_score,
                                                             int32_t* __restrict__ out_idx,
                                                             float* __restrict__ out_score) {
  pdl_wait();
  constexpr int KM = 8, NCM = 2 * KM, WM = KM + 3;
  // each thread builds its row in shared memory; the block then writes its
  // rows out contiguously
  __shared__ int32_t si[256 * WM];
  __shared__ float ss[256 * WM];
  const int64_t nq = pr.B * pr.Hkv * pr.N;
  const int64_t q0 = (int64_t)blockIdx.x * blockDim.x;
  const int64_t qi = q0 + threadIdx.x;
  const int K = pr.K, W = K + 3;
  if (qi < nq) {
    // pair counts are below 2^31, so query indices fit 32 bits
    const uint32_t t = (uint32_t)qi % (uint32_t)pr.N;
    const int32_t qb = (int32_t)(t / (uint32_t)pr.C);
    float sc[NCM];
    int32_t lf[NCM];
    bool val[NCM];
    // K = 8: the query's nodes and leaf scores are two and four aligned
    // 16-byte vectors (rows of 32 and 64 bytes)
    int32_t pv[KM];
    float rv[NCM];
    if (K == KM) {
      const int4* kp = reinterpret_cast<const int4*>(kept2 + qi * KM);
      const float4* lp = reinterpret_cast<const float4*>(leaf_score + qi * NCM);
#pragma unroll
      for (int j = 0; j < KM / 4; ++j) {
        const int4 v = kp[j];
        pv[4 * j] = v.x; pv[4 * j + 1] = v.y; pv[4 * j + 2] = v.z; pv[4 * j + 3] = v.w;
      }
#pragma unroll
      for (int j = 0; j < NCM / 4; ++j) {
        const float4 v = lp[j];
        rv[4 * j] = v.x; rv[4 * j + 1] = v.y; rv[4 * j + 2] = v.z; rv[4 * j + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < KM; ++j) pv[j] = j < K ? kept2[qi * K + j] : -1;
#pragma unroll
      for (int c = 0; c < NCM; ++c) rv[c] = (c >> 1) < K ? leaf_score[(qi * K + (c >> 1)) * 2 + (c & 1)] : 0.0f;
    }
#pragma unroll
    for (int c = 0; c < NCM; ++c) {
      const int32_t p = pv[c >> 1];
      lf[c] = p >= 0 ? 2 * p + (c & 1) : -1;
      val[c] = p >= 0 && lf[c] >= 1 && lf[c] <= qb - 2;
      // a score slot whose node is not eligible was never written: ignored
      const float v = val[c] ? rv[c] : -INFINITY;
      sc[c] = v != v ? -INFINITY : v;  // NaN ranks as -inf (a total order)
    }
    // rank keys: the orderable score with its low 4 bits replaced by the
    // reversed candidate slot, so keys are distinct and, among scores equal to
    // 2^-19 relative (far inside the 1e-3 tie margin), the lower slot -- the
    // lower leaf, candidates running in ascending leaf order -- ranks first;
    // candidates outside E get key 0 and never rank above a valid one
    uint32_t key[NCM];
#pragma unroll
    for (int c = 0; c < NCM; ++c) {
      const uint32_t u = __float_as_uint(sc[c]);
      const uint32_t ok = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
      key[c] = val[c] ? ((ok & ~15u) | (uint32_t)(15 - c)) : 0u;
    }
    // the K-th largest key: a bitonic sort (descending) of a copy in
    // registers, 80 compare-exchanges with indices fixed at compile time;
    // with fewer than K valid candidates it is an invalid key (0)
    uint32_t sk[NCM];
#pragma unroll
    for (int c = 0; c < NCM; ++c) sk[c] = key[c];
#pragma unroll
    for (int kb = 2; kb <= NCM; kb <<= 1) {
#pragma unroll
      for (int j = kb >> 1; j > 0; j >>= 1) {
#pragma unroll
        for (int i = 0; i < NCM; ++i) {
          const int l = i ^ j;
          if (l > i) {
            const uint32_t a = sk[i], b = sk[l];
            const bool desc = (i & kb) == 0;
            sk[i] = desc ? max(a, b) : min(a, b);
            sk[l] = desc ? min(a, b) : max(a, b);
          }
        }
      }
    }
    uint32_t thr = 0;
#pragma unroll
    for (int j = 0; j < KM; ++j)
      if (j == K - 1) thr = sk[j];
    int32_t* oi = si + threadIdx.x * W;
    float* os = ss + threadIdx.x * W;
    int pos = 1;
#pragma unroll
    for (int c = 0; c < NCM; ++c) {
      // valid keys are distinct and non-zero: exactly min(K, valid) reach thr
      if (val[c] && key[c] >= thr && pos <= K) {  // candidates run in ascending leaf order
        oi[pos] = lf[c];
        os[pos] = sc[c] * kLn2;
        ++pos;
      }
    }
    oi[0] = 0;
    os[0] = INFINITY;
    if (qb - 1 > 0) { oi[pos] = qb - 1; os[pos] = INFINITY; ++pos; }
    if (qb > 0) { oi[pos] = qb; os[pos] = INFINITY; ++pos; }
    for (; pos < W; ++pos) { oi[pos] = -1; os[pos] = -INFINITY; }
  }
  __syncthreads();
  const int64_t nrow = (nq - q0 < (int64_t)blockDim.x ? nq - q0 : (int64_t)blockDim.x);
  const int n = (int)nrow * W;
  int32_t* gi = out_idx + q0 * W;
  for (int e = threadIdx.x; e < n; e += blockDim.x) gi[e] = si[e];
  if (out_score) {
    float* gs = out_score + q0 * W;
    for (int e = threadIdx.x; e < n; e += blockDim.x) gs[e] = ss[e];
  }
}

// ------------------------------------------------------------------ host
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2D view [rows, d] of a bf16 [.., d] tensor; box = 64 columns x box_rows,
// 128-byte swizzle (the K-major operand layout of the MMA).
bool make_tmap_rows(CUtensorMap* m, const void* base, int64_t rows, int d, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int G>
static cudaError_t launch_leaf_tc_t(const Prob& pr, const PrefillWs& w, char* ws, const CUtensorMap& kmap,
                                    const void* q, int grid, cudaStream_t st) {
  const size_t smem = sizeof(LeafTcSmem<D>) + 1024;
  const uint64_t tw = g_test_wait_ns.load(std::memory_order_relaxed);
  const LeafWaits waits{tw ? tw : kWaitLimitNs, g_test_drop_tile.load(std::memory_order_relaxed)};
  auto kern = leaf_tc_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  note_launch();
  e = launch_pdl(true, kern, dim3(grid), dim3(kLeafTcThreads), smem, st, pr, kmap, (const uint16_t*)q,
                 (const int4*)(ws + w.tile_info), (const int32_t*)(ws + w.tile_off) + w.nbuckets,
                 (const int32_t*)(ws + w.pairs), (float*)(ws + w.leaf_score), (int32_t*)(ws + w.status), waits);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_buckets(const BucketJob& j, int num_sms, cudaStream_t st) {
  BucketArgs a{j.nq, j.N, j.n2, j.nchunk, j.width, j.shift, j.dedup};
  // counts, offsets and cursor are contiguous: clear all three at once (the
  // first counting kernel follows this memset as a plain launch; the later
  // ones overlap their launch with the kernel before them)
  cudaError_t e = cudaMemsetAsync(j.counts, 0, j.clear_bytes, st);
  if (e != cudaSuccess) return e;
  const int64_t n = j.nq * j.width;
  const unsigned g1 = (unsigned)std::min<int64_t>(ceil_div64(n, 256), (int64_t)num_sms * 16);
  const bool smem_bins = j.n2 <= kSmemBins;
  const dim3 gs((unsigned)ceil_div64(j.N, kQueriesPerCta), (unsigned)(j.nq / j.N));
  const size_t hbytes = (size_t)j.n2 * sizeof(int32_t);
  if (smem_bins) {
    e = cudaFuncSetAttribute(count_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(kSmemBins * 4));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(scatter_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)(kSmemBins * 4));
    if (e != cudaSuccess) return e;
  }
  note_launch();
  if (smem_bins) count_smem_kernel<<<gs, kBucketThreads, hbytes, st>>>(a, j.lists, j.counts);
  else count_kernel<<<g1, 256, 0, st>>>(a, j.lists, j.counts);
  note_launch();
  e = launch_pdl(true, scan_kernel, dim3(1), dim3(1024), 0, st, j.nbuckets, j.Q, j.counts, j.offsets, j.tile_off);
  if (e != cudaSuccess) return e;
  note_launch();
  if (smem_bins)
    e = launch_pdl(true, scatter_smem_kernel, gs, dim3(kBucketThreads), hbytes, st, a, j.lists, j.offsets, j.cursor,
                   j.pairs);
  else
    e = launch_pdl(true, scatter_kernel, dim3(g1), dim3(256), 0, st, a, j.lists, j.offsets, j.cursor, j.pairs);
  if (e != cudaSuccess) return e;
  const unsigned g2 = (unsigned)std::min<int64_t>(ceil_div64(j.nbuckets, 256), (int64_t)num_sms * 8);
  note_launch();
  return launch_pdl(true, tiles_kernel, dim3(g2), dim3(256), 0, st, j.nbuckets, j.n2, j.nchunk, j.Q, j.counts,
                    j.offsets, j.tile_off, j.tile_info);
}

cudaError_t launch_leaf_tc(const Prob& pr, const Pyr& s, const PrefillWs& w, char* ws, const void* q,
                           const void* k, int32_t* out_idx, float* out_score, int num_sms, cudaStream_t st) {
  const int64_t nq = pr.B * pr.Hkv * pr.N;
  const int32_t* kept2 = (const int32_t*)(ws + w.kept2);
  cudaError_t e;
  if (w.nbuckets > 0) {
    const int32_t Q = kTileRows / pr.G;
    BucketJob j{};
    j.lists = kept2;
    j.nq = nq; j.N = pr.N; j.n2 = w.n2; j.nchunk = w.nchunk; j.nbuckets = w.nbuckets;
    j.width = pr.K; j.shift = 5; j.Q = Q;
    j.counts = (int32_t*)(ws + w.counts);
    j.offsets = (int32_t*)(ws + w.offsets);
    j.cursor = (int32_t*)(ws + w.cursor);
    j.tile_off = (int32_t*)(ws + w.tile_off);
    j.pairs = (int32_t*)(ws + w.pairs);
    j.tile_info = (int4*)(ws + w.tile_info);
    j.clear_bytes = w.tile_off - w.counts;
    e = launch_buckets(j, num_sms, st);
    if (e != cudaSuccess) return e;
    CUtensorMap kmap;
    if (!make_tmap_rows(&kmap, k, pr.B * pr.Hkv * pr.N, pr.d, kTileKeys)) return cudaErrorInvalidValue;
    const int grid = num_sms > 0 ? num_sms : 148;
#define PISA_LEAF_TC_CASE(DD, GG) \
    if (pr.d == DD && pr.G == GG) e = launch_leaf_tc_t<DD, GG>(pr, w, ws, kmap, q, grid, st); else
    PISA_LEAF_TC_CASE(128, 1) PISA_LEAF_TC_CASE(128, 2) PISA_LEAF_TC_CASE(128, 4) PISA_LEAF_TC_CASE(128, 8)
    PISA_LEAF_TC_CASE(64, 1) PISA_LEAF_TC_CASE(64, 2) PISA_LEAF_TC_CASE(64, 4) PISA_LEAF_TC_CASE(64, 8)
    e = cudaErrorInvalidValue;
#undef PISA_LEAF_TC_CASE
    if (e != cudaSuccess) return e;
  }
  note_launch();
  if (pr.K <= 8)
    return launch_pdl(true, finalize_small_kernel, dim3((unsigned)ceil_div64(nq, 256)), dim3(256), 0, st, pr, kept2,
                      (const float*)(ws + w.leaf_score), out_idx, out_score);
  return launch_pdl(true, finalize_kernel, dim3((unsigned)ceil_div64(nq, 8)), dim3(256), 0, st, pr, kept2,
                    (const float*)(ws + w.leaf_score), out_idx, out_score);
}

}  // namespace pisa

extern "C" void pisa_test_inject_leaf_timeout(uint64_t wait_limit_ns, int32_t drop_first_key_tile) {
  pisa::g_test_wait_ns.store(wait_limit_ns, std::memory_order_relaxed);
  pisa::g_test_drop_tile.store(drop_first_key_tile ? 1 : 0, std::memory_order_relaxed);
}
