// attend.cu -- block-sparse attention over the selected leaf blocks, on the
// tcgen05 tensor cores.  agihunt.info summary of "Block Sparse Attention with
// Log-Linear Complexity", opening paragraph: each query reads only its
// selected tiles of C keys, so the attention pass is linear in N; rcap.io
// post, "Selection walks the tree top-down": the kept leaf indices drive
// sparse attention over the original keys (and their values).
//
// For query position t of key head h and each query head of its group, the
// output is softmax(s q . k_i) v_i over the keys i <= t of the union of the
// query's selected blocks (s: the selection's score scale).
//
// GB300 design: block-centric, like the leaf stage.  Pairs (query, selected
// block j) are counting-sorted by (sequence, key head, query chunk, j).  One
// tile is 128 rows = 128/G queries x G heads of one bucket against the 64
// keys and values of block j:
//   - a loader warp brings the 64 x d key and value tiles by TMA (128-byte
//     swizzle) once per run of consecutive tiles with the same block;
//   - eight producer warps gather the query-head rows with cp.async;
//   - one thread issues S = Q K^T (M = 128, N = 64, K = d) into TMEM and,
//     once the probabilities are in shared memory, O = P V (M = 128, N = d,
//     K = 64; V is read in its natural key-major layout as an MN-major
//     operand) into a second TMEM region; two TMEM slots alternate, and the
//     S MMA of a tile is issued before the O MMA of the tile before it;
//   - two groups of four softmax warps take alternate tiles; a thread owns
//     one row: it reads the row's 64 scores, masks the keys after t (only the
//     query's own block has any), writes exp2(s - m) in bf16 into the
//     swizzled P tile, then reads its O row and stores O / l in bf16 with
//     lse = m + log2(l) -- one partial result per (query head, block).
// A combine kernel merges the partials of each query head (weights
// exp2(lse_b - max)) into the bf16 output.  The partials are the price of
// the block-centric order (each key/value tile is read once per query
// chunk); with blocks chosen independently per query there is no
// query-centric order that shares tiles.
#include <cudaTypedefs.h>

#include <algorithm>

#include "pisa_common.cuh"
#include "pisa_internal.h"
#include "tc_ptx.cuh"

namespace pisa {

namespace {

constexpr int kRows = 128;     // MMA M: queries x heads
constexpr int kKeys = 64;      // one leaf block
constexpr int kProdWarps = 8;  // warps 0-7 gather 16 query-head rows each
constexpr int kProdRows = kRows / kProdWarps;
constexpr int kLoadWarp = kProdWarps;
constexpr int kMmaWarp = kLoadWarp + 1;
constexpr int kSoftWarps = 8;  // two groups of four (one warp per TMEM lane quadrant)
constexpr int kThreads = 32 * (kMmaWarp + 1 + kSoftWarps);
constexpr int kGroup = 4;      // consecutive tiles per CTA turn
constexpr int kPairShift = 6;  // a pair is (t << 6) | slot
constexpr uint64_t kWaitLimitNs = 4000000000ull;

template <int D>
struct Cfg {
  static constexpr int SA = D == 128 ? 3 : 4;  // query-row stages
  static constexpr int SB = D == 128 ? 2 : 3;  // key/value stages (>= 2: see the MMA loop)
  static constexpr uint32_t kTmemCols = D == 128 ? 512 : 256;
};

template <int D>
struct AttnSmem {
  uint8_t a[Cfg<D>::SA][kRows * D * 2];
  uint8_t kv[Cfg<D>::SB][2][kKeys * D * 2];  // [stage][keys, values]
  uint8_t p[2][kRows * kKeys * 2];
  uint64_t full_a[Cfg<D>::SA], empty_a[Cfg<D>::SA], full_b[Cfg<D>::SB], empty_b[Cfg<D>::SB];
  uint64_t sfull[2], pfull[2], ofull[2], tempty[2], done;
  uint32_t tmem_base;
  int32_t abort;
  int32_t zero;
};

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
  __device__ int peek() const {
    if (i + 1 < gend) return i + 1;
    const int j = (g + (int)gridDim.x) * kGroup;
    return j < T ? j : -1;
  }
};

// Descriptor of an MN-major bf16 operand in the 128-byte swizzled layout:
// each 128-byte row holds 64 consecutive MN elements of one K index, 8-row
// atoms of 1024 bytes follow each other along K, and the next 64 MN elements
// start `lbo` bytes further.
__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;  // next 64 MN elements
  d |= (uint64_t)(1024u >> 4) << 32;            // next 8 K rows
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
    attend_tc_kernel(Prob pr, const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                     const uint16_t* __restrict__ q, const int4* __restrict__ tile_info,
                     const int32_t* __restrict__ tile_total, const int32_t* __restrict__ pairs,
                     float* __restrict__ part_lse, uint16_t* __restrict__ part_o, int32_t* __restrict__ status) {
  constexpr int SA = Cfg<D>::SA, SB = Cfg<D>::SB;
  extern __shared__ unsigned char smem_raw[];
  AttnSmem<D>& sm = *reinterpret_cast<AttnSmem<D>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr int kHalfA = kRows * 128;  // bytes of one 64-column slice of the query rows
  constexpr int kHalfB = kKeys * 128;  // bytes of one 64-column slice of a key or value tile
  constexpr uint32_t kKvBytes = 2u * kKeys * D * 2;
  constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(kRows, kKeys);
  constexpr uint32_t kIdescO = ptx::idesc_bf16_f32(kRows, D) | (1u << 16);  // B (values) MN-major
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  volatile int32_t* abort = &sm.abort;
  const int W = pr.K + 3;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SA; ++s) {
      ptx::mbar_init(ptx::smem_u32(&sm.full_a[s]), 32 * kProdWarps);
      ptx::mbar_init(ptx::smem_u32(&sm.empty_a[s]), 1);
    }
    for (int s = 0; s < SB; ++s) {
      ptx::mbar_init(ptx::smem_u32(&sm.full_b[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&sm.empty_b[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(ptx::smem_u32(&sm.sfull[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&sm.pfull[s]), 4);
      ptx::mbar_init(ptx::smem_u32(&sm.ofull[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&sm.tempty[s]), 4);
    }
    ptx::mbar_init(ptx::smem_u32(&sm.done), 1);
    sm.abort = 0;
    sm.zero = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(&sm.tmem_base), Cfg<D>::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int T = *tile_total;

  if (warp < kProdWarps) {
    // ------------------------------------------------------------ producers
    // warp w gathers rows [16w, 16w + 16) of every tile with cp.async, into
    // the 128-byte swizzled K-major layout
    constexpr int CPR = D / 8;     // 16-byte chunks per row
    constexpr int RPI = 32 / CPR;  // rows per warp instruction
    const int ch = lane % CPR, hi = lane / CPR;
    const int row0 = warp * kProdRows;
    const int64_t ND = pr.N * D;
    int it = 0;
    bool ok = true;
    for (TileIter ti(T); ti.valid(); ti.next()) {
      const int4 info = tile_info[ti.i];
      const int b = info.x / (int)pr.Hkv, h = info.x - b * (int)pr.Hkv;
      // this warp's (at most 16 / G, or one) query positions, one per lane
      const int nq_w = (kProdRows + G - 1) / G;
      const int qn = row0 / G + lane;
      const int32_t tq = (lane < nq_w && qn < info.z) ? (int32_t)((uint32_t)pairs[info.y + qn] >> kPairShift) : 0;
      const int sa = it % SA, use = it / SA;
      ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sm.empty_a[sa]), (use & 1) ^ 1, abort, kWaitLimitNs);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      const uint32_t abase = ptx::smem_u32(sm.a[sa]);
#pragma unroll
      for (int r0 = 0; r0 < kProdRows; r0 += RPI) {
        const int rl = r0 + hi;  // row within the warp's 16
        const int r = row0 + rl;
        const int qw = r / G - row0 / G;  // query index within the warp
        const int32_t t = __shfl_sync(0xffffffffu, tq, qw);
        if (r / G < info.z) {
          const int g = r % G;
          const uint16_t* src = q + (((int64_t)b * pr.Hq + h * G + g) * ND + (int64_t)t * D + ch * 8);
          ptx::cp_async_16(abase + (ch >> 3) * kHalfA + r * 128 + (((ch & 7) ^ (r & 7)) << 4), src);
        }
      }
      ptx::cp_async_arrive_noinc(ptx::smem_u32(&sm.full_a[sa]));
      ++it;
    }
    ptx::cp_async_wait_all();
    if (!ok) *abort = 1;
  } else if (warp == kLoadWarp) {
    // ------------------------------------------------- key / value tiles
    if (lane == 0) {
      int bcount = 0, last_bh = -1, last_j = -1;
      bool ok = true;
      for (TileIter ti(T); ti.valid(); ti.next()) {
        const int4 info = tile_info[ti.i];
        if (info.x == last_bh && info.w == last_j) continue;
        const int sb = bcount % SB, ub = bcount / SB;
        ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sm.empty_b[sb]), (ub & 1) ^ 1, abort, kWaitLimitNs);
        if (!ok) break;
        const uint32_t fb = ptx::smem_u32(&sm.full_b[sb]);
        ptx::mbar_arrive_expect_tx(fb, kKvBytes);
        const int32_t y = (int32_t)(info.x * pr.N + (int64_t)kKeys * info.w);
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh) {
          ptx::tma_load_2d(ptx::smem_u32(sm.kv[sb][0]) + hh * kHalfB, &kmap, 64 * hh, y, fb);
          ptx::tma_load_2d(ptx::smem_u32(sm.kv[sb][1]) + hh * kHalfB, &vmap, 64 * hh, y, fb);
        }
        ++bcount;
        last_bh = info.x;
        last_j = info.w;
      }
      if (!ok) *abort = 1;
      // every issued load lands before the CTA can exit, whoever gave up
      for (int k = bcount > SB ? bcount - SB : 0; k < bcount; ++k)
        ptx::mbar_wait_bounded(ptx::smem_u32(&sm.full_b[k % SB]), (k / SB) & 1, &sm.zero, kWaitLimitNs);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      int it = 0, bcount = 0, last_bh = -1, last_j = -1, sb = 0, prev_sb = 0;
      bool ok = true, prev_last = false;
      // O = P V of tile j (slot j & 1); releases the key/value stage after
      // the last tile of its run
      auto issue_o = [&](int j, int sbj, bool lastj) -> bool {
        const int e = j & 1;
        if (!ptx::mbar_wait_bounded(ptx::smem_u32(&sm.pfull[e]), (j >> 1) & 1, abort, kWaitLimitNs)) return false;
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_after();
        const uint32_t p0 = ptx::smem_u32(sm.p[e]), v0 = ptx::smem_u32(sm.kv[sbj][1]);
        const uint32_t d = tmem + 128 + e * D;
#pragma unroll
        for (int k = 0; k < kKeys / 16; ++k)
          ptx::mma_bf16(d, ptx::desc_sw128(p0 + k * 32), desc_mn_sw128(v0 + k * 2048, kHalfB), kIdescO,
                        k > 0 ? 1u : 0u);
        ptx::mma_commit(ptx::smem_u32(&sm.ofull[e]));
        if (lastj) ptx::mma_commit(ptx::smem_u32(&sm.empty_b[sbj]));
        return true;
      };
      TileIter ti(T);
      int4 info = ti.valid() ? tile_info[ti.i] : make_int4(-1, 0, 0, 0);
      for (; ti.valid(); ti.next()) {
        const int nx = ti.peek();
        const int4 ninfo = nx >= 0 ? tile_info[nx] : make_int4(-1, 0, 0, 0);
        const int sa = it % SA, use = it / SA, e = it & 1;
        if (info.x != last_bh || info.w != last_j) {
          sb = bcount % SB;
          ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sm.full_b[sb]), (bcount / SB) & 1, abort, kWaitLimitNs);
          if (!ok) break;
          ++bcount;
          last_bh = info.x;
          last_j = info.w;
        }
        ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sm.full_a[sa]), use & 1, abort, kWaitLimitNs) &&
             ptx::mbar_wait_bounded(ptx::smem_u32(&sm.tempty[e]), ((it >> 1) & 1) ^ 1, abort, kWaitLimitNs);
        if (!ok) break;
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_after();
        const uint32_t a0 = ptx::smem_u32(sm.a[sa]), k0 = ptx::smem_u32(sm.kv[sb][0]);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t oa = (k >> 2) * kHalfA + (k & 3) * 32, ob = (k >> 2) * kHalfB + (k & 3) * 32;
          ptx::mma_bf16(tmem + e * kKeys, ptx::desc_sw128(a0 + oa), ptx::desc_sw128(k0 + ob), kIdescS,
                        k > 0 ? 1u : 0u);
        }
        ptx::mma_commit(ptx::smem_u32(&sm.empty_a[sa]));
        ptx::mma_commit(ptx::smem_u32(&sm.sfull[e]));
        // S of this tile is queued; now O of the previous one
        if (it > 0 && !(ok = issue_o(it - 1, prev_sb, prev_last))) break;
        prev_sb = sb;
        prev_last = ninfo.x != info.x || ninfo.w != info.w;
        info = ninfo;
        ++it;
      }
      if (ok && it > 0) ok = issue_o(it - 1, prev_sb, prev_last);
      if (!ok) *abort = 1;
      ptx::mma_commit(ptx::smem_u32(&sm.done));
      ptx::mbar_wait_bounded(ptx::smem_u32(&sm.done), 0, &sm.zero, kWaitLimitNs);
    }
    __syncwarp();
  } else {
    // --------------------------------------------- softmax and partials
    const int grp = (warp - (kMmaWarp + 1)) / 4;  // takes tiles it % 2 == grp
    const int q4 = warp & 3;                      // TMEM lane quadrant
    const int r = q4 * 32 + lane;
    const int qr = r / G, g = r % G;
    const float sc = pr.scale2;
    const uint32_t prow = ptx::smem_u32(sm.p[grp]) + r * 128;
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    int it = 0;
    for (TileIter ti(T); ti.valid(); ti.next(), ++it) {
      if ((it & 1) != grp) continue;
      const int4 info = tile_info[ti.i];
      const bool valid = qr < info.z;
      const uint32_t pe = valid ? (uint32_t)pairs[info.y + qr] : 0u;
      const int64_t t = pe >> kPairShift;
      const int slot = (int)(pe & ((1u << kPairShift) - 1));
      const int uph = (it >> 1) & 1;
      bool okw = ptx::mbar_wait_bounded(ptx::smem_u32(&sm.sfull[grp]), uph, abort, kWaitLimitNs);
      if (!__all_sync(0xffffffffu, okw)) { *abort = 1; break; }
      ptx::tc_fence_after();
      float x[64];
      {
        uint32_t v0[32], v1[32];
        ptx::tmem_ld32(lane_base + grp * kKeys, v0);
        ptx::tmem_ld32(lane_base + grp * kKeys + 32, v1);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          x[j] = __uint_as_float(v0[j]);
          x[32 + j] = __uint_as_float(v1[j]);
        }
      }
      // keys j*64 + c with c <= lim are at or before t (lim >= 63: all)
      const int64_t lim64 = valid ? t - (int64_t)info.w * kKeys : 63;
      const int lim = lim64 > 63 ? 63 : (int)lim64;
      float m = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; ++c) m = fmaxf(m, c <= lim ? x[c] : -INFINITY);
      m *= sc;
      const bool any = lim >= 0;
      float l = 0.0f;
      {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float p0 = (any && c <= lim) ? ptx::ex2(fmaf(x[c], sc, -m)) : 0.0f;
          const float p1 = (any && c + 1 <= lim) ? ptx::ex2(fmaf(x[c + 1], sc, -m)) : 0.0f;
          l += p0 + p1;
          pk[c / 2] = pack_bf16(p0, p1);
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t dst = prow + ((c ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(pk[4 * c]), "r"(pk[4 * c + 1]),
                       "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                       : "memory");
        }
      }
      // the MMA reads P through the async proxy
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&sm.pfull[grp]));
      okw = ptx::mbar_wait_bounded(ptx::smem_u32(&sm.ofull[grp]), uph, abort, kWaitLimitNs);
      if (!__all_sync(0xffffffffu, okw)) { *abort = 1; break; }
      ptx::tc_fence_after();
      const float inv = any ? 1.0f / l : 0.0f;
      const int64_t bh = info.x;
      // this row's partial; the rows are written four at a time below
      uint16_t* dst = valid ? part_o + ((((bh * pr.N + t) * W + slot) * G + g) * D) : nullptr;
      const uint32_t srow = ptx::smem_u32(sm.p[grp]) + (q4 * 32) * 128;
#pragma unroll
      for (int half = 0; half < D / 64; ++half) {
        if (half > 0) __syncwarp();  // the previous half has been read back
        // stage the 64 bf16 of this half in this warp's 32 rows of the P
        // tile (free: the O MMA that read it has completed), swizzled so the
        // 16-byte writes of 8 consecutive rows hit distinct banks
#pragma unroll
        for (int piece = 0; piece < 2; ++piece) {
          uint32_t v0[32];
          ptx::tmem_ld32(lane_base + 128 + grp * D + half * 64 + piece * 32, v0);
          ptx::tmem_ld_wait();
          if (half == D / 64 - 1 && piece == 1) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&sm.tempty[grp]));
          }
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pk[j] = pack_bf16(__uint_as_float(v0[2 * j]) * inv, __uint_as_float(v0[2 * j + 1]) * inv);
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const int c = piece * 4 + c4;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(srow + lane * 128 + ((c ^ (lane & 7)) << 4)),
                         "r"(pk[4 * c4]), "r"(pk[4 * c4 + 1]), "r"(pk[4 * c4 + 2]), "r"(pk[4 * c4 + 3])
                         : "memory");
          }
        }
        __syncwarp();
        // read back four rows per instruction (eight lanes per 128-byte row)
        // and store full 128-byte lines
        const int c = lane & 7;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int rr = 4 * k + (lane >> 3);
          const uint64_t dp = __shfl_sync(0xffffffffu, reinterpret_cast<uint64_t>(dst), rr);
          uint32_t a0, a1, a2, a3;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                       : "r"(srow + rr * 128 + ((c ^ (rr & 7)) << 4))
                       : "memory");
          if (dp) reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(dp) + half * 64)[c] = make_uint4(a0, a1, a2, a3);
        }
      }
      if (valid) part_lse[((bh * pr.N + t) * W + slot) * G + g] = any ? m + ptx::lg2(l) : -INFINITY;
      __syncwarp();  // the staged rows are read before the next tile's P overwrites them
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, Cfg<D>::kTmemCols);
  if (threadIdx.x == 0 && sm.abort) set_status(status, PISA_DEV_TIMEOUT);
}

// One thread per (query, head, 8 output dims): merges the query head's block
// partials with weights exp2(lse_b - max_b lse_b).  The bucketing dropped
// empty, out-of-range and repeated slots, whose lse keeps the NaN fill of
// the workspace; slots whose block held no key at or before t have lse =
// -inf.  Both are skipped, so no index row is read and every load of a
// query head's partials is issued at once (BATCH slots in flight; a running
// maximum when the row is longer).  A query with no attended key gets zeros.
template <int D, int BATCH>
__global__ void __launch_bounds__(256) attend_combine_kernel(Prob pr, const float* __restrict__ part_lse,
                                                              const uint16_t* __restrict__ part_o,
                                                              uint16_t* __restrict__ out) {
  constexpr int CH = D / 8;
  const int G = pr.G, W = pr.K + 3;
  const int64_t total = pr.B * pr.Hkv * pr.N * G * CH;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int ch = (int)(i % CH);
    const int64_t rg = i / CH;
    const int g = (int)(rg % G);
    const int64_t qi = rg / G;  // (b * Hkv + h) * N + t
    const float* lrow = part_lse + qi * W * G + g;
    const uint16_t* orow = part_o + (qi * W * G + g) * D + ch * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, l = 0.0f, m = -INFINITY;
    for (int s0 = 0; s0 < W; s0 += BATCH) {
      float ls[BATCH];
      uint4 v[BATCH];
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        const int s = s0 + u;
        ls[u] = s < W ? lrow[(int64_t)s * G] : -INFINITY;
        v[u] = s < W ? *reinterpret_cast<const uint4*>(orow + (int64_t)s * G * D) : make_uint4(0u, 0u, 0u, 0u);
      }
      float bm = -INFINITY;
#pragma unroll
      for (int u = 0; u < BATCH; ++u)
        if (ls[u] > bm) bm = ls[u];  // NaN (empty slot) never wins
      if (bm > m) {
        const float f = m == -INFINITY ? 0.0f : ptx::ex2(m - bm);
        l *= f;
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] *= f;
        m = bm;
      }
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        if (!(ls[u] > -INFINITY)) continue;  // empty (NaN) or keyless (-inf)
        const float w = ptx::ex2(ls[u] - m);
        l += w;
        const uint32_t u4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[2 * j] = fmaf(w, __uint_as_float(u4[j] << 16), acc[2 * j]);
          acc[2 * j + 1] = fmaf(w, __uint_as_float(u4[j] & 0xFFFF0000u), acc[2 * j + 1]);
        }
      }
    }
    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
    const int64_t bh = qi / pr.N, t = qi - bh * pr.N;
    const int64_t b = bh / pr.Hkv, h = bh - b * pr.Hkv;
    uint4 o;
    o.x = pack_bf16(acc[0] * inv, acc[1] * inv);
    o.y = pack_bf16(acc[2] * inv, acc[3] * inv);
    o.z = pack_bf16(acc[4] * inv, acc[5] * inv);
    o.w = pack_bf16(acc[6] * inv, acc[7] * inv);
    *reinterpret_cast<uint4*>(out + (((b * pr.Hq + h * G + g) * pr.N + t) * D + ch * 8)) = o;
  }
}

template <int D, int G>
cudaError_t launch_attend_t(const Prob& pr, const AttendWs& w, char* ws, const CUtensorMap& kmap,
                            const CUtensorMap& vmap, const void* q, int grid, cudaStream_t st) {
  const size_t smem = sizeof(AttnSmem<D>) + 1024;
  auto kern = attend_tc_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  note_launch();
  kern<<<grid, kThreads, smem, st>>>(pr, kmap, vmap, (const uint16_t*)q, (const int4*)(ws + w.tile_info),
                                     (const int32_t*)(ws + w.tile_off) + w.nbuckets,
                                     (const int32_t*)(ws + w.pairs), (float*)(ws + w.part_lse),
                                     (uint16_t*)(ws + w.part_o), (int32_t*)(ws + w.status));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attend(const Prob& pr, const Pyr& s, const AttendWs& w, char* ws, const void* q, const void* k,
                          const void* v, const int32_t* idx, void* out, int num_sms, cudaStream_t st) {
  const int64_t nq = pr.B * pr.Hkv * pr.N;
  cudaError_t e;
  if (w.nbuckets > 0) {
    BucketJob j{};
    j.lists = idx;
    j.nq = nq; j.N = pr.N; j.n2 = s.nb; j.nchunk = w.nchunk; j.nbuckets = w.nbuckets;
    j.width = pr.K + 3; j.shift = kPairShift; j.dedup = 1; j.Q = kRows / pr.G;
    j.counts = (int32_t*)(ws + w.counts);
    j.offsets = (int32_t*)(ws + w.offsets);
    j.cursor = (int32_t*)(ws + w.cursor);
    j.tile_off = (int32_t*)(ws + w.tile_off);
    j.pairs = (int32_t*)(ws + w.pairs);
    j.tile_info = (int4*)(ws + w.tile_info);
    j.clear_bytes = w.tile_off - w.counts;
    e = launch_buckets(j, num_sms, st);
    if (e != cudaSuccess) return e;
    // slots the kernel does not write keep a NaN lse: the combine skips them
    e = cudaMemsetAsync(ws + w.part_lse, 0xFF, (size_t)nq * (pr.K + 3) * pr.G * sizeof(float), st);
    if (e != cudaSuccess) return e;
    CUtensorMap kmap, vmap;
    if (!make_tmap_rows(&kmap, k, nq, pr.d, kKeys) || !make_tmap_rows(&vmap, v, nq, pr.d, kKeys))
      return cudaErrorInvalidValue;
    const int grid = num_sms > 0 ? num_sms : 148;
#define PISA_ATTEND_CASE(DD, GG) \
    if (pr.d == DD && pr.G == GG) e = launch_attend_t<DD, GG>(pr, w, ws, kmap, vmap, q, grid, st); else
    PISA_ATTEND_CASE(128, 1) PISA_ATTEND_CASE(128, 2) PISA_ATTEND_CASE(128, 4) PISA_ATTEND_CASE(128, 8)
    PISA_ATTEND_CASE(64, 1) PISA_ATTEND_CASE(64, 2) PISA_ATTEND_CASE(64, 4) PISA_ATTEND_CASE(64, 8)
    e = cudaErrorInvalidValue;
#undef PISA_ATTEND_CASE
    if (e != cudaSuccess) return e;
  }
  const int64_t threads = nq * pr.G * (pr.d / 8);
  const unsigned blocks = (unsigned)std::min<int64_t>(ceil_div64(threads, 256), (int64_t)num_sms * 64);
  const float* pl = (const float*)(ws + w.part_lse);
  const uint16_t* po = (const uint16_t*)(ws + w.part_o);
  uint16_t* o = (uint16_t*)out;
  note_launch();
  const bool short_row = pr.K + 3 <= 12;
  if (pr.d == 128) {
    if (short_row) attend_combine_kernel<128, 12><<<blocks, 256, 0, st>>>(pr, pl, po, o);
    else attend_combine_kernel<128, 20><<<blocks, 256, 0, st>>>(pr, pl, po, o);
  } else {
    if (short_row) attend_combine_kernel<64, 12><<<blocks, 256, 0, st>>>(pr, pl, po, o);
    else attend_combine_kernel<64, 20><<<blocks, 256, 0, st>>>(pr, pl, po, o);
  }
  return cudaGetLastError();
}

}  // namespace pisa
