// decode.cu -- one decode step in a single launch: incremental pyramid update
// along the new key's path, then the top-down walk and leaf scoring for that
// one query.  agihunt.info summary of "Block Sparse Attention with Log-Linear
// Complexity": "Decode routing is O(log N) per step" (pyramid paragraph) and
// the single-stage decode kernel that avoids relaunches (kernel paragraph);
// rcap.io post, kernel paragraph (one fused kernel per step for decode).
//
// One CTA (4 warps) per (sequence, key head).  Phases:
//  1. update: the new key's leaf is re-averaged from its raw keys (staged in
//     shared memory by cp.async), then each ancestor is recombined from its
//     two children with the exact fp32 steps of the pyramid build, so the
//     state equals a fresh build bit for bit; siblings are prefetched at once.
//  2. walk: per level the needed child rows are fetched with one bulk copy
//     each into shared memory (one HBM round trip per level), the four warps
//     form the G-head dot products, and candidate scoring / Top-K / expansion
//     run on shared-memory lists (at most 2K candidates).
//  3. leaves: each warp streams its candidate leaves in 4 KB chunks (one bulk
//     copy each, three buffers per warp) and keeps an online log2-sum-exp2 per
//     head; bf16 keys are scored by warp-level m16n8k16 MMAs (16 keys x the G
//     heads per tile), fp32 keys by CUDA-core FMAs; then the Top-K with the
//     forced blocks.
// The step is bound by HBM: it reads ~2K leaf tiles per (sequence, key head).
#include "pisa_common.cuh"
#include "pisa_internal.h"
#include "tc_ptx.cuh"

namespace pisa {

constexpr int kDecWarps = 4;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kStageBytes = 12288;  // per warp: three 4 KB leaf chunks
constexpr int kChunkBytes = 4096;
constexpr int kNBuf = kStageBytes / kChunkBytes;
constexpr uint64_t kDecWaitNs = 4000000000ull;

template <int G>
struct DecSmem {
  alignas(128) unsigned char stage[kDecWarps][kStageBytes];  // 48 KB staging
  int32_t cand[kMaxCand], nxt[kMaxCand];
  float x[kMaxCand][G], xn[kMaxCand][G];
  int32_t has_x[kMaxCand], has_xn[kMaxCand];
  int32_t work[2 * kMaxCand];
  int32_t slot0[kMaxCand], slot1[kMaxCand];
  float y[2 * kMaxCand][G];
  float score[kMaxCand];
  int32_t kept2[kMaxK];
  int32_t leaf[kMaxCand];
  float lscore[kMaxCand];
  alignas(16) uint32_t key[kMaxCand];  // rank keys of the current list (0 past its end)
  int32_t scan[4];
  int32_t nkept2, nl;
  uint64_t bar_rows, bar_leaf[kDecWarps][kNBuf];
  int32_t abort;
  int32_t zero;  // stays 0
};

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Rank key of list entry `slot` (lists run in ascending node / leaf order):
// the orderable score with its low 6 bits replaced by the reversed slot, so
// keys are distinct and non-zero, a higher score ranks first, and among
// scores equal to 2^-17 relative (far inside the 1e-3 tie margin) the lower
// slot -- the lower index -- ranks first.  NaN ranks as -inf, -0 as +0.
__device__ __forceinline__ uint32_t rank_key(float sc, int slot) {
  if (sc != sc) sc = -INFINITY;
  if (sc == 0.0f) sc = 0.0f;
  const uint32_t u = __float_as_uint(sc);
  const uint32_t ok = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (ok & ~63u) | (uint32_t)(63 - slot);
}

// Number of keys of sm_keys[0, 64) above k (16-byte loads; unused entries
// hold 0, below every key).
__device__ __forceinline__ int rank_above(const uint32_t* sm_keys, int n, uint32_t k) {
  const uint4* kv = reinterpret_cast<const uint4*>(sm_keys);
  int rank = 0;
  for (int j = 0; j < (n + 3) / 4; ++j) {
    const uint4 v = kv[j];
    rank += (v.x > k ? 1 : 0) + (v.y > k ? 1 : 0) + (v.z > k ? 1 : 0) + (v.w > k ? 1 : 0);
  }
  return rank;
}

// Exclusive scan of one value per thread over threads [0, 64).
__device__ __forceinline__ int scan64(int v, int32_t* scratch, int* total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31 && warp < 2) scratch[warp] = x;
  __syncthreads();
  const int w0 = scratch[0], w1 = scratch[1];
  __syncthreads();
  *total = w0 + w1;
  return (warp == 1 ? w0 : 0) + x - v;
}

template <int D, int G>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(Prob pr, Pyr s, const void* __restrict__ q,
                                                             const void* __restrict__ kc, KeyPages kp,
                                                             const int32_t* __restrict__ seq_lens, float* pyr,
                                                             int32_t* __restrict__ status, int32_t* __restrict__ out_idx,
                                                             float* __restrict__ out_score, int32_t* __restrict__ trace) {
  constexpr int DPL = D / 32;
  constexpr int NB = 32 / G;
  extern __shared__ unsigned char dsm_raw[];
  DecSmem<G>& sm = *reinterpret_cast<DecSmem<G>*>((reinterpret_cast<uintptr_t>(dsm_raw) + 127) & ~(uintptr_t)127);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t bh = blockIdx.x, b = bh / pr.Hkv, h = bh % pr.Hkv;
  const int K = pr.K, W = K + 3;
  int32_t* oi = out_idx + bh * W;
  float* os = out_score ? out_score + bh * W : nullptr;
  int32_t* trow = trace ? trace + bh * (int64_t)s.L * K : nullptr;
  if (trow)
    for (int i = tid; i < s.L * K; i += kDecThreads) trow[i] = -1;
  const int64_t len = seq_lens[b];
  if (len < 1 || len > s.N) {
    if (tid == 0) set_status(status, PISA_DEV_BAD_SEQ_LEN);
    for (int i = tid; i < W; i += kDecThreads) { oi[i] = -1; if (os) os[i] = -INFINITY; }
    return;
  }
  const bool bf16 = pr.dtype == PISA_BF16;
  const int esz = bf16 ? 2 : 4;
  const int64_t t = len - 1, qb = t / s.C;
  if (kp.table) {
    // every page the step can read (leaves 0..qb) must be in the pool
    bool bad = false;
    for (int64_t j = tid; j <= qb; j += kDecThreads) {
      const int32_t pg = kp.table[b * kp.max_pages + j];
      bad |= pg < 0 || pg >= kp.num_pages;
    }
    if (__syncthreads_or(bad)) {
      if (tid == 0) set_status(status, PISA_DEV_BAD_INDEX);
      for (int i = tid; i < W; i += kDecThreads) { oi[i] = -1; if (os) os[i] = -INFINITY; }
      return;
    }
  }
  float* ph = pyr + bh * s.P * D;
  volatile int32_t* abort = &sm.abort;

  if (tid == 0) {
    ptx::mbar_init(ptx::smem_u32(&sm.bar_rows), 1);
    for (int w = 0; w < kDecWarps; ++w)
      for (int u = 0; u < kNBuf; ++u) ptx::mbar_init(ptx::smem_u32(&sm.bar_leaf[w][u]), 1);
    sm.abort = 0;
    sm.zero = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }

  // ---------------------------------------------------------------- 1. update
  {
    unsigned char* keys = &sm.stage[0][0];  // up to C*D*4 = 32 KB
    float* sib = reinterpret_cast<float*>(&sm.stage[0][0] + 32768);  // one row per level (16 KB)
    const int64_t n_leaf = len - qb * s.C;
    const char* src = reinterpret_cast<const char*>(kc) + (leaf_row(kp, pr.Hkv, s.N, s.C, b, h, qb) * D) * esz;
    const int chunks = (int)(n_leaf * D * esz / 16);
    for (int c = tid; c < chunks; c += kDecThreads) ptx::cp_async_16(ptx::smem_u32(keys + 16 * c), src + 16 * c);
    for (int w = tid; w < s.L * (D / 4); w += kDecThreads) {
      const int level = 2 + w / (D / 4);
      const int c4 = w % (D / 4);
      if (level > s.L) continue;
      const int64_t cpath = qb >> (level - 2), sibling = cpath ^ 1;
      if (sibling < s.size[level - 2])
        ptx::cp_async_16(ptx::smem_u32(sib + (level - 2) * D + 4 * c4), ph + (s.off[level - 2] + sibling) * D + 4 * c4);
    }
    ptx::cp_async_commit();
    ptx::cp_async_wait<0>();
    __syncthreads();
    if (tid < D) {
      // leaf: keys in index order, IEEE fp32 adds, one division (as the build)
      float acc = 0.0f;
      for (int64_t i = 0; i < n_leaf; ++i) {
        const float v = bf16 ? bf16_to_f(reinterpret_cast<const uint16_t*>(keys)[i * D + tid])
                             : reinterpret_cast<const float*>(keys)[i * D + tid];
        acc = __fadd_rn(acc, v);
      }
      float m = __fdiv_rn(acc, (float)n_leaf);
      ph[(s.off[0] + qb) * D + tid] = m;
      for (int level = 2; level <= s.L; ++level) {
        const int64_t j = qb >> (level - 1), cpath = qb >> (level - 2), sibling = cpath ^ 1;
        const int64_t npath = node_count(s, level - 1, cpath, len);
        const int64_t nsib = sibling < s.size[level - 2] ? node_count(s, level - 1, sibling, len) : 0;
        const float vs = nsib > 0 ? sib[(level - 2) * D + tid] : 0.0f;
        m = (cpath & 1) ? combine_children(vs, nsib, m, npath) : combine_children(m, npath, vs, nsib);
        ph[(s.off[level - 1] + j) * D + tid] = m;
      }
      ptx::fence_proxy_async_global();  // the walk below reads these rows by bulk copy
    }
  }
  // query heads, scaled by s * log2(e), staged through the (now idle)
  // staging area on their way into registers
  float(*qs)[D] = reinterpret_cast<float(*)[D]>(&sm.stage[0][0]);
  __syncthreads();  // the update phase is done with the staging area
  for (int i = tid; i < G * D; i += kDecThreads) {
    const int g = i / D, c = i % D;
    const int64_t off = (b * pr.Hq + h * G + g) * D + c;
    const float v = bf16 ? bf16_to_f(reinterpret_cast<const uint16_t*>(q)[off]) : reinterpret_cast<const float*>(q)[off];
    qs[g][c] = v * pr.scale2;
  }
  __syncthreads();

  // ------------------------------------------------------------------ 2. walk
  int L_len = 0;
  {
    int64_t n = ceil_div64(len, s.C);
    for (;;) { ++L_len; if (n == 1) break; n = ceil_div64(n, 2); }
  }
  float qr[G][DPL];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int c = 0; c < DPL; ++c) qr[g][c] = qs[g][lane * DPL + c];

  if (tid == 0) sm.nkept2 = 0;
  __syncthreads();
  if (qb - 2 >= 1) {
    int l0 = 0;
    for (int level = L_len; level >= 2; --level)
      if (eligible_count(level, qb) > K) { l0 = level; break; }
    if (trow)
      for (int level = L_len; level >= 2 && level > l0; --level) {
        const int64_t n = eligible_count(level, qb);
        for (int i = tid; i < n; i += kDecThreads) trow[(level - 1) * K + i] = i;
      }
    if (l0 == 0) {
      const int n2 = (int)eligible_count(2, qb);
      for (int i = tid; i < n2; i += kDecThreads) sm.kept2[i] = i;
      if (tid == 0) sm.nkept2 = n2;
    } else {
      int nc = (int)eligible_count(l0, qb);
      for (int i = tid; i < nc; i += kDecThreads) { sm.cand[i] = i; sm.has_x[i] = 0; }
      __syncthreads();
      uint32_t rphase = 0;
      float* rows = reinterpret_cast<float*>(&sm.stage[0][0]);
      for (int level = l0; level >= 2; --level) {
        const int64_t ncap = s.size[level - 2];
        // work list (threads 0..63 own one candidate each)
        int nwork = 0, e0 = 0, e1 = 0, der = 0;
        int64_t c0 = 0;
        if (tid < nc) {
          c0 = 2 * (int64_t)sm.cand[tid];
          e0 = c0 < ncap && node_eligible(level - 1, c0, qb);
          e1 = c0 + 1 < ncap && node_eligible(level - 1, c0 + 1, qb);
          der = e0 && e1 && sm.has_x[tid];
          nwork = e0 + (e1 && !der);
        }
        int nwork_all;
        const int pos = scan64(tid < 64 ? nwork : 0, sm.scan, &nwork_all);
        if (tid < nc) {
          int p = pos;
          sm.slot0[tid] = e0 ? p : -1;
          if (e0) sm.work[p++] = (int32_t)c0;
          sm.slot1[tid] = e1 ? (der ? -2 : p) : -1;
          if (e1 && !der) sm.work[p++] = (int32_t)(c0 + 1);
        }
        // child rows, fetched in batches that fit the staging area: one bulk
        // copy per row, then the four warps form the dot products
        constexpr int kRowsPerBatch = kDecWarps * kStageBytes / (D * 4);
        for (int b0 = 0; b0 < nwork_all && !*abort; b0 += kRowsPerBatch) {
          const int nrow = nwork_all - b0 < kRowsPerBatch ? nwork_all - b0 : kRowsPerBatch;
          if (tid == 0) ptx::mbar_arrive_expect_tx(ptx::smem_u32(&sm.bar_rows), (uint32_t)(nrow * D * 4));
          __syncthreads();
          for (int w = tid; w < nrow; w += kDecThreads)
            ptx::bulk_g2s(ptx::smem_u32(rows + w * D), ph + (s.off[level - 2] + sm.work[b0 + w]) * D, D * 4,
                          ptx::smem_u32(&sm.bar_rows));
          if (!ptx::mbar_wait_bounded(ptx::smem_u32(&sm.bar_rows), rphase, abort, kDecWaitNs)) *abort = 1;
          rphase ^= 1;
          __syncthreads();
          if (*abort) break;
          // dot products: warp w takes batches w, w+4, ... of NB child rows
          for (int w0 = warp * NB; w0 < nrow; w0 += kDecWarps * NB) {
            float v[32];
#pragma unroll
            for (int n = 0; n < NB; ++n) {
              float mu[DPL];
              const int w = w0 + n;
              if (w < nrow) {
                if (DPL == 4) {
                  const float4 m4 = *reinterpret_cast<const float4*>(rows + w * D + lane * 4);
                  mu[0] = m4.x; mu[1] = m4.y; mu[2] = m4.z; mu[3] = m4.w;
                } else {
                  const float2 m2 = *reinterpret_cast<const float2*>(rows + w * D + lane * 2);
                  mu[0] = m2.x; mu[1] = m2.y;
                }
              } else {
#pragma unroll
                for (int c = 0; c < DPL; ++c) mu[c] = 0.0f;
              }
#pragma unroll
              for (int g = 0; g < G; ++g) {
                float acc = 0.0f;
#pragma unroll
                for (int c = 0; c < DPL; ++c) acc = fmaf(qr[g][c], mu[c], acc);
                v[n * G + g] = acc;
              }
            }
            const float r = warp_transpose_sum32(v);
            const int w = w0 + lane / G;
            if (w < nrow) sm.y[b0 + w][lane % G] = r;
          }
          __syncthreads();  // the next batch overwrites the staging area
        }
        if (*abort) break;
        // candidate scores
        if (tid < nc) {
          const int s0 = sm.slot0[tid], s1 = sm.slot1[tid];
          float n0 = 0.0f, n1 = 0.0f;
          if (s1 == -2) {
            n0 = (float)node_count(s, level - 1, c0, len);
            n1 = (float)node_count(s, level - 1, c0 + 1, len);
          }
          float sc = 0.0f;
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float a = s0 >= 0 ? sm.y[s0][g] : 0.0f;
            float bb = 0.0f;
            if (s1 >= 0) bb = sm.y[s1][g];
            else if (s1 == -2) bb = ((n0 + n1) * sm.x[tid][g] - n0 * a) / n1;
            sc += (s0 >= 0 && s1 != -1) ? pair_score(pr.scorer, a, bb) : (s0 >= 0 ? a : bb);
          }
          sm.score[tid] = sc != sc ? -INFINITY : sc;  // NaN ranks as -inf
        }
        if (tid < kMaxCand) sm.key[tid] = tid < nc ? rank_key(sm.score[tid], tid) : 0u;
        __syncthreads();
        // Top-K and expansion, in index order
        int keep = 0, nchild = 0;
        if (tid < nc) {
          keep = rank_above(sm.key, nc, sm.key[tid]) < K;
          nchild = keep ? (level > 2 ? e0 + e1 : 1) : 0;
        }
        int total;
        const int p2 = scan64(tid < 64 ? nchild : 0, sm.scan, &total);
        if (keep) {
          if (level == 2) {
            sm.kept2[p2] = sm.cand[tid];
          } else {
            int p = p2;
            const int s0 = sm.slot0[tid], s1 = sm.slot1[tid];
            float n0 = 0.0f, n1 = 0.0f;
            if (s1 == -2) {
              n0 = (float)node_count(s, level - 1, c0, len);
              n1 = (float)node_count(s, level - 1, c0 + 1, len);
            }
            if (e0) {
              sm.nxt[p] = (int32_t)c0;
#pragma unroll
              for (int g = 0; g < G; ++g) sm.xn[p][g] = sm.y[s0][g];
              sm.has_xn[p] = 1;
              ++p;
            }
            if (e1) {
              sm.nxt[p] = (int32_t)(c0 + 1);
#pragma unroll
              for (int g = 0; g < G; ++g) {
                const float a = e0 ? sm.y[s0][g] : 0.0f;
                sm.xn[p][g] = s1 >= 0 ? sm.y[s1][g] : ((n0 + n1) * sm.x[tid][g] - n0 * a) / n1;
              }
              sm.has_xn[p] = 1;
            }
          }
        }
        // kept set in index order for the trace
        int kt;
        const int kpos = scan64(tid < 64 ? keep : 0, sm.scan, &kt);
        if (keep && trow) trow[(level - 1) * K + kpos] = sm.cand[tid];
        if (level == 2) {
          if (tid == 0) sm.nkept2 = total;
          break;
        }
        __syncthreads();
        nc = total;
        if (tid < nc) {
          sm.cand[tid] = sm.nxt[tid];
          sm.has_x[tid] = sm.has_xn[tid];
#pragma unroll
          for (int g = 0; g < G; ++g) sm.x[tid][g] = sm.xn[tid][g];
        }
        __syncthreads();
      }
    }
  }
  __syncthreads();

  // ----------------------------------------------------------- 3. leaf stage
  {
    const int nk2 = sm.nkept2;
    int e0 = 0, e1 = 0;
    int32_t p = -1;
    if (tid < nk2) {
      p = sm.kept2[tid];
      e0 = node_eligible(1, 2 * (int64_t)p, qb);
      e1 = node_eligible(1, 2 * (int64_t)p + 1, qb);
    }
    int nl;
    const int pos = scan64(tid < 64 ? e0 + e1 : 0, sm.scan, &nl);
    if (tid < nk2) {
      int pp = pos;
      if (e0) sm.leaf[pp++] = 2 * p;
      if (e1) sm.leaf[pp++] = 2 * p + 1;
    }
    __syncthreads();
    // each warp streams its leaves in 4 KB chunks through three buffers: the
    // copies of chunks c+1 and c+2 are in flight while chunk c is scored
    if (bf16) {
      // bf16 keys: one bulk copy per chunk (row-major key rows; bulk copies
      // stream faster here than two-dimensional TMA tiles); warp-level
      // m16n8k16 MMAs give 16 keys x 8 columns (the G heads) per tile, and
      // every lane keeps an online max / sum for its two heads (2t, 2t+1)
      // over its keys (rows g and g+8 of each tile).
      constexpr int KPC = kChunkBytes / (D * 2);  // keys per chunk: 16 (d = 128) or 32 (d = 64)
      const int cpl = s.C / KPC;
      const int nlw = nl > warp ? (nl - warp + kDecWarps - 1) / kDecWarps : 0;
      const int nch = nlw * cpl;
      unsigned char* st = &sm.stage[warp][0];
      const int grp = lane >> 2, tig = lane & 3;
      uint32_t bq[D / 32][4];  // B fragments: column grp = head grp (zero past G)
      {
        const int64_t qoff = (b * pr.Hq + h * G + (grp < G ? grp : 0)) * D;
#pragma unroll
        for (int bb = 0; bb < D / 32; ++bb) {
          uint4 v = grp < G ? *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(q) + qoff + 32 * bb +
                                                               8 * tig)
                            : make_uint4(0u, 0u, 0u, 0u);
          bq[bb][0] = v.x; bq[bb][1] = v.y; bq[bb][2] = v.z; bq[bb][3] = v.w;
        }
      }
      uint32_t lphase = 0u;
      auto issue = [&](int c) {
        if (lane == 0) {
          const int64_t leaf = sm.leaf[warp + (c / cpl) * kDecWarps];
          const uint32_t bar = ptx::smem_u32(&sm.bar_leaf[warp][c % kNBuf]);
          ptx::mbar_arrive_expect_tx(bar, KPC * D * 2);
          ptx::bulk_g2s(ptx::smem_u32(st + (c % kNBuf) * kChunkBytes),
                        reinterpret_cast<const uint16_t*>(kc) +
                            (leaf_row(kp, pr.Hkv, s.N, s.C, b, h, leaf) + (c % cpl) * KPC) * D,
                        KPC * D * 2, bar);
        }
      };
      int issued = 0, waited = 0;
      for (; issued < nch && issued < kNBuf - 1; ++issued) issue(issued);
      float m0 = -INFINITY, s0 = 0.0f, m1 = -INFINITY, s1 = 0.0f;  // heads 2t, 2t+1
      Moments w0{0.0f, 0.0f, 0.0f}, w1{0.0f, 0.0f, 0.0f};            // PISA-1 / PISA-2
      const bool lse_scorer = pr.scorer == PISA_SCORER_LSE;
      const float sc = pr.scale2;
      for (int c = 0; c < nch; ++c) {
        if (c + kNBuf - 1 < nch) {
          __syncwarp();  // every lane is done with the buffer this copy overwrites
          issue(c + kNBuf - 1);
          issued = c + kNBuf;
        }
        const int bf = c % kNBuf;
        const bool ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sm.bar_leaf[warp][bf]), (lphase >> bf) & 1u, abort,
                                               kDecWaitNs);
        lphase ^= 1u << bf;
        waited = c + 1;
        if (!__all_sync(0xffffffffu, ok)) { *abort = 1; break; }
        if (c % cpl == 0) {
          m0 = -INFINITY; s0 = 0.0f; m1 = -INFINITY; s1 = 0.0f;
          w0 = Moments{0.0f, 0.0f, 0.0f};
          w1 = Moments{0.0f, 0.0f, 0.0f};
        }
        const unsigned char* buf = st + bf * kChunkBytes;
#pragma unroll
        for (int mt = 0; mt < KPC / 16; ++mt) {
          float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          const int r0 = 16 * mt + grp, r1 = r0 + 8;
#pragma unroll
          for (int bb = 0; bb < D / 32; ++bb) {
            // dims 32 bb + 8 t + {0..7} of keys r0 and r1 (the k-step mapping of the B fragments)
            const uint4 a0 = *reinterpret_cast<const uint4*>(buf + r0 * D * 2 + 64 * bb + 16 * tig);
            const uint4 a1 = *reinterpret_cast<const uint4*>(buf + r1 * D * 2 + 64 * bb + 16 * tig);
            mma_bf16_16816(d, a0.x, a1.x, a0.y, a1.y, bq[bb][0], bq[bb][1]);
            mma_bf16_16816(d, a0.z, a1.z, a0.w, a1.w, bq[bb][2], bq[bb][3]);
          }
          // d[0], d[1]: key r0, heads 2t, 2t+1; d[2], d[3]: key r1
          const float x00 = d[0] * sc, x01 = d[1] * sc, x10 = d[2] * sc, x11 = d[3] * sc;
          if (lse_scorer) {
            const float n0 = fmaxf(m0, fmaxf(x00, x10)), n1 = fmaxf(m1, fmaxf(x01, x11));
            s0 = s0 * ptx::ex2(m0 - n0) + ptx::ex2(x00 - n0) + ptx::ex2(x10 - n0);
            s1 = s1 * ptx::ex2(m1 - n1) + ptx::ex2(x01 - n1) + ptx::ex2(x11 - n1);
            m0 = n0;
            m1 = n1;
          } else {
            mom_add(w0, x00);
            mom_add(w0, x10);
            mom_add(w1, x01);
            mom_add(w1, x11);
          }
        }
        if (c % cpl == cpl - 1) {
          // combine the 8 lanes (groups) of each head, then sum the G heads
          float lse = 0.0f;
          if (lse_scorer) {
#pragma unroll
            for (int o = 4; o <= 16; o <<= 1) {
              const float mo0 = __shfl_xor_sync(0xffffffffu, m0, o), so0 = __shfl_xor_sync(0xffffffffu, s0, o);
              const float mo1 = __shfl_xor_sync(0xffffffffu, m1, o), so1 = __shfl_xor_sync(0xffffffffu, s1, o);
              const float a0 = fmaxf(m0, mo0), a1 = fmaxf(m1, mo1);
              s0 = s0 * ptx::ex2(m0 - a0) + so0 * ptx::ex2(mo0 - a0);
              s1 = s1 * ptx::ex2(m1 - a1) + so1 * ptx::ex2(mo1 - a1);
              m0 = a0;
              m1 = a1;
            }
            if (2 * tig < G) lse += m0 + ptx::lg2(s0);
            if (2 * tig + 1 < G) lse += m1 + ptx::lg2(s1);
          } else {
#pragma unroll
            for (int o = 4; o <= 16; o <<= 1) {
              const float n0o = __shfl_xor_sync(0xffffffffu, w0.n, o), u0 = __shfl_xor_sync(0xffffffffu, w0.mean, o),
                          v0 = __shfl_xor_sync(0xffffffffu, w0.m2, o);
              const float n1o = __shfl_xor_sync(0xffffffffu, w1.n, o), u1 = __shfl_xor_sync(0xffffffffu, w1.mean, o),
                          v1 = __shfl_xor_sync(0xffffffffu, w1.m2, o);
              mom_merge(w0, n0o, u0, v0);
              mom_merge(w1, n1o, u1, v1);
            }
            if (2 * tig < G) lse += moment_score(pr.scorer, w0.n, w0.mean, w0.m2);
            if (2 * tig + 1 < G) lse += moment_score(pr.scorer, w1.n, w1.mean, w1.m2);
          }
          lse += __shfl_xor_sync(0xffffffffu, lse, 1);
          lse += __shfl_xor_sync(0xffffffffu, lse, 2);
          if (lane == 0) sm.lscore[warp + (c / cpl) * kDecWarps] = lse != lse ? -INFINITY : lse;
        }
      }
      // after an early exit, let copies already issued land before the CTA ends
      for (int c = waited; c < issued; ++c) {
        const int bf = c % kNBuf;
        ptx::mbar_wait_bounded(ptx::smem_u32(&sm.bar_leaf[warp][bf]), (lphase >> bf) & 1u, &sm.zero, kDecWaitNs);
        lphase ^= 1u << bf;
      }
    } else {
    const int kpc = kChunkBytes / (D * esz) < s.C ? kChunkBytes / (D * esz) : s.C;  // keys per chunk
    const int cpl = s.C / kpc;                                                      // chunks per leaf
    const int nlw = nl > warp ? (nl - warp + kDecWarps - 1) / kDecWarps : 0;        // this warp's leaves
    const int nch = nlw * cpl;
    unsigned char* st = &sm.stage[warp][0];
    const uint32_t chunk_bytes = (uint32_t)(kpc * D * esz);
    uint32_t lphase = 0u;  // bit b: phase parity of buffer b
    auto issue = [&](int c) {
      if (lane == 0) {
        const int64_t leaf = sm.leaf[warp + (c / cpl) * kDecWarps];
        const int k0 = (c % cpl) * kpc;
        const uint32_t bar = ptx::smem_u32(&sm.bar_leaf[warp][c % kNBuf]);
        ptx::mbar_arrive_expect_tx(bar, chunk_bytes);
        ptx::bulk_g2s(ptx::smem_u32(st + (c % kNBuf) * kChunkBytes),
                      reinterpret_cast<const char*>(kc) + ((leaf_row(kp, pr.Hkv, s.N, s.C, b, h, leaf) + k0) * D) * esz,
                      chunk_bytes, bar);
      }
    };
    int issued = 0, waited = 0;
    for (; issued < nch && issued < kNBuf - 1; ++issued) issue(issued);
    float m = -INFINITY, ssum = 0.0f;  // this lane's head: lane % G
    Moments wm{0.0f, 0.0f, 0.0f};      // PISA-1 / PISA-2
    for (int c = 0; c < nch; ++c) {
      if (c + kNBuf - 1 < nch) {
        __syncwarp();  // every lane is done with the buffer this copy overwrites
        issue(c + kNBuf - 1);
        issued = c + kNBuf;
      }
      const int bf = c % kNBuf;
      const bool ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sm.bar_leaf[warp][bf]), (lphase >> bf) & 1u, abort,
                                             kDecWaitNs);
      lphase ^= 1u << bf;
      waited = c + 1;
      if (!__all_sync(0xffffffffu, ok)) { *abort = 1; break; }
      if (c % cpl == 0) { m = -INFINITY; ssum = 0.0f; wm = Moments{0.0f, 0.0f, 0.0f}; }
      const unsigned char* buf = st + bf * kChunkBytes;
      for (int k1 = 0; k1 < kpc; k1 += NB) {
        float v[32];
#pragma unroll
        for (int n = 0; n < NB; ++n) {
          float kv[DPL];
          const unsigned char* row = buf + (k1 + n) * D * esz + lane * DPL * esz;
          if (bf16) {
            if (DPL == 4) {
              const uint2 u = *reinterpret_cast<const uint2*>(row);
              kv[0] = __uint_as_float(u.x << 16); kv[1] = __uint_as_float(u.x & 0xffff0000u);
              kv[2] = __uint_as_float(u.y << 16); kv[3] = __uint_as_float(u.y & 0xffff0000u);
            } else {
              const uint32_t u = *reinterpret_cast<const uint32_t*>(row);
              kv[0] = __uint_as_float(u << 16); kv[1] = __uint_as_float(u & 0xffff0000u);
            }
          } else {
#pragma unroll
            for (int cc = 0; cc < DPL; ++cc) kv[cc] = reinterpret_cast<const float*>(row)[cc];
          }
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float acc = 0.0f;
#pragma unroll
            for (int cc = 0; cc < DPL; ++cc) acc = fmaf(qr[g][cc], kv[cc], acc);
            v[n * G + g] = acc;
          }
        }
        const float x = warp_transpose_sum32(v);  // key k1 + lane/G, head lane%G
        if (k1 + lane / G < kpc) {  // a batch may run past a short chunk
          if (pr.scorer == PISA_SCORER_LSE) {
            const float mn = fmaxf(m, x);
            ssum = ssum * ptx::ex2(m - mn) + ptx::ex2(x - mn);
            m = mn;
          } else {
            mom_add(wm, x);
          }
        }
      }
      if (c % cpl == cpl - 1) {
        // combine the lanes of each head, then sum the heads
        float lse;
        if (pr.scorer == PISA_SCORER_LSE) {
          float mh = m, sh = ssum;
#pragma unroll
          for (int o = 16; o >= G; o >>= 1) {
            const float mo = __shfl_xor_sync(0xffffffffu, mh, o), so = __shfl_xor_sync(0xffffffffu, sh, o);
            const float mn = fmaxf(mh, mo);
            sh = sh * ptx::ex2(mh - mn) + so * ptx::ex2(mo - mn);
            mh = mn;
          }
          lse = mh + ptx::lg2(sh);
        } else {
#pragma unroll
          for (int o = 16; o >= G; o >>= 1)
            mom_merge(wm, __shfl_xor_sync(0xffffffffu, wm.n, o), __shfl_xor_sync(0xffffffffu, wm.mean, o),
                      __shfl_xor_sync(0xffffffffu, wm.m2, o));
          lse = moment_score(pr.scorer, wm.n, wm.mean, wm.m2);
        }
#pragma unroll
        for (int o = G / 2; o >= 1; o >>= 1) lse += __shfl_xor_sync(0xffffffffu, lse, o);
        if (lane == 0) sm.lscore[warp + (c / cpl) * kDecWarps] = lse != lse ? -INFINITY : lse;
      }
    }
    // after an early exit, let copies already issued land before the CTA ends
    for (int c = waited; c < issued; ++c) {
      const int bf = c % kNBuf;
      ptx::mbar_wait_bounded(ptx::smem_u32(&sm.bar_leaf[warp][bf]), (lphase >> bf) & 1u, &sm.zero, kDecWaitNs);
      lphase ^= 1u << bf;
    }
    }  // fp32 keys
    __syncthreads();
    if (*abort) {
      if (tid == 0) set_status(status, PISA_DEV_TIMEOUT);
      for (int i = tid; i < W; i += kDecThreads) { oi[i] = -1; if (os) os[i] = -INFINITY; }
      return;
    }
    // Top-K of the candidate leaves plus the forced blocks, ascending
    if (tid < kMaxCand) sm.key[tid] = tid < nl ? rank_key(sm.lscore[tid], tid) : 0u;
    __syncthreads();
    int keep = 0;
    if (tid < nl) keep = rank_above(sm.key, nl, sm.key[tid]) < K;
    int nkept;
    const int kp = scan64(tid < 64 ? keep : 0, sm.scan, &nkept);
    if (keep && kp < K) {  // the ranking order is total: at most K are kept
      oi[1 + kp] = sm.leaf[tid];
      if (os) os[1 + kp] = sm.lscore[tid] * kLn2;
    }
    if (tid == 0) {
      oi[0] = 0;
      if (os) os[0] = INFINITY;
      int ps = 1 + nkept;
      if (qb - 1 > 0) { oi[ps] = (int32_t)(qb - 1); if (os) os[ps] = INFINITY; ++ps; }
      if (qb > 0) { oi[ps] = (int32_t)qb; if (os) os[ps] = INFINITY; ++ps; }
      for (; ps < W; ++ps) { oi[ps] = -1; if (os) os[ps] = -INFINITY; }
    }
  }
}

template <int D, int G>
static cudaError_t launch_decode_t(const Prob& pr, const Pyr& s, const void* q, const void* kc,
                                   const KeyPages& kp, const int32_t* seq_lens, float* pyr, int32_t* status, int32_t* out_idx,
                                   float* out_score, int32_t* trace, cudaStream_t st) {
  const size_t smem = sizeof(DecSmem<G>) + 128;
  auto kern = decode_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  note_launch();
  kern<<<(unsigned)(pr.B * pr.Hkv), kDecThreads, smem, st>>>(pr, s, q, kc, kp, seq_lens, pyr, status, out_idx,
                                                              out_score, trace);
  return cudaGetLastError();
}

cudaError_t launch_decode(const Prob& pr, const Pyr& s, const void* q, const void* kc, const KeyPages& kp,
                          const int32_t* seq_lens,
                          float* pyr, int32_t* status, int32_t* out_idx, float* out_score, int32_t* trace,
                          cudaStream_t st) {
  if (s.L * pr.d * 4 > 16384) return cudaErrorInvalidValue;  // sibling rows must fit their staging slot
#define PISA_DEC_CASE(DD, GG) \
  if (pr.d == DD && pr.G == GG)  \
    return launch_decode_t<DD, GG>(pr, s, q, kc, kp, seq_lens, pyr, status, out_idx, out_score, trace, st);
  PISA_DEC_CASE(128, 1) PISA_DEC_CASE(128, 2) PISA_DEC_CASE(128, 4) PISA_DEC_CASE(128, 8)
  PISA_DEC_CASE(64, 1) PISA_DEC_CASE(64, 2) PISA_DEC_CASE(64, 4) PISA_DEC_CASE(64, 8)
#undef PISA_DEC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pisa
