// route_mma.cu -- top-down pyramid routing with the child dot products on
// the tensor cores (bf16 inputs, GQA groups of 4 query heads).  Same walk and
// scoring as route.cu (rcap.io post on "Block Sparse Attention with
// Log-Linear Complexity": "Selection walks the tree top-down", "The scoring
// rule matters"; agihunt.info summary, kernel paragraph: one selection per
// GQA group, the heads' scores summed).
//
// A warp walks two queries.  Per level, the child summary rows each query
// needs (one per candidate whose own dot is known, two at the start level)
// are multiplied against its four query-head vectors as warp-level m16n8k16
// MMAs with fp32 accumulation: for one query, A = 16 rows = 8 child nodes x
// the two halves of the d dims, B = 8 columns = the 4 heads x the two halves;
// only the blocks where row half = column half are used, and one shuffle
// pair adds a node's two halves.  With the rows stored half-interleaved,
// the eight lanes of a node read one whole 128-byte line per load.  The
// query rows are bf16, so they are exact in the MMA; each fp32 summary is
// split into bf16 hi + lo (mu = hi + lo to about 2^-16 relative) and
// multiplied twice, so the dots match an fp32 computation to ~1e-6.  The two
// pieces are prepared once per call by split_pyramid_kernel.
//
// The candidate bookkeeping (work list by ballot prefix sums, scores, Top-K
// by 32-bit orderable keys with the slot order breaking ties, expansion
// into ascending ping-pong lists) runs on 16 lanes per query.
#include <algorithm>

#include "pisa_common.cuh"
#include "pisa_internal.h"

namespace pisa {

template <int NC>
struct RouteMmaQ {
  float4 x[2][NC];  // own dot per head of each candidate (known below the start level)
  float4 y[2 * NC];  // child dots per head, by work-list position
  int32_t cand[2][NC];
  int32_t work[2 * NC];
};

template <int NC>
struct RouteMmaQPad : RouteMmaQ<NC> {
  // the two queries of a warp start 16 banks apart
  static constexpr int kWords = (int)(sizeof(RouteMmaQ<NC>) / 4);
  static constexpr int kPad = (16 - kWords % 32 + 64) % 32;
  int32_t pad[kPad > 0 ? kPad : 4];
};

__device__ __forceinline__ uint32_t orderable_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum of v in {0, 1, 2} over the 16 lanes of this lane's half
// of the warp (two ballots, no shuffles); *tot receives the half's total.
__device__ __forceinline__ int prefix16(int v, int lane, int* tot) {
  const unsigned b0 = __ballot_sync(0xffffffffu, v & 1);
  const unsigned b1 = __ballot_sync(0xffffffffu, v & 2);
  const unsigned hm = (lane & 16) ? 0xffff0000u : 0x0000ffffu;
  const unsigned lt = hm & ((1u << lane) - 1u);
  *tot = __popc(b0 & hm) + 2 * __popc(b1 & hm);
  return __popc(b0 & lt) + 2 * __popc(b1 & lt);
}

__device__ __forceinline__ bool elig_node(int level, int j, int e_hi) {
  return (j << (level - 1)) <= e_hi && (((j + 1) << (level - 1)) - 1) >= 1;
}

__device__ __forceinline__ int count_node(int C, int level, int j, int64_t N) {
  const int64_t w = (int64_t)C << (level - 1);
  const int64_t c = N - (int64_t)j * w;
  return (int)(c < 0 ? 0 : (c > w ? w : c));
}

__device__ __forceinline__ float sib_dot(float x, float a, int n0, int n1) {
  if (n0 == n1) return 2.0f * x - a;
  return ((float)(n0 + n1) * x - (float)n0 * a) / (float)n1;
}

__device__ __forceinline__ float comp(const float4& v, int g) {
  return g == 0 ? v.x : (g == 1 ? v.y : (g == 2 ? v.z : v.w));
}

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// fp32 pyramid -> bf16 hi (rounded) and lo (rounded residual).  Within each
// row of D dims the elements are permuted so that 128-byte line bb holds dims
// [32 bb, 32 bb + 32) of the first half followed by the same 32 dims of the
// second half: eight lanes then read one line per node (see the dot phase).
__global__ void split_pyramid_kernel(int64_t n, int D, const float* __restrict__ pyr,
                                     __nv_bfloat16* __restrict__ hi, __nv_bfloat16* __restrict__ lo) {
  const int hd = D / 2;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % D);
    const int64_t pos = (i - c) + ((c % hd) / 32) * 64 + (c / hd) * 32 + (c & 31);
    const float v = pyr[i];
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    hi[pos] = h;
    lo[pos] = __float2bfloat16_rn(v - __bfloat162float(h));
  }
}

// MMA layout.  One m16n8k16 sequence serves one query and 8 child nodes:
// A row r is (node r/2 of rows 0..7 or 4 + (r-8)/2, half r%2 of the D dims),
// B column j is (query head j%4, half j/4), so only the blocks where the row
// half equals the column half are used and a node's dot is the sum of its two
// halves' results.  K-block mapping: k-step pair bb, thread-in-group t covers
// dims 32 bb + 8 t + {0..7} of its half (one 16-byte load; words x, y for the
// first step and z, w for the second).  With the permuted row layout the
// eight lanes of a node read one contiguous 128-byte line per load.
// kLse: the log-sum-exp scorer (the PISA default), compiled on its own so the
// truncated scorers cost it nothing.
template <int D, int KM, int WARPS, bool kLse>
__global__ void __launch_bounds__(WARPS * 32, 16 / WARPS) route_mma_kernel(Prob pr, Pyr s, const uint16_t* __restrict__ q,
                                                               const uint16_t* __restrict__ phi,
                                                               const uint16_t* __restrict__ plo,
                                                               int32_t* __restrict__ kept2,
                                                               int32_t* __restrict__ trace) {
  constexpr int G = 4;
  constexpr int NC = 2 * KM;
  constexpr int CPL = NC / 16;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  RouteMmaQPad<NC>& sm = reinterpret_cast<RouteMmaQPad<NC>*>(smem_raw)[threadIdx.x / 16];
  RouteMmaQPad<NC>* smw = reinterpret_cast<RouteMmaQPad<NC>*>(smem_raw) + (threadIdx.x / 32) * 2;
  const int lane = threadIdx.x & 31, ll = lane & 15, half = lane >> 4;
  const int grp = lane >> 2, tig = lane & 3;  // MMA group id / thread in group
  // query counts are below 2^31 (the prefill size limit), so 32-bit index math
  const uint32_t nq = (uint32_t)(pr.B * pr.Hkv * pr.N), N32 = (uint32_t)pr.N;
  const uint32_t qi = (blockIdx.x * WARPS + threadIdx.x / 32) * 2 + half;
  const bool live = qi < nq;
  const uint32_t qc = live ? qi : nq - 1;
  const int64_t t = qc % N32;
  const int K = pr.K;
  const int64_t qb = t / s.C;
  int32_t* kout = kept2 + (int64_t)qc * K;
  int32_t* trow = (trace && live) ? trace + (int64_t)qc * s.L * K : nullptr;
  if (trow)
    for (int i = ll; i < s.L * K; i += 16) trow[i] = -1;

  int l0 = 0;
  if (live && qb - 2 >= 1) {
    // start level: the highest level with more than K eligible nodes, i.e.
    // the largest l <= L with (qb - 2) >> (l - 1) >= K
    const uint32_t xk = (uint32_t)(qb - 2) / (uint32_t)K;
    if (xk >= 2) l0 = min((int)s.L, 32 - __clz(xk));
    if (l0 < 2) l0 = 0;
    if (trow)
      for (int level = s.L; level >= 2 && level > l0; --level) {
        const int64_t n = eligible_count(level, qb);
        for (int i = ll; i < n; i += 16) trow[(level - 1) * K + i] = i;
      }
    if (l0 == 0) {
      const int64_t n2 = eligible_count(2, qb);
      for (int i = ll; i < K; i += 16) kout[i] = i < n2 ? i : -1;
    }
  } else if (live) {
    for (int i = ll; i < K; i += 16) kout[i] = -1;
  }
  const int l0w = max(l0, __shfl_xor_sync(0xffffffffu, l0, 16));
  if (l0w == 0) return;  // warp-uniform

  // B fragments of both queries: column grp = (head grp % 4, half grp / 4)
  constexpr int NB = D / 64;  // k-step pairs per half
  const uint32_t qw = (blockIdx.x * WARPS + threadIdx.x / 32) * 2;
  uint32_t bq[2][NB][4];
  int64_t pbase[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const uint32_t qu = min(qw + u, nq - 1);
    const uint32_t tu = qu % N32, bhu = qu / N32;
    const uint32_t Hkv = (uint32_t)pr.Hkv;
    const int64_t qrow = ((int64_t)((bhu / Hkv) * (uint32_t)pr.Hq + (bhu % Hkv) * G + (grp & 3)) * pr.N + tu) * D +
                         (grp >> 2) * (D / 2) + 8 * tig;
#pragma unroll
    for (int bb = 0; bb < NB; ++bb) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(q + qrow + 32 * bb));
      bq[u][bb][0] = v.x; bq[u][bb][1] = v.y; bq[u][bb][2] = v.z; bq[u][bb][3] = v.w;
    }
    // the two queries of a warp may belong to different (b, h) rows of the pyramid
    pbase[u] = (int64_t)bhu * s.P * D;
  }

  int cur = 0;
  int nc = l0 > 0 ? (int)eligible_count(l0, qb) : 0;
  for (int i = ll; i < nc; i += 16) sm.cand[0][i] = i;
  const int e_hi = (int)(qb - 2);
  __syncwarp();

  for (int level = l0w; level >= 2; --level) {
    const bool act = level <= l0;
    const int ncur = act ? nc : 0;
    const int ncap = (int)s.size[level - 2];
    const bool hx = level < l0;  // candidates made by expansion carry their own dot

    // 1. work list: the first child of every candidate, and the second one
    //    unless it follows from the candidate's own dot
    int c0v[CPL], e0v[CPL], e1v[CPL], s0v[CPL], s1v[CPL];
    int nwork = 0;
#pragma unroll
    for (int sl = 0; sl < CPL; ++sl) {
      const int i = sl * 16 + ll;
      const bool valid = i < ncur;
      const int c0 = valid ? 2 * sm.cand[cur][i] : 0;
      const int e0 = valid && c0 < ncap && elig_node(level - 1, c0, e_hi);
      const int e1 = valid && c0 + 1 < ncap && elig_node(level - 1, c0 + 1, e_hi);
      const int der = e0 && e1 && hx;
      int tot;
      int p = nwork + prefix16(e0 + (e1 && !der), lane, &tot);
      s0v[sl] = e0 ? p : -1;
      if (e0) sm.work[p++] = c0;
      s1v[sl] = e1 ? (der ? -2 : p) : -1;
      if (e1 && !der) sm.work[p] = c0 + 1;
      nwork += tot;
      c0v[sl] = c0; e0v[sl] = e0; e1v[sl] = e1;
    }
    __syncwarp();

    // 2. dot products: per query, 8 child nodes per m16n8k16 sequence
    {
      const int nw[2] = {__shfl_sync(0xffffffffu, nwork, 0), __shfl_sync(0xffffffffu, nwork, 16)};
      const int nmax = max(nw[0], nw[1]);
      // per-level row bases of both queries (hi and lo pyramids); a row adds node * D
      const int64_t loff = s.off[level - 2] * D + (grp & 1) * 32 + 8 * tig;
      const uint16_t* hbase[2] = {phi + pbase[0] + loff, phi + pbase[1] + loff};
      const uint16_t* lbase[2] = {plo + pbase[0] + loff, plo + pbase[1] + loff};
      // lanes (even group, t < 2) finish node grp/2, lanes (odd group, t >= 2) node 4 + grp/2
      const bool roleA = !(grp & 1) && tig < 2, roleB = (grp & 1) && tig >= 2;
      const float sc = pr.scale2;
      for (int r0 = 0; r0 < nmax; r0 += 8) {
        uint4 hv[2][2][NB], lv[2][2][NB];  // [query][row grp / grp + 8][pair]
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int w = r0 + 4 * rr + (grp >> 1);
            const uint32_t ro = (uint32_t)(w < nw[u] ? smw[u].work[w] : 0) * (uint32_t)D;  // < 2^27
#pragma unroll
            for (int bb = 0; bb < NB; ++bb) {
              hv[u][rr][bb] = __ldg(reinterpret_cast<const uint4*>(hbase[u] + ro + 64 * bb));
              lv[u][rr][bb] = __ldg(reinterpret_cast<const uint4*>(lbase[u] + ro + 64 * bb));
            }
          }
        // four independent accumulator chains: (query) x (hi, lo)
        float dh[2][4], dl[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int e = 0; e < 4; ++e) dh[u][e] = dl[u][e] = 0.0f;
#pragma unroll
        for (int bb = 0; bb < NB; ++bb)
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const uint4 h0 = hv[u][0][bb], h1 = hv[u][1][bb], l0v = lv[u][0][bb], l1v = lv[u][1][bb];
            mma_16816(dh[u], h0.x, h1.x, h0.y, h1.y, bq[u][bb][0], bq[u][bb][1]);
            mma_16816(dl[u], l0v.x, l1v.x, l0v.y, l1v.y, bq[u][bb][0], bq[u][bb][1]);
            mma_16816(dh[u], h0.z, h1.z, h0.w, h1.w, bq[u][bb][2], bq[u][bb][3]);
            mma_16816(dl[u], l0v.z, l1v.z, l0v.w, l1v.w, bq[u][bb][2], bq[u][bb][3]);
          }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          float d[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) d[e] = dh[u][e] + dl[u][e];
          // add the two halves: partner lane = lane ^ 6 (group ^ 1, t ^ 2)
          const float x0 = __shfl_xor_sync(0xffffffffu, roleA ? d[2] : d[0], 6);
          const float x1 = __shfl_xor_sync(0xffffffffu, roleA ? d[3] : d[1], 6);
          const int w = r0 + (roleA ? 0 : 4) + (grp >> 1);
          if ((roleA || roleB) && w < nw[u]) {
            const float2 v = roleA ? make_float2((d[0] + x0) * sc, (d[1] + x1) * sc)
                                   : make_float2((d[2] + x0) * sc, (d[3] + x1) * sc);
            *reinterpret_cast<float2*>(reinterpret_cast<float*>(&smw[u].y[w]) + 2 * (tig & 1)) = v;
          }
        }
      }
    }
    __syncwarp();

    // 3. scores and rank keys (higher score first, then lower index)
    uint32_t key[CPL];
    float4 ya[CPL], yb[CPL];
#pragma unroll
    for (int sl = 0; sl < CPL; ++sl) {
      const int i = sl * 16 + ll;
      key[sl] = 0;
      ya[sl] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      yb[sl] = ya[sl];
      if (i < ncur) {
        const int s0 = s0v[sl], s1 = s1v[sl];
        if (s0 >= 0) ya[sl] = sm.y[s0];
        if (s1 >= 0) {
          yb[sl] = sm.y[s1];
        } else if (s1 == -2) {
          // only the last node of a level can hold fewer keys than the others
          const bool full = c0v[sl] + 2 < ncap;
          const int n0 = full ? 1 : count_node(s.C, level - 1, c0v[sl], s.N);
          const int n1 = full ? 1 : count_node(s.C, level - 1, c0v[sl] + 1, s.N);
          const float4 xv = sm.x[cur][i];
          yb[sl] = make_float4(sib_dot(xv.x, ya[sl].x, n0, n1), sib_dot(xv.y, ya[sl].y, n0, n1),
                               sib_dot(xv.z, ya[sl].z, n0, n1), sib_dot(xv.w, ya[sl].w, n0, n1));
        }
        float scv = 0.0f;
        if constexpr (kLse) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float a = comp(ya[sl], g), bb = comp(yb[sl], g);
            scv += (s0 >= 0 && s1 != -1) ? lse2_pair(a, bb) : (s0 >= 0 ? a : bb);
          }
        } else {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float a = comp(ya[sl], g), bb = comp(yb[sl], g);
            scv += (s0 >= 0 && s1 != -1) ? pair_score(pr.scorer, a, bb) : (s0 >= 0 ? a : bb);
          }
        }
        if (scv == 0.0f) scv = 0.0f;        // -0 ranks like +0
        if (scv != scv) scv = -INFINITY;     // NaN ranks last (keys stay <= 0xff800000)
        key[sl] = orderable_key(scv);
      }
    }
    int rank[CPL];
#pragma unroll
    for (int sl = 0; sl < CPL; ++sl) rank[sl] = 0;
#pragma unroll
    for (int sj = 0; sj < CPL; ++sj) {
#pragma unroll
      for (int l = 0; l < 16; ++l) {
        const uint32_t kj = __shfl_sync(0xffffffffu, key[sj], l, 16);
#pragma unroll
        for (int sl = 0; sl < CPL; ++sl) {
          // equal scores: the lower slot (the lower node index) ranks first.
          // Keys of real scores are at most 0xff800000, so kj + 1 cannot wrap.
          const uint32_t before = (sj < sl || (sj == sl && l < ll)) ? 1u : 0u;
          rank[sl] += (kj + before > key[sl]) ? 1 : 0;
        }
      }
    }

    // 4. kept set (index order), next candidates (ascending) or the kept level-2 nodes
    const int nxt = cur ^ 1;
    int nkept = 0, nchild = 0;
#pragma unroll
    for (int sl = 0; sl < CPL; ++sl) {
      const int i = sl * 16 + ll;
      const int keep = (i < ncur && rank[sl] < K) ? 1 : 0;
      const int nch = keep && level > 2 ? e0v[sl] + e1v[sl] : 0;
      int ktot, ctot;
      const int kp = nkept + prefix16(keep, lane, &ktot);
      int cp = nchild + prefix16(nch, lane, &ctot);
      if (keep) {
        const int32_t ci = sm.cand[cur][i];
        if (trow) trow[(level - 1) * K + kp] = ci;
        if (level == 2) kout[kp] = ci;
        if (e0v[sl] && nch) {
          sm.cand[nxt][cp] = c0v[sl];
          sm.x[nxt][cp] = ya[sl];
          ++cp;
        }
        if (e1v[sl] && nch) {
          sm.cand[nxt][cp] = c0v[sl] + 1;
          sm.x[nxt][cp] = yb[sl];
        }
      }
      nkept += ktot;
      nchild += ctot;
    }
    if (level == 2 && act)
      for (int i = nkept + ll; i < K; i += 16) kout[i] = -1;
    if (act) {
      nc = nchild;
      cur = nxt;
    }
    __syncwarp();
  }
}

template <int D, int KM, int WARPS, bool kLse>
static cudaError_t launch_route_mma_t(const Prob& pr, const Pyr& s, const void* q, const uint16_t* phi,
                                      const uint16_t* plo, int32_t* kept2, int32_t* trace, cudaStream_t st) {
  const size_t smem = sizeof(RouteMmaQPad<2 * KM>) * 2 * WARPS;
  auto kern = route_mma_kernel<D, KM, WARPS, kLse>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t nq = pr.B * pr.Hkv * pr.N;
  note_launch();
  kern<<<(unsigned)ceil_div64(nq, 2 * WARPS), WARPS * 32, smem, st>>>(pr, s, (const uint16_t*)q, phi, plo, kept2,
                                                                        trace);
  return cudaGetLastError();
}

bool route_mma_supported(const Prob& pr) {
  return pr.dtype == PISA_BF16 && pr.G == 4 && (pr.d == 64 || pr.d == 128);
}

cudaError_t launch_route_mma(const Prob& pr, const Pyr& s, const void* q, const float* pyr, uint16_t* phi,
                             uint16_t* plo, int32_t* kept2, int32_t* trace, cudaStream_t st) {
  const int64_t n = pr.B * pr.Hkv * s.P * pr.d;
  if (n == 0) return cudaSuccess;
  note_launch();
  split_pyramid_kernel<<<(unsigned)std::min<int64_t>(ceil_div64(n, 256), 8192), 256, 0, st>>>(
      n, pr.d, pyr, (__nv_bfloat16*)phi, (__nv_bfloat16*)plo);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
#define PISA_RM_CASE(DD, LSE)                                                                             \
  if (pr.d == DD && (pr.scorer == PISA_SCORER_LSE) == LSE) {                                              \
    if (pr.K <= 8) return launch_route_mma_t<DD, 8, 8, LSE>(pr, s, q, phi, plo, kept2, trace, st);        \
    if (pr.K <= 16) return launch_route_mma_t<DD, 16, 8, LSE>(pr, s, q, phi, plo, kept2, trace, st);      \
    return launch_route_mma_t<DD, 32, 4, LSE>(pr, s, q, phi, plo, kept2, trace, st);                      \
  }
  PISA_RM_CASE(128, true) PISA_RM_CASE(64, true) PISA_RM_CASE(128, false) PISA_RM_CASE(64, false)
#undef PISA_RM_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pisa
