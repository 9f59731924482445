// route.cu -- top-down pyramid routing over the intermediate levels
// (levels L .. 2).  rcap.io post on "Block Sparse Attention with Log-Linear
// Complexity": "Selection walks the tree top-down" (score a bounded set of at
// most g*K candidates, keep Top-K, expand the kept nodes' children) and "The
// scoring rule matters" (a candidate's score is the LogSumExp over its child
// summaries); agihunt.info summary, kernel paragraph (the heads of a GQA group
// share one selection: their scores are summed).
//
// Layout.  A warp walks 32/LQ queries, LQ lanes each (LQ = 8, or 16 when a
// child row needs more lanes).  Within a query's lanes, each child summary
// row is split over LPN consecutive lanes; a
// lane keeps DQ = 64/G dims of all G query heads in registers (64 floats),
// multiplies them against its slice of the row with packed fp32x2 FMAs, and
// the LPN lanes reduce their G partial sums with a transposing butterfly.
// Candidates (at most 2K per level) live in per-query shared-memory lists in
// ascending node order; a candidate's rank is computed with shuffles over a
// 64-bit key (score, then lower index first), and the kept nodes' eligible
// children form the next list (ping-pong buffers).
//
// Work saving that does not change the result: a candidate c whose two
// children c0, c1 are both eligible already knows x = s q . mu_c from the
// level above (c was a child there), and mu_c = (n0 mu_c0 + n1 mu_c1) /
// (n0 + n1), so s q . mu_c1 = ((n0 + n1) x - n0 (s q . mu_c0)) / n1: one dot
// per candidate instead of two below the first scored level.
#include "pisa_common.cuh"
#include "pisa_internal.h"

namespace pisa {

template <int G, int NC>
struct RouteQData {
  int32_t cand[2][NC];    // ping-pong candidate lists (ascending node order)
  float x[2][NC][G];      // s2 * q_g . mu_cand, when known
  int32_t hasx[2][NC];
  int32_t work[2 * NC];   // child rows whose dots are computed this level
  float y[2 * NC][G];     // their dots (s2 units)
};

// Per-query slice, padded so that the slices of the QPW queries sharing a
// warp start 32/QPW banks apart: their lanes then never collide on a bank.
template <int G, int NC, int QPW>
struct RouteQ : RouteQData<G, NC> {
  static constexpr int kWords = (int)(sizeof(RouteQData<G, NC>) / 4);
  static constexpr int kPad = ((32 / QPW) - kWords % 32 + 64) % 32;
  int32_t pad[kPad > 0 ? kPad : 1];
};

__device__ __forceinline__ uint32_t orderable(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum within an LQ-lane segment.
template <int LQ>
__device__ __forceinline__ int scan_seg(int v, int ll, int* tot) {
  int x = v;
#pragma unroll
  for (int o = 1; o < LQ; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o, LQ);
    if (ll >= o) x += y;
  }
  *tot = __shfl_sync(0xffffffffu, x, LQ - 1, LQ);
  return x - v;
}

// Max over the warp's query groups (lanes LQ apart).
template <int LQ>
__device__ __forceinline__ int warp_max_groups(int v) {
#pragma unroll
  for (int o = LQ; o < 32; o <<= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Dot of the second child from the candidate's own dot (see the header):
// exact 2x - a for equal counts, the count-weighted form otherwise.
__device__ __forceinline__ float sibling_dot(float x, float a, int n0, int n1) {
  if (n0 == n1) return 2.0f * x - a;
  return ((float)(n0 + n1) * x - (float)n0 * a) / (float)n1;
}

// Keys present in node (level, j) of a prefill of N keys (32-bit form).
__device__ __forceinline__ int node_count32(int C, int level, int j, int64_t N) {
  const int64_t w = (int64_t)C << (level - 1);
  const int64_t c = N - (int64_t)j * w;
  return (int)(c < 0 ? 0 : (c > w ? w : c));
}

// Level-`level` node j meets E = [1, e_hi] (e_hi = qb - 2 >= 1).
__device__ __forceinline__ bool elig32(int level, int j, int e_hi) {
  return (j << (level - 1)) <= e_hi && (((j + 1) << (level - 1)) - 1) >= 1;
}

// Dots (s2 units) of the two children of a query's path node at `level`
// under prefix-consistent summaries: a complete left child and the path
// child's prefix summary (see prefix_path.cu).  path: [nq, L, 2, G].
template <int G>
__device__ __forceinline__ void path_children(const float* __restrict__ path, int64_t qc, int L, int64_t qb,
                                              int level, int g, float* a, float* bb) {
  const float* pp = path + qc * L * 2 * G;
  const float pc = pp[(level - 2) * 2 * G + g];
  if ((qb >> (level - 2)) & 1) {
    *a = pp[(level - 1) * 2 * G + G + g];
    *bb = pc;
  } else {
    *a = pc;
    *bb = pc;
  }
}

template <int D, int G, int KM, int WARPS, int LQ>
__global__ void __launch_bounds__(WARPS * 32) route_kernel(Prob pr, Pyr s, const void* __restrict__ q,
                                                           const float* __restrict__ pyr,
                                                           const float* __restrict__ path,
                                                           int32_t* __restrict__ kept2,
                                                           int32_t* __restrict__ trace) {
  constexpr int NC = 2 * KM;
  constexpr int CPL = NC / LQ;                  // candidates per lane
  constexpr int DQ = (64 / G) < D ? 64 / G : D; // dims per lane (DQ * G <= 64 registers)
  constexpr int LPN = D / DQ;                   // lanes per child row
  constexpr int NPP = LQ / LPN;                 // rows per pass per query
  constexpr int QPW = 32 / LQ;                  // queries per warp
  static_assert(LPN <= LQ && NC % LQ == 0, "lane split");
  extern __shared__ __align__(16) unsigned char smem_raw[];
  RouteQ<G, NC, QPW>& sm = reinterpret_cast<RouteQ<G, NC, QPW>*>(smem_raw)[threadIdx.x / LQ];
  const int lane = threadIdx.x & 31, ll = lane % LQ;
  const int64_t nq = pr.B * pr.Hkv * pr.N;
  const int64_t qi = ((int64_t)blockIdx.x * WARPS + threadIdx.x / 32) * QPW + lane / LQ;
  const bool live = qi < nq;
  const int64_t qc = live ? qi : nq - 1;
  const int64_t t = qc % pr.N, bh = qc / pr.N;
  const int64_t b = bh / pr.Hkv, h = bh % pr.Hkv;
  const int K = pr.K;
  const int64_t qb = t / s.C;
  int32_t* kout = kept2 + qc * K;
  int32_t* trow = (trace && live) ? trace + qc * (int64_t)s.L * K : nullptr;
  if (trow)
    for (int i = ll; i < s.L * K; i += LQ) trow[i] = -1;

  int l0 = 0;
  if (live && qb - 2 >= 1) {
    for (int level = s.L; level >= 2; --level)
      if (eligible_count(level, qb) > K) { l0 = level; break; }
    if (trow)
      for (int level = s.L; level >= 2 && level > l0; --level) {
        const int64_t n = eligible_count(level, qb);
        for (int i = ll; i < n; i += LQ) trow[(level - 1) * K + i] = i;
      }
    if (l0 == 0) {
      const int64_t n2 = eligible_count(2, qb);
      for (int i = ll; i < K; i += LQ) kout[i] = i < n2 ? i : -1;
    }
  } else if (live) {
    for (int i = ll; i < K; i += LQ) kout[i] = -1;
  }
  const int l0w = warp_max_groups<LQ>(l0);
  if (l0w == 0) return;  // warp-uniform

  // This lane's slice of the query heads, scaled by s * log2(e), as pairs.
  // Its i-th group of 4 dims is [(i * LPN + chunk) * 4, +4): the LPN lanes of
  // a row read consecutive 16-byte pieces, so each load of a row group is one
  // contiguous 16 * LPN-byte span (few L1 wavefronts per warp load).
  const int chunk = ll % LPN;
  float2 q2[G][DQ / 2];
  {
    const bool bf16 = pr.dtype == PISA_BF16;
    const size_t esz = bf16 ? 2 : 4;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const char* p = reinterpret_cast<const char*>(q) + (((b * pr.Hq + h * G + g) * pr.N + t) * D) * esz;
#pragma unroll
      for (int c = 0; c < DQ; c += 4) {
        float v[4];
        load4(p + ((c / 4) * LPN + chunk) * 4 * esz, bf16, v);
        q2[g][c / 2] = make_float2(v[0] * pr.scale2, v[1] * pr.scale2);
        q2[g][c / 2 + 1] = make_float2(v[2] * pr.scale2, v[3] * pr.scale2);
      }
    }
  }
  const float* ph = pyr + bh * s.P * D;

  int cur = 0;
  int nc = l0 > 0 ? (int)eligible_count(l0, qb) : 0;
  for (int i = ll; i < nc; i += LQ) { sm.cand[0][i] = i; sm.hasx[0][i] = 0; }
  const int e_hi = (int)(qb - 2);
  __syncwarp();

  for (int level = l0w; level >= 2; --level) {
    const bool act = level <= l0;
    const int ncur = act ? nc : 0;
    const int ncap = (int)s.size[level - 2];

    // 1. work list: the children whose dot products are needed
    int c0v[CPL];
    int e0v[CPL], e1v[CPL], s0v[CPL], s1v[CPL];
    int nwork = 0;
#pragma unroll
    for (int sl = 0; sl < CPL; ++sl) {
      const int i = sl * LQ + ll;
      const bool valid = i < ncur;
      const int c0 = valid ? 2 * sm.cand[cur][i] : 0;
      const int e0 = valid && c0 < ncap && elig32(level - 1, c0, e_hi);
      const int e1 = valid && c0 + 1 < ncap && elig32(level - 1, c0 + 1, e_hi);
      const int der = e0 && e1 && sm.hasx[cur][i];
      int tot;
      int p = nwork + scan_seg<LQ>(e0 + (e1 && !der), ll, &tot);
      s0v[sl] = e0 ? p : -1;
      if (e0) sm.work[p++] = c0;
      s1v[sl] = e1 ? (der ? -2 : p) : -1;
      if (e1 && !der) sm.work[p] = c0 + 1;
      nwork += tot;
      c0v[sl] = c0; e0v[sl] = e0; e1v[sl] = e1;
    }
    __syncwarp();

    // 2. dot products, NPP child rows per pass per query
    {
      const float* lvl = ph + s.off[level - 2] * D + chunk * 4;
      const int nmax = warp_max_groups<LQ>(nwork);
#pragma unroll 2
      for (int w0 = 0; w0 < nmax; w0 += NPP) {
        const int w = w0 + ll / LPN;
        const bool ok = w < nwork;
        const float* row = lvl + (int64_t)(ok ? sm.work[w] : 0) * D;
        float2 acc[G];
#pragma unroll
        for (int g = 0; g < G; ++g) acc[g] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int c = 0; c < DQ; c += 4) {
          const float4 m =
              ok ? __ldg(reinterpret_cast<const float4*>(row + (c / 4) * LPN * 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
          const float2 m01 = make_float2(m.x, m.y), m23 = make_float2(m.z, m.w);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            acc[g] = __ffma2_rn(q2[g][c / 2], m01, acc[g]);
            acc[g] = __ffma2_rn(q2[g][c / 2 + 1], m23, acc[g]);
          }
        }
        float v[G];
#pragma unroll
        for (int g = 0; g < G; ++g) v[g] = acc[g].x + acc[g].y;
        // reduce over the LPN lanes of the row; each lane ends with one head
        int hbase = 0, nv = G;
#pragma unroll
        for (int o = LPN / 2; o >= 1; o >>= 1) {
          if (nv > 1) {
            const int hf = nv / 2;
            const bool up = (ll & o) != 0;
#pragma unroll
            for (int i = 0; i < G / 2; ++i) {
              if (i < hf) {
                const float send = up ? v[i] : v[i + hf];
                const float keep = up ? v[i + hf] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o, LQ);
              }
            }
            if (up) hbase += hf;
            nv = hf;
          } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], o, LQ);
          }
        }
        if (ok) sm.y[w][hbase] = v[0];
      }
    }
    __syncwarp();

    // 3. scores and 64-bit rank keys (higher score first, then lower index)
    uint64_t key[CPL];
#pragma unroll
    for (int sl = 0; sl < CPL; ++sl) {
      const int i = sl * LQ + ll;
      key[sl] = 0;
      if (i < ncur) {
        const int s0 = s0v[sl], s1 = s1v[sl];
        int n0 = 0, n1 = 0;
        if (s1 == -2) {
          n0 = node_count32(s.C, level - 1, c0v[sl], s.N);
          n1 = node_count32(s.C, level - 1, c0v[sl] + 1, s.N);
        }
        const bool onpath = path && sm.cand[cur][i] == (int)(qb >> (level - 1));
        float sc = 0.0f;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float a = s0 >= 0 ? sm.y[s0][g] : 0.0f;
          float bb = 0.0f;
          if (s1 >= 0) bb = sm.y[s1][g];
          else if (s1 == -2) bb = sibling_dot(sm.x[cur][i][g], a, n0, n1);
          if (onpath) path_children<G>(path, qc, s.L, qb, level, g, &a, &bb);
          sc += (s0 >= 0 && s1 != -1) ? pair_score(pr.scorer, a, bb) : (s0 >= 0 ? a : bb);
        }
        if (sc != sc) sc = -INFINITY;  // NaN ranks last
        key[sl] = ((uint64_t)orderable(sc) << 32) | (uint32_t)(~(uint32_t)sm.cand[cur][i]);
      }
    }
    int rank[CPL];
#pragma unroll
    for (int sl = 0; sl < CPL; ++sl) rank[sl] = 0;
#pragma unroll
    for (int sj = 0; sj < CPL; ++sj) {
      const uint32_t khi = (uint32_t)(key[sj] >> 32), klo = (uint32_t)key[sj];
#pragma unroll
      for (int l = 0; l < LQ; ++l) {
        const uint64_t kj = ((uint64_t)__shfl_sync(0xffffffffu, khi, l, LQ) << 32) |
                            __shfl_sync(0xffffffffu, klo, l, LQ);
#pragma unroll
        for (int sl = 0; sl < CPL; ++sl) rank[sl] += kj > key[sl] ? 1 : 0;
      }
    }

    // 4. kept set (index order), next candidates or the kept level-2 nodes
    const int nxt = cur ^ 1;
    int nkept = 0, nchild = 0;
#pragma unroll
    for (int sl = 0; sl < CPL; ++sl) {
      const int i = sl * LQ + ll;
      const int keep = (i < ncur && rank[sl] < K) ? 1 : 0;
      const int nch = keep && level > 2 ? e0v[sl] + e1v[sl] : 0;
      int ktot, ctot;
      const int kp = nkept + scan_seg<LQ>(keep, ll, &ktot);
      int cp = nchild + scan_seg<LQ>(nch, ll, &ctot);
      if (keep) {
        const int32_t ci = sm.cand[cur][i];
        if (trow) trow[(level - 1) * K + kp] = ci;
        if (level == 2) kout[kp] = ci;
        if (nch) {
          const int s0 = s0v[sl], s1 = s1v[sl];
          int n0 = 0, n1 = 0;
          if (s1 == -2) {
            n0 = node_count32(s.C, level - 1, c0v[sl], s.N);
            n1 = node_count32(s.C, level - 1, c0v[sl] + 1, s.N);
          }
          const bool onpath = path && ci == (int)(qb >> (level - 1));
          if (e0v[sl]) {
            sm.cand[nxt][cp] = c0v[sl];
#pragma unroll
            for (int g = 0; g < G; ++g) {
              float a = sm.y[s0][g], bb = 0.0f;
              if (onpath) path_children<G>(path, qc, s.L, qb, level, g, &a, &bb);
              sm.x[nxt][cp][g] = a;
            }
            sm.hasx[nxt][cp] = 1;
            ++cp;
          }
          if (e1v[sl]) {
            sm.cand[nxt][cp] = c0v[sl] + 1;
#pragma unroll
            for (int g = 0; g < G; ++g) {
              float a = e0v[sl] ? sm.y[s0][g] : 0.0f;
              float bb = s1 >= 0 ? sm.y[s1][g] : sibling_dot(sm.x[cur][i][g], a, n0, n1);
              if (onpath) path_children<G>(path, qc, s.L, qb, level, g, &a, &bb);
              sm.x[nxt][cp][g] = bb;
            }
            sm.hasx[nxt][cp] = 1;
          }
        }
      }
      nkept += ktot;
      nchild += ctot;
    }
    if (level == 2 && act)
      for (int i = nkept + ll; i < K; i += LQ) kout[i] = -1;
    if (act) {
      nc = nchild;
      cur = nxt;
    }
    __syncwarp();
  }
}

template <int D, int G, int KM, int WARPS>
static cudaError_t launch_route_t(const Prob& pr, const Pyr& s, const void* q, const float* pyr, const float* path,
                                  int32_t* kept2, int32_t* trace, cudaStream_t st) {
  constexpr int DQ = (64 / G) < D ? 64 / G : D;
  constexpr int LQ = (D / DQ) > 8 ? 16 : 8;  // lanes per query
  const size_t smem = sizeof(RouteQ<G, 2 * KM, 32 / LQ>) * (32 / LQ) * WARPS;
  auto kern = route_kernel<D, G, KM, WARPS, LQ>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t nq = pr.B * pr.Hkv * pr.N;
  const int64_t grid = ceil_div64(nq, (32 / LQ) * WARPS);
  note_launch();
  kern<<<(unsigned)grid, WARPS * 32, smem, st>>>(pr, s, q, pyr, path, kept2, trace);
  return cudaGetLastError();
}

template <int D, int G>
static cudaError_t launch_route_k(const Prob& pr, const Pyr& s, const void* q, const float* pyr, const float* path,
                                  int32_t* kept2, int32_t* trace, cudaStream_t st) {
  if (pr.K <= 8) return launch_route_t<D, G, 8, 8>(pr, s, q, pyr, path, kept2, trace, st);
  if (pr.K <= 16) return launch_route_t<D, G, 16, 8>(pr, s, q, pyr, path, kept2, trace, st);
  return launch_route_t<D, G, 32, 4>(pr, s, q, pyr, path, kept2, trace, st);
}

cudaError_t launch_route(const Prob& pr, const Pyr& s, const void* q, const float* pyr, const float* path,
                         int32_t* kept2, int32_t* trace, int32_t* /*status*/, cudaStream_t st) {
  if (pr.B * pr.Hkv * pr.N == 0) return cudaSuccess;
#define PISA_ROUTE_CASE(DD, GG) \
  if (pr.d == DD && pr.G == GG) return launch_route_k<DD, GG>(pr, s, q, pyr, path, kept2, trace, st);
  PISA_ROUTE_CASE(128, 1) PISA_ROUTE_CASE(128, 2) PISA_ROUTE_CASE(128, 4) PISA_ROUTE_CASE(128, 8)
  PISA_ROUTE_CASE(64, 1) PISA_ROUTE_CASE(64, 2) PISA_ROUTE_CASE(64, 4) PISA_ROUTE_CASE(64, 8)
#undef PISA_ROUTE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pisa
