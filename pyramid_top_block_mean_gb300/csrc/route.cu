// route.cu -- top-down pyramid routing over the intermediate levels
// (levels L .. 2).  rcap.io post on "Block Sparse Attention with Log-Linear
// Complexity": "Selection walks the tree top-down" (score a bounded set of at
// most g*K candidates, keep Top-K, expand the kept nodes' children) and "The
// scoring rule matters" (a candidate's score is the LogSumExp over its child
// summaries); agihunt.info summary, kernel paragraph (the heads of a GQA group
// share one selection: their scores are summed).
//
// One warp walks one (sequence, key head, query position).  The query's G
// head vectors live in registers, lane l holding dims [l*D/32, (l+1)*D/32);
// each child summary is read once per walk with one coalesced vector load per
// lane, all G heads are multiplied against it, and a transposing butterfly
// reduces 32 (node, head) partial sums at once.  Candidate lists, their dot
// products and scores stay in the warp's slice of shared memory.
//
// Work saving that does not change the result: a candidate c whose two
// children c0, c1 are both eligible already knows x = s q . mu_c from the
// level above (c was a child there), and mu_c = (n0 mu_c0 + n1 mu_c1) /
// (n0 + n1), so s q . mu_c1 = ((n0 + n1) x - n0 (s q . mu_c0)) / n1: one dot
// per candidate instead of two below the first scored level.
#include "pisa_common.cuh"
#include "pisa_internal.h"

namespace pisa {

constexpr int kRouteWarps = 8;

template <int G>
struct RouteWarpSm {
  int32_t cand[kMaxCand];          // candidate nodes at the current level
  int32_t nxt[kMaxCand];           // next level's candidates
  float x[kMaxCand][G];            // s2 * q . mu_cand, if known
  float xn[kMaxCand][G];
  int32_t has_x[kMaxCand];
  int32_t has_xn[kMaxCand];
  int32_t work[2 * kMaxCand];      // child nodes whose dot is computed
  float y[2 * kMaxCand][G];        // their dots (s2 units)
  int32_t slot0[kMaxCand], slot1[kMaxCand];  // work slot of each child (-1: none)
  float score[kMaxCand];
};

__device__ __forceinline__ int warp_excl_scan(int v, int* total) {
  const int lane = threadIdx.x & 31;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  *total = __shfl_sync(0xffffffffu, x, 31);
  return x - v;
}

template <int D, int G>
__global__ void __launch_bounds__(kRouteWarps * 32) route_kernel(Prob pr, Pyr s, const void* __restrict__ q,
                                                                 const float* __restrict__ pyr,
                                                                 int32_t* __restrict__ kept2,
                                                                 int32_t* __restrict__ trace) {
  constexpr int DPL = D / 32;   // dims per lane
  constexpr int NB = 32 / G;    // nodes per reduction batch
  extern __shared__ __align__(16) unsigned char smem_raw[];
  RouteWarpSm<G>& sm = reinterpret_cast<RouteWarpSm<G>*>(smem_raw)[threadIdx.x / 32];
  const int lane = threadIdx.x & 31;
  const int64_t qi = (int64_t)blockIdx.x * kRouteWarps + threadIdx.x / 32;
  const int64_t total_q = pr.B * pr.Hkv * pr.N;
  if (qi >= total_q) return;
  const int64_t t = qi % pr.N;
  const int64_t bh = qi / pr.N;          // b * Hkv + h
  const int64_t b = bh / pr.Hkv, h = bh % pr.Hkv;
  const int K = pr.K;
  const int64_t qb = t / s.C;
  int32_t* kout = kept2 + qi * K;
  int32_t* trow = trace ? trace + qi * (int64_t)s.L * K : nullptr;
  if (trow)
    for (int i = lane; i < s.L * K; i += 32) trow[i] = -1;

  const int64_t nE = qb - 2;
  if (nE < 1) {
    for (int i = lane; i < K; i += 32) kout[i] = -1;
    return;
  }

  // First level with more than K eligible nodes (levels above keep all).
  int l0 = 0;
  for (int level = s.L; level >= 2; --level)
    if (eligible_count(level, qb) > K) { l0 = level; break; }
  if (trow) {
    for (int level = s.L; level >= 2 && level > l0; --level) {
      const int64_t n = eligible_count(level, qb);
      for (int i = lane; i < n; i += 32) trow[(level - 1) * K + i] = i;
    }
  }
  if (l0 == 0) {
    const int64_t n2 = eligible_count(2, qb);
    for (int i = lane; i < K; i += 32) kout[i] = i < n2 ? i : -1;
    return;
  }

  // query heads, pre-scaled by s * log2(e)
  float qr[G][DPL];
  {
    const bool bf16 = pr.dtype == PISA_BF16;
    const size_t esz = bf16 ? 2 : 4;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int64_t hq = h * G + g;
      const char* p = reinterpret_cast<const char*>(q) + (((b * pr.Hq + hq) * pr.N + t) * D + lane * DPL) * esz;
      if (DPL == 4) load4(p, bf16, qr[g]);
      else load2(p, bf16, qr[g]);
#pragma unroll
      for (int c = 0; c < DPL; ++c) qr[g][c] *= pr.scale2;
    }
  }
  const float* ph = pyr + bh * s.P * D;

  int nc = (int)eligible_count(l0, qb);  // <= 2K
  for (int i = lane; i < nc; i += 32) { sm.cand[i] = i; sm.has_x[i] = 0; }
  __syncwarp();

  for (int level = l0; level >= 2; --level) {
    const int64_t ncap = s.size[level - 2];   // nodes of the child level
    // 1. work list: the children whose dot products are needed
    int base = 0;
    for (int i0 = 0; i0 < nc; i0 += 32) {
      const int i = i0 + lane;
      int nwork = 0, e0 = 0, e1 = 0, der = 0;
      int64_t c0 = 0;
      if (i < nc) {
        c0 = 2 * (int64_t)sm.cand[i];
        e0 = c0 < ncap && node_eligible(level - 1, c0, qb);
        e1 = c0 + 1 < ncap && node_eligible(level - 1, c0 + 1, qb);
        der = e0 && e1 && sm.has_x[i];
        nwork = e0 + (e1 && !der);
      }
      int tot;
      const int pos = base + warp_excl_scan(nwork, &tot);
      if (i < nc) {
        int p = pos;
        sm.slot0[i] = e0 ? p : -1;
        if (e0) sm.work[p++] = (int32_t)c0;
        // slot1 >= 0: computed; -2: derived from x; -1: not eligible
        sm.slot1[i] = e1 ? (der ? -2 : p) : -1;
        if (e1 && !der) sm.work[p++] = (int32_t)(c0 + 1);
      }
      base += tot;
    }
    __syncwarp();
    const int nwork_all = base;

    // 2. dot products, NB nodes x G heads per transposing reduction
    const float* lvl = ph + s.off[level - 2] * D + lane * DPL;
    for (int w0 = 0; w0 < nwork_all; w0 += NB) {
      float v[32];
#pragma unroll
      for (int n = 0; n < NB; ++n) {
        float mu[DPL];
        const int w = w0 + n;
        if (w < nwork_all) {
          const float* row = lvl + (int64_t)sm.work[w] * D;
          if (DPL == 4) {
            const float4 m4 = __ldg(reinterpret_cast<const float4*>(row));
            mu[0] = m4.x; mu[1] = m4.y; mu[2] = m4.z; mu[3] = m4.w;
          } else {
            const float2 m2 = __ldg(reinterpret_cast<const float2*>(row));
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
      if (w < nwork_all) sm.y[w][lane % G] = r;
    }
    __syncwarp();

    // 3. candidate scores: sum over heads of log2-sum-exp2 over eligible children
    for (int i = lane; i < nc; i += 32) {
      const int s0 = sm.slot0[i], s1 = sm.slot1[i];
      const int64_t c0 = 2 * (int64_t)sm.cand[i];
      float sc = 0.0f;
      float n0 = 0.0f, n1 = 0.0f;
      if (s1 == -2) {
        n0 = (float)node_count(s, level - 1, c0, s.N);
        n1 = (float)node_count(s, level - 1, c0 + 1, s.N);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float a = s0 >= 0 ? sm.y[s0][g] : 0.0f;
        float bb;
        if (s1 >= 0) bb = sm.y[s1][g];
        else if (s1 == -2) bb = ((n0 + n1) * sm.x[i][g] - n0 * a) / n1;
        else bb = 0.0f;
        float l;
        if (s0 >= 0 && s1 != -1) l = lse2_pair(a, bb);
        else l = s0 >= 0 ? a : bb;
        sc += l;
      }
      sm.score[i] = sc;
    }
    __syncwarp();

    // 4. Top-K (ties to the lower index), kept set compacted in index order
    int base2 = 0;
    for (int i0 = 0; i0 < nc; i0 += 32) {
      const int i = i0 + lane;
      int keep = 0, nchild = 0;
      int64_t c0 = 0;
      int e0 = 0, e1 = 0;
      if (i < nc) {
        const float si = sm.score[i];
        const int32_t ci = sm.cand[i];
        int rank = 0;
        for (int j = 0; j < nc; ++j) rank += beats(sm.score[j], sm.cand[j], si, ci) ? 1 : 0;
        keep = rank < K;
        c0 = 2 * (int64_t)ci;
        e0 = c0 < ncap && node_eligible(level - 1, c0, qb);
        e1 = c0 + 1 < ncap && node_eligible(level - 1, c0 + 1, qb);
        nchild = keep ? (level > 2 ? e0 + e1 : 1) : 0;
      }
      int tot;
      const int pos = base2 + warp_excl_scan(nchild, &tot);
      if (keep) {
        if (level == 2) {
          kout[pos] = sm.cand[i];
        } else {
          int p = pos;
          const int s0 = sm.slot0[i], s1 = sm.slot1[i];
          float n0 = 0.0f, n1 = 0.0f;
          if (s1 == -2) {
            n0 = (float)node_count(s, level - 1, c0, s.N);
            n1 = (float)node_count(s, level - 1, c0 + 1, s.N);
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
              sm.xn[p][g] = s1 >= 0 ? sm.y[s1][g] : ((n0 + n1) * sm.x[i][g] - n0 * a) / n1;
            }
            sm.has_xn[p] = 1;
          }
        }
        if (trow) {
          // kept set in index order: position among kept candidates
          int kpos = 0;
          for (int j = 0; j < i; ++j) {
            int rj = 0;
            for (int m = 0; m < nc; ++m) rj += beats(sm.score[m], sm.cand[m], sm.score[j], sm.cand[j]) ? 1 : 0;
            kpos += rj < K;
          }
          trow[(level - 1) * K + kpos] = sm.cand[i];
        }
      }
      base2 += tot;
    }
    __syncwarp();
    if (level == 2) {
      for (int i = base2 + lane; i < K; i += 32) kout[i] = -1;
      break;
    }
    nc = base2;
    for (int i = lane; i < nc; i += 32) {
      sm.cand[i] = sm.nxt[i];
      sm.has_x[i] = sm.has_xn[i];
#pragma unroll
      for (int g = 0; g < G; ++g) sm.x[i][g] = sm.xn[i][g];
    }
    __syncwarp();
  }
}

template <int D, int G>
static cudaError_t launch_route_t(const Prob& pr, const Pyr& s, const void* q, const float* pyr, int32_t* kept2,
                                  int32_t* trace, cudaStream_t st) {
  const size_t smem = sizeof(RouteWarpSm<G>) * kRouteWarps;
  auto kern = route_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t nq = pr.B * pr.Hkv * pr.N;
  const int64_t grid = ceil_div64(nq, kRouteWarps);
  kern<<<(unsigned)grid, kRouteWarps * 32, smem, st>>>(pr, s, q, pyr, kept2, trace);
  return cudaGetLastError();
}

cudaError_t launch_route(const Prob& pr, const Pyr& s, const void* q, const float* pyr, int32_t* kept2,
                         int32_t* trace, int32_t* /*status*/, cudaStream_t st) {
  if (pr.B * pr.Hkv * pr.N == 0) return cudaSuccess;
#define PISA_ROUTE_CASE(DD, GG) \
  if (pr.d == DD && pr.G == GG) return launch_route_t<DD, GG>(pr, s, q, pyr, kept2, trace, st);
  PISA_ROUTE_CASE(128, 1) PISA_ROUTE_CASE(128, 2) PISA_ROUTE_CASE(128, 4) PISA_ROUTE_CASE(128, 8)
  PISA_ROUTE_CASE(64, 1) PISA_ROUTE_CASE(64, 2) PISA_ROUTE_CASE(64, 4) PISA_ROUTE_CASE(64, 8)
#undef PISA_ROUTE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pisa
