// route_mma.cu -- top-down pyramid routing with the child dot products on
// the tensor cores (bf16 inputs, GQA groups of 4 query heads).  Same walk and
// scoring as route.cu (rcap.io post on "Block Sparse Attention with
// Log-Linear Complexity": "Selection walks the tree top-down", "The scoring
// rule matters"; agihunt.info summary, kernel paragraph: one selection per
// GQA group, the heads' scores summed).
//
// A warp walks two queries.  Per level, the child summary rows each query
// needs (at most 2K) are multiplied against its four query-head vectors as a
// sequence of warp-level m16n8k16 MMAs: A = 16 child rows (8 per query),
// B = 8 columns (the 2 x 4 query heads), fp32 accumulation.  Only the two
// diagonal 8 x 4 blocks are used.  Each lane loads two 16-byte slices per row
// and K block with no shuffles or reductions.  The query rows are bf16, so they
// are exact in the MMA; each fp32 summary is split into bf16 hi + lo
// (mu = hi + lo to about 2^-16 relative) and multiplied twice, so the dots
// match an fp32 computation to ~1e-6.  The two pieces are prepared once per
// call by split_pyramid_kernel into the workspace.
//
// The candidate bookkeeping (work list, scores, Top-K by a 64-bit rank key,
// expansion into ascending ping-pong lists) runs on 16 lanes per query.
#include <algorithm>

#include "pisa_common.cuh"
#include "pisa_internal.h"

namespace pisa {

template <int NC>
struct RouteMmaQ {
  int32_t cand[2][NC];
  float x[2][NC][4];
  int32_t hasx[2][NC];
  int32_t work[2 * NC];
  float y[2 * NC][4];
};

template <int NC>
struct RouteMmaQPad : RouteMmaQ<NC> {
  // the two queries of a warp start 16 banks apart
  static constexpr int kWords = (int)(sizeof(RouteMmaQ<NC>) / 4);
  static constexpr int kPad = (16 - kWords % 32 + 64) % 32;
  int32_t pad[kPad > 0 ? kPad : 1];
};

__device__ __forceinline__ uint32_t orderable_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int scan16_seg(int v, int ll, int* tot) {
  int x = v;
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o, 16);
    if (ll >= o) x += y;
  }
  *tot = __shfl_sync(0xffffffffu, x, 15, 16);
  return x - v;
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

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// fp32 pyramid -> bf16 hi (rounded) and lo (rounded residual), same layout.
__global__ void split_pyramid_kernel(int64_t n, const float* __restrict__ pyr, __nv_bfloat16* __restrict__ hi,
                                     __nv_bfloat16* __restrict__ lo) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float v = pyr[i];
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    hi[i] = h;
    lo[i] = __float2bfloat16_rn(v - __bfloat162float(h));
  }
}

// K-block mapping: MMA k-step s of a lane with thread-in-group t uses the
// physical dims 32 (s/2) + 8t + 4 (s%2) + {0..3}; for each pair of steps the
// lane's dims are 8 contiguous elements (one 16-byte load), and the same
// mapping is applied to A (child rows) and B (query heads).
template <int D, int KM, int WARPS>
__global__ void __launch_bounds__(WARPS * 32) route_mma_kernel(Prob pr, Pyr s, const uint16_t* __restrict__ q,
                                                               const uint16_t* __restrict__ phi,
                                                               const uint16_t* __restrict__ plo,
                                                               int32_t* __restrict__ kept2,
                                                               int32_t* __restrict__ trace) {
  constexpr int G = 4;
  constexpr int NC = 2 * KM;
  constexpr int CPL = NC / 16;
  constexpr int NBLK = D / 32;  // 16-byte slices per row per lane
  extern __shared__ __align__(16) unsigned char smem_raw[];
  RouteMmaQPad<NC>& sm = reinterpret_cast<RouteMmaQPad<NC>*>(smem_raw)[threadIdx.x / 16];
  RouteMmaQPad<NC>* smw = reinterpret_cast<RouteMmaQPad<NC>*>(smem_raw) + (threadIdx.x / 32) * 2;
  const int lane = threadIdx.x & 31, ll = lane & 15, half = lane >> 4;
  const int grp = lane >> 2, tig = lane & 3;  // MMA group id / thread in group
  const int64_t nq = pr.B * pr.Hkv * pr.N;
  const int64_t qi = ((int64_t)blockIdx.x * WARPS + threadIdx.x / 32) * 2 + half;
  const bool live = qi < nq;
  const int64_t qc = live ? qi : nq - 1;
  const int64_t t = qc % pr.N, bh = qc / pr.N;
  const int64_t b = bh / pr.Hkv, h = bh % pr.Hkv;
  const int K = pr.K;
  const int64_t qb = t / s.C;
  int32_t* kout = kept2 + qc * K;
  int32_t* trow = (trace && live) ? trace + qc * (int64_t)s.L * K : nullptr;
  if (trow)
    for (int i = ll; i < s.L * K; i += 16) trow[i] = -1;

  int l0 = 0;
  if (live && qb - 2 >= 1) {
    for (int level = s.L; level >= 2; --level)
      if (eligible_count(level, qb) > K) { l0 = level; break; }
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

  // B fragments: column grp = (query half, head grp % 4); unscaled bf16 pairs
  uint32_t bq[D / 16][2];
  {
    const int64_t qrow = ((b * pr.Hq + h * G + (grp & 3)) * pr.N + t) * D;
#pragma unroll
    for (int blk = 0; blk < NBLK; ++blk) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(q + qrow + 32 * blk + 8 * tig));
      bq[2 * blk][0] = v.x; bq[2 * blk][1] = v.y;
      bq[2 * blk + 1][0] = v.z; bq[2 * blk + 1][1] = v.w;
    }
  }
  // the two queries of a warp may belong to different (b, h) rows of the pyramid
  const int64_t qw = ((int64_t)blockIdx.x * WARPS + threadIdx.x / 32) * 2;
  const int64_t pbase0 = (min(qw, nq - 1) / pr.N) * s.P * D;
  const int64_t pbase1 = (min(qw + 1, nq - 1) / pr.N) * s.P * D;

  int cur = 0;
  int nc = l0 > 0 ? (int)eligible_count(l0, qb) : 0;
  for (int i = ll; i < nc; i += 16) { sm.cand[0][i] = i; sm.hasx[0][i] = 0; }
  const int e_hi = (int)(qb - 2);
  __syncwarp();

  for (int level = l0w; level >= 2; --level) {
    const bool act = level <= l0;
    const int ncur = act ? nc : 0;
    const int ncap = (int)s.size[level - 2];

    // 1. work list
    int c0v[CPL], e0v[CPL], e1v[CPL], s0v[CPL], s1v[CPL];
    int nwork = 0;
#pragma unroll
    for (int sl = 0; sl < CPL; ++sl) {
      const int i = sl * 16 + ll;
      const bool valid = i < ncur;
      const int c0 = valid ? 2 * sm.cand[cur][i] : 0;
      const int e0 = valid && c0 < ncap && elig_node(level - 1, c0, e_hi);
      const int e1 = valid && c0 + 1 < ncap && elig_node(level - 1, c0 + 1, e_hi);
      const int der = e0 && e1 && sm.hasx[cur][i];
      int tot;
      int p = nwork + scan16_seg(e0 + (e1 && !der), ll, &tot);
      s0v[sl] = e0 ? p : -1;
      if (e0) sm.work[p++] = c0;
      s1v[sl] = e1 ? (der ? -2 : p) : -1;
      if (e1 && !der) sm.work[p] = c0 + 1;
      nwork += tot;
      c0v[sl] = c0; e0v[sl] = e0; e1v[sl] = e1;
    }
    __syncwarp();

    // 2. dot products: 8 rows of each query per m16n8k16 tile sequence
    {
      const int nw0 = __shfl_sync(0xffffffffu, nwork, 0), nw1 = __shfl_sync(0xffffffffu, nwork, 16);
      const int nmax = max(nw0, nw1);
      const int64_t loff = s.off[level - 2] * D + 8 * tig;
      for (int r0 = 0; r0 < nmax; r0 += 8) {
        const int wa = r0 + grp;  // work row of query 0 (MMA row grp) and of query 1 (row grp + 8)
        const bool oka = wa < nw0, okb = wa < nw1;
        const int64_t ra = pbase0 + loff + (int64_t)(oka ? smw[0].work[wa] : 0) * D;
        const int64_t rb = pbase1 + loff + (int64_t)(okb ? smw[1].work[wa] : 0) * D;
        uint4 ha[NBLK], la[NBLK], hb[NBLK], lb[NBLK];
#pragma unroll
        for (int blk = 0; blk < NBLK; ++blk) {
          ha[blk] = __ldg(reinterpret_cast<const uint4*>(phi + ra + 32 * blk));
          la[blk] = __ldg(reinterpret_cast<const uint4*>(plo + ra + 32 * blk));
          hb[blk] = __ldg(reinterpret_cast<const uint4*>(phi + rb + 32 * blk));
          lb[blk] = __ldg(reinterpret_cast<const uint4*>(plo + rb + 32 * blk));
        }
        float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int blk = 0; blk < NBLK; ++blk) {
          // step 2*blk: dims 8t + 0..3 (words x, y); step 2*blk+1: dims 8t + 4..7 (z, w)
          mma_16816(d, ha[blk].x, hb[blk].x, ha[blk].y, hb[blk].y, bq[2 * blk][0], bq[2 * blk][1]);
          mma_16816(d, la[blk].x, lb[blk].x, la[blk].y, lb[blk].y, bq[2 * blk][0], bq[2 * blk][1]);
          mma_16816(d, ha[blk].z, hb[blk].z, ha[blk].w, hb[blk].w, bq[2 * blk + 1][0], bq[2 * blk + 1][1]);
          mma_16816(d, la[blk].z, lb[blk].z, la[blk].w, lb[blk].w, bq[2 * blk + 1][0], bq[2 * blk + 1][1]);
        }
        // lanes with tig < 2 hold (query 0 row wa, heads 2tig, 2tig+1);
        // lanes with tig >= 2 hold (query 1 row wa, heads 2tig-4, 2tig-3)
        const float sc = pr.scale2;
        if (tig < 2) {
          if (oka) { smw[0].y[wa][2 * tig] = d[0] * sc; smw[0].y[wa][2 * tig + 1] = d[1] * sc; }
        } else {
          if (okb) { smw[1].y[wa][2 * tig - 4] = d[2] * sc; smw[1].y[wa][2 * tig - 3] = d[3] * sc; }
        }
      }
    }
    __syncwarp();

    // 3. scores and rank keys
    uint64_t key[CPL];
#pragma unroll
    for (int sl = 0; sl < CPL; ++sl) {
      const int i = sl * 16 + ll;
      key[sl] = 0;
      if (i < ncur) {
        const int s0 = s0v[sl], s1 = s1v[sl];
        int n0 = 0, n1 = 0;
        if (s1 == -2) {
          n0 = count_node(s.C, level - 1, c0v[sl], s.N);
          n1 = count_node(s.C, level - 1, c0v[sl] + 1, s.N);
        }
        float scv = 0.0f;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float a = s0 >= 0 ? sm.y[s0][g] : 0.0f;
          float bb = 0.0f;
          if (s1 >= 0) bb = sm.y[s1][g];
          else if (s1 == -2) bb = sib_dot(sm.x[cur][i][g], a, n0, n1);
          scv += (s0 >= 0 && s1 != -1) ? lse2_pair(a, bb) : (s0 >= 0 ? a : bb);
        }
        key[sl] = ((uint64_t)orderable_key(scv) << 32) | (uint32_t)(~(uint32_t)sm.cand[cur][i]);
      }
    }
    int rank[CPL];
#pragma unroll
    for (int sl = 0; sl < CPL; ++sl) rank[sl] = 0;
#pragma unroll
    for (int sj = 0; sj < CPL; ++sj) {
      const uint32_t khi = (uint32_t)(key[sj] >> 32), klo = (uint32_t)key[sj];
#pragma unroll
      for (int l = 0; l < 16; ++l) {
        const uint64_t kj = ((uint64_t)__shfl_sync(0xffffffffu, khi, l, 16) << 32) |
                            __shfl_sync(0xffffffffu, klo, l, 16);
#pragma unroll
        for (int sl = 0; sl < CPL; ++sl) rank[sl] += kj > key[sl] ? 1 : 0;
      }
    }

    // 4. kept set, expansion
    const int nxt = cur ^ 1;
    int nkept = 0, nchild = 0;
#pragma unroll
    for (int sl = 0; sl < CPL; ++sl) {
      const int i = sl * 16 + ll;
      const int keep = (i < ncur && rank[sl] < K) ? 1 : 0;
      const int nch = keep && level > 2 ? e0v[sl] + e1v[sl] : 0;
      int ktot, ctot;
      const int kp = nkept + scan16_seg(keep, ll, &ktot);
      int cp = nchild + scan16_seg(nch, ll, &ctot);
      if (keep) {
        const int32_t ci = sm.cand[cur][i];
        if (trow) trow[(level - 1) * K + kp] = ci;
        if (level == 2) kout[kp] = ci;
        if (nch) {
          const int s0 = s0v[sl], s1 = s1v[sl];
          int n0 = 0, n1 = 0;
          if (s1 == -2) {
            n0 = count_node(s.C, level - 1, c0v[sl], s.N);
            n1 = count_node(s.C, level - 1, c0v[sl] + 1, s.N);
          }
          if (e0v[sl]) {
            sm.cand[nxt][cp] = c0v[sl];
#pragma unroll
            for (int g = 0; g < G; ++g) sm.x[nxt][cp][g] = sm.y[s0][g];
            sm.hasx[nxt][cp] = 1;
            ++cp;
          }
          if (e1v[sl]) {
            sm.cand[nxt][cp] = c0v[sl] + 1;
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const float a = e0v[sl] ? sm.y[s0][g] : 0.0f;
              sm.x[nxt][cp][g] = s1 >= 0 ? sm.y[s1][g] : sib_dot(sm.x[cur][i][g], a, n0, n1);
            }
            sm.hasx[nxt][cp] = 1;
          }
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

template <int D, int KM, int WARPS>
static cudaError_t launch_route_mma_t(const Prob& pr, const Pyr& s, const void* q, const uint16_t* phi,
                                      const uint16_t* plo, int32_t* kept2, int32_t* trace, cudaStream_t st) {
  const size_t smem = sizeof(RouteMmaQPad<2 * KM>) * 2 * WARPS;
  auto kern = route_mma_kernel<D, KM, WARPS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t nq = pr.B * pr.Hkv * pr.N;
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
  split_pyramid_kernel<<<(unsigned)std::min<int64_t>(ceil_div64(n, 256), 8192), 256, 0, st>>>(
      n, pyr, (__nv_bfloat16*)phi, (__nv_bfloat16*)plo);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
#define PISA_RM_CASE(DD)                                                                                  \
  if (pr.d == DD) {                                                                                       \
    if (pr.K <= 8) return launch_route_mma_t<DD, 8, 8>(pr, s, q, phi, plo, kept2, trace, st);             \
    if (pr.K <= 16) return launch_route_mma_t<DD, 16, 8>(pr, s, q, phi, plo, kept2, trace, st);           \
    return launch_route_mma_t<DD, 32, 4>(pr, s, q, phi, plo, kept2, trace, st);                           \
  }
  PISA_RM_CASE(128) PISA_RM_CASE(64)
#undef PISA_RM_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pisa
