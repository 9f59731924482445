// prefix_path.cu -- the prefix-consistent summaries of a prefill query's
// path (pisa_summaries PISA_SUMMARIES_PREFIX).
//
// Reading (agihunt.info summary, pyramid paragraph: decode routing walks the
// pyramid of the keys seen so far; rcap.io post, the pisa_select sketch): a
// query at position t reads every node summary as the mean of the node's
// keys at positions <= t.  Only the nodes on t's path reach past t: at level
// l the node j_l = qb >> (l-1), qb = t / C.  Every other eligible node lies
// wholly before the path and reads as in the full pyramid.  The walk needs
// the path nodes only through their children's dots, so this kernel hands it,
// per query and level l,
//   P_l = s2 (q_g . prefix(l) - q_g . ref)   the path node's own prefix dot
//   S_l = s2 (q_g . mu(l-1, j_{l-1} - 1) - q_g . ref)
//         the dot of its complete left child when the path child j_{l-1} is
//         a right child (odd), unused otherwise,
// with prefix(1) the mean of the keys [qb C, t] and, going up,
//   prefix(l) = (n_s mu_s + c prefix(l-1)) / (n_s + c)   when j_{l-1} is odd
//   prefix(l) = prefix(l-1)                               otherwise,
// mu_s the left sibling (complete, n_s = C 2^(l-2) keys) and c the keys of
// prefix(l-1), which is the count-weighted mean of the keys <= t in the span.
// The dots follow from linearity: q . prefix(l) is the same recurrence over
// q . (key sum) / n and q . mu_s.  ref is the finite-masked root summary (the
// reference of the routing over difference rows) or zero.
//
// One CTA per (sequence, key head, leaf block); a thread per (query, head)
// pair of the block (two per thread for G = 4).  The CTA stages in shared
// memory the prefix sums of the block's keys (row t = the sum of keys
// t0 .. t0 + t), the path's complete left siblings of the odd levels, and the
// reference row; each thread then takes its pair's whole dots in one pass
// over its query row, one accumulator per dot (no cross-lane reductions):
// the prefix-sum row of its position, the reference, and every staged
// sibling.  The level recurrence and the output row follow per thread.
#include "pisa_common.cuh"
#include "pisa_internal.h"

namespace pisa {

constexpr int kPathThreads = 128;
constexpr int kPathMaxOdd = 20;  // odd levels of a path: at most L - 1 <= 20 (N <= 2^26)

// Where the CTA's staged rows are, and what its pairs share.
struct PathBlock {
  const float* ksum;  // [C][D + 4]: prefix sums of the block's keys
  const float* sib;   // [ns][D]: left siblings of the odd levels in level order, zero rows after the last
  const float* refr;  // [D]
  float* dsh;         // [kPathThreads][kPathMaxOdd + 1]: a thread's sibling dots, read back by level
  int64_t bh, b, h, qb, t0;
  int nt;
};

// The (query, head) pairs of one thread: whole dots in one pass over the
// query row (NS sibling slots, the zero-padded ones costing only their FMAs:
// no per-level branch in the pass), then the level recurrence.
template <int D, int G, int NS>
__device__ __forceinline__ void path_pairs(const Prob& pr, const Pyr& s, const void* __restrict__ q, bool bf16,
                                           const PathBlock& pb, float* __restrict__ out) {
  constexpr int DP = D + 4;
  const int tid = threadIdx.x;
  const int L = s.L;
  const size_t esz = bf16 ? 2 : 4;
  for (int pi = tid; pi < s.C * G; pi += kPathThreads) {
    const int t = pi / G, g = pi % G;
    if (t >= pb.nt) continue;
    const char* qr =
        reinterpret_cast<const char*>(q) + (((pb.b * pr.Hq + pb.h * G + g) * pr.N + pb.t0 + t) * D) * esz;
    const float* kr = pb.ksum + t * DP;
    float dk = 0.0f, dr = 0.0f;
    float ds[NS];
#pragma unroll
    for (int j = 0; j < NS; ++j) ds[j] = 0.0f;
    for (int c = 0; c < D; c += 8) {
      // eight query elements per load (16 bytes of bf16)
      float qv[8];
      if (bf16) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(qr + (size_t)c * 2));
        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          qv[2 * e] = __uint_as_float(wv[e] << 16);
          qv[2 * e + 1] = __uint_as_float(wv[e] & 0xffff0000u);
        }
      } else {
        load4(qr + (size_t)c * 4, false, qv);
        load4(qr + (size_t)(c + 4) * 4, false, qv + 4);
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const float* qh = qv + 4 * hh;
        const float4 kk = *reinterpret_cast<const float4*>(kr + c + 4 * hh);
        const float4 rr = *reinterpret_cast<const float4*>(pb.refr + c + 4 * hh);
        dk = fmaf(qh[0], kk.x, fmaf(qh[1], kk.y, fmaf(qh[2], kk.z, fmaf(qh[3], kk.w, dk))));
        dr = fmaf(qh[0], rr.x, fmaf(qh[1], rr.y, fmaf(qh[2], rr.z, fmaf(qh[3], rr.w, dr))));
#pragma unroll
        for (int j = 0; j < NS; ++j) {
          const float4 sv = *reinterpret_cast<const float4*>(pb.sib + j * D + c + 4 * hh);
          ds[j] = fmaf(qh[0], sv.x, fmaf(qh[1], sv.y, fmaf(qh[2], sv.z, fmaf(qh[3], sv.w, ds[j]))));
        }
      }
    }
    float* dst = pb.dsh + tid * (kPathMaxOdd + 1);  // odd stride: no bank conflicts
#pragma unroll
    for (int j = 0; j < NS; ++j) dst[j] = ds[j];
    // level recurrence (see the file comment), outputs [L][2] of this head
    const float n1 = (float)(t + 1);
    float P = dk / n1 - dr;  // q . (prefix(1) - ref)
    float cnt = n1;
    float* orow = out + ((pb.bh * s.N + pb.t0 + t) * L) * 2 * G;
    orow[g] = P * pr.scale2;
    orow[G + g] = 0.0f;
    int j = 0;
    for (int l = 2; l <= L; ++l) {
      const int64_t jc = pb.qb >> (l - 2);
      float S = 0.0f;
      if (jc & 1) {  // CTA-uniform
        S = dst[j++] - dr;
        const float ns = (float)((int64_t)s.C << (l - 2));
        P = (ns * S + cnt * P) / (ns + cnt);
        cnt += ns;
      }
      orow[(l - 1) * 2 * G + g] = P * pr.scale2;
      orow[(l - 1) * 2 * G + G + g] = S * pr.scale2;
    }
  }
}

template <int D, int G>
__global__ void __launch_bounds__(kPathThreads) path_dots_kernel(Prob pr, Pyr s, const void* __restrict__ q,
                                                                const void* __restrict__ k,
                                                                const float* __restrict__ pyr, int ref_root,
                                                                float* __restrict__ out) {
  constexpr int DP = D + 4;  // padded row stride: the rows of consecutive positions start 4 banks apart
  extern __shared__ __align__(16) float path_smem[];
  float* ksum = path_smem;                      // [C][DP]
  float* sib = ksum + (size_t)s.C * DP;         // [kPathMaxOdd][D]
  float* refr = sib + (size_t)kPathMaxOdd * D;  // [D]
  float* dsh = refr + D;                        // [kPathThreads][kPathMaxOdd + 1]
  const int tid = threadIdx.x;
  const int L = s.L;
  const int64_t nblk = pr.B * pr.Hkv * s.nb;
  const int64_t w = blockIdx.x;
  if (w >= nblk) return;  // CTA-uniform
  PathBlock pb;
  pb.bh = w / s.nb;
  pb.qb = w % s.nb;
  pb.b = pb.bh / pr.Hkv;
  pb.h = pb.bh % pr.Hkv;
  const float* ph = pyr + pb.bh * s.P * D;
  const bool bf16 = pr.dtype == PISA_BF16;
  const size_t esz = bf16 ? 2 : 4;
  pb.t0 = pb.qb * s.C;
  pb.nt = (int)(s.N - pb.t0 < s.C ? s.N - pb.t0 : s.C);

  // left siblings of the odd levels (which: CTA-uniform) in level order, then
  // zero rows up to the slot count of the pass
  int nodd = 0;
  for (int l = 2; l <= L; ++l) {
    const int64_t jc = pb.qb >> (l - 2);
    if (jc & 1) {
      const float* row = ph + (s.off[l - 2] + jc - 1) * D;
      for (int c = tid; c < D; c += kPathThreads) sib[nodd * D + c] = row[c];
      ++nodd;
    }
  }
  const int nslot = nodd <= 4 ? 4 : (nodd <= 8 ? 8 : (nodd <= 12 ? 12 : (nodd <= 16 ? 16 : kPathMaxOdd)));
  for (int i = nodd * D + tid; i < nslot * D; i += kPathThreads) sib[i] = 0.0f;
  for (int c = tid; c < D; c += kPathThreads) {
    const float r = ref_root ? ph[(s.P - 1) * D + c] : 0.0f;
    refr[c] = isfinite(r) ? r : 0.0f;
  }
  // prefix sums of the block's keys, one thread per dim
  const char* kb = reinterpret_cast<const char*>(k) + (pb.bh * s.N + pb.t0) * D * esz;
  for (int c = tid; c < D; c += kPathThreads) {
    float run = 0.0f;
    for (int t = 0; t < pb.nt; ++t) {
      const char* e = kb + ((size_t)t * D + c) * esz;
      run += bf16 ? bf16_to_f(*reinterpret_cast<const uint16_t*>(e)) : *reinterpret_cast<const float*>(e);
      ksum[t * DP + c] = run;
    }
  }
  __syncthreads();
  pb.ksum = ksum;
  pb.sib = sib;
  pb.refr = refr;
  pb.dsh = dsh;
  switch (nslot) {  // CTA-uniform
    case 4: path_pairs<D, G, 4>(pr, s, q, bf16, pb, out); break;
    case 8: path_pairs<D, G, 8>(pr, s, q, bf16, pb, out); break;
    case 12: path_pairs<D, G, 12>(pr, s, q, bf16, pb, out); break;
    case 16: path_pairs<D, G, 16>(pr, s, q, bf16, pb, out); break;
    default: path_pairs<D, G, kPathMaxOdd>(pr, s, q, bf16, pb, out); break;
  }
}

size_t path_dots_bytes(const Prob& pr, const Pyr& s) {
  return pr.prefix ? (size_t)pr.B * pr.Hkv * pr.N * s.L * 2 * pr.G * sizeof(float) : 0;
}

template <int D, int G>
static cudaError_t launch_path_t(const Prob& pr, const Pyr& s, const void* q, const void* k, const float* pyr,
                                 int ref_root, float* out, cudaStream_t st) {
  if (s.L - 1 > kPathMaxOdd) return cudaErrorInvalidValue;  // beyond the size limit
  const size_t smem =
      ((size_t)s.C * (D + 4) + (size_t)(kPathMaxOdd + 1) * D + (size_t)kPathThreads * (kPathMaxOdd + 1)) * sizeof(float);
  auto kern = path_dots_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t nblk = pr.B * pr.Hkv * s.nb;
  note_launch();
  kern<<<(unsigned)nblk, kPathThreads, smem, st>>>(pr, s, q, k, pyr, ref_root, out);
  return cudaGetLastError();
}

cudaError_t launch_path_dots(const Prob& pr, const Pyr& s, const void* q, const void* k, const float* pyr,
                             int ref_root, float* out, cudaStream_t st) {
  if (pr.B * pr.Hkv * pr.N == 0) return cudaSuccess;
#define PISA_PATH_CASE(DD, GG) \
  if (pr.d == DD && pr.G == GG) return launch_path_t<DD, GG>(pr, s, q, k, pyr, ref_root, out, st);
  PISA_PATH_CASE(128, 1) PISA_PATH_CASE(128, 2) PISA_PATH_CASE(128, 4) PISA_PATH_CASE(128, 8)
  PISA_PATH_CASE(64, 1) PISA_PATH_CASE(64, 2) PISA_PATH_CASE(64, 4) PISA_PATH_CASE(64, 8)
#undef PISA_PATH_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pisa
