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

template <int D, int G>
__global__ void __launch_bounds__(kPathThreads) path_dots_kernel(Prob pr, Pyr s, const void* __restrict__ q,
                                                                const void* __restrict__ k,
                                                                const float* __restrict__ pyr, int ref_root,
                                                                float* __restrict__ out) {
  constexpr int DP = D + 4;  // padded row stride: the rows of consecutive positions start 4 banks apart
  extern __shared__ __align__(16) float path_smem[];
  float* ksum = path_smem;                      // [C][DP]: prefix sums of the block's keys
  float* sib = ksum + (size_t)s.C * DP;         // [kPathMaxOdd][D]: row l - 2 = level l's sibling (odd levels)
  float* refr = sib + (size_t)kPathMaxOdd * D;  // [D]
  const int tid = threadIdx.x;
  const int L = s.L;
  const int64_t nblk = pr.B * pr.Hkv * s.nb;
  const int64_t w = blockIdx.x;
  if (w >= nblk) return;  // CTA-uniform
  const int64_t bh = w / s.nb, qb = w % s.nb;
  const int64_t b = bh / pr.Hkv, h = bh % pr.Hkv;
  const float* ph = pyr + bh * s.P * D;
  const bool bf16 = pr.dtype == PISA_BF16;
  const size_t esz = bf16 ? 2 : 4;
  const int64_t t0 = qb * s.C;
  const int nt = (int)(s.N - t0 < s.C ? s.N - t0 : s.C);

  // siblings of the odd levels (which levels: CTA-uniform), the reference row
  for (int l = 2; l <= L; ++l) {
    const int64_t jc = qb >> (l - 2);
    if (jc & 1) {
      const float* row = ph + (s.off[l - 2] + jc - 1) * D;
      for (int c = tid; c < D; c += kPathThreads) sib[(l - 2) * D + c] = row[c];
    }
  }
  for (int c = tid; c < D; c += kPathThreads) {
    const float r = ref_root ? ph[(s.P - 1) * D + c] : 0.0f;
    refr[c] = isfinite(r) ? r : 0.0f;
  }
  // prefix sums of the block's keys, one thread per dim
  const char* kb = reinterpret_cast<const char*>(k) + (bh * s.N + t0) * D * esz;
  for (int c = tid; c < D; c += kPathThreads) {
    float run = 0.0f;
    for (int t = 0; t < nt; ++t) {
      const char* e = kb + ((size_t)t * D + c) * esz;
      run += bf16 ? bf16_to_f(*reinterpret_cast<const uint16_t*>(e)) : *reinterpret_cast<const float*>(e);
      ksum[t * DP + c] = run;
    }
  }
  __syncthreads();

  for (int pi = tid; pi < s.C * G; pi += kPathThreads) {
    const int t = pi / G, g = pi % G;
    if (t >= nt) continue;
    const char* qr = reinterpret_cast<const char*>(q) + (((b * pr.Hq + h * G + g) * pr.N + t0 + t) * D) * esz;
    const float* kr = ksum + t * DP;
    float dk = 0.0f, dr = 0.0f;
    float ds[kPathMaxOdd];
#pragma unroll
    for (int i = 0; i < kPathMaxOdd; ++i) ds[i] = 0.0f;
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
        const float4 rr = *reinterpret_cast<const float4*>(refr + c + 4 * hh);
        dk = fmaf(qh[0], kk.x, fmaf(qh[1], kk.y, fmaf(qh[2], kk.z, fmaf(qh[3], kk.w, dk))));
        dr = fmaf(qh[0], rr.x, fmaf(qh[1], rr.y, fmaf(qh[2], rr.z, fmaf(qh[3], rr.w, dr))));
#pragma unroll
        for (int i = 0; i < kPathMaxOdd; ++i)
          if (i + 2 <= L && ((qb >> i) & 1)) {  // level i + 2 has a left sibling (CTA-uniform)
            const float4 sv = *reinterpret_cast<const float4*>(sib + i * D + c + 4 * hh);
            ds[i] = fmaf(qh[0], sv.x, fmaf(qh[1], sv.y, fmaf(qh[2], sv.z, fmaf(qh[3], sv.w, ds[i]))));
          }
      }
    }
    // level recurrence (see the file comment), outputs [L][2] of this head
    const float n1 = (float)(t + 1);
    float P = dk / n1 - dr;  // q . (prefix(1) - ref)
    float cnt = n1;
    float* orow = out + ((bh * s.N + t0 + t) * L) * 2 * G;
    orow[g] = P * pr.scale2;
    orow[G + g] = 0.0f;
#pragma unroll
    for (int l = 2; l <= kPathMaxOdd + 1; ++l) {
      if (l > L) break;
      const int64_t jc = qb >> (l - 2);
      float S = 0.0f;
      if (jc & 1) {
        S = ds[l - 2] - dr;
        const float ns = (float)((int64_t)s.C << (l - 2));
        P = (ns * S + cnt * P) / (ns + cnt);
        cnt += ns;
      }
      orow[(l - 1) * 2 * G + g] = P * pr.scale2;
      orow[(l - 1) * 2 * G + G + g] = S * pr.scale2;
    }
  }
}

size_t path_dots_bytes(const Prob& pr, const Pyr& s) {
  return pr.prefix ? (size_t)pr.B * pr.Hkv * pr.N * s.L * 2 * pr.G * sizeof(float) : 0;
}

template <int D, int G>
static cudaError_t launch_path_t(const Prob& pr, const Pyr& s, const void* q, const void* k, const float* pyr,
                                 int ref_root, float* out, cudaStream_t st) {
  if (s.L - 1 > kPathMaxOdd) return cudaErrorInvalidValue;  // beyond the size limit
  const size_t smem = ((size_t)s.C * (D + 4) + (size_t)(kPathMaxOdd + 1) * D) * sizeof(float);
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
