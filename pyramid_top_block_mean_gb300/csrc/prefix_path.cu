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
// One warp per (sequence, key head, leaf block); its 64 queries share the
// block's path siblings, which are staged in shared memory.  Lanes split
// into G heads x 32/G dim groups: each lane keeps a running sum of the
// block's keys over its dims, takes its partial dots with its head's query
// row, and the dim groups reduce with shuffles.
#include "pisa_common.cuh"
#include "pisa_internal.h"

namespace pisa {

template <int D, int G>
__global__ void __launch_bounds__(128) path_dots_kernel(Prob pr, Pyr s, const void* __restrict__ q,
                                                        const void* __restrict__ k,
                                                        const float* __restrict__ pyr, int ref_root,
                                                        float* __restrict__ out) {
  constexpr int DG = 32 / G;   // dim groups (lanes per head)
  constexpr int DPL = D / DG;  // dims per lane: 4 .. 32
  extern __shared__ __align__(16) float sib_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x / 32;
  const int g = lane / DG, dg = lane % DG;
  const int L = s.L;
  float* sib = sib_smem + (size_t)warp * L * D;  // [L][D]; row l - 1 for level l >= 2
  const int64_t nblk = pr.B * pr.Hkv * s.nb;
  const int64_t w = (int64_t)blockIdx.x * (blockDim.x / 32) + warp;
  if (w >= nblk) return;  // warp-uniform
  const int64_t bh = w / s.nb, qb = w % s.nb;
  const int64_t b = bh / pr.Hkv, h = bh % pr.Hkv;
  const float* ph = pyr + bh * s.P * D;
  const bool bf16 = pr.dtype == PISA_BF16;
  const int d0 = dg * DPL;

  // reference row and the path's left siblings (complete nodes), lane's dims
  float ref[DPL];
#pragma unroll
  for (int c = 0; c < DPL; ++c) {
    const float r = ref_root ? ph[(s.P - 1) * D + d0 + c] : 0.0f;
    ref[c] = isfinite(r) ? r : 0.0f;
  }
  for (int l = 2; l <= L; ++l) {
    const int64_t jc = qb >> (l - 2);
    if (jc & 1) {
      const float* row = ph + (s.off[l - 2] + jc - 1) * D;
      for (int c = lane; c < D; c += 32) sib[(l - 1) * D + c] = row[c];
    }
  }
  __syncwarp();

  float ks[DPL];
#pragma unroll
  for (int c = 0; c < DPL; ++c) ks[c] = 0.0f;
  const int64_t t0 = qb * s.C;
  const int nt = (int)(s.N - t0 < s.C ? s.N - t0 : s.C);
  const size_t esz = bf16 ? 2 : 4;
  const char* krow0 = reinterpret_cast<const char*>(k) + ((bh * s.N + t0) * D + d0) * esz;
  const char* qrow0 = reinterpret_cast<const char*>(q) + (((b * pr.Hq + h * G + g) * pr.N + t0) * D + d0) * esz;
  for (int r = 0; r < nt; ++r) {
    const int64_t t = t0 + r;
    float qv[DPL];
    if constexpr (DPL >= 4) {
#pragma unroll
      for (int c = 0; c < DPL; c += 4) {
        float kv[4];
        load4(krow0 + ((int64_t)r * D + c) * esz, bf16, kv);
        load4(qrow0 + ((int64_t)r * D + c) * esz, bf16, qv + c);
#pragma unroll
        for (int e = 0; e < 4; ++e) ks[c + e] += kv[e];
      }
    } else {
      float kv[2];
      load2(krow0 + (int64_t)r * D * esz, bf16, kv);
      load2(qrow0 + (int64_t)r * D * esz, bf16, qv);
      ks[0] += kv[0];
      ks[1] += kv[1];
    }
    // partial dots: q . key sum, q . ref, q . sibling of every odd level
    float dk = 0.0f, dr = 0.0f;
#pragma unroll
    for (int c = 0; c < DPL; ++c) {
      dk = fmaf(qv[c], ks[c], dk);
      dr = fmaf(qv[c], ref[c], dr);
    }
#pragma unroll
    for (int o = DG / 2; o >= 1; o >>= 1) {
      dk += __shfl_xor_sync(0xffffffffu, dk, o);
      dr += __shfl_xor_sync(0xffffffffu, dr, o);
    }
    const float n1 = (float)(r + 1);
    float P = dk / n1 - dr;  // q . (prefix(1) - ref)
    float cnt = n1;
    float* orow = out + (((w / s.nb) * s.N + t) * L) * 2 * G;  // [L][2][G] of this query
    if (dg == 0) {
      orow[0 * 2 * G + 0 * G + g] = P * pr.scale2;
      orow[0 * 2 * G + 1 * G + g] = 0.0f;
    }
    for (int l = 2; l <= L; ++l) {
      const int64_t jc = qb >> (l - 2);
      float S = 0.0f;
      if (jc & 1) {  // warp-uniform
        float ds = 0.0f;
        const float* srow = sib + (l - 1) * D + d0;
#pragma unroll
        for (int c = 0; c < DPL; ++c) ds = fmaf(qv[c], srow[c], ds);
#pragma unroll
        for (int o = DG / 2; o >= 1; o >>= 1) ds += __shfl_xor_sync(0xffffffffu, ds, o);
        S = ds - dr;
        const float ns = (float)((int64_t)s.C << (l - 2));
        P = (ns * S + cnt * P) / (ns + cnt);
        cnt += ns;
      }
      if (dg == 0) {
        orow[(l - 1) * 2 * G + 0 * G + g] = P * pr.scale2;
        orow[(l - 1) * 2 * G + 1 * G + g] = S * pr.scale2;
      }
    }
  }
}

size_t path_dots_bytes(const Prob& pr, const Pyr& s) {
  return pr.prefix ? (size_t)pr.B * pr.Hkv * pr.N * s.L * 2 * pr.G * sizeof(float) : 0;
}

template <int D, int G>
static cudaError_t launch_path_t(const Prob& pr, const Pyr& s, const void* q, const void* k, const float* pyr,
                                 int ref_root, float* out, cudaStream_t st) {
  constexpr int WARPS = 4;
  const size_t smem = (size_t)WARPS * s.L * D * sizeof(float);
  auto kern = path_dots_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t nblk = pr.B * pr.Hkv * s.nb;
  note_launch();
  kern<<<(unsigned)ceil_div64(nblk, WARPS), WARPS * 32, smem, st>>>(pr, s, q, k, pyr, ref_root, out);
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
