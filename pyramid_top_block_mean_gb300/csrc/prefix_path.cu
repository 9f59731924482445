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
// One CTA of four warps per (sequence, key head, leaf block): the block's
// queries are split among the warps (a quarter each, in order), which share
// the block's path siblings staged in shared memory.  A warp starts its
// running key sum from the sums of the earlier warps' key rows, exchanged
// through shared memory, so the four walk their queries concurrently.
// Lanes split into G heads x 32/G dim groups: each lane keeps the running
// sum over its dims, takes its partial dots with its head's query row, and
// the dim groups reduce with shuffles.
#include "pisa_common.cuh"
#include "pisa_internal.h"

namespace pisa {

constexpr int kPathWarps = 4;

// Dim of a lane's j-th element: with at least four dims per lane, lane dg of
// the DG lanes of a head owns the 4-dim chunks dg, dg + DG, dg + 2 DG, ...,
// so that the DG lanes of a head read consecutive 16-byte chunks of a row
// (coalesced in global memory, conflict-free in shared memory); with two, the
// pair 2 dg, 2 dg + 1.
template <int D, int DG, int DPL>
__device__ __forceinline__ int path_dim(int dg, int j) {
  if constexpr (DPL >= 4) return 4 * (dg + DG * (j >> 2)) + (j & 3);
  return dg * DPL + j;
}

// Loads the lane's DPL elements of one row (bf16 or fp32) as floats.
template <int D, int DG, int DPL>
__device__ __forceinline__ void path_row(const char* row, bool bf16, size_t esz, int dg, float (&v)[DPL]) {
  if constexpr (DPL >= 4) {
#pragma unroll
    for (int m = 0; m < DPL / 4; ++m) load4(row + (size_t)path_dim<D, DG, DPL>(dg, 4 * m) * esz, bf16, v + 4 * m);
  } else {
    load2(row + (size_t)path_dim<D, DG, DPL>(dg, 0) * esz, bf16, v);
  }
}

template <int D, int G>
__global__ void __launch_bounds__(kPathWarps * 32) path_dots_kernel(Prob pr, Pyr s, const void* __restrict__ q,
                                                                    const void* __restrict__ k,
                                                                    const float* __restrict__ pyr, int ref_root,
                                                                    float* __restrict__ out) {
  constexpr int DG = 32 / G;   // dim groups (lanes per head)
  constexpr int DPL = D / DG;  // dims per lane: 2 .. 32
  extern __shared__ __align__(16) float sib_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x / 32;
  const int g = lane / DG, dg = lane % DG;
  const int L = s.L;
  float* sib = sib_smem;                           // [L][D]; row l - 1 for level l >= 2
  float* ksw = sib + (size_t)L * D;                // [kPathWarps][D]: each warp's key-row sum
  float* obuf = ksw + (size_t)kPathWarps * D;      // [kPathWarps][L][2][G]: a query's outputs
  const int64_t nblk = pr.B * pr.Hkv * s.nb;
  const int64_t w = blockIdx.x;
  if (w >= nblk) return;  // CTA-uniform
  const int64_t bh = w / s.nb, qb = w % s.nb;
  const int64_t b = bh / pr.Hkv, h = bh % pr.Hkv;
  const float* ph = pyr + bh * s.P * D;
  const bool bf16 = pr.dtype == PISA_BF16;

  // the path's left siblings (complete nodes), staged once per block
  for (int l = 2; l <= L; ++l) {
    const int64_t jc = qb >> (l - 2);
    if (jc & 1) {
      const float* row = ph + (s.off[l - 2] + jc - 1) * D;
      for (int c = threadIdx.x; c < D; c += kPathWarps * 32) sib[(l - 1) * D + c] = row[c];
    }
  }
  // reference row, lane's dims
  float ref[DPL];
#pragma unroll
  for (int j = 0; j < DPL; ++j) {
    const float r = ref_root ? ph[(s.P - 1) * D + path_dim<D, DG, DPL>(dg, j)] : 0.0f;
    ref[j] = isfinite(r) ? r : 0.0f;
  }

  const int64_t t0 = qb * s.C;
  const int nt = (int)(s.N - t0 < s.C ? s.N - t0 : s.C);
  const int per = (s.C + kPathWarps - 1) / kPathWarps;
  const int r0 = min(nt, warp * per), r1 = min(nt, r0 + per);
  const size_t esz = bf16 ? 2 : 4;
  const char* krow0 = reinterpret_cast<const char*>(k) + (bh * s.N + t0) * D * esz;
  const char* qrow0 = reinterpret_cast<const char*>(q) + ((b * pr.Hq + h * G + g) * pr.N + t0) * D * esz;

  // this warp's key rows summed, then the sums of the earlier warps' rows
  float ks[DPL];
#pragma unroll
  for (int j = 0; j < DPL; ++j) ks[j] = 0.0f;
  for (int r = r0; r < r1; ++r) {
    float kv[DPL];
    path_row<D, DG, DPL>(krow0 + (size_t)r * D * esz, bf16, esz, dg, kv);
#pragma unroll
    for (int j = 0; j < DPL; ++j) ks[j] += kv[j];
  }
  if (g == 0)
#pragma unroll
    for (int j = 0; j < DPL; ++j) ksw[warp * D + path_dim<D, DG, DPL>(dg, j)] = ks[j];
  __syncthreads();
#pragma unroll
  for (int j = 0; j < DPL; ++j) {
    float sacc = 0.0f;  // the earlier warps' sums, in warp order
    for (int u = 0; u < warp; ++u) sacc += ksw[u * D + path_dim<D, DG, DPL>(dg, j)];
    ks[j] = sacc;
  }

  float* ob = obuf + (size_t)warp * L * 2 * G;
  const int nout = L * 2 * G;  // floats per query
  for (int r = r0; r < r1; ++r) {
    const int64_t t = t0 + r;
    float qv[DPL], kv[DPL];
    path_row<D, DG, DPL>(krow0 + (size_t)r * D * esz, bf16, esz, dg, kv);
    path_row<D, DG, DPL>(qrow0 + (size_t)r * D * esz, bf16, esz, dg, qv);
#pragma unroll
    for (int j = 0; j < DPL; ++j) ks[j] += kv[j];
    // partial dots: q . key sum, q . ref, q . sibling of every odd level
    float dk = 0.0f, dr = 0.0f;
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      dk = fmaf(qv[j], ks[j], dk);
      dr = fmaf(qv[j], ref[j], dr);
    }
#pragma unroll
    for (int o = DG / 2; o >= 1; o >>= 1) {
      dk += __shfl_xor_sync(0xffffffffu, dk, o);
      dr += __shfl_xor_sync(0xffffffffu, dr, o);
    }
    const float n1 = (float)(r + 1);
    float P = dk / n1 - dr;  // q . (prefix(1) - ref)
    float cnt = n1;
    if (dg == 0) {
      ob[0 * 2 * G + 0 * G + g] = P * pr.scale2;
      ob[0 * 2 * G + 1 * G + g] = 0.0f;
    }
    for (int l = 2; l <= L; ++l) {
      const int64_t jc = qb >> (l - 2);
      float S = 0.0f;
      if (jc & 1) {  // warp-uniform
        float ds = 0.0f;
        const float* srow = sib + (l - 1) * D;
#pragma unroll
        for (int j = 0; j < DPL; ++j) ds = fmaf(qv[j], srow[path_dim<D, DG, DPL>(dg, j)], ds);
#pragma unroll
        for (int o = DG / 2; o >= 1; o >>= 1) ds += __shfl_xor_sync(0xffffffffu, ds, o);
        S = ds - dr;
        const float ns = (float)((int64_t)s.C << (l - 2));
        P = (ns * S + cnt * P) / (ns + cnt);
        cnt += ns;
      }
      if (dg == 0) {
        ob[(l - 1) * 2 * G + 0 * G + g] = P * pr.scale2;
        ob[(l - 1) * 2 * G + 1 * G + g] = S * pr.scale2;
      }
    }
    // the query's [L][2][G] outputs leave as whole rows
    __syncwarp();
    float* orow = out + ((bh * s.N + t) * L) * 2 * G;
    for (int e = lane; e < nout; e += 32) orow[e] = ob[e];
    __syncwarp();
  }
}

size_t path_dots_bytes(const Prob& pr, const Pyr& s) {
  return pr.prefix ? (size_t)pr.B * pr.Hkv * pr.N * s.L * 2 * pr.G * sizeof(float) : 0;
}

template <int D, int G>
static cudaError_t launch_path_t(const Prob& pr, const Pyr& s, const void* q, const void* k, const float* pyr,
                                 int ref_root, float* out, cudaStream_t st) {
  const size_t smem = ((size_t)(s.L + kPathWarps) * D + (size_t)kPathWarps * s.L * 2 * G) * sizeof(float);
  auto kern = path_dots_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t nblk = pr.B * pr.Hkv * s.nb;
  note_launch();
  kern<<<(unsigned)nblk, kPathWarps * 32, smem, st>>>(pr, s, q, k, pyr, ref_root, out);
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
