// pyramid.cu -- key pyramid build (mean-pooled leaves, then g = 2 pooling of
// every coarser level).  agihunt.info summary of "Block Sparse Attention with
// Log-Linear Complexity", pyramid paragraph; rcap.io post, "Think of the keys
// as leaves of a tree".
//
// The keys are the contiguous cache or a pool of pages (KeyPages).
//
// Two launches per call:
//  build_lower: one CTA per 16 consecutive leaves of one (sequence, key head).
//    It streams the CTA's 1024 keys once (16-byte vector loads, 16 threads per
//    key row), writes the 16 leaf means and the 8 + 4 + 2 + 1 nodes of levels
//    2..5 above them from shared memory.  This pass reads the whole key tensor
//    once and is HBM-bound.
//  build_upper: one CTA per (sequence, key head) for levels 6..L (1/16 of the
//    nodes; reads level 5 from L2).
#include "pisa_common.cuh"
#include "pisa_internal.h"

namespace pisa {

constexpr int kLeavesPerCta = 16;
constexpr int kLowerLevels = 5;  // levels 1..5 live inside one CTA's subtree

__device__ __forceinline__ int64_t seq_len_of(const int32_t* seq_lens, int64_t b, int64_t N) {
  if (!seq_lens) return N;
  int64_t v = seq_lens[b];
  return v < 0 ? 0 : (v > N ? N : v);
}

// Mean of the `count` keys starting at `keys` for DPT consecutive dims, summed
// in key order with IEEE fp32 adds (the decode update uses the same routine).
template <int DPT>
__device__ __forceinline__ void leaf_mean_dims(const void* keys, int64_t row_stride_elems,
                                               bool bf16, int64_t count, float (&out)[DPT]) {
#pragma unroll
  for (int c = 0; c < DPT; ++c) out[c] = 0.0f;
  if (count <= 0) return;
#pragma unroll 4
  for (int64_t i = 0; i < count; ++i) {
    float v[DPT];
    if (bf16) {
      const uint16_t* p = reinterpret_cast<const uint16_t*>(keys) + i * row_stride_elems;
#pragma unroll
      for (int c = 0; c < DPT; c += 4) load4(p + c, true, v + c);
    } else {
      const float* p = reinterpret_cast<const float*>(keys) + i * row_stride_elems;
#pragma unroll
      for (int c = 0; c < DPT; c += 4) load4(p + c, false, v + c);
    }
#pragma unroll
    for (int c = 0; c < DPT; ++c) out[c] = __fadd_rn(out[c], v[c]);
  }
  const float n = (float)count;
#pragma unroll
  for (int c = 0; c < DPT; ++c) out[c] = __fdiv_rn(out[c], n);
}

// kPaged: keys through a page table (compiled separately, so the contiguous
// kernel keeps its registers and occupancy).
template <int D, bool kPaged>
__global__ void __launch_bounds__(256) build_lower_kernel(Prob pr, Pyr s, const void* __restrict__ k, KeyPages kp,
                                                          const int32_t* __restrict__ seq_lens,
                                                          float* __restrict__ pyr, int32_t* __restrict__ status) {
  constexpr int TPL = 16;            // threads per leaf row
  constexpr int DPT = D / TPL;       // dims per thread (8 or 4)
  __shared__ float sm[kLeavesPerCta][D];
  const int64_t b = blockIdx.z, h = blockIdx.y;
  const int64_t leaf0 = (int64_t)blockIdx.x * kLeavesPerCta;
  const int64_t len = seq_len_of(seq_lens, b, s.N);
  const bool bf16 = pr.dtype == PISA_BF16;
  const int tid = threadIdx.x;
  const int ll = tid / TPL, c0 = (tid % TPL) * DPT;
  const int64_t leaf = leaf0 + ll;
  const int64_t bh = b * pr.Hkv + h;
  float* ph = pyr + bh * s.P * D;

  // level 1: leaf means
  {
    int64_t cnt = leaf < s.nb ? node_count(s, 1, leaf, len) : 0;
    const size_t esz = bf16 ? 2 : 4;
    if (kPaged && cnt > 0) {
      const int32_t pg = kp.table[b * kp.max_pages + leaf];
      if (pg < 0 || pg >= kp.num_pages) {  // a page outside the pool is not read
        if (c0 == 0) set_status(status, PISA_DEV_BAD_INDEX);
        cnt = 0;
      }
    }
    const int64_t row = kPaged ? (cnt > 0 ? leaf_row(kp, pr.Hkv, s.N, s.C, b, h, leaf) : 0) : bh * s.N + leaf * s.C;
    const char* kb = reinterpret_cast<const char*>(k) + (row * D + c0) * esz;
    float m[DPT];
    leaf_mean_dims<DPT>(kb, D, bf16, cnt, m);
#pragma unroll
    for (int c = 0; c < DPT; ++c) sm[ll][c0 + c] = m[c];
    if (leaf < s.nb) {
      float* dst = ph + (s.off[0] + leaf) * D + c0;
#pragma unroll
      for (int c = 0; c < DPT; c += 4)
        *reinterpret_cast<float4*>(dst + c) = make_float4(m[c], m[c + 1], m[c + 2], m[c + 3]);
    }
  }
  __syncthreads();

  // levels 2..5 inside the subtree, in place in shared memory
  int nodes = kLeavesPerCta;
  for (int level = 2; level <= kLowerLevels && level <= s.L; ++level) {
    nodes >>= 1;
    const int64_t j0 = leaf0 >> (level - 1);
    float tmp[(kLeavesPerCta / 2) * D / 256 > 0 ? (kLeavesPerCta / 2) * D / 256 : 1];
    const int work = nodes * D;
    int n_my = 0;
    for (int w = tid; w < work; w += 256) {
      const int jl = w / D, c = w % D;
      const int64_t j = j0 + jl;
      const int64_t n0 = node_count(s, level - 1, 2 * j, len);
      const int64_t n1 = node_count(s, level - 1, 2 * j + 1, len);
      tmp[n_my++] = combine_children(sm[2 * jl][c], n0, sm[2 * jl + 1][c], n1);
    }
    __syncthreads();
    n_my = 0;
    for (int w = tid; w < work; w += 256) {
      const int jl = w / D, c = w % D;
      const int64_t j = j0 + jl;
      const float v = tmp[n_my++];
      sm[jl][c] = v;
      if (j < s.size[level - 1]) ph[(s.off[level - 1] + j) * D + c] = v;
    }
    __syncthreads();
  }
}

template <int D>
__global__ void __launch_bounds__(256) build_upper_kernel(Prob pr, Pyr s, const int32_t* __restrict__ seq_lens,
                                                          float* __restrict__ pyr) {
  // D / 4 threads per node, four consecutive dims each (float4); the node
  // counts are computed once per node, and the loop over a level's nodes is
  // unrolled so several child loads are in flight
  constexpr int TPN = D / 4, NPP = 256 / TPN;  // threads per node, nodes per pass
  const int64_t b = blockIdx.y, h = blockIdx.x;
  const int64_t len = seq_len_of(seq_lens, b, s.N);
  float* ph = pyr + (b * pr.Hkv + h) * s.P * D;
  const int c4 = (threadIdx.x % TPN) * 4, jl = threadIdx.x / TPN;
  for (int level = kLowerLevels + 1; level <= s.L; ++level) {
    const int n = (int)s.size[level - 1];
    const int nc = (int)s.size[level - 2];
    const float* child = ph + s.off[level - 2] * D;
    float* out = ph + s.off[level - 1] * D;
#pragma unroll 4
    for (int j = jl; j < n; j += NPP) {
      const int64_t n0 = node_count(s, level - 1, 2 * (int64_t)j, len);
      const bool has1 = 2 * j + 1 < nc;
      const int64_t n1 = has1 ? node_count(s, level - 1, 2 * (int64_t)j + 1, len) : 0;
      const float4 m0 = *reinterpret_cast<const float4*>(child + (int64_t)(2 * j) * D + c4);
      const float4 m1 = has1 ? *reinterpret_cast<const float4*>(child + (int64_t)(2 * j + 1) * D + c4)
                             : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      float4 r;
      r.x = combine_children(m0.x, n0, m1.x, n1);
      r.y = combine_children(m0.y, n0, m1.y, n1);
      r.z = combine_children(m0.z, n0, m1.z, n1);
      r.w = combine_children(m0.w, n0, m1.w, n1);
      *reinterpret_cast<float4*>(out + (int64_t)j * D + c4) = r;
    }
    __syncthreads();
  }
}

cudaError_t launch_build_pyramid(const Prob& pr, const Pyr& s, const void* k, const KeyPages& kp,
                                 const int32_t* seq_lens, float* pyr, int32_t* status, cudaStream_t st) {
  if (pr.B == 0 || pr.Hkv == 0 || s.nb == 0) return cudaSuccess;
  dim3 g1((unsigned)ceil_div64(s.nb, kLeavesPerCta), (unsigned)pr.Hkv, (unsigned)pr.B);
  note_launch();
  if (kp.table) {
    if (pr.d == 128) build_lower_kernel<128, true><<<g1, 256, 0, st>>>(pr, s, k, kp, seq_lens, pyr, status);
    else build_lower_kernel<64, true><<<g1, 256, 0, st>>>(pr, s, k, kp, seq_lens, pyr, status);
  } else {
    if (pr.d == 128) build_lower_kernel<128, false><<<g1, 256, 0, st>>>(pr, s, k, kp, seq_lens, pyr, status);
    else build_lower_kernel<64, false><<<g1, 256, 0, st>>>(pr, s, k, kp, seq_lens, pyr, status);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || s.L <= kLowerLevels) return e;
  dim3 g2((unsigned)pr.Hkv, (unsigned)pr.B);
  note_launch();
  if (pr.d == 128) build_upper_kernel<128><<<g2, 256, 0, st>>>(pr, s, seq_lens, pyr);
  else build_upper_kernel<64><<<g2, 256, 0, st>>>(pr, s, seq_lens, pyr);
  return cudaGetLastError();
}

}  // namespace pisa
