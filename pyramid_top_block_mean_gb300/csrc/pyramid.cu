// pyramid.cu -- key pyramid build (mean-pooled leaves, then g = 2 pooling of
// every coarser level).  agihunt.info summary of "Block Sparse Attention with
// Log-Linear Complexity", pyramid paragraph; rcap.io post, "Think of the keys
// as leaves of a tree".
//
// The keys are the contiguous cache or a pool of pages (KeyPages).
//
// Two launches per call:
//  build_lower: one CTA per 16 consecutive leaves of one (sequence, key head).
//    It copies the CTA's 1024 keys once into shared memory (one bulk copy per
//    leaf, two rounds of leaves in flight), sums them there, and writes the
//    16 leaf means and the 8 + 4 + 2 + 1 nodes of levels 2..5 above them.
//    This pass reads the whole key tensor once and is HBM-bound.
//  build_upper: one CTA per (sequence, key head) for levels 6..L (1/16 of the
//    nodes; reads level 5 from L2).
#include "pisa_common.cuh"
#include "pisa_internal.h"
#include "tc_ptx.cuh"

namespace pisa {

constexpr int kLeavesPerCta = 16;
constexpr int kLowerLevels = 5;  // levels 1..5 live inside one CTA's subtree

__device__ __forceinline__ int64_t seq_len_of(const int32_t* seq_lens, int64_t b, int64_t N) {
  if (!seq_lens) return N;
  int64_t v = seq_lens[b];
  return v < 0 ? 0 : (v > N ? N : v);
}

// Shared memory of build_lower: two stages of one round's leaves (the raw
// keys, copied whole), the CTA's 16 leaf means, and the stages' barriers.
constexpr int kBuildThreads = 256;
constexpr int kBuildStages = 2;
constexpr uint64_t kBuildWaitNs = 4000000000ull;

template <int D>
constexpr int leaves_per_round() { return kBuildThreads / D; }  // one thread per (leaf, dim)

static size_t build_lower_smem(int d, bool bf16, int C) {
  const size_t stage = (size_t)(kBuildThreads / d) * C * d * (bf16 ? 2 : 4);
  return 128 + kBuildStages * stage + (size_t)kLeavesPerCta * d * 4 + 64;
}

// kPaged: keys through a page table (compiled separately, so the contiguous
// kernel keeps its registers and occupancy).
//
// The CTA's leaves are taken in rounds of 256 / D (one thread per leaf and
// dimension).  Thread 0 copies a round's raw keys into a shared-memory stage
// with one bulk copy per leaf (a leaf's C rows are contiguous in the cache
// and in a page), two rounds ahead of the reduction, so each CTA keeps tens
// of kilobytes of HBM reads in flight; every thread then sums its dimension
// over the leaf's keys in key order with IEEE fp32 adds and one division,
// as the decode step recomputes its current leaf (decode.cu), so an
// incrementally updated pyramid equals a fresh build bit for bit.
template <int D, bool kPaged>
__global__ void __launch_bounds__(kBuildThreads) build_lower_kernel(Prob pr, Pyr s, const void* __restrict__ k,
                                                                   KeyPages kp, const int32_t* __restrict__ seq_lens,
                                                                   float* __restrict__ pyr, int32_t* __restrict__ status) {
  pdl_wait();
  constexpr int LPR = leaves_per_round<D>();
  constexpr int kRounds = kLeavesPerCta / LPR;
  extern __shared__ unsigned char bsm_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(bsm_raw) + 127) & ~(uintptr_t)127);
  const bool bf16 = pr.dtype == PISA_BF16;
  const uint32_t esz = bf16 ? 2u : 4u;
  const uint32_t leaf_bytes = (uint32_t)s.C * D * esz;
  const uint32_t stage_bytes = LPR * leaf_bytes;
  float (*sm)[D] = reinterpret_cast<float (*)[D]>(base + kBuildStages * stage_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + kBuildStages * stage_bytes + kLeavesPerCta * D * 4);
  __shared__ int32_t abort_flag;
  const int64_t b = blockIdx.z, h = blockIdx.y;
  const int64_t leaf0 = (int64_t)blockIdx.x * kLeavesPerCta;
  const int64_t len = seq_len_of(seq_lens, b, s.N);
  const int tid = threadIdx.x;
  const int lr = tid / D, c = tid % D;  // leaf within the round, dimension
  const int64_t bh = b * pr.Hkv + h;
  float* ph = pyr + bh * s.P * D;
  const unsigned char* kbytes = reinterpret_cast<const unsigned char*>(k);

  // keys of a leaf present in this call (0 past the sequence or for a page
  // outside the pool, which is reported and not read)
  auto leaf_count = [&](int64_t leaf, bool report) -> int64_t {
    int64_t cnt = leaf < s.nb ? node_count(s, 1, leaf, len) : 0;
    if (kPaged && cnt > 0) {
      const int32_t pg = kp.table[b * kp.max_pages + leaf];
      if (pg < 0 || pg >= kp.num_pages) {
        if (report) set_status(status, PISA_DEV_BAD_INDEX);
        cnt = 0;
      }
    }
    return cnt;
  };
  // thread 0: one bulk copy per leaf of round r into stage r % 2
  auto issue = [&](int r) {
    const int st = r % kBuildStages;
    uint32_t total = 0;
    int64_t cnts[LPR];
#pragma unroll
    for (int j = 0; j < LPR; ++j) {
      cnts[j] = leaf_count(leaf0 + r * LPR + j, true);
      total += (uint32_t)cnts[j] * D * esz;
    }
    const uint32_t bar = ptx::smem_u32(&full[st]);
    ptx::mbar_arrive_expect_tx(bar, total);
#pragma unroll
    for (int j = 0; j < LPR; ++j) {
      if (cnts[j] == 0) continue;
      const int64_t row = leaf_row(kp, pr.Hkv, s.N, s.C, b, h, leaf0 + r * LPR + j);
      ptx::bulk_g2s(ptx::smem_u32(base + st * stage_bytes + j * leaf_bytes), kbytes + row * D * esz,
                    (uint32_t)cnts[j] * D * esz, bar);
    }
  };

  if (tid == 0) {
    for (int st = 0; st < kBuildStages; ++st) ptx::mbar_init(ptx::smem_u32(&full[st]), 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int r = 0; r < kBuildStages && r < kRounds; ++r) issue(r);

  // level 1: leaf means
  for (int r = 0; r < kRounds; ++r) {
    const int st = r % kBuildStages;
    const int64_t leaf = leaf0 + r * LPR + lr;
    const int64_t cnt = leaf_count(leaf, false);
    const bool ok = ptx::mbar_wait_bounded(ptx::smem_u32(&full[st]), (r / kBuildStages) & 1, &abort_flag, kBuildWaitNs);
    if (!ok) abort_flag = 1;
    float m = 0.0f;
    if (ok && cnt > 0) {
      const unsigned char* src = base + st * stage_bytes + lr * leaf_bytes + c * esz;
      if (bf16) {
#pragma unroll 8
        for (int64_t i = 0; i < cnt; ++i)
          m = __fadd_rn(m, __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t*>(src + i * D * 2) << 16));
      } else {
#pragma unroll 8
        for (int64_t i = 0; i < cnt; ++i) m = __fadd_rn(m, *reinterpret_cast<const float*>(src + i * D * 4));
      }
      m = __fdiv_rn(m, (float)cnt);
    }
    sm[r * LPR + lr][c] = m;
    if (leaf < s.nb) ph[(s.off[0] + leaf) * D + c] = m;
    __syncthreads();  // the stage is read: thread 0 refills it two rounds ahead
    if (tid == 0 && r + kBuildStages < kRounds && !abort_flag) issue(r + kBuildStages);
  }
  if (tid == 0 && abort_flag) set_status(status, PISA_DEV_TIMEOUT);

  // levels 2..5 inside the subtree, in place in shared memory
  int nodes = kLeavesPerCta;
  for (int level = 2; level <= kLowerLevels && level <= s.L; ++level) {
    nodes >>= 1;
    const int64_t j0 = leaf0 >> (level - 1);
    float tmp[(kLeavesPerCta / 2) * D / kBuildThreads > 0 ? (kLeavesPerCta / 2) * D / kBuildThreads : 1];
    const int work = nodes * D;
    int n_my = 0;
    for (int w = tid; w < work; w += kBuildThreads) {
      const int jl = w / D, cc = w % D;
      const int64_t j = j0 + jl;
      const int64_t n0 = node_count(s, level - 1, 2 * j, len);
      const int64_t n1 = node_count(s, level - 1, 2 * j + 1, len);
      tmp[n_my++] = combine_children(sm[2 * jl][cc], n0, sm[2 * jl + 1][cc], n1);
    }
    __syncthreads();
    n_my = 0;
    for (int w = tid; w < work; w += kBuildThreads) {
      const int jl = w / D, cc = w % D;
      const int64_t j = j0 + jl;
      const float v = tmp[n_my++];
      sm[jl][cc] = v;
      if (j < s.size[level - 1]) ph[(s.off[level - 1] + j) * D + cc] = v;
    }
    __syncthreads();
  }
}

template <int D>
__global__ void __launch_bounds__(256) build_upper_kernel(Prob pr, Pyr s, const int32_t* __restrict__ seq_lens,
                                                          float* __restrict__ pyr) {
  pdl_wait();
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

// Levels 6..L with the whole of level 5 in shared memory (when it fits):
// each level is computed from the previous one in shared memory, into the
// other of two buffers, and written out; one CTA of 1024 threads per
// (sequence, key head), one __syncthreads per level instead of a round trip
// through L2.
constexpr size_t kUpperSmemMax = 200 * 1024;

static size_t build_upper_smem(int d, int64_t n5) { return (size_t)(n5 + (n5 + 1) / 2) * d * 4; }

constexpr int kUpperThreads = 1024;

template <int D>
__global__ void __launch_bounds__(kUpperThreads) build_upper_smem_kernel(Prob pr, Pyr s,
                                                                         const int32_t* __restrict__ seq_lens,
                                                                         float* __restrict__ pyr) {
  pdl_wait();
  extern __shared__ float4 usm4[];
  float* usm = reinterpret_cast<float*>(usm4);
  constexpr int TPN = D / 4, NPP = kUpperThreads / TPN;  // threads per node (four dims each), nodes per pass
  const int64_t b = blockIdx.y, h = blockIdx.x;
  const int64_t len = seq_len_of(seq_lens, b, s.N);
  float* ph = pyr + (b * pr.Hkv + h) * s.P * D;
  const int c4 = (threadIdx.x % TPN) * 4, jl = threadIdx.x / TPN;
  const int n5 = (int)s.size[kLowerLevels - 1];
  float* const buf0 = usm;                     // level 5, then 7, 9, ...
  float* const buf1 = usm + (int64_t)n5 * D;    // levels 6, 8, ...
  __shared__ uint64_t bar;
  __shared__ int32_t abort_flag;
  {
    // level 5 by bulk copies of at most 32 KB (rows are 16-byte multiples)
    const uint32_t bytes = (uint32_t)n5 * D * 4;
    if (threadIdx.x == 0) {
      abort_flag = 0;
      ptx::mbar_init(ptx::smem_u32(&bar), 1);
      ptx::fence_mbar_init();
      ptx::mbar_arrive_expect_tx(ptx::smem_u32(&bar), bytes);
      const unsigned char* src = reinterpret_cast<const unsigned char*>(ph + s.off[kLowerLevels - 1] * D);
      for (uint32_t o = 0; o < bytes; o += 32768)
        ptx::bulk_g2s(ptx::smem_u32(reinterpret_cast<unsigned char*>(buf0) + o), src + o,
                      bytes - o < 32768 ? bytes - o : 32768, ptx::smem_u32(&bar));
    }
    __syncthreads();
    if (!ptx::mbar_wait_bounded(ptx::smem_u32(&bar), 0, &abort_flag, kBuildWaitNs)) abort_flag = 1;
    __syncthreads();
    if (abort_flag) return;  // a copy that never lands leaves levels >= 6 unwritten
  }
  int cur = 0;
  for (int level = kLowerLevels + 1; level <= s.L; ++level) {
    const int n = (int)s.size[level - 1];
    const int nc = (int)s.size[level - 2];
    const float* child = cur ? buf1 : buf0;
    float* nxt = cur ? buf0 : buf1;
    float* out = ph + s.off[level - 1] * D;
    for (int j = jl; j < n; j += NPP) {
      const int64_t n0 = node_count(s, level - 1, 2 * (int64_t)j, len);
      const bool has1 = 2 * j + 1 < nc;
      const int64_t n1 = has1 ? node_count(s, level - 1, 2 * (int64_t)j + 1, len) : 0;
      const float4 m0 = *reinterpret_cast<const float4*>(child + (2 * j) * D + c4);
      const float4 m1 = has1 ? *reinterpret_cast<const float4*>(child + (2 * j + 1) * D + c4)
                             : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      float4 r;
      r.x = combine_children(m0.x, n0, m1.x, n1);
      r.y = combine_children(m0.y, n0, m1.y, n1);
      r.z = combine_children(m0.z, n0, m1.z, n1);
      r.w = combine_children(m0.w, n0, m1.w, n1);
      *reinterpret_cast<float4*>(nxt + j * D + c4) = r;
      *reinterpret_cast<float4*>(out + (int64_t)j * D + c4) = r;
    }
    __syncthreads();
    cur ^= 1;
  }
}

cudaError_t launch_build_pyramid(const Prob& pr, const Pyr& s, const void* k, const KeyPages& kp,
                                 const int32_t* seq_lens, float* pyr, int32_t* status, cudaStream_t st) {
  if (pr.B == 0 || pr.Hkv == 0 || s.nb == 0) return cudaSuccess;
  dim3 g1((unsigned)ceil_div64(s.nb, kLeavesPerCta), (unsigned)pr.Hkv, (unsigned)pr.B);
  const size_t smem = build_lower_smem(pr.d, pr.dtype == PISA_BF16, (int)s.C);
  auto kern = kp.table ? (pr.d == 128 ? build_lower_kernel<128, true> : build_lower_kernel<64, true>)
                       : (pr.d == 128 ? build_lower_kernel<128, false> : build_lower_kernel<64, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  note_launch();
  e = launch_pdl(false, kern, g1, dim3(kBuildThreads), smem, st, pr, s, k, kp, seq_lens, pyr, status);
  if (e != cudaSuccess || s.L <= kLowerLevels) return e;
  dim3 g2((unsigned)pr.Hkv, (unsigned)pr.B);
  const size_t usmem = build_upper_smem(pr.d, s.size[kLowerLevels - 1]);
  if (usmem <= kUpperSmemMax) {
    auto ukern = pr.d == 128 ? build_upper_smem_kernel<128> : build_upper_smem_kernel<64>;
    e = cudaFuncSetAttribute(ukern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)usmem);
    if (e != cudaSuccess) return e;
    note_launch();
    return launch_pdl(true, ukern, g2, dim3(kUpperThreads), usmem, st, pr, s, seq_lens, pyr);
  }
  note_launch();
  return launch_pdl(true, pr.d == 128 ? build_upper_kernel<128> : build_upper_kernel<64>, g2, dim3(256), 0, st, pr, s,
                    seq_lens, pyr);
}

}  // namespace pisa
