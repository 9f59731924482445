// pisa_common.cuh -- device helpers shared by the selector's kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pisa.h"

namespace pisa {

constexpr int kMaxLevels = 40;
constexpr int kMaxK = 32;      // blocks kept per level
constexpr int kMaxCand = 2 * kMaxK;  // candidates per level (g = 2)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Shape of the key pyramid for a capacity of N keys (see pisa.h).
struct Pyr {
  int32_t L;                  // levels
  int32_t C;                  // keys per leaf
  int64_t N;                  // key capacity
  int64_t nb;                 // leaves
  int64_t P;                  // nodes per (sequence, key head)
  int64_t size[kMaxLevels];   // size[l-1] = nodes of level l
  int64_t off[kMaxLevels];    // off[l-1]  = first row of level l
};

// Problem description passed by value to the kernels.
struct Prob {
  int64_t B, N;
  int32_t Hq, Hkv, G, d, C, K;
  float scale2;     // score scale times log2(e): exponents are taken base 2
  int32_t dtype;    // PISA_BF16 / PISA_FP32
  int32_t scorer;   // pisa_scorer
  int32_t prefix;   // prefill walks read prefix-consistent summaries (PISA_SUMMARIES_PREFIX)
};

__host__ __device__ inline int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Keys present in node (level, j) when the sequence holds `len` keys.
__host__ __device__ inline int64_t node_count(const Pyr& s, int level, int64_t j, int64_t len) {
  const int64_t w = (int64_t)s.C << (level - 1);
  int64_t c = len - j * w;
  return c < 0 ? 0 : (c > w ? w : c);
}

// E = [1, qb-2]: a level-`level` node is eligible when its leaf range meets E.
__host__ __device__ inline bool node_eligible(int level, int64_t j, int64_t qb) {
  const int64_t e_hi = qb - 2;
  if (e_hi < 1) return false;
  const int64_t lo = j << (level - 1);
  const int64_t hi = ((j + 1) << (level - 1)) - 1;
  return lo <= e_hi && hi >= 1;
}

// Number of eligible nodes at `level` (level >= 2: nodes 0..(qb-2)>>(l-1);
// level 1: leaves 1..qb-2).
__host__ __device__ inline int64_t eligible_count(int level, int64_t qb) {
  if (qb - 2 < 1) return 0;
  if (level == 1) return qb - 2;
  return ((qb - 2) >> (level - 1)) + 1;
}

// Parent summary from its two children, count-weighted, IEEE round-to-nearest
// steps in a fixed order.  Used by the build and by the decode update so the
// two agree bit for bit.
__device__ __forceinline__ float combine_children(float m0, int64_t n0, float m1, int64_t n1) {
  if (n1 == 0) return m0;
  if (n0 == 0) return 0.0f;
  const float a = __fmul_rn((float)n0, m0);
  const float b = __fmul_rn((float)n1, m1);
  return __fdiv_rn(__fadd_rn(a, b), (float)(n0 + n1));
}

__device__ __forceinline__ float bf16_to_f(uint16_t v) {
  return __uint_as_float(((uint32_t)v) << 16);
}

// Load 4 consecutive elements (bf16 or fp32) as floats; `p` points at the
// first element (8-byte aligned for bf16, 16-byte for fp32).
__device__ __forceinline__ void load4(const void* p, bool bf16, float out[4]) {
  if (bf16) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
    out[0] = __uint_as_float(v.x << 16);
    out[1] = __uint_as_float(v.x & 0xffff0000u);
    out[2] = __uint_as_float(v.y << 16);
    out[3] = __uint_as_float(v.y & 0xffff0000u);
  } else {
    const float4 v = __ldg(reinterpret_cast<const float4*>(p));
    out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
  }
}

__device__ __forceinline__ void load2(const void* p, bool bf16, float out[2]) {
  if (bf16) {
    const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(p));
    out[0] = __uint_as_float(v << 16);
    out[1] = __uint_as_float(v & 0xffff0000u);
  } else {
    const float2 v = __ldg(reinterpret_cast<const float2*>(p));
    out[0] = v.x; out[1] = v.y;
  }
}

// Sum 32 per-lane partial values over the warp so that lane L ends with the
// total of value index L (a transposing butterfly: 31 shuffles in all).
__device__ __forceinline__ float warp_transpose_sum32(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = upper ? v[i] : v[i + o];
      const float keep = upper ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0];
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// log2(2^a + 2^b) without overflow.
__device__ __forceinline__ float lse2_pair(float a, float b) {
  const float m = fmaxf(a, b), n = fminf(a, b);
  return m + __log2f(1.0f + exp2f(n - m));
}

// Block scorers (agihunt.info summary, LSE paragraph: PISA-1 keeps only the
// mean, PISA-2 adds the variance term of the LSE Taylor expansion; rcap.io,
// "The scoring rule matters": truncations at first and second order).  Over
// n summands y_i in log2 units (scaled dots times log2 e):
//   PISA_SCORER_LSE:      log2 sum 2^y_i
//   PISA_SCORER_MEAN:     log2 n + mean(y)
//   PISA_SCORER_MEAN_VAR: log2 n + mean(y) + (ln 2 / 2) var(y)
// which are the natural-log log n + mean(x) (+ var(x) / 2) times log2 e.
constexpr float kHalfLn2 = 0.34657359027997264f;

// Score of a node from the scaled dots (log2 units) of its two eligible children.
__device__ __forceinline__ float pair_score(int scorer, float a, float b) {
  if (scorer == PISA_SCORER_LSE) return lse2_pair(a, b);
  const float mean = 0.5f * (a + b);
  if (scorer == PISA_SCORER_MEAN) return 1.0f + mean;
  const float h = 0.5f * (a - b);
  return 1.0f + mean + kHalfLn2 * (h * h);
}

// PISA-1 / PISA-2 score from n summands with mean `mean` and centred second
// moment m2 = sum (y_i - mean)^2 (log2 units).
__device__ __forceinline__ float moment_score(int scorer, float n, float mean, float m2) {
  const float r = __log2f(n) + mean;
  return scorer == PISA_SCORER_MEAN_VAR ? r + kHalfLn2 * (m2 / n) : r;
}

// Running count, mean and centred second moment (Welford's update; Chan's
// merge of two partial sets).
struct Moments {
  float n, mean, m2;
};
__device__ __forceinline__ void mom_add(Moments& s, float y) {
  s.n += 1.0f;
  const float d = y - s.mean;
  s.mean += d / s.n;
  s.m2 = fmaf(d, y - s.mean, s.m2);
}
__device__ __forceinline__ void mom_merge(Moments& a, float nb, float meanb, float m2b) {
  const float n = a.n + nb;
  if (nb == 0.0f || n == 0.0f) return;
  const float d = meanb - a.mean;
  a.mean = fmaf(d, nb / n, a.mean);
  a.m2 = a.m2 + m2b + d * d * (a.n * nb / n);
  a.n = n;
}

// Where the raw keys of leaf `leaf` of (sequence b, key head h) start, in rows
// of d elements: the contiguous cache [B, Hkv, N, d], or a pool of pages of C
// keys laid out [num_pages, Hkv, C, d] and addressed through a page table
// [B, max_pages] (page j of a sequence holds its leaf j).
struct KeyPages {
  const int32_t* table;  // null: contiguous
  int64_t max_pages, num_pages;
};
__device__ __forceinline__ int64_t leaf_row(const KeyPages& kp, int64_t Hkv, int64_t N, int64_t C, int64_t b,
                                            int64_t h, int64_t leaf) {
  if (!kp.table) return (b * Hkv + h) * N + leaf * C;
  return ((int64_t)kp.table[b * kp.max_pages + leaf] * Hkv + h) * C;
}

// Kernels launched with launch_pdl start here: wait until the previous grid
// on the stream has completed and its memory operations are visible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Record the first device fault in the workspace status word.
__device__ __forceinline__ void set_status(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

// Higher score first; equal scores go to the lower node index.
// Ranking order of every Top-K: higher score first, then lower index.  The
// callers map a NaN score to -inf when they load it, so the order is total
// whatever the inputs hold and a Top-K keeps exactly min(K, n) candidates.
__device__ __forceinline__ bool beats(float sa, int32_t ia, float sb, int32_t ib) {
  return sa > sb || (sa == sb && ia < ib);
}

}  // namespace pisa
