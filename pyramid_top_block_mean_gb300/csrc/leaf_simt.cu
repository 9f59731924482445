// leaf_simt.cu -- leaf LSE scoring on the CUDA cores, fused with the final
// Top-K: the path for fp32 inputs (which the bf16 tensor-core kernel does not
// take).  agihunt.info summary of "Block Sparse Attention with Log-Linear
// Complexity", kernel paragraph ("leaf LSE scoring") and LSE paragraph (first,
// previous and current blocks forced in).
//
// One warp per (sequence, key head, query).  The candidate leaves are the
// eligible children of the query's kept level-2 nodes (at most 2K).  For each
// leaf the warp streams its C raw keys (lane l holds dims [l*D/32, ...)),
// forms the G head dot products, reduces 32 (key, head) partials per
// transposing butterfly, and takes the per-head log2-sum-exp2 over the C keys.
#include "pisa_common.cuh"
#include "pisa_internal.h"

namespace pisa {

constexpr int kLeafWarps = 8;

struct LeafWarpSm {
  int32_t leaf[kMaxCand];
  float score[kMaxCand];
};

template <int D, int G>
__global__ void __launch_bounds__(kLeafWarps * 32) leaf_simt_kernel(Prob pr, Pyr s, const void* __restrict__ q,
                                                                    const void* __restrict__ k,
                                                                    const int32_t* __restrict__ kept2,
                                                                    int32_t* __restrict__ out_idx,
                                                                    float* __restrict__ out_score) {
  constexpr int DPL = D / 32;
  constexpr int NB = 32 / G;         // keys per reduction batch
  __shared__ LeafWarpSm smw[kLeafWarps];
  LeafWarpSm& sm = smw[threadIdx.x / 32];
  const int lane = threadIdx.x & 31;
  const int64_t qi = (int64_t)blockIdx.x * kLeafWarps + threadIdx.x / 32;
  if (qi >= pr.B * pr.Hkv * pr.N) return;
  const int64_t t = qi % pr.N, bh = qi / pr.N;
  const int64_t b = bh / pr.Hkv, h = bh % pr.Hkv;
  const int K = pr.K, W = K + 3;
  const int64_t qb = t / s.C;
  const bool bf16 = pr.dtype == PISA_BF16;
  const size_t esz = bf16 ? 2 : 4;

  // candidate leaves (ascending)
  int nl = 0;
  for (int i0 = 0; i0 < K; i0 += 32) {
    const int i = i0 + lane;
    const int32_t p = i < K ? kept2[qi * K + i] : -1;
    int e0 = 0, e1 = 0;
    if (p >= 0) {
      e0 = node_eligible(1, 2 * (int64_t)p, qb);
      e1 = node_eligible(1, 2 * (int64_t)p + 1, qb);
    }
    const int c = e0 + e1;
    int x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    const int tot = __shfl_sync(0xffffffffu, x, 31);
    int pos = nl + x - c;
    if (e0) sm.leaf[pos++] = 2 * p;
    if (e1) sm.leaf[pos++] = 2 * p + 1;
    nl += tot;
  }
  __syncwarp();

  float qr[G][DPL];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const char* p = reinterpret_cast<const char*>(q) + (((b * pr.Hq + h * G + g) * pr.N + t) * D + lane * DPL) * esz;
    if (DPL == 4) load4(p, bf16, qr[g]);
    else load2(p, bf16, qr[g]);
#pragma unroll
    for (int c = 0; c < DPL; ++c) qr[g][c] *= pr.scale2;
  }
  const char* kh = reinterpret_cast<const char*>(k) + (bh * pr.N * D + lane * DPL) * esz;

  for (int li = 0; li < nl; ++li) {
    const int64_t leaf = sm.leaf[li];
    // C = 64 keys, processed NB at a time
    constexpr int NBAT = 64 / NB;
    float vals[NBAT];
#pragma unroll
    for (int bt = 0; bt < NBAT; ++bt) {
      float v[32];
#pragma unroll
      for (int n = 0; n < NB; ++n) {
        const int64_t key = leaf * 64 + bt * NB + n;
        float kv[DPL];
        const char* p = kh + key * D * esz;
        if (DPL == 4) load4(p, bf16, kv);
        else load2(p, bf16, kv);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float acc = 0.0f;
#pragma unroll
          for (int c = 0; c < DPL; ++c) acc = fmaf(qr[g][c], kv[c], acc);
          v[n * G + g] = acc;
        }
      }
      vals[bt] = warp_transpose_sum32(v);  // lane: key bt*NB + lane/G, head lane%G
    }
    float lse;
    if (pr.scorer == PISA_SCORER_LSE) {
      // per head (lanes sharing lane % G): log2-sum-exp2 over the 64 keys
      float m = vals[0];
#pragma unroll
      for (int bt = 1; bt < NBAT; ++bt) m = fmaxf(m, vals[bt]);
#pragma unroll
      for (int o = 16; o >= G; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float sum = 0.0f;
#pragma unroll
      for (int bt = 0; bt < NBAT; ++bt) sum += exp2f(vals[bt] - m);
#pragma unroll
      for (int o = 16; o >= G; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      lse = m + __log2f(sum);
    } else {
      // PISA-1 / PISA-2: mean, then centred second moment, of the 64 scaled dots
      float s1 = 0.0f;
#pragma unroll
      for (int bt = 0; bt < NBAT; ++bt) s1 += vals[bt];
#pragma unroll
      for (int o = 16; o >= G; o >>= 1) s1 += __shfl_xor_sync(0xffffffffu, s1, o);
      const float mean = s1 * (1.0f / 64.0f);
      float s2 = 0.0f;
#pragma unroll
      for (int bt = 0; bt < NBAT; ++bt) s2 = fmaf(vals[bt] - mean, vals[bt] - mean, s2);
#pragma unroll
      for (int o = 16; o >= G; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
      lse = moment_score(pr.scorer, 64.0f, mean, s2);
    }
    // sum over the G heads (lanes 0..G-1 hold distinct heads)
#pragma unroll
    for (int o = G / 2; o >= 1; o >>= 1) lse += __shfl_xor_sync(0xffffffffu, lse, o);
    if (lane == 0) sm.score[li] = lse != lse ? -INFINITY : lse;  // NaN ranks as -inf
  }
  __syncwarp();

  // Top-K of the candidate leaves (ties to the lower index) plus F, ascending.
  int32_t* oi = out_idx + qi * W;
  float* os = out_score ? out_score + qi * W : nullptr;
  int nkept = 0;
  for (int i0 = 0; i0 < nl; i0 += 32) {
    const int i = i0 + lane;
    int keep = 0;
    if (i < nl) {
      int rank = 0;
      for (int j = 0; j < nl; ++j) rank += beats(sm.score[j], sm.leaf[j], sm.score[i], sm.leaf[i]) ? 1 : 0;
      keep = rank < K;
    }
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    const int pos = 1 + nkept + __popc(bal & ((1u << lane) - 1));
    if (keep && pos <= K) {  // the ranking order is total: at most K are kept
      oi[pos] = sm.leaf[i];
      if (os) os[pos] = sm.score[i] * kLn2;
    }
    nkept += __popc(bal);
  }
  if (lane == 0) {
    int pos = 0;
    oi[pos] = 0;
    if (os) os[pos] = INFINITY;
    pos = 1 + nkept;
    if (qb - 1 > 0) { oi[pos] = (int32_t)(qb - 1); if (os) os[pos] = INFINITY; ++pos; }
    if (qb > 0) { oi[pos] = (int32_t)qb; if (os) os[pos] = INFINITY; ++pos; }
    for (; pos < W; ++pos) { oi[pos] = -1; if (os) os[pos] = -INFINITY; }
  }
}

cudaError_t launch_leaf_simt(const Prob& pr, const Pyr& s, const void* q, const void* k, const int32_t* kept2,
                             int32_t* out_idx, float* out_score, cudaStream_t st) {
  const int64_t nq = pr.B * pr.Hkv * pr.N;
  if (nq == 0) return cudaSuccess;
  const unsigned grid = (unsigned)ceil_div64(nq, kLeafWarps);
#define PISA_LEAF_CASE(DD, GG)                                                                         \
  if (pr.d == DD && pr.G == GG) {                                                                      \
    note_launch();                                                                                     \
    leaf_simt_kernel<DD, GG><<<grid, kLeafWarps * 32, 0, st>>>(pr, s, q, k, kept2, out_idx, out_score); \
    return cudaGetLastError();                                                                         \
  }
  PISA_LEAF_CASE(128, 1) PISA_LEAF_CASE(128, 2) PISA_LEAF_CASE(128, 4) PISA_LEAF_CASE(128, 8)
  PISA_LEAF_CASE(64, 1) PISA_LEAF_CASE(64, 2) PISA_LEAF_CASE(64, 4) PISA_LEAF_CASE(64, 8)
#undef PISA_LEAF_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pisa
