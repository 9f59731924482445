// route_haar.cu -- top-down pyramid routing over a difference ("Haar")
// form of the pyramid, with the dot products on the tensor cores (bf16
// queries, GQA groups of 4 query heads).  Same walk and scores as route.cu
// (rcap.io post on "Block Sparse Attention with Log-Linear Complexity":
// "Selection walks the tree top-down", "The scoring rule matters";
// agihunt.info summary, kernel paragraph: one selection per GQA group, the
// heads' scores summed).
//
// Summary rows.  For every node (l, j) of level l >= 2 the preparation
// kernel stores two rows, each as fp16 with a power-of-two scale of its own
// (so that the row's largest element lands in [2^14, 2^15)):
//   MU  = mu(l, j) - mu(root)            (the summary relative to the root's)
//   DD  = mu(l-1, 2j) - mu(l-1, 2j+1)    (the difference of its two children;
//                                         zero when the node has one child)
// plus the fp16 rounding residual of each (lo) and its 2-norm.  Because the
// parent is the count-weighted mean of its children,
//   q.mu(child 0) = q.mu(node) + n1/(n0+n1) q.DD,
//   q.mu(child 1) = q.mu(node) - n0/(n0+n1) q.DD,
// so one DD row per candidate gives both of its children's dots from the
// candidate's own dot, and the rounding errors of the levels only add up
// (no factor grows along the path).  Dots relative to the root differ from
// the true ones by one constant per head, which shifts every candidate's
// group score by the same amount and leaves each Top-K unchanged.
//
// Precision.  An fp16 row moves half the bytes of the bf16 hi + lo pair that
// an fp32-faithful dot needs.  Its rounding error in a dot is at most
// s |q_h| |residual| (Cauchy-Schwarz); when that bound, summed over the
// group's heads, exceeds kLoTau (log2 units) the residual row is fetched too
// and multiplied in the same accumulators (rows with unusually large
// summaries, such as the ancestors of a block of planted keys).  Otherwise the
// error stays a few 1e-5 in the group score, two orders of magnitude below
// the 1e-3 margin within which two candidates count as tied.
//
// A warp walks two queries (16 lanes of bookkeeping each).  Per level and
// query, every candidate needs one DD row (and, at the start level, its MU
// row); eight rows at a time are multiplied against the query's four head
// vectors as m16n8k16 MMAs with A = the 8 rows' first halves (MMA rows 0-7)
// and second halves (rows 8-15) and B = the 4 heads x the two halves, of which
// the two half-diagonal blocks are used.  Rows are stored so that a lane's A
// fragments of two consecutive MMAs are one 32-byte load (the four lanes of a
// row read one whole 128-byte line per load, and no fragment register is
// moved before its MMA), and the lane of (row r, head h) ends with that row's
// whole dot with head h.
#include <cuda_fp16.h>

#include <algorithm>

#include "pisa_common.cuh"
#include "pisa_internal.h"

namespace pisa {

namespace {

// Residual fetch threshold: the bound on a row's fp16 rounding error in the
// group score, in log2 units (2e-3 in natural-log units).
constexpr float kLoTau = 2.0e-3f * kLog2e;

__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

// Exponent e such that max * 2^e lies in [2^14, 2^15) (0 for zero or
// non-finite max), clamped so that 2^e and 2^-e are normal floats.
__device__ __forceinline__ int row_exponent(float mx) {
  if (!(mx > 0.0f) || !(mx < INFINITY)) return 0;
  const int E = (int)((__float_as_uint(mx) >> 23) & 0xffu) - 127;
  return min(126, max(-126, 14 - E));
}

// Stored row layout (D elements).  For k-step kk (16 dims of each half,
// hd = D / 2) and quad thread t, the f16 pairs
//   {c0, c0+1}, {hd+c0, hd+c0+1}, {c0+8, c0+9}, {hd+c0+8, hd+c0+9},  c0 = 16 kk + 2 t,
// are that thread's A fragment (a0, a1, a2, a3) of the MMA in which row r
// holds the first half of node r and row r + 8 its second half.  The 16-byte
// fragments of k-steps 2m and 2m + 1 of thread t are adjacent, at byte
// 128 m + 32 t: one 32-byte load per thread and k-step pair, and the quad's
// four loads cover one whole 128-byte line.  inv_row_pos(p) is the dim held
// at position p (so the prep kernel writes each lane's piece contiguously):
// p = 8 chunk + 2 word + (kp & 1) with chunk = 8 (kk >> 1) + 2 t + (kk & 1),
// word = 2 (kp >> 3) + (half of the row), kp = dim within the k-step.
__device__ __forceinline__ int inv_row_pos(int p, int D) {
  const int chunk = p >> 3, word = (p >> 1) & 3;
  const int kk = ((chunk >> 3) << 1) | (chunk & 1);
  const int t = (chunk >> 1) & 3;
  const int kp = ((word >> 1) << 3) | (t << 1) | (p & 1);
  return (word & 1) * (D / 2) + kk * 16 + kp;
}

// 32 bytes from global memory (read-only path), as two 16-byte fragments.
__device__ __forceinline__ void ldg_frag2(const void* p, uint4& a, uint4& b) {
  asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
               : "l"(p));
}

__device__ __forceinline__ uint32_t orderable_key_h(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum of v in {0, 1, 2} over the 16 lanes of this lane's
// half of the warp (two ballots); *tot receives the half's total.
__device__ __forceinline__ int prefix16h(int v, int lane, int* tot) {
  const unsigned b0 = __ballot_sync(0xffffffffu, v & 1);
  const unsigned b1 = __ballot_sync(0xffffffffu, v & 2);
  const unsigned hm = (lane & 16) ? 0xffff0000u : 0x0000ffffu;
  const unsigned lt = hm & ((1u << lane) - 1u);
  *tot = __popc(b0 & hm) + 2 * __popc(b1 & hm);
  return __popc(b0 & lt) + 2 * __popc(b1 & lt);
}

__device__ __forceinline__ bool elig_node_h(int level, int j, int e_hi) {
  return (j << (level - 1)) <= e_hi && (((j + 1) << (level - 1)) - 1) >= 1;
}

__device__ __forceinline__ int count_node_h(int C, int level, int j, int64_t N) {
  const int64_t w = (int64_t)C << (level - 1);
  const int64_t c = N - (int64_t)j * w;
  return (int)(c < 0 ? 0 : (c > w ? w : c));
}

__device__ __forceinline__ float comp4(const float4& v, int g) {
  return g == 0 ? v.x : (g == 1 ? v.y : (g == 2 ? v.z : v.w));
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint4& a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2_fast(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace

// One warp per stored row: row w of [BH, P2, 2] is (node r = w / 2 of the
// levels >= 2, kind w % 2: MU or DD).  P2 = P - n_1 rows per (sequence, key
// head); node (l, j) is row off_l - n_1 + j.  meta[r] = {2^-e of MU, norm of
// the MU residual, 2^-e of DD, norm of the DD residual} (residual norms in
// the pyramid's units).
__global__ void haar_prep_kernel(int64_t BH, Pyr s, int D, const float* __restrict__ pyr, __half* __restrict__ mu_hi,
                                 __half* __restrict__ mu_lo, __half* __restrict__ dd_hi, __half* __restrict__ dd_lo,
                                 float2* __restrict__ meta) {
  pdl_wait();
  const int64_t n1 = s.size[0];
  const int64_t P2 = s.P - n1;
  const int64_t nrow = BH * P2 * 2;
  const int lane = threadIdx.x & 31;
  const int per = D / 32;  // elements per lane (2 or 4)
  for (int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) / 32; w < nrow;
       w += (int64_t)gridDim.x * blockDim.x / 32) {
    const int kind = (int)(w & 1);
    const int64_t r = w >> 1;
    const int64_t bh = r / P2, r2 = r % P2;
    int l = 2;
    while (l < s.L && r2 >= s.off[l] - n1) ++l;  // s.off[l] is the first row of level l + 1
    const int64_t j = r2 - (s.off[l - 1] - n1);
    const float* pb = pyr + bh * s.P * D;
    // lane L produces stored positions [per L, per L + per) of the row, so
    // each row is written with one coalesced store per array
    float v[4];
    float mx = 0.0f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      if (m >= per) break;
      const int c = inv_row_pos(per * lane + m, D);
      float x;
      if (kind == 0) {
        const float ref = pb[(s.P - 1) * D + c];
        x = pb[(s.off[l - 1] + j) * D + c] - (isfinite(ref) ? ref : 0.0f);
      } else {
        const int64_t c0 = 2 * j, c1 = 2 * j + 1;
        x = c1 < s.size[l - 2] ? pb[(s.off[l - 2] + c0) * D + c] - pb[(s.off[l - 2] + c1) * D + c] : 0.0f;
      }
      v[m] = x;
      mx = fmaxf(mx, fabsf(x));
    }
    mx = warp_max(mx);
    const int e = row_exponent(mx);
    const float sc = pow2f(e);
    float ss = 0.0f;
    __half* hi = (kind == 0 ? mu_hi : dd_hi) + r * D;
    __half* lo = (kind == 0 ? mu_lo : dd_lo) + r * D;
    uint32_t hw[2] = {0u, 0u}, lw2[2] = {0u, 0u};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      if (m >= per) break;
      const float xs = v[m] * sc;
      const __half h = __float2half_rn(xs);
      const __half lw = __float2half_rn(xs - __half2float(h));
      const float lf = __half2float(lw);
      ss = fmaf(lf, lf, ss);
      hw[m >> 1] |= (uint32_t)__half_as_ushort(h) << (16 * (m & 1));
      lw2[m >> 1] |= (uint32_t)__half_as_ushort(lw) << (16 * (m & 1));
    }
    if (per == 4) {
      reinterpret_cast<uint2*>(hi)[lane] = make_uint2(hw[0], hw[1]);
      reinterpret_cast<uint2*>(lo)[lane] = make_uint2(lw2[0], lw2[1]);
    } else {
      reinterpret_cast<uint32_t*>(hi)[lane] = hw[0];
      reinterpret_cast<uint32_t*>(lo)[lane] = lw2[0];
    }
    ss = warp_sum(ss);
    if (lane == 0) meta[r * 2 + kind] = make_float2(pow2f(-e), sqrtf(ss) * pow2f(-e));
  }
}

template <int NC>
struct HaarQ {
  float4 x[2][NC];  // own dots per head of the candidate lists (log2 units, root-relative)
  float4 y[NC];     // raw MMA dots of the current pass, by slot
  int32_t cand[2][NC];
};

template <int NC>
struct HaarQPad : HaarQ<NC> {
  // the two queries of a warp start 16 banks apart
  static constexpr int kWords = (int)(sizeof(HaarQ<NC>) / 4);
  static constexpr int kPad = (16 - kWords % 32 + 64) % 32;
  int32_t pad[kPad > 0 ? kPad : 4];
};

struct HaarView {
  const uint16_t* mu_hi;
  const uint16_t* mu_lo;
  const uint16_t* dd_hi;
  const uint16_t* dd_lo;
  const float4* meta;
  int64_t P2;
};

// Dots of fp16 rows of the candidates of both queries of the warp: query
// u's candidates are slots [0, nw[u]), slot i held by lane 16 u + i % 16 as
// its cv[i / 16].  The raw MMA results (row
// and query scales not yet applied) go to sm[u].y[slot]; with kAdd they are
// added to it instead, and only the groups of eight slots whose bit is set in
// gmask (one bit per group, both queries) are done: the residual pass.
// For a group of eight slots, lane (r, t) loads its A fragments from slot r's
// row (one 16-byte chunk per k-step) and, after the k-steps, holds
// D[r][2t] + D[r + 8][2t + 1]: the dot of slot r's row with head t.
template <int D, int NC, bool kAdd>
__device__ __forceinline__ void haar_pass(HaarQPad<NC>* smw, const int (&cv)[NC / 16], const uint16_t* __restrict__ rows,
                                          const int64_t (&pbase)[2], int64_t rowoff, const int (&nw)[2],
                                          uint32_t gmask, const uint32_t (&bq)[2][D / 32][2], int lane) {
  constexpr int NK = D / 32;
  const int grp = lane >> 2, tig = lane & 3;
  const int nmax = max(nw[0], nw[1]);
  const int64_t loff = rowoff * D + 16 * tig;
#pragma unroll
  for (int r0 = 0; r0 < NC; r0 += 8) {
    if (r0 >= nmax) break;
    if (kAdd && !((gmask >> (r0 / 8)) & 1u)) continue;  // warp-uniform
    const int w = r0 + grp;
    uint4 a[2][NK];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      // slot w of query u is lane 16 u + w % 16's candidate w / 16 (uniform per group)
      const int node = __shfl_sync(0xffffffffu, cv[r0 >> 4], 16 * u + (w & 15));
      const uint32_t ro = (uint32_t)(w < nw[u] ? node : 0) * (uint32_t)D;
      const uint16_t* rp = rows + pbase[u] + loff + ro;
#pragma unroll
      for (int m = 0; m < NK / 2; ++m) ldg_frag2(rp + 64 * m, a[u][2 * m], a[u][2 * m + 1]);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int kk = 0; kk < NK; ++kk) mma_f16_16816(d, a[u][kk], bq[u][kk][0], bq[u][kk][1]);
      if (w < nw[u]) {
        float* dst = reinterpret_cast<float*>(&smw[u].y[w]) + tig;
        const float v = d[0] + d[3];
        *dst = kAdd ? *dst + v : v;
      }
    }
  }
}

// Groups of eight slots (bit i: slots [8i, 8i + 8) of either query) in which
// some candidate's residual bound bnd exceeds kLoTau.
template <int CPL>
__device__ __forceinline__ uint32_t lo_groups(const float (&bnd)[CPL], int ncur, int ll) {
  uint32_t gm = 0;
#pragma unroll
  for (int sl = 0; sl < CPL; ++sl) {
    const unsigned b = __ballot_sync(0xffffffffu, sl * 16 + ll < ncur && bnd[sl] > kLoTau);
    const unsigned m = (b | (b >> 16)) & 0xffffu;  // slots of either query
    gm |= ((m & 0xffu) ? 1u : 0u) << (2 * sl);
    gm |= ((m >> 8) ? 1u : 0u) << (2 * sl + 1);
  }
  return gm;
}

// Occupancy: K <= 8 runs three 8-warp CTAs per SM (a register budget of 80;
// the walk is latency- and issue-bound, and 24 resident warps beat 16 warps
// with more registers); larger K keep 16 warps per SM.
template <int D, int KM, int WARPS, bool kLse>
__global__ void __launch_bounds__(WARPS * 32, (KM <= 8 ? 24 : 16) / WARPS)
    route_haar_kernel(Prob pr, Pyr s, const uint16_t* __restrict__ q, HaarView hv, const float* __restrict__ path,
                      int32_t* __restrict__ kept2, int32_t* __restrict__ trace) {
  pdl_wait();
  constexpr int G = 4;
  constexpr int NC = 2 * KM;
  constexpr int CPL = NC / 16;
  constexpr int NK = D / 32;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  HaarQPad<NC>& sm = reinterpret_cast<HaarQPad<NC>*>(smem_raw)[threadIdx.x / 16];
  HaarQPad<NC>* smw = reinterpret_cast<HaarQPad<NC>*>(smem_raw) + (threadIdx.x / 32) * 2;
  const int lane = threadIdx.x & 31, ll = lane & 15, half = lane >> 4;
  const int grp = lane >> 2, tig = lane & 3;
  // query counts are below 2^31 (the prefill size limit), so 32-bit index math
  const uint32_t nq = (uint32_t)(pr.B * pr.Hkv * pr.N), N32 = (uint32_t)pr.N;
  const uint32_t qi = (blockIdx.x * WARPS + threadIdx.x / 32) * 2 + half;
  const bool live = qi < nq;
  const uint32_t qc = live ? qi : nq - 1;
  const int64_t t = qc % N32;
  const int K = pr.K;
  const int64_t qb = t / s.C;
  int32_t* kout = kept2 + (int64_t)qc * K;
  int32_t* trow = (trace && live) ? trace + (int64_t)qc * s.L * K : nullptr;
  if (trow)
    for (int i = ll; i < s.L * K; i += 16) trow[i] = -1;

  int l0 = 0;
  if (live && qb - 2 >= 1) {
    // start level: the highest level with more than K eligible nodes, i.e.
    // the largest l <= L with (qb - 2) >> (l - 1) >= K
    const uint32_t xk = (uint32_t)(qb - 2) / (uint32_t)K;
    if (xk >= 2) l0 = min((int)s.L, 32 - __clz(xk));
    if (l0 < 2) l0 = 0;
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
  const int l0o = __shfl_xor_sync(0xffffffffu, l0, 16);
  const int l0w = max(l0, l0o);
  if (l0w == 0) return;  // warp-uniform

  // B fragments of both queries: lane (r, t) holds column r = 2 h + s (half s
  // of head h) at k = 2t, 2t+1 and 2t+8, 2t+9 of every k-step, converted to
  // fp16 with one power-of-two scale per query (exact for bf16 inputs in
  // range); per-query head norms for the residual bound.
  const uint32_t qw = (blockIdx.x * WARPS + threadIdx.x / 32) * 2;
  uint32_t bq[2][NK][2];
  int64_t pbase[2], mbase[2];
  float qfac[2], bfac[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const uint32_t qu = min(qw + u, nq - 1);
    const uint32_t tu = qu % N32, bhu = qu / N32;
    const uint32_t Hkv = (uint32_t)pr.Hkv;
    const int64_t head = (int64_t)((bhu / Hkv) * (uint32_t)pr.Hq + (bhu % Hkv) * G + (grp >> 1));
    const uint16_t* qp = q + (head * pr.N + tu) * D + (grp & 1) * (D / 2) + 2 * tig;
    float f[NK][4];
    float mx = 0.0f, ss = 0.0f;
#pragma unroll
    for (int kk = 0; kk < NK; ++kk) {
      const uint32_t w0 = __ldg(reinterpret_cast<const uint32_t*>(qp + 16 * kk));
      const uint32_t w1 = __ldg(reinterpret_cast<const uint32_t*>(qp + 16 * kk + 8));
      f[kk][0] = __uint_as_float(w0 << 16);
      f[kk][1] = __uint_as_float(w0 & 0xffff0000u);
      f[kk][2] = __uint_as_float(w1 << 16);
      f[kk][3] = __uint_as_float(w1 & 0xffff0000u);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        mx = fmaxf(mx, fabsf(f[kk][e]));
        ss = fmaf(f[kk][e], f[kk][e], ss);
      }
    }
    mx = warp_max(mx);
    const int e = row_exponent(mx);
    const float sc = pow2f(e);
#pragma unroll
    for (int kk = 0; kk < NK; ++kk) {
      bq[u][kk][0] = pack_f16x2(f[kk][0] * sc, f[kk][1] * sc);
      bq[u][kk][1] = pack_f16x2(f[kk][2] * sc, f[kk][3] * sc);
    }
    qfac[u] = pow2f(-e) * pr.scale2;
    // |q_h|^2 over the lanes of head h (quad threads and both halves), then
    // the sum of the four heads' norms
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    ss += __shfl_xor_sync(0xffffffffu, ss, 4);
    float hn = sqrtf(ss);
    hn += __shfl_xor_sync(0xffffffffu, hn, 8);
    hn += __shfl_xor_sync(0xffffffffu, hn, 16);
    bfac[u] = hn * pr.scale2;  // bound per unit of residual norm: sum over heads of s |q_h| (log2 units)
    pbase[u] = (int64_t)bhu * hv.P2 * D;
    mbase[u] = (int64_t)bhu * hv.P2;
  }
  const float myq = half ? qfac[1] : qfac[0], mybf = half ? bfac[1] : bfac[0];
  const int64_t mymb = half ? mbase[1] : mbase[0];

  int cur = 0;
  int nc = l0 > 0 ? (int)eligible_count(l0, qb) : 0;
  for (int i = ll; i < nc; i += 16) sm.cand[0][i] = i;
  const int e_hi = (int)(qb - 2);
  const int64_t n1 = s.size[0];
  __syncwarp();

  for (int level = l0w; level >= 2; --level) {
    const bool act = level <= l0;
    const int ncur = act ? nc : 0;
    const bool start = act && level == l0;
    const int ncap = (int)s.size[level - 2];
    const int64_t rowoff = s.off[level - 1] - n1;

    int cv[CPL];
    float4 mt[CPL];
    float4 xv[CPL];
#pragma unroll
    for (int sl = 0; sl < CPL; ++sl) {
      const int i = sl * 16 + ll;
      const bool valid = i < ncur;
      cv[sl] = valid ? sm.cand[cur][i] : 0;
      mt[sl] = valid ? __ldg(hv.meta + mymb + rowoff + cv[sl]) : make_float4(0.f, 0.f, 0.f, 0.f);
      xv[sl] = (valid && !start) ? sm.x[cur][i] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int nwu[2] = {__shfl_sync(0xffffffffu, ncur, 0), __shfl_sync(0xffffffffu, ncur, 16)};

    // start level: the candidates' own dots from their MU rows (hi pass,
    // then the residual pass for the groups whose rounding bound is too wide)
    const unsigned st_b = __ballot_sync(0xffffffffu, start);
    if (st_b) {
      const int ns[2] = {(st_b & 1u) ? nwu[0] : 0, (st_b >> 16) ? nwu[1] : 0};
      haar_pass<D, NC, false>(smw, cv, hv.mu_hi, pbase, rowoff, ns, 0u, bq, lane);
      float bnd[CPL];
#pragma unroll
      for (int sl = 0; sl < CPL; ++sl) bnd[sl] = start ? mybf * mt[sl].y : 0.0f;
      const uint32_t gm = lo_groups<CPL>(bnd, ncur, ll);
      __syncwarp();
      if (gm) haar_pass<D, NC, true>(smw, cv, hv.mu_lo, pbase, rowoff, ns, gm, bq, lane);
      __syncwarp();
#pragma unroll
      for (int sl = 0; sl < CPL; ++sl) {
        const int i = sl * 16 + ll;
        if (start && i < ncur) {
          const float4 r = sm.y[i];
          const float f = mt[sl].x * myq;
          xv[sl] = make_float4(r.x * f, r.y * f, r.z * f, r.w * f);
        }
      }
      __syncwarp();
    }

    // every level: the candidates' DD rows give both children's dots
    haar_pass<D, NC, false>(smw, cv, hv.dd_hi, pbase, rowoff, nwu, 0u, bq, lane);
    {
      float bnd[CPL];
#pragma unroll
      for (int sl = 0; sl < CPL; ++sl) bnd[sl] = mybf * mt[sl].w;
      const uint32_t gm = lo_groups<CPL>(bnd, ncur, ll);
      __syncwarp();
      if (gm) haar_pass<D, NC, true>(smw, cv, hv.dd_lo, pbase, rowoff, nwu, gm, bq, lane);
    }
    __syncwarp();

    // scores and rank keys (higher score first, then lower index)
    uint32_t key[CPL];
    float4 ya[CPL], yb[CPL];
    int e0v[CPL], e1v[CPL];
#pragma unroll
    for (int sl = 0; sl < CPL; ++sl) {
      const int i = sl * 16 + ll;
      key[sl] = 0;
      e0v[sl] = e1v[sl] = 0;
      ya[sl] = yb[sl] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < ncur) {
        const int c0 = 2 * cv[sl];
        const bool has1 = c0 + 1 < ncap;
        e0v[sl] = elig_node_h(level - 1, c0, e_hi);
        e1v[sl] = has1 && elig_node_h(level - 1, c0 + 1, e_hi);
        // child weights: only the last node of a level can hold fewer keys
        float w0 = 0.5f, w1 = 0.5f;
        if (c0 + 2 >= ncap) {
          const float n0 = (float)count_node_h(s.C, level - 1, c0, s.N);
          const float nn1 = has1 ? (float)count_node_h(s.C, level - 1, c0 + 1, s.N) : 0.0f;
          w0 = nn1 / (n0 + nn1);
          w1 = n0 / (n0 + nn1);
        }
        const float4 r = sm.y[i];
        const float f = mt[sl].z * myq;
        const float4 x = xv[sl];
        const float yv[4] = {r.x * f, r.y * f, r.z * f, r.w * f};
        ya[sl] = make_float4(fmaf(w0, yv[0], x.x), fmaf(w0, yv[1], x.y), fmaf(w0, yv[2], x.z), fmaf(w0, yv[3], x.w));
        yb[sl] = make_float4(fmaf(-w1, yv[0], x.x), fmaf(-w1, yv[1], x.y), fmaf(-w1, yv[2], x.z),
                             fmaf(-w1, yv[3], x.w));
        if (path && cv[sl] == (int)(qb >> (level - 1))) {
          // the query's path node: its children read the prefix-consistent
          // summaries (the path child's prefix dot; a complete left sibling)
          const float4* pp = reinterpret_cast<const float4*>(path + (int64_t)qc * s.L * 2 * G);
          const float4 pc = __ldg(pp + (level - 2) * 2);
          if ((qb >> (level - 2)) & 1) {
            ya[sl] = __ldg(pp + (level - 1) * 2 + 1);
            yb[sl] = pc;
          } else {
            ya[sl] = pc;
            yb[sl] = pc;
          }
        }
        const bool both = e0v[sl] && e1v[sl];
        float scv = 0.0f;
        if constexpr (kLse) {
          // sum over heads of log2(2^a + 2^b) = sum of maxima + log2 of the
          // product of (1 + 2^(min - max)), each factor in (1, 2]
          if (both) {
            float pr4 = 1.0f;
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const float a = comp4(ya[sl], g), bb = comp4(yb[sl], g);
              const float mx = fmaxf(a, bb);
              scv += mx;
              pr4 *= 1.0f + ex2_fast(fminf(a, bb) - mx);
            }
            scv += lg2_fast(pr4);
          } else {
#pragma unroll
            for (int g = 0; g < G; ++g) scv += e0v[sl] ? comp4(ya[sl], g) : comp4(yb[sl], g);
          }
        } else {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float a = comp4(ya[sl], g), bb = comp4(yb[sl], g);
            scv += both ? pair_score(pr.scorer, a, bb) : (e0v[sl] ? a : bb);
          }
        }
        if (scv == 0.0f) scv = 0.0f;     // -0 ranks like +0
        if (scv != scv) scv = -INFINITY;  // NaN ranks last
        // rank key: the orderable score with its low 6 bits replaced by the
        // reversed slot, so keys are distinct and, among scores equal to 2^-17
        // relative (ties far inside the 1e-3 tie margin), the lower slot --
        // the lower node index -- ranks first
        key[sl] = (orderable_key_h(scv) & ~63u) | (uint32_t)(63 - i);
      }
    }
    int rank[CPL];
#pragma unroll
    for (int sl = 0; sl < CPL; ++sl) rank[sl] = 0;
#pragma unroll
    for (int sj = 0; sj < CPL; ++sj) {
#pragma unroll
      for (int l = 0; l < 16; ++l) {
        const uint32_t kj = __shfl_sync(0xffffffffu, key[sj], l, 16);
#pragma unroll
        for (int sl = 0; sl < CPL; ++sl) rank[sl] += kj > key[sl] ? 1 : 0;
      }
    }

    // kept set (index order), next candidates (ascending) or the kept level-2 nodes
    const int nxt = cur ^ 1;
    int nkept = 0, nchild = 0;
#pragma unroll
    for (int sl = 0; sl < CPL; ++sl) {
      const int i = sl * 16 + ll;
      const int keep = (i < ncur && rank[sl] < K) ? 1 : 0;
      const int nch = keep && level > 2 ? e0v[sl] + e1v[sl] : 0;
      int ktot, ctot;
      const int kp = nkept + prefix16h(keep, lane, &ktot);
      int cp = nchild + prefix16h(nch, lane, &ctot);
      if (keep) {
        const int32_t ci = cv[sl];
        if (trow) trow[(level - 1) * K + kp] = ci;
        if (level == 2) kout[kp] = ci;
        if (e0v[sl] && nch) {
          sm.cand[nxt][cp] = 2 * ci;
          sm.x[nxt][cp] = ya[sl];
          ++cp;
        }
        if (e1v[sl] && nch) {
          sm.cand[nxt][cp] = 2 * ci + 1;
          sm.x[nxt][cp] = yb[sl];
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

template <int D, int KM, int WARPS, bool kLse>
static cudaError_t launch_route_haar_t(const Prob& pr, const Pyr& s, const void* q, const HaarView& hv,
                                       const float* path, int32_t* kept2, int32_t* trace, bool after_prep,
                                       cudaStream_t st) {
  const size_t smem = sizeof(HaarQPad<2 * KM>) * 2 * WARPS;
  auto kern = route_haar_kernel<D, KM, WARPS, kLse>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t nq = pr.B * pr.Hkv * pr.N;
  note_launch();
  return launch_pdl(after_prep, kern, dim3((unsigned)ceil_div64(nq, 2 * WARPS)), dim3(WARPS * 32), smem, st, pr, s,
                    (const uint16_t*)q, hv, path, kept2, trace);
}

bool route_haar_supported(const Prob& pr) {
  return pr.dtype == PISA_BF16 && pr.G == 4 && (pr.d == 64 || pr.d == 128);
}

size_t haar_rows_bytes(const Prob& pr, const Pyr& s) {
  const int64_t P2 = s.L >= 2 ? s.P - s.size[0] : 0;
  return (size_t)pr.B * pr.Hkv * P2 * pr.d * 2;  // one fp16 array (of four)
}

size_t haar_meta_bytes(const Prob& pr, const Pyr& s) {
  const int64_t P2 = s.L >= 2 ? s.P - s.size[0] : 0;
  return (size_t)pr.B * pr.Hkv * P2 * 16;
}

cudaError_t launch_route_haar(const Prob& pr, const Pyr& s, const void* q, const float* pyr, char* rows,
                              float4* meta, const float* path, int32_t* kept2, int32_t* trace, cudaStream_t st) {
  const int64_t BH = pr.B * pr.Hkv;
  const int64_t P2 = s.L >= 2 ? s.P - s.size[0] : 0;
  const size_t arr = haar_rows_bytes(pr, s);
  HaarView hv{(const uint16_t*)rows, (const uint16_t*)(rows + arr), (const uint16_t*)(rows + 2 * arr),
              (const uint16_t*)(rows + 3 * arr), meta, P2};
  if (P2 > 0) {
    const int64_t warps = BH * P2 * 2;
    note_launch();
    cudaError_t e = launch_pdl(false, haar_prep_kernel, dim3((unsigned)std::min<int64_t>(ceil_div64(warps, 8), 16384)),
                               dim3(256), 0, st, BH, s, pr.d, pyr, (__half*)rows, (__half*)(rows + arr),
                               (__half*)(rows + 2 * arr), (__half*)(rows + 3 * arr), reinterpret_cast<float2*>(meta));
    if (e != cudaSuccess) return e;
  }
#define PISA_RH_CASE(DD, LSE)                                                                            \
  if (pr.d == DD && (pr.scorer == PISA_SCORER_LSE) == LSE) {                                             \
    if (pr.K <= 8) return launch_route_haar_t<DD, 8, 8, LSE>(pr, s, q, hv, path, kept2, trace, P2 > 0, st);            \
    if (pr.K <= 16) return launch_route_haar_t<DD, 16, 8, LSE>(pr, s, q, hv, path, kept2, trace, P2 > 0, st);          \
    return launch_route_haar_t<DD, 32, 4, LSE>(pr, s, q, hv, path, kept2, trace, P2 > 0, st);                          \
  }
  PISA_RH_CASE(128, true) PISA_RH_CASE(64, true) PISA_RH_CASE(128, false) PISA_RH_CASE(64, false)
#undef PISA_RH_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pisa
