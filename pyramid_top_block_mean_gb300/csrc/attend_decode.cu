// attend_decode.cu -- attention of one decode query over its selected blocks.
// agihunt.info summary of "Block Sparse Attention with Log-Linear
// Complexity", opening paragraph (each query reads only its selected tiles of
// C keys) and pyramid paragraph (decode routing per step); rcap.io post,
// "Selection walks the tree top-down" (the kept leaves drive sparse attention
// over the original keys and values).
//
// One CTA (4 warps) per (sequence, key head); the query sits at position
// t = seq_lens[b] - 1 and its G query heads share the blocks of idx[b, h, :].
// The warps take the distinct valid blocks round-robin and stream each block
// in chunks of 16 keys (one bulk copy for the keys, one for the values, three
// stages per warp).  Per chunk, warp-level m16n8k16 bf16 MMAs give
// S = K q (16 keys x 8 columns: the G heads, zero-padded), an online softmax
// per head rescales the running output, and O^T += V^T P (8 or 4 tiles of 16
// dims; V^T fragments by ldmatrix.trans from the key-major chunk, P moved
// from accumulator to operand layout through 256 bytes of shared memory).
// The four warps' (max, sum, output) are merged in shared memory at the end,
// so nothing but the output row reaches HBM.  Bound by HBM: (K+3) x 64 keys
// x d x 2 (keys and values) bf16 per (sequence, key head).
#include "pisa_common.cuh"
#include "pisa_internal.h"
#include "tc_ptx.cuh"

namespace pisa {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kKeysPerChunk = 16;
constexpr int kStages = 3;
constexpr int kMaxSlots = 64;
constexpr uint64_t kWaitNs = 4000000000ull;

template <int D>
struct AdSmem {
  union {
    uint16_t kv[kWarps][kStages][2][kKeysPerChunk * D];  // [warp][stage][keys, values]
    float o[kWarps][8][D];                               // after the stream: each warp's output
  } u;
  uint16_t p[kWarps][kKeysPerChunk][8];  // P tile: [key][head]
  float m[kWarps][8], l[kWarps][8];
  int64_t chunk_key[kWarps][(kMaxSlots / kWarps) * 4];  // first key of each chunk a warp streams
  int32_t blocks[kMaxSlots];
  int32_t nblocks;
  uint64_t bar[kWarps][kStages];
  int32_t abort;
  int32_t zero;
};

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads) attend_decode_kernel(Prob pr, Pyr s, const uint16_t* __restrict__ q,
                                                                  const uint16_t* __restrict__ kc,
                                                                  const uint16_t* __restrict__ vc,
                                                                  const int32_t* __restrict__ seq_lens,
                                                                  const int32_t* __restrict__ idx,
                                                                  uint16_t* __restrict__ out,
                                                                  int32_t* __restrict__ status) {
  constexpr int KT = D / 32;  // 32-dim steps of the S MMAs (two k16 MMAs each)
  constexpr int MT = D / 16;  // 16-dim tiles of the output
  constexpr uint32_t kChunkBytes = kKeysPerChunk * D * 2;
  extern __shared__ unsigned char smem_raw[];
  AdSmem<D>& sm = *reinterpret_cast<AdSmem<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~(uintptr_t)127);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grp = lane >> 2, tig = lane & 3;
  const int64_t bh = blockIdx.x, b = bh / pr.Hkv, h = bh % pr.Hkv;
  const int W = pr.K + 3;
  uint16_t* orow = out + (b * pr.Hq + h * G) * D;  // G rows of D
  const int64_t len = seq_lens[b];
  if (len < 1 || len > s.N) {
    if (tid == 0) set_status(status, PISA_DEV_BAD_SEQ_LEN);
    for (int i = tid; i < G * D; i += kThreads) orow[i] = 0;
    return;
  }
  const int64_t t = len - 1, qb = t / s.C;
  volatile int32_t* abort = &sm.abort;
  if (warp == 0) {
    // the distinct blocks of the row that hold a key at or before t, in slot
    // order: lane i takes slots i and i + 32; a slot repeating an earlier
    // one is dropped
    const int32_t* row = idx + bh * W;
    const int32_t r0 = lane < W ? row[lane] : -1, r1 = lane + 32 < W ? row[lane + 32] : -1;
    const bool ok0 = r0 >= 0 && r0 <= qb, ok1 = r1 >= 0 && r1 <= qb;
    const unsigned below = (1u << lane) - 1u;
    const unsigned m0 = __match_any_sync(0xffffffffu, ok0 ? r0 : -1 - lane);  // invalid slots match nothing
    const unsigned m1 = __match_any_sync(0xffffffffu, ok1 ? r1 : -1 - lane);
    bool dup1 = (m1 & below) != 0u;
    for (int u = 0; u < 32; ++u) {
      const int32_t o = __shfl_sync(0xffffffffu, ok0 ? r0 : -1, u);  // every lane takes part
      dup1 |= ok1 && o == r1;
    }
    const bool keep0 = ok0 && (m0 & below) == 0u, keep1 = ok1 && !dup1;
    const unsigned b0 = __ballot_sync(0xffffffffu, keep0), b1 = __ballot_sync(0xffffffffu, keep1);
    if (keep0) sm.blocks[__popc(b0 & below)] = r0;
    if (keep1) sm.blocks[__popc(b0) + __popc(b1 & below)] = r1;
    if (lane == 0) {
      sm.nblocks = __popc(b0) + __popc(b1);
      for (int w = 0; w < kWarps; ++w)
        for (int u = 0; u < kStages; ++u) ptx::mbar_init(ptx::smem_u32(&sm.bar[w][u]), 1);
      sm.abort = 0;
      sm.zero = 0;
      ptx::fence_mbar_init();
      ptx::fence_proxy_async_smem();
    }
  }
  __syncthreads();
  // the blocks are dealt round-robin to the warps; lane k of a warp lists the
  // 16-key chunks of the warp's k-th block, up to the chunk that holds t (the
  // capacity is a multiple of 16, so no chunk runs past it)
  int nch;
  {
    const int i = warp + kWarps * lane;
    int cnt = 0;
    int64_t k0 = 0;
    if (i < sm.nblocks) {
      k0 = (int64_t)sm.blocks[i] * s.C;
      const int64_t kend = k0 + s.C - 1 < t ? k0 + s.C - 1 : t;  // last key read
      cnt = (int)((kend - k0) / kKeysPerChunk) + 1;
    }
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    for (int c = 0; c < cnt; ++c) sm.chunk_key[warp][x - cnt + c] = k0 + (int64_t)kKeysPerChunk * c;
    nch = __shfl_sync(0xffffffffu, x, 31);
    __syncwarp();
  }

  // q fragments (the B operand of S = K q): head grp (zero past G), dims
  // 32 kk + 8 tig + {0..7}
  uint32_t bq[KT][4];
#pragma unroll
  for (int kk = 0; kk < KT; ++kk) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (grp < G) v = *reinterpret_cast<const uint4*>(q + (b * pr.Hq + h * G + grp) * D + 32 * kk + 8 * tig);
    bq[kk][0] = v.x; bq[kk][1] = v.y; bq[kk][2] = v.z; bq[kk][3] = v.w;
  }
  auto issue = [&](int c) {
    if (lane == 0) {
      const int64_t row0 = (bh * s.N + sm.chunk_key[warp][c]) * D;
      const uint32_t bar = ptx::smem_u32(&sm.bar[warp][c % kStages]);
      ptx::mbar_arrive_expect_tx(bar, 2 * kChunkBytes);
      ptx::bulk_g2s(ptx::smem_u32(sm.u.kv[warp][c % kStages][0]), kc + row0, kChunkBytes, bar);
      ptx::bulk_g2s(ptx::smem_u32(sm.u.kv[warp][c % kStages][1]), vc + row0, kChunkBytes, bar);
    }
  };
  float oacc[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.0f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;  // heads 2 tig, 2 tig + 1
  const float sc = pr.scale2;
  uint32_t phase = 0u;
  int issued = 0, waited = 0;
  for (; issued < nch && issued < kStages - 1; ++issued) issue(issued);
  for (int c = 0; c < nch; ++c) {
    if (c + kStages - 1 < nch) {
      __syncwarp();  // every lane is done with the buffers this copy overwrites
      issue(c + kStages - 1);
      issued = c + kStages;
    }
    const int st = c % kStages;
    const bool ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sm.bar[warp][st]), (phase >> st) & 1u, abort, kWaitNs);
    phase ^= 1u << st;
    waited = c + 1;
    if (!__all_sync(0xffffffffu, ok)) { *abort = 1; break; }
    const unsigned char* kbuf = reinterpret_cast<const unsigned char*>(sm.u.kv[warp][st][0]);
    const int64_t key0 = sm.chunk_key[warp][c];
    // S = K q: keys grp and grp + 8 of the chunk, heads 2 tig and 2 tig + 1
    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f}, e[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // two independent chains
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      const uint4 a0 = *reinterpret_cast<const uint4*>(kbuf + grp * D * 2 + 64 * kk + 16 * tig);
      const uint4 a1 = *reinterpret_cast<const uint4*>(kbuf + (grp + 8) * D * 2 + 64 * kk + 16 * tig);
      mma16816(d, a0.x, a1.x, a0.y, a1.y, bq[kk][0], bq[kk][1]);
      mma16816(e, a0.z, a1.z, a0.w, a1.w, bq[kk][2], bq[kk][3]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) d[j] += e[j];
    // causal mask inside the query's own block, then the online softmax
    const bool v0 = key0 + grp <= t, v1 = key0 + grp + 8 <= t;
    const float x00 = v0 ? d[0] * sc : -INFINITY, x01 = v0 ? d[1] * sc : -INFINITY;
    const float x10 = v1 ? d[2] * sc : -INFINITY, x11 = v1 ? d[3] * sc : -INFINITY;
    float c0 = fmaxf(x00, x10), c1 = fmaxf(x01, x11);
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
      c0 = fmaxf(c0, __shfl_xor_sync(0xffffffffu, c0, o));
      c1 = fmaxf(c1, __shfl_xor_sync(0xffffffffu, c1, o));
    }
    const float n0 = fmaxf(m0, c0), n1 = fmaxf(m1, c1);  // finite: key t or an earlier key is valid
    const float a0s = m0 == -INFINITY ? 0.0f : ptx::ex2(m0 - n0), a1s = m1 == -INFINITY ? 0.0f : ptx::ex2(m1 - n1);
    m0 = n0;
    m1 = n1;
    const float p00 = n0 == -INFINITY ? 0.0f : ptx::ex2(x00 - n0), p10 = n0 == -INFINITY ? 0.0f : ptx::ex2(x10 - n0);
    const float p01 = n1 == -INFINITY ? 0.0f : ptx::ex2(x01 - n1), p11 = n1 == -INFINITY ? 0.0f : ptx::ex2(x11 - n1);
    l0 = l0 * a0s + p00 + p10;
    l1 = l1 * a1s + p01 + p11;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      oacc[mt][0] *= a0s; oacc[mt][2] *= a0s;  // head 2 tig
      oacc[mt][1] *= a1s; oacc[mt][3] *= a1s;  // head 2 tig + 1
    }
    // P from accumulator layout (key, head pair) to operand layout (key pair, head)
    __syncwarp();
    {
      uint32_t* prow = reinterpret_cast<uint32_t*>(&sm.p[warp][0][0]);
      prow[grp * 4 + tig] = pack2(p00, p01);        // key grp, heads 2 tig, 2 tig + 1
      prow[(grp + 8) * 4 + tig] = pack2(p10, p11);  // key grp + 8
    }
    __syncwarp();
    const uint16_t* pt = &sm.p[warp][0][0];
    const uint32_t pb0 = (uint32_t)pt[(2 * tig) * 8 + grp] | ((uint32_t)pt[(2 * tig + 1) * 8 + grp] << 16);
    const uint32_t pb1 = (uint32_t)pt[(2 * tig + 8) * 8 + grp] | ((uint32_t)pt[(2 * tig + 9) * 8 + grp] << 16);
    // O^T += V^T P: V^T tiles (16 dims x 16 keys) by ldmatrix.trans from the key-major chunk
    const uint32_t vbase = ptx::smem_u32(sm.u.kv[warp][st][1]);
    const int mrow = lane & 7, msel = lane >> 3;  // matrix msel: keys 8 (msel >> 1) + mrow, dims + 8 (msel & 1)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      uint32_t r0, r1, r2, r3;
      ldmatrix_x4_trans(vbase + ((8 * (msel >> 1) + mrow) * D + 16 * mt + 8 * (msel & 1)) * 2, r0, r1, r2, r3);
      mma16816(oacc[mt], r0, r1, r2, r3, pb0, pb1);
    }
  }
  // after an early exit, let copies already issued land before the CTA ends
  for (int c = waited; c < issued; ++c) {
    const int st = c % kStages;
    ptx::mbar_wait_bounded(ptx::smem_u32(&sm.bar[warp][st]), (phase >> st) & 1u, &sm.zero, kWaitNs);
    phase ^= 1u << st;
  }
  // per warp: (max, sum, output) of heads 2 tig, 2 tig + 1
#pragma unroll
  for (int o = 4; o <= 16; o <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o);
  }
  if (grp == 0) {
    sm.m[warp][2 * tig] = m0; sm.m[warp][2 * tig + 1] = m1;
    sm.l[warp][2 * tig] = l0; sm.l[warp][2 * tig + 1] = l1;
  }
  __syncthreads();  // every warp is done with the staging buffers the outputs overlay
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    sm.u.o[warp][2 * tig][16 * mt + grp] = oacc[mt][0];
    sm.u.o[warp][2 * tig + 1][16 * mt + grp] = oacc[mt][1];
    sm.u.o[warp][2 * tig][16 * mt + grp + 8] = oacc[mt][2];
    sm.u.o[warp][2 * tig + 1][16 * mt + grp + 8] = oacc[mt][3];
  }
  __syncthreads();
  // merge the warps: head g, two dims per thread
  for (int e = tid; e < G * (D / 2); e += kThreads) {
    const int g = e / (D / 2), c2 = 2 * (e % (D / 2));
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, sm.m[w][g]);
    float L = 0.0f, o0 = 0.0f, o1 = 0.0f;
    if (mx > -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        if (sm.m[w][g] == -INFINITY) continue;
        const float f = ptx::ex2(sm.m[w][g] - mx);
        L = fmaf(sm.l[w][g], f, L);
        o0 = fmaf(sm.u.o[w][g][c2], f, o0);
        o1 = fmaf(sm.u.o[w][g][c2 + 1], f, o1);
      }
    }
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    *reinterpret_cast<uint32_t*>(orow + g * D + c2) = pack2(o0 * inv, o1 * inv);
  }
  if (tid == 0 && sm.abort) set_status(status, PISA_DEV_TIMEOUT);
}

template <int D, int G>
cudaError_t launch_t(const Prob& pr, const Pyr& s, const void* q, const void* k, const void* v,
                     const int32_t* seq_lens, const int32_t* idx, void* out, int32_t* status, cudaStream_t st) {
  const size_t smem = sizeof(AdSmem<D>) + 128;
  auto kern = attend_decode_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  note_launch();
  kern<<<(unsigned)(pr.B * pr.Hkv), kThreads, smem, st>>>(pr, s, (const uint16_t*)q, (const uint16_t*)k,
                                                          (const uint16_t*)v, seq_lens, idx, (uint16_t*)out, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attend_decode(const Prob& pr, const Pyr& s, const void* q, const void* k, const void* v,
                                 const int32_t* seq_lens, const int32_t* idx, void* out, int32_t* status,
                                 cudaStream_t st) {
  if (pr.K + 3 > kMaxSlots) return cudaErrorInvalidValue;
#define PISA_AD_CASE(DD, GG) \
  if (pr.d == DD && pr.G == GG) return launch_t<DD, GG>(pr, s, q, k, v, seq_lens, idx, out, status, st);
  PISA_AD_CASE(128, 1) PISA_AD_CASE(128, 2) PISA_AD_CASE(128, 4) PISA_AD_CASE(128, 8)
  PISA_AD_CASE(64, 1) PISA_AD_CASE(64, 2) PISA_AD_CASE(64, 4) PISA_AD_CASE(64, 8)
#undef PISA_AD_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pisa
