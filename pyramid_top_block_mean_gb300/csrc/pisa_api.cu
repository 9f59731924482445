// pisa_api.cu -- the C ABI of include/pisa.h: argument checks, workspace
// layout and kernel launches.  Every check runs on the host before the first
// launch; a failing call launches nothing.
#include <atomic>
#include <math.h>
#include <mutex>

#include "pisa_common.cuh"
#include "pisa_internal.h"

namespace pisa {

constexpr int64_t kMaxN = (int64_t)1 << 26;  // keeps t*K + slot inside int32

bool make_pyr(int64_t N, int32_t C, Pyr* s) {
  if (N < 0 || C <= 0) return false;
  s->C = C;
  s->N = N;
  s->nb = ceil_div64(N, C);
  s->L = 0;
  s->P = 0;
  if (s->nb == 0) return true;
  int64_t n = s->nb;
  for (;;) {
    if (s->L >= kMaxLevels) return false;
    s->size[s->L] = n;
    s->off[s->L] = s->P;
    s->P += n;
    s->L++;
    if (n == 1) break;
    n = ceil_div64(n, 2);
  }
  for (int l = s->L; l < kMaxLevels; ++l) { s->size[l] = 0; s->off[l] = s->P; }
  return true;
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

PrefillWs prefill_ws_layout(const Prob& pr, const Pyr& s) {
  PrefillWs w{};
  const int64_t nq = pr.B * pr.Hkv * pr.N;
  const int64_t n2 = s.L >= 2 ? s.size[1] : 0;
  w.n2 = n2;
  w.nchunk = ceil_div64(pr.N, (int64_t)1 << kChunkShift);
  w.nbuckets = pr.B * pr.Hkv * w.nchunk * n2;
  w.max_tiles = w.nbuckets + ceil_div64(nq * pr.K, 128 / 8);
  size_t o = 0;
  w.status = o; o += 256;
  w.kept2 = o; o = align_up(o + (size_t)nq * pr.K * 4, 256);
  w.leaf_score = o; o = align_up(o + (size_t)nq * pr.K * 2 * 4, 256);
  w.counts = o; o = align_up(o + (size_t)(w.nbuckets + 1) * 4, 256);
  w.offsets = o; o = align_up(o + (size_t)(w.nbuckets + 1) * 4, 256);
  w.cursor = o; o = align_up(o + (size_t)(w.nbuckets + 1) * 4, 256);
  w.tile_off = o; o = align_up(o + (size_t)(w.nbuckets + 1) * 4, 256);
  w.pairs = o; o = align_up(o + (size_t)nq * pr.K * 4, 256);
  w.tile_info = o; o = align_up(o + (size_t)w.max_tiles * 16, 256);
  w.haar_rows = o; o = align_up(o + 4 * haar_rows_bytes(pr, s), 256);
  w.haar_meta = o; o = align_up(o + haar_meta_bytes(pr, s), 256);
  w.path = o; o = align_up(o + path_dots_bytes(pr, s), 256);
  w.total = o;
  return w;
}

AttendWs attend_ws_layout(const Prob& pr, const Pyr& s) {
  AttendWs w{};
  const int64_t nq = pr.B * pr.Hkv * pr.N;
  const int64_t W = pr.K + 3;
  w.nchunk = ceil_div64(pr.N, (int64_t)1 << kChunkShift);
  w.nbuckets = pr.B * pr.Hkv * w.nchunk * s.nb;
  w.max_tiles = w.nbuckets + ceil_div64(nq * W, 128 / 8);
  size_t o = 0;
  w.status = o; o += 256;
  w.counts = o; o = align_up(o + (size_t)(w.nbuckets + 1) * 4, 256);
  w.offsets = o; o = align_up(o + (size_t)(w.nbuckets + 1) * 4, 256);
  w.cursor = o; o = align_up(o + (size_t)(w.nbuckets + 1) * 4, 256);
  w.tile_off = o; o = align_up(o + (size_t)(w.nbuckets + 1) * 4, 256);
  w.pairs = o; o = align_up(o + (size_t)nq * W * 4, 256);
  w.tile_info = o; o = align_up(o + (size_t)w.max_tiles * 16, 256);
  w.part_lse = o; o = align_up(o + (size_t)nq * W * pr.G * 4, 256);
  w.part_o = o; o = align_up(o + (size_t)nq * W * pr.G * pr.d * 2, 256);
  w.total = o;
  return w;
}

size_t decode_ws_bytes(const Prob&, const Pyr&) { return 256; }

size_t flat_ws_bytes(const Prob& pr, const Pyr& s) {
  // status word + leaf means rounded to bf16 [B, Hkv, nb, d]
  return 256 + align_up((size_t)pr.B * pr.Hkv * s.nb * pr.d * 2, 256);
}

int sm_count(int device) {
  static std::mutex mu;
  static int cache[64] = {0};
  if (device < 0 || device >= 64) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (cache[device] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) == cudaSuccess) cache[device] = v;
  }
  return cache[device];
}

// Shared validation of the problem description.
static pisa_status check_params(const pisa_params* p, Prob* pr, Pyr* s) {
  if (!p || p->struct_size < sizeof(pisa_params)) return PISA_ERR_INVALID_ARG;
  if (p->B < 0 || p->N < 0 || p->H_q < 1 || p->H_kv < 1 || p->d < 1 || p->C < 1 || p->g < 1 ||
      p->K < 1 || p->qtile < 1)
    return PISA_ERR_INVALID_ARG;
  if (p->H_q % p->H_kv != 0) return PISA_ERR_INVALID_ARG;
  if (!(p->scale >= 0.0f) || isinf(p->scale)) return PISA_ERR_INVALID_ARG;
  if (p->scorer < PISA_SCORER_LSE || p->scorer > PISA_SCORER_MEAN_VAR) return PISA_ERR_INVALID_ARG;
  if (p->summaries != PISA_SUMMARIES_ALL && p->summaries != PISA_SUMMARIES_PREFIX) return PISA_ERR_INVALID_ARG;
  if (p->dtype != PISA_BF16 && p->dtype != PISA_FP32) return PISA_ERR_UNSUPPORTED;
  const int G = p->H_q / p->H_kv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return PISA_ERR_UNSUPPORTED;
  if (p->d != 64 && p->d != 128) return PISA_ERR_UNSUPPORTED;
  if (p->C != 64 || p->g != 2 || p->K > kMaxK) return PISA_ERR_UNSUPPORTED;
  if (p->N > kMaxN) return PISA_ERR_UNSUPPORTED;
  if (!make_pyr(p->N, p->C, s)) return PISA_ERR_INVALID_ARG;
  pr->B = p->B; pr->N = p->N; pr->Hq = p->H_q; pr->Hkv = p->H_kv; pr->G = G;
  pr->d = p->d; pr->C = p->C; pr->K = p->K; pr->dtype = p->dtype; pr->scorer = p->scorer;
  pr->prefix = p->summaries == PISA_SUMMARIES_PREFIX ? 1 : 0;
  const float sc = p->scale > 0.0f ? p->scale : 1.0f / sqrtf((float)p->d);
  pr->scale2 = sc * kLog2e;
  return PISA_OK;
}

static bool aligned16(const void* x) { return ((uintptr_t)x & 15u) == 0; }

static pisa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PISA_OK : PISA_ERR_CUDA; }

static std::atomic<unsigned long long> g_launches{0};

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

}  // namespace pisa

using namespace pisa;

extern "C" {

int pisa_abi_version(void) { return PISA_ABI_VERSION; }

uint64_t pisa_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

const char* pisa_status_string(pisa_status s) {
  switch (s) {
    case PISA_OK: return "PISA_OK";
    case PISA_ERR_INVALID_ARG: return "PISA_ERR_INVALID_ARG: null pointer, bad size or shape";
    case PISA_ERR_UNSUPPORTED: return "PISA_ERR_UNSUPPORTED: d, C, g, G, K, N or dtype outside the built set";
    case PISA_ERR_MISALIGNED: return "PISA_ERR_MISALIGNED: a pointer is not 16-byte aligned";
    case PISA_ERR_WORKSPACE: return "PISA_ERR_WORKSPACE: workspace smaller than pisa_workspace_bytes()";
    case PISA_ERR_CUDA: return "PISA_ERR_CUDA: a CUDA call or launch failed";
    case PISA_ERR_DEVICE: return "PISA_ERR_DEVICE: a kernel reported a fault in the status word";
  }
  return "unknown pisa_status";
}

int32_t pisa_pyramid_levels(const pisa_params* p) {
  Prob pr; Pyr s;
  if (check_params(p, &pr, &s) != PISA_OK) return 0;
  return s.L;
}

int64_t pisa_pyramid_nodes(const pisa_params* p) {
  Prob pr; Pyr s;
  if (check_params(p, &pr, &s) != PISA_OK) return 0;
  return s.P;
}

size_t pisa_pyramid_bytes(const pisa_params* p) {
  Prob pr; Pyr s;
  if (check_params(p, &pr, &s) != PISA_OK) return 0;
  return (size_t)pr.B * pr.Hkv * s.P * pr.d * sizeof(float);
}

size_t pisa_workspace_bytes(const pisa_params* p, int32_t mode) {
  Prob pr; Pyr s;
  if (check_params(p, &pr, &s) != PISA_OK) return 0;
  switch (mode) {
    case PISA_MODE_PREFILL: return prefill_ws_layout(pr, s).total;
    case PISA_MODE_DECODE: return decode_ws_bytes(pr, s);
    case PISA_MODE_FLAT: return flat_ws_bytes(pr, s);
    case PISA_MODE_ATTEND: return attend_ws_layout(pr, s).total;
  }
  return 0;
}

pisa_status pisa_build_pyramid(const pisa_params* p, const void* k, const int32_t* seq_lens, float* pyramid,
                               void* stream) {
  Prob pr; Pyr s;
  pisa_status rc = check_params(p, &pr, &s);
  if (rc != PISA_OK) return rc;
  if (pr.B * pr.Hkv * pr.N == 0) return PISA_OK;
  if (!k || !pyramid) return PISA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(pyramid)) return PISA_ERR_MISALIGNED;
  return cuda_status(launch_build_pyramid(pr, s, k, KeyPages{nullptr, 0, 0}, seq_lens, pyramid, nullptr,
                                          (cudaStream_t)stream));
}

// Checks of a paged key pool shared by the paged entry points.
static pisa_status paged_checks(const Prob& pr, const Pyr& s, const void* k_pages, int64_t num_pages,
                                const int32_t* page_table, KeyPages* kp) {
  if (!k_pages || !page_table || num_pages < 1) return PISA_ERR_INVALID_ARG;
  if (!aligned16(k_pages) || ((uintptr_t)page_table & 3u)) return PISA_ERR_MISALIGNED;
  if (num_pages > ((int64_t)1 << 31) - 1) return PISA_ERR_UNSUPPORTED;
  kp->table = page_table;
  kp->max_pages = s.nb;
  kp->num_pages = num_pages;
  (void)pr;
  return PISA_OK;
}

pisa_status pisa_build_pyramid_paged(const pisa_params* p, const void* k_pages, int64_t num_pages,
                                     const int32_t* page_table, const int32_t* seq_lens, float* pyramid, void* ws,
                                     size_t ws_bytes, void* stream) {
  Prob pr; Pyr s;
  pisa_status rc = check_params(p, &pr, &s);
  if (rc != PISA_OK) return rc;
  if (pr.B * pr.Hkv * pr.N == 0) return PISA_OK;
  if (!pyramid || !ws) return PISA_ERR_INVALID_ARG;
  if (!aligned16(pyramid) || !aligned16(ws) || ((uintptr_t)seq_lens & 3u)) return PISA_ERR_MISALIGNED;
  if (ws_bytes < decode_ws_bytes(pr, s)) return PISA_ERR_WORKSPACE;
  KeyPages kp;
  rc = paged_checks(pr, s, k_pages, num_pages, page_table, &kp);
  if (rc != PISA_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(ws, 0, 256, st) != cudaSuccess) return PISA_ERR_CUDA;
  return cuda_status(launch_build_pyramid(pr, s, k_pages, kp, seq_lens, pyramid, (int32_t*)ws, st));
}

// Checks shared by the prefill entry points.
static pisa_status prefill_checks(const pisa_params* p, Prob* pr, Pyr* s, PrefillWs* w, const void* q, const void* k,
                                  const float* pyramid, const void* ws, size_t ws_bytes, bool need_k, bool need_pyr,
                                  const int32_t* out_idx, bool need_out, const float* out_score,
                                  const int32_t* trace) {
  pisa_status rc = check_params(p, pr, s);
  if (rc != PISA_OK) return rc;
  *w = prefill_ws_layout(*pr, *s);
  if (pr->B * pr->Hkv * pr->N == 0) return PISA_OK;
  if (!q || !ws || (need_k && !k) || (need_pyr && !pyramid) || (need_out && !out_idx)) return PISA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(ws) || (need_k && !aligned16(k)) || (need_pyr && !aligned16(pyramid)))
    return PISA_ERR_MISALIGNED;
  if (((uintptr_t)out_idx & 3u) || ((uintptr_t)out_score & 3u) || ((uintptr_t)trace & 3u))
    return PISA_ERR_MISALIGNED;
  if (ws_bytes < w->total) return PISA_ERR_WORKSPACE;
  // pair counts, tile indices and TMA row coordinates are 32-bit; the bucket
  // grid (query chunks x level-2 nodes) grows with N^2
  if (pr->B * pr->Hkv * pr->N * pr->K >= ((int64_t)1 << 31)) return PISA_ERR_UNSUPPORTED;
  if (w->max_tiles >= ((int64_t)1 << 31)) return PISA_ERR_UNSUPPORTED;
  return PISA_OK;
}

// k is needed only for prefix-consistent summaries (the partial leaf of each
// query's path).
static pisa_status run_route(const Prob& pr, const Pyr& s, const PrefillWs& w, const void* q, const void* k,
                             const float* pyramid, char* base, int32_t* trace, cudaStream_t st) {
  int32_t* status = (int32_t*)(base + w.status);
  if (cudaMemsetAsync(status, 0, 256, st) != cudaSuccess) return PISA_ERR_CUDA;
  const bool haar = route_haar_supported(pr);
  float* path = nullptr;
  if (pr.prefix) {
    path = (float*)(base + w.path);
    const cudaError_t e = launch_path_dots(pr, s, q, k, pyramid, haar ? 1 : 0, path, st);
    if (e != cudaSuccess) return PISA_ERR_CUDA;
  }
  if (haar)
    return cuda_status(launch_route_haar(pr, s, q, pyramid, base + w.haar_rows, (float4*)(base + w.haar_meta), path,
                                         (int32_t*)(base + w.kept2), trace, st));
  return cuda_status(launch_route(pr, s, q, pyramid, path, (int32_t*)(base + w.kept2), trace, status, st));
}

static pisa_status run_leaves(const Prob& pr, const Pyr& s, const PrefillWs& w, const void* q, const void* k,
                              char* base, int32_t* out_idx, float* out_score, cudaStream_t st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PISA_ERR_CUDA;
  cudaError_t e;
  if (pr.dtype == PISA_BF16)
    e = launch_leaf_tc(pr, s, w, base, q, k, out_idx, out_score, sm_count(dev), st);
  else
    e = launch_leaf_simt(pr, s, q, k, (const int32_t*)(base + w.kept2), out_idx, out_score, st);
  return cuda_status(e);
}

pisa_status pisa_select_prefill(const pisa_params* p, const void* q, const void* k, const float* pyramid, void* ws,
                                size_t ws_bytes, int32_t* out_idx, float* out_score, int32_t* trace,
                                void* stream) {
  Prob pr; Pyr s; PrefillWs w;
  pisa_status rc = prefill_checks(p, &pr, &s, &w, q, k, pyramid, ws, ws_bytes, true, true, out_idx, true, out_score,
                                  trace);
  if (rc != PISA_OK || pr.B * pr.Hkv * pr.N == 0) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  rc = run_route(pr, s, w, q, k, pyramid, (char*)ws, trace, st);
  if (rc != PISA_OK) return rc;
  return run_leaves(pr, s, w, q, k, (char*)ws, out_idx, out_score, st);
}

pisa_status pisa_prefill_route(const pisa_params* p, const void* q, const float* pyramid, void* ws, size_t ws_bytes,
                               int32_t* trace, void* stream) {
  Prob pr; Pyr s; PrefillWs w;
  pisa_status rc = prefill_checks(p, &pr, &s, &w, q, nullptr, pyramid, ws, ws_bytes, false, true, nullptr, false,
                                  nullptr, trace);
  if (rc != PISA_OK || pr.B * pr.Hkv * pr.N == 0) return rc;
  if (pr.prefix) return PISA_ERR_UNSUPPORTED;  // prefix-consistent walks need the keys: pisa_select_prefill
  return run_route(pr, s, w, q, nullptr, pyramid, (char*)ws, trace, (cudaStream_t)stream);
}

pisa_status pisa_prefill_leaves(const pisa_params* p, const void* q, const void* k, void* ws, size_t ws_bytes,
                                int32_t* out_idx, float* out_score, void* stream) {
  Prob pr; Pyr s; PrefillWs w;
  pisa_status rc = prefill_checks(p, &pr, &s, &w, q, k, nullptr, ws, ws_bytes, true, false, out_idx, true, out_score,
                                  nullptr);
  if (rc != PISA_OK || pr.B * pr.Hkv * pr.N == 0) return rc;
  return run_leaves(pr, s, w, q, k, (char*)ws, out_idx, out_score, (cudaStream_t)stream);
}

pisa_status pisa_select_decode(const pisa_params* p, const void* q, const void* k_cache, const int32_t* seq_lens,
                               float* pyramid, void* ws, size_t ws_bytes, int32_t* out_idx, float* out_score,
                               int32_t* trace, void* stream) {
  Prob pr; Pyr s;
  pisa_status rc = check_params(p, &pr, &s);
  if (rc != PISA_OK) return rc;
  if (pr.B * pr.Hkv == 0) return PISA_OK;
  if (pr.N == 0) return PISA_ERR_INVALID_ARG;
  if (!q || !k_cache || !seq_lens || !pyramid || !ws || !out_idx) return PISA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(pyramid) || !aligned16(ws)) return PISA_ERR_MISALIGNED;
  if (((uintptr_t)out_idx & 3u) || ((uintptr_t)out_score & 3u) || ((uintptr_t)seq_lens & 3u) ||
      ((uintptr_t)trace & 3u))
    return PISA_ERR_MISALIGNED;
  if (ws_bytes < decode_ws_bytes(pr, s)) return PISA_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  int32_t* status = (int32_t*)ws;
  cudaError_t e = cudaMemsetAsync(status, 0, 256, st);
  if (e != cudaSuccess) return PISA_ERR_CUDA;
  return cuda_status(launch_decode(pr, s, q, k_cache, KeyPages{nullptr, 0, 0}, seq_lens, pyramid, status, out_idx,
                                   out_score, trace, st));
}

pisa_status pisa_select_decode_paged(const pisa_params* p, const void* q, const void* k_pages, int64_t num_pages,
                                     const int32_t* page_table, const int32_t* seq_lens, float* pyramid, void* ws,
                                     size_t ws_bytes, int32_t* out_idx, float* out_score, int32_t* trace,
                                     void* stream) {
  Prob pr; Pyr s;
  pisa_status rc = check_params(p, &pr, &s);
  if (rc != PISA_OK) return rc;
  if (pr.B * pr.Hkv == 0) return PISA_OK;
  if (pr.N == 0) return PISA_ERR_INVALID_ARG;
  if (!q || !seq_lens || !pyramid || !ws || !out_idx) return PISA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(pyramid) || !aligned16(ws)) return PISA_ERR_MISALIGNED;
  if (((uintptr_t)out_idx & 3u) || ((uintptr_t)out_score & 3u) || ((uintptr_t)seq_lens & 3u) ||
      ((uintptr_t)trace & 3u))
    return PISA_ERR_MISALIGNED;
  if (ws_bytes < decode_ws_bytes(pr, s)) return PISA_ERR_WORKSPACE;
  KeyPages kp;
  rc = paged_checks(pr, s, k_pages, num_pages, page_table, &kp);
  if (rc != PISA_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  int32_t* status = (int32_t*)ws;
  if (cudaMemsetAsync(status, 0, 256, st) != cudaSuccess) return PISA_ERR_CUDA;
  return cuda_status(launch_decode(pr, s, q, k_pages, kp, seq_lens, pyramid, status, out_idx, out_score, trace, st));
}

pisa_status pisa_select_flat(const pisa_params* p, const void* q, const float* pyramid, void* ws, size_t ws_bytes,
                             int32_t* out_idx, float* out_score, void* stream) {
  Prob pr; Pyr s;
  pisa_status rc = check_params(p, &pr, &s);
  if (rc != PISA_OK) return rc;
  if (pr.B * pr.Hkv * pr.N == 0) return PISA_OK;
  if (pr.dtype != PISA_BF16) return PISA_ERR_UNSUPPORTED;  // the comparator is built for bf16 inputs
  if (!q || !pyramid || !ws || !out_idx) return PISA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(pyramid) || !aligned16(ws)) return PISA_ERR_MISALIGNED;
  if (((uintptr_t)out_idx & 3u) || ((uintptr_t)out_score & 3u)) return PISA_ERR_MISALIGNED;
  if (ws_bytes < flat_ws_bytes(pr, s)) return PISA_ERR_WORKSPACE;
  if (pr.B * pr.Hkv * s.nb >= ((int64_t)1 << 31)) return PISA_ERR_UNSUPPORTED;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaMemsetAsync(ws, 0, 256, st);
  if (e != cudaSuccess) return PISA_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PISA_ERR_CUDA;
  return cuda_status(launch_flat(pr, s, q, pyramid, (char*)ws, out_idx, out_score, sm_count(dev), st));
}

pisa_status pisa_attend_prefill(const pisa_params* p, const void* q, const void* k, const void* v,
                                const int32_t* idx, void* ws, size_t ws_bytes, void* out, void* stream) {
  Prob pr; Pyr s;
  pisa_status rc = check_params(p, &pr, &s);
  if (rc != PISA_OK) return rc;
  if (pr.B * pr.Hkv * pr.N == 0) return PISA_OK;
  if (pr.dtype != PISA_BF16) return PISA_ERR_UNSUPPORTED;  // built for bf16 inputs
  if (!q || !k || !v || !idx || !ws || !out) return PISA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(ws) || !aligned16(out) ||
      ((uintptr_t)idx & 3u))
    return PISA_ERR_MISALIGNED;
  const AttendWs w = attend_ws_layout(pr, s);
  if (ws_bytes < w.total) return PISA_ERR_WORKSPACE;
  // pair counts, tile indices and TMA row coordinates are 32-bit; the bucket
  // grid (query chunks x blocks) grows with N^2
  if (pr.B * pr.Hkv * pr.N * (pr.K + 3) >= ((int64_t)1 << 31)) return PISA_ERR_UNSUPPORTED;
  if (w.max_tiles >= ((int64_t)1 << 31)) return PISA_ERR_UNSUPPORTED;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(ws, 0, 256, st) != cudaSuccess) return PISA_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PISA_ERR_CUDA;
  return cuda_status(launch_attend(pr, s, w, (char*)ws, q, k, v, idx, out, sm_count(dev), st));
}

pisa_status pisa_attend_decode(const pisa_params* p, const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* seq_lens, const int32_t* idx, void* ws, size_t ws_bytes, void* out,
                               void* stream) {
  Prob pr; Pyr s;
  pisa_status rc = check_params(p, &pr, &s);
  if (rc != PISA_OK) return rc;
  if (pr.B * pr.Hkv == 0) return PISA_OK;
  if (pr.N == 0) return PISA_ERR_INVALID_ARG;
  if (pr.dtype != PISA_BF16 || pr.N % 16 != 0) return PISA_ERR_UNSUPPORTED;  // 16-key chunks never pass N
  if (!q || !k_cache || !v_cache || !seq_lens || !idx || !ws || !out) return PISA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(ws) || !aligned16(out) ||
      ((uintptr_t)seq_lens & 3u) || ((uintptr_t)idx & 3u))
    return PISA_ERR_MISALIGNED;
  if (ws_bytes < decode_ws_bytes(pr, s)) return PISA_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(ws, 0, 256, st) != cudaSuccess) return PISA_ERR_CUDA;
  return cuda_status(launch_attend_decode(pr, s, q, k_cache, v_cache, seq_lens, idx, out, (int32_t*)ws, st));
}

pisa_status pisa_read_device_status(const void* ws, int32_t* device_code, void* stream) {
  if (!ws || !device_code) return PISA_ERR_INVALID_ARG;
  int32_t v = 0;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess) return PISA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return PISA_ERR_CUDA;
  *device_code = v;
  return v == 0 ? PISA_OK : PISA_ERR_DEVICE;
}

}  // extern "C"
