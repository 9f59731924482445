/*
 * pisa.h -- C ABI of the GB300 (sm_103a) PISA pyramid Top-K block selector.
 *
 * The operation (web pages about arXiv 2609.31093, "Block Sparse Attention
 * with Log-Linear Complexity"):
 *  - agihunt.info summary, pyramid paragraph: keys are mean-pooled into leaf
 *    blocks of C keys, and coarser levels mean-pool adjacent nodes with
 *    branching factor g = 2, giving O(log N) levels; selection starts at the
 *    coarsest level, scores a bounded candidate set with LogSumExp, keeps
 *    Top-K and expands only the kept nodes; decode routing is O(log N) a step.
 *  - same page, LSE paragraph: the first, previous and current leaf blocks are
 *    always selected; kernel paragraph: query heads of one GQA group share the
 *    selected blocks; leaf blocks are scored by LSE over their raw keys.
 *  - rcap.io post, "Selection walks the tree top-down" and "The scoring rule
 *    matters": at most g*K candidates per level; a candidate's score is the
 *    LogSumExp over its child summaries.
 *
 * Readings fixed by this library where the pages are silent: the walk starts
 * at the root and keeps all candidates while a level has at most K; a node is
 * eligible when its leaf range meets E = [1, qb-2] (qb = t / C); summaries are
 * plain means of the keys present in a node's span (not masked by the query
 * position, unless PISA_SUMMARIES_PREFIX is asked for); the group score is the sum of the heads' natural-log LSEs; the
 * scale is 1/sqrt(d) unless given; Top-K ties go to the lower node index;
 * the forced blocks F = {0, qb-1, qb} are added to the Top-K of E.
 *
 * Conventions shared by every call
 *  - All tensors are caller-owned DEVICE memory, contiguous, row-major.
 *    q      prefill [B, H_q, N, d];   decode [B, H_q, d]
 *    k      prefill [B, H_kv, N, d];  decode: key cache [B, H_kv, N, d] with
 *           N the capacity (N_max)
 *    pyramid fp32 [B, H_kv, P, d], P = pisa_pyramid_nodes(); node (l, j) of
 *           level l >= 1 sits at row off_l + j, off_1 = 0, off_{l+1} = off_l +
 *           n_l, n_1 = ceil(N / C), n_{l+1} = ceil(n_l / 2), up to n_L = 1.
 *           Node (l, j) covers leaves [j 2^(l-1), (j+1) 2^(l-1)).
 *    out_idx int32 [.., K+3]: Top-K leaf blocks of E together with F, in
 *           ascending order, padded with -1.
 *    out_score fp32 [.., K+3] (nullable): the group-summed leaf LSE of each
 *           Top-K block, +INFINITY for forced blocks, -INFINITY for padding.
 *  - q, k, pyramid and the workspace must be 16-byte aligned.
 *  - dtype PISA_BF16 or PISA_FP32 (q and k alike); d in {64, 128}; C = 64;
 *    g = 2; 1 <= K <= 32; H_q % H_kv == 0 with G = H_q / H_kv in {1,2,4,8};
 *    qtile >= 1 (it only changes data reuse, never results).
 *  - Every call validates its arguments on the host before any launch and,
 *    on failure, returns a negative status and launches nothing.  Launch
 *    failures return PISA_ERR_CUDA.  Calls are asynchronous on `stream`
 *    (a cudaStream_t; NULL is the legacy default stream), never allocate
 *    memory and never synchronise, except pisa_read_device_status and
 *    pisa_read_static_status.
 *  - The workspace is caller-owned scratch of at least
 *    pisa_workspace_bytes(params, mode) bytes.  Its first 256 bytes hold a
 *    device status word that kernels set on faults they detect (a decode
 *    sequence length outside [1, N], an exhausted bounded wait); each call
 *    clears it first.  Calls that share a workspace must not overlap.
 *  - The library holds no global state besides the loaded kernels, a
 *    per-device cache of SM counts, a process-wide launch counter and the
 *    fixed scratch of pisa_select_prefill_static; it is safe to call from
 *    several threads on different streams with different workspaces.
 */
#ifndef PISA_H_
#define PISA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PISA_ABI_VERSION 3

typedef enum {
  PISA_OK = 0,
  PISA_ERR_INVALID_ARG = -1,  /* null pointer, bad size or shape */
  PISA_ERR_UNSUPPORTED = -2,  /* valid but not built: d, C, g, G, K, dtype */
  PISA_ERR_MISALIGNED = -3,   /* a pointer is not 16-byte aligned */
  PISA_ERR_WORKSPACE = -4,    /* workspace smaller than required */
  PISA_ERR_CUDA = -5,         /* a CUDA runtime call or launch failed */
  PISA_ERR_DEVICE = -6        /* a kernel reported a fault (status word) */
} pisa_status;

typedef enum { PISA_BF16 = 0, PISA_FP32 = 1 } pisa_dtype;

/* Block scorer of the walk and the leaves (agihunt.info summary, LSE
 * paragraph; rcap.io, "The scoring rule matters").  Over the n summands x_i
 * of a candidate (scaled dots with its eligible children's summaries above
 * the leaves, with its raw keys at the leaves):
 *   PISA_SCORER_LSE       log sum_i exp(x_i)                 (PISA)
 *   PISA_SCORER_MEAN      log n + mean(x)                    (PISA-1)
 *   PISA_SCORER_MEAN_VAR  log n + mean(x) + var(x) / 2        (PISA-2)
 * the first- and second-order truncations of the cumulant expansion of the
 * log-sum-exp around the mean (var: population variance).  The flat
 * comparator and the attention ignore it. */
typedef enum {
  PISA_SCORER_LSE = 0,
  PISA_SCORER_MEAN = 1,
  PISA_SCORER_MEAN_VAR = 2
} pisa_scorer;

/* Which keys a prefill query's node summaries cover (agihunt.info summary,
 * pyramid paragraph: decode routing walks the pyramid of the keys seen so
 * far; rcap.io, the pisa_select sketch walks summaries without a mask).
 *   PISA_SUMMARIES_ALL     every key of the node's span (the pyramid of the
 *                          whole sequence; a summary straddling position t
 *                          includes keys after t)
 *   PISA_SUMMARIES_PREFIX  the span's keys at positions <= t only, i.e. the
 *                          pyramid of the first t + 1 keys, which is what the
 *                          decode step at length t + 1 walks (prefix-
 *                          consistent, leak-free)
 * Leaf scores read complete past blocks under both, and the decode, flat and
 * attention calls ignore the field. */
typedef enum {
  PISA_SUMMARIES_ALL = 0,
  PISA_SUMMARIES_PREFIX = 1
} pisa_summaries;

typedef enum {
  PISA_MODE_PREFILL = 0,
  PISA_MODE_DECODE = 1,
  PISA_MODE_FLAT = 2,
  PISA_MODE_ATTEND = 3
} pisa_mode;

/* Device status codes written into the workspace status word. */
#define PISA_DEV_OK 0
#define PISA_DEV_BAD_SEQ_LEN 1   /* decode: seq_lens[b] outside [1, N] */
#define PISA_DEV_TIMEOUT 2       /* a bounded device wait ran out */
#define PISA_DEV_BAD_INDEX 3     /* an internal index check failed */

typedef struct {
  uint32_t struct_size; /* sizeof(pisa_params), for forward compatibility */
  int32_t dtype;        /* pisa_dtype of q and k */
  int64_t B;            /* sequences */
  int64_t N;            /* prefill: tokens per sequence; decode: capacity */
  int32_t H_q;          /* query heads */
  int32_t H_kv;         /* key heads */
  int32_t d;            /* head dimension */
  int32_t C;            /* leaf block size (keys per leaf) */
  int32_t g;            /* branching factor */
  int32_t K;            /* blocks kept per level */
  int32_t qtile;        /* queries sharing one leaf tile (reuse only) */
  float scale;          /* score scale inside exp(); 0 means 1/sqrt(d) */
  int32_t scorer;       /* pisa_scorer (0: the log-sum-exp of PISA) */
  int32_t summaries;    /* pisa_summaries of prefill walks (0: all keys) */
} pisa_params;

/* ABI version of the loaded library (PISA_ABI_VERSION). */
int pisa_abi_version(void);

/* Number of kernel launches this library has issued in this process, over
 * all devices and streams (a relaxed atomic counter, for launch accounting in
 * benchmarks).  Host only; never fails. */
uint64_t pisa_kernel_launches(void);

/* Human-readable name of a status. */
const char* pisa_status_string(pisa_status s);

/* Number of pyramid levels L and nodes P per (sequence, key head); 0 on bad
 * params.  Host only. */
int32_t pisa_pyramid_levels(const pisa_params* p);
int64_t pisa_pyramid_nodes(const pisa_params* p);

/* Bytes of the fp32 pyramid [B, H_kv, P, d]; 0 on bad params. */
size_t pisa_pyramid_bytes(const pisa_params* p);

/* Workspace bytes needed by pisa_select_prefill (PISA_MODE_PREFILL),
 * pisa_select_decode (PISA_MODE_DECODE), pisa_select_flat (PISA_MODE_FLAT)
 * or pisa_attend_prefill (PISA_MODE_ATTEND); 0 on bad params. */
size_t pisa_workspace_bytes(const pisa_params* p, int32_t mode);

/* Key pyramid (agihunt.info summary, pyramid paragraph; rcap.io, "Think of
 * the keys as leaves of a tree").  Writes every node of the capacity-N layout:
 * node (l, j) = mean of the keys k[b, h, i], i in its span and below
 * len_b = seq_lens[b] (or N when seq_lens is NULL); a node with no key is
 * zero.  seq_lens: DEVICE int32 [B] or NULL; values outside [0, N] are
 * clamped.  Leaves are sums over keys in index order divided by the count;
 * each parent is (n0 m0 + n1 m1) / (n0 + n1) of its children, all in
 * IEEE round-to-nearest fp32, so pisa_select_decode's incremental update
 * reproduces it bit for bit. */
pisa_status pisa_build_pyramid(const pisa_params* p, const void* k,
                               const int32_t* seq_lens, float* pyramid,
                               void* stream);

/* Prefill / training selection for every query position t in [0, N) of every
 * sequence and key head (agihunt.info summary, kernel paragraph: the
 * two-stage prefill kernel; rcap.io, the pisa_select sketch).  `pyramid`
 * must hold pisa_build_pyramid(p, k, NULL, ...).  Outputs:
 *   out_idx   int32 [B, H_kv, N, K+3] (required)
 *   out_score fp32  [B, H_kv, N, K+3] (nullable)
 *   trace     int32 [B, H_kv, N, L, K] (nullable, for tests): for each level
 *             l = 2..L the kept node set (ascending, -1 padded) of the walk,
 *             row l-1; rows of levels above the first level with more than
 *             K eligible nodes hold all eligible nodes; row 0 is left -1. */
pisa_status pisa_select_prefill(const pisa_params* p, const void* q,
                                const void* k, const float* pyramid, void* ws,
                                size_t ws_bytes, int32_t* out_idx,
                                float* out_score, int32_t* trace, void* stream);

/* The two stages of pisa_select_prefill, for callers that time or inspect
 * them separately; run back to back on one stream with one workspace they
 * are exactly pisa_select_prefill.
 *   pisa_prefill_route: clears the status word and walks levels L..2 for
 *     every query (rcap.io, "Selection walks the tree top-down"), leaving the
 *     kept level-2 nodes of each query in the workspace; writes `trace`.
 *     With PISA_SUMMARIES_PREFIX it returns PISA_ERR_UNSUPPORTED (that walk
 *     reads the raw keys of each query's own leaf): use pisa_select_prefill.
 *   pisa_prefill_leaves: scores the leaf candidates (the two children of each
 *     kept level-2 node) by LSE over their raw keys and writes out_idx and
 *     out_score.  It must follow pisa_prefill_route on the same workspace
 *     with the same params, q and pyramid. */
pisa_status pisa_prefill_route(const pisa_params* p, const void* q,
                               const float* pyramid, void* ws, size_t ws_bytes,
                               int32_t* trace, void* stream);
pisa_status pisa_prefill_leaves(const pisa_params* p, const void* q,
                                const void* k, void* ws, size_t ws_bytes,
                                int32_t* out_idx, float* out_score,
                                void* stream);

/* One decode step (agihunt.info summary: "Decode routing is O(log N) per
 * step"; kernel paragraph: a single-stage decode kernel).  For each sequence
 * b the caller has already written its new key at position seq_lens[b]-1 of
 * k_cache.  In one launch the call first updates `pyramid` in place along the
 * path of that position (the leaf from its raw keys, every ancestor from its
 * two children), then selects for the query at position seq_lens[b]-1.
 *   q        [B, H_q, d];  seq_lens DEVICE int32 [B], each in [1, N]
 *   pyramid  must hold the pyramid of the keys [0, seq_lens[b]-1) (e.g. from
 *            pisa_build_pyramid with those lengths, or from the previous step)
 *   out_idx  int32 [B, H_kv, K+3];  out_score fp32 [B, H_kv, K+3] (nullable)
 *   trace    int32 [B, H_kv, L, K] (nullable): the kept sets of the walk, as
 *            for pisa_select_prefill, with L the levels of capacity N.
 * A sequence length outside [1, N] sets PISA_DEV_BAD_SEQ_LEN in the status
 * word and leaves that sequence's outputs at -1 / -INFINITY. */
pisa_status pisa_select_decode(const pisa_params* p, const void* q,
                               const void* k_cache, const int32_t* seq_lens,
                               float* pyramid, void* ws, size_t ws_bytes,
                               int32_t* out_idx, float* out_score,
                               int32_t* trace, void* stream);

/* Paged key cache (the usual layout of a serving decode cache).  The raw
 * keys live in a pool of pages of C keys,
 *   k_pages  [num_pages, H_kv, C, d] (DEVICE, dtype of p): page j of
 *            sequence b is page_table[b * ceil(N / C) + j] and holds that
 *            sequence's keys [j C, (j + 1) C) for every key head;
 *   page_table int32 [B, ceil(N / C)] (DEVICE), N the capacity of p.
 * Only the pages of leaves that hold keys (j C < seq_lens[b]) are read.  A
 * page index outside [0, num_pages) sets PISA_DEV_BAD_INDEX in the status
 * word and is never dereferenced: the build treats that leaf as empty, the
 * decode step writes -1 / -INFINITY for that sequence.  The pyramid stays
 * in its capacity layout [B, H_kv, P, d].  Results equal those of the
 * contiguous calls on the same keys bit for bit.
 *   pisa_build_pyramid_paged: pisa_build_pyramid from pages; ws holds the
 *     status word (at least pisa_workspace_bytes(p, PISA_MODE_DECODE)).
 *   pisa_select_decode_paged: pisa_select_decode from pages. */
pisa_status pisa_build_pyramid_paged(const pisa_params* p, const void* k_pages,
                                     int64_t num_pages,
                                     const int32_t* page_table,
                                     const int32_t* seq_lens, float* pyramid,
                                     void* ws, size_t ws_bytes, void* stream);
pisa_status pisa_select_decode_paged(const pisa_params* p, const void* q,
                                     const void* k_pages, int64_t num_pages,
                                     const int32_t* page_table,
                                     const int32_t* seq_lens, float* pyramid,
                                     void* ws, size_t ws_bytes,
                                     int32_t* out_idx, float* out_score,
                                     int32_t* trace, void* stream);

/* Flat BSA-style comparator (agihunt.info summary, model paragraph: "BSA
 * (NSA's selected branch with mean summaries)"; rcap.io: "scores every query
 * against every block summary", O(N^2/C)).  Every query head h' scores every
 * complete past block i in [0, qb-1] by softmax_i(s q_h' . mu(1, i)); a block's
 * score is the sum over the group's heads; Top-K over E plus F, output as
 * pisa_select_prefill.  Reads only level 1 (the leaf means) of `pyramid`;
 * uses them rounded to bf16 on the tensor-core path. */
pisa_status pisa_select_flat(const pisa_params* p, const void* q,
                             const float* pyramid, void* ws, size_t ws_bytes,
                             int32_t* out_idx, float* out_score, void* stream);

/* Prefill selection without a caller workspace, for callers that cannot
 * allocate device memory when they select blocks (code running inside a
 * runtime that owns every device allocation, such as a plug-in or a host
 * callback that may not call cudaMalloc or a framework allocator).  The paper
 * has no counterpart: this is a deployment convenience around
 * pisa_select_prefill.  Arguments and outputs are those of
 * pisa_select_prefill without ws, ws_bytes and trace.
 *  - The workspace is one fixed 64 MiB device array inside the library, held
 *    on every GPU that loads it until the process exits.  Problems needing
 *    more (pisa_workspace_bytes(p, PISA_MODE_PREFILL) > 64 MiB) get
 *    PISA_ERR_WORKSPACE and nothing is launched.
 *  - The array's 64 MiB are reserved when the CUDA module holding it is
 *    loaded on a device.  Under CUDA's default lazy module loading that
 *    happens inside the first call of this function (or of
 *    pisa_read_static_status) on that device, which also looks up and caches
 *    the array's device address with the device current; under eager loading
 *    it happens when the library is loaded.  Make that first call where
 *    allocation is still allowed (at initialisation, for instance) and before
 *    any stream capture on the device.
 *  - Later calls never allocate.  All calls on a device share the array, and
 *    each call clears what must start at zero; calls that overlap on the GPU
 *    (other streams, other threads) race on it and must be serialised by the
 *    caller.
 *  - The array starts with the same device status word as any workspace;
 *    pisa_read_static_status reads it. */
pisa_status pisa_select_prefill_static(const pisa_params* p, const void* q,
                                       const void* k, const float* pyramid,
                                       int32_t* out_idx, float* out_score,
                                       void* stream);

/* Device status word of the current device's fixed array used by
 * pisa_select_prefill_static (faults its kernels detected, such as an
 * exhausted bounded wait): synchronises `stream`, then copies the word into
 * *device_code (PISA_DEV_*).  Returns PISA_ERR_DEVICE when it is non-zero.
 * The paper has no counterpart. */
pisa_status pisa_read_static_status(int32_t* device_code, void* stream);

/* Block-sparse attention over a selection (agihunt.info summary, opening
 * paragraph: each query reads only its selected tiles of C keys, so the
 * attention pass is linear in N; rcap.io, "Selection walks the tree
 * top-down": the kept leaf indices drive sparse attention over the original
 * keys).  For query position t of key head h, each query head g of its GQA
 * group (head h*G + g) gets
 *   out[b, h*G+g, t] = sum_i softmax_i(s q . k_i) v_i
 * over the key positions i <= t of the blocks listed in idx[b, h, t, :]
 * (s: the score scale of the params, 1/sqrt(d) when 0).
 *   q    bf16 [B, H_q, N, d];  k, v  bf16 [B, H_kv, N, d]  (DEVICE)
 *   idx  int32 [B, H_kv, N, K+3] (DEVICE): block indices, e.g. the out_idx of
 *        pisa_select_prefill or pisa_select_flat.  Entries outside [0, nb)
 *        are empty slots; a block listed twice counts once; blocks after the
 *        query's own block contribute nothing.
 *   out  bf16 [B, H_q, N, d] (DEVICE).  A query with no key at or before t
 *        in its blocks gets a zero row.
 *   ws   at least pisa_workspace_bytes(p, PISA_MODE_ATTEND) bytes; it holds
 *        one bf16 partial row per (query head, slot): about
 *        2 * B * H_q * N * (K+3) * d bytes.
 * dtype must be PISA_BF16 (PISA_ERR_UNSUPPORTED otherwise); q, k, v, out and
 * ws 16-byte aligned, idx 4-byte aligned.  Inputs are assumed finite.  A
 * bounded device wait that runs out sets PISA_DEV_TIMEOUT in the status
 * word. */
pisa_status pisa_attend_prefill(const pisa_params* p, const void* q,
                                const void* k, const void* v,
                                const int32_t* idx, void* ws, size_t ws_bytes,
                                void* out, void* stream);

/* Attention of one decode step over its selection (the decode counterpart
 * of pisa_attend_prefill).  For sequence b the query sits at position
 * t = seq_lens[b] - 1; each query head g of key head h's group gets
 *   out[b, h*G+g] = sum_i softmax_i(s q . k_i) v_i
 * over the key positions i <= t of the blocks listed in idx[b, h, :].
 *   q    bf16 [B, H_q, d];  k_cache, v_cache bf16 [B, H_kv, N, d] (DEVICE)
 *   idx  int32 [B, H_kv, K+3] (DEVICE), e.g. out_idx of pisa_select_decode;
 *        the same entry rules as pisa_attend_prefill
 *   out  bf16 [B, H_q, d] (DEVICE); ws at least
 *        pisa_workspace_bytes(p, PISA_MODE_DECODE) bytes (status word).
 * dtype must be PISA_BF16 and the capacity N a multiple of 16
 * (PISA_ERR_UNSUPPORTED otherwise).  A sequence length outside [1, N] sets
 * PISA_DEV_BAD_SEQ_LEN and writes a zero row. */
pisa_status pisa_attend_decode(const pisa_params* p, const void* q,
                               const void* k_cache, const void* v_cache,
                               const int32_t* seq_lens, const int32_t* idx,
                               void* ws, size_t ws_bytes, void* out,
                               void* stream);

/* TEST ONLY: fault injection for the bounded device waits of the tcgen05
 * leaf stage (the leaf kernel of pisa_select_prefill and
 * pisa_prefill_leaves with bf16 inputs).  wait_limit_ns replaces the 4 s
 * limit of every wait in later launches (0 restores it); with
 * drop_first_key_tile != 0 the first CTA announces its first key tile on the
 * stage barrier but never issues the copy, so its first MMA wait can only run
 * out.  The kernel then sets PISA_DEV_TIMEOUT in the status word, lets every
 * copy and MMA it issued complete, frees its tensor memory and returns; the
 * call's outputs are then undefined.  Process-wide, not synchronised with
 * launches in flight; never needed outside tests. */
void pisa_test_inject_leaf_timeout(uint64_t wait_limit_ns, int32_t drop_first_key_tile);

/* Synchronises `stream`, then copies the workspace status word into
 * *device_code (PISA_DEV_*).  Returns PISA_ERR_DEVICE when it is non-zero. */
pisa_status pisa_read_device_status(const void* ws, int32_t* device_code,
                                    void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PISA_H_ */
