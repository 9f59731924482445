// pisa_internal.h -- host-side declarations shared by the library's units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pisa_common.cuh"

namespace pisa {

// Pairs (query, kept level-2 node) are bucketed by (sequence, key head,
// query chunk of 2^kChunkShift positions, level-2 node) so that the leaf
// stage sweeps one chunk of queries at a time and their rows stay in L2.
constexpr int kChunkShift = 16;

// Workspace layout of one call (byte offsets from the workspace base).
struct PrefillWs {
  size_t status;      // int32 status word (first 256 bytes)
  size_t kept2;       // int32 [B, Hkv, N, K] kept level-2 nodes (-1 padded)
  size_t leaf_score;  // fp32  [B, Hkv, N, K, 2] group LSE (log2 units)
  size_t counts;      // int32 [nbuckets + 1] pairs per level-2 node
  size_t offsets;     // int32 [nbuckets + 1] exclusive scan of counts
  size_t cursor;      // int32 [nbuckets]
  size_t tile_off;    // int32 [nbuckets + 1] exclusive scan of tiles per bucket
  size_t pairs;       // int32 [B * Hkv * N * K] (t << 5 | slot) grouped by bucket
  size_t tile_info;   // int4  [max_tiles] {bucket, first pair, pairs, 0}
  size_t haar_rows;   // fp16 4 x [B, Hkv, P2, d]: summary and child-difference rows, hi and lo (P2 = P - n_1)
  size_t haar_meta;   // fp32 [B, Hkv, P2, 4]: row scales and residual norms
  size_t path;        // fp32 [B, Hkv, N, L, 2, G] prefix-consistent path dots (only with PISA_SUMMARIES_PREFIX)
  size_t total;
  int64_t nbuckets;   // B * Hkv * nchunk * n_2
  int64_t nchunk;     // ceil(N / 2^kChunkShift)
  int64_t n2;         // level-2 nodes
  int64_t max_tiles;  // nbuckets + B * Hkv * N * K / Q, Q the smallest tile
};

// Counting sort of (query, entry) pairs into buckets (sequence, key head,
// query chunk, node) and the tile list over them (leaf_tc.cu).  lists holds
// `width` entries per query (negative or >= n2: none; with dedup, an entry
// equal to an earlier one of its query is dropped too); a pair is stored as
// (t << shift) | slot; tiles hold at most Q pairs.
struct BucketJob {
  const int32_t* lists;
  int64_t nq, N, n2, nchunk, nbuckets;
  int32_t width, shift, dedup, Q;
  int32_t *counts, *offsets, *cursor, *tile_off, *pairs;
  int4* tile_info;
  size_t clear_bytes;  // bytes from counts to the end of cursor
};
cudaError_t launch_buckets(const BucketJob& j, int num_sms, cudaStream_t st);

// Workspace layout of pisa_attend_prefill.
struct AttendWs {
  size_t status;      // int32 status word (first 256 bytes)
  size_t counts;      // int32 [nbuckets + 1] pairs per (bucket, block)
  size_t offsets;     // int32 [nbuckets + 1]
  size_t cursor;      // int32 [nbuckets + 1]
  size_t tile_off;    // int32 [nbuckets + 1]
  size_t pairs;       // int32 [B * Hkv * N * (K+3)] (t << 6 | slot) grouped by bucket
  size_t tile_info;   // int4  [max_tiles]
  size_t part_lse;    // fp32 [B, Hkv, N, K+3, G] log2-sum-exp2 of each block's scores
  size_t part_o;      // bf16 [B, Hkv, N, K+3, G, d] softmax-weighted values of each block
  size_t total;
  int64_t nbuckets;   // B * Hkv * nchunk * nb
  int64_t nchunk;
  int64_t max_tiles;
};

bool make_pyr(int64_t N, int32_t C, Pyr* s);
PrefillWs prefill_ws_layout(const Prob& pr, const Pyr& s);
AttendWs attend_ws_layout(const Prob& pr, const Pyr& s);
size_t decode_ws_bytes(const Prob& pr, const Pyr& s);
size_t flat_ws_bytes(const Prob& pr, const Pyr& s);

int sm_count(int device);

// Counts one kernel launch (process-wide, relaxed atomic); called before every launch.
void note_launch();

// Launches a kernel of the prefill chain.  With pdl (every kernel of a call
// but its first) the launch uses programmatic stream serialization: its
// launch and prologue may overlap the tail of the kernel before it, which
// is part of the same call.  A call's first kernel is launched plainly, so
// it keeps full ordering after whatever the caller queued on the stream
// (copies, event waits).  Every kernel launched here calls pdl_wait()
// before it touches memory; it blocks until the previous grid has
// completed and its writes are visible, and returns at once after a plain
// launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// 2D TMA view [rows, d] of a bf16 tensor: box of 64 columns x box_rows rows,
// 128-byte swizzle (the K-major operand layout of the tcgen05 MMAs).
bool make_tmap_rows(CUtensorMap* m, const void* base, int64_t rows, int d, int box_rows);

cudaError_t launch_build_pyramid(const Prob& pr, const Pyr& s, const void* k, const KeyPages& kp,
                                 const int32_t* seq_lens, float* pyr, int32_t* status, cudaStream_t st);
// path: the prefix-consistent path dots of every query (launch_path_dots) or
// null for summaries over all keys.
cudaError_t launch_route(const Prob& pr, const Pyr& s, const void* q, const float* pyr, const float* path,
                         int32_t* kept2, int32_t* trace, int32_t* status, cudaStream_t st);
size_t path_dots_bytes(const Prob& pr, const Pyr& s);
// ref_root: dots relative to the finite-masked root summary (the difference-row
// routing) rather than absolute (the fp32 routing).
cudaError_t launch_path_dots(const Prob& pr, const Pyr& s, const void* q, const void* k, const float* pyr,
                             int ref_root, float* out, cudaStream_t st);
bool route_haar_supported(const Prob& pr);
size_t haar_rows_bytes(const Prob& pr, const Pyr& s);  // one of the four fp16 row arrays
size_t haar_meta_bytes(const Prob& pr, const Pyr& s);
cudaError_t launch_route_haar(const Prob& pr, const Pyr& s, const void* q, const float* pyr, char* rows,
                              float4* meta, const float* path, int32_t* kept2, int32_t* trace, cudaStream_t st);
cudaError_t launch_leaf_simt(const Prob& pr, const Pyr& s, const void* q, const void* k, const int32_t* kept2,
                             int32_t* out_idx, float* out_score, cudaStream_t st);
cudaError_t launch_leaf_tc(const Prob& pr, const Pyr& s, const PrefillWs& w, char* ws, const void* q,
                           const void* k, int32_t* out_idx, float* out_score, int num_sms, cudaStream_t st);
cudaError_t launch_decode(const Prob& pr, const Pyr& s, const void* q, const void* kc, const KeyPages& kp,
                          const int32_t* seq_lens,
                          float* pyr, int32_t* status, int32_t* out_idx, float* out_score, int32_t* trace,
                          cudaStream_t st);
cudaError_t launch_attend(const Prob& pr, const Pyr& s, const AttendWs& w, char* ws, const void* q, const void* k,
                          const void* v, const int32_t* idx, void* out, int num_sms, cudaStream_t st);
cudaError_t launch_attend_decode(const Prob& pr, const Pyr& s, const void* q, const void* k, const void* v,
                                 const int32_t* seq_lens, const int32_t* idx, void* out, int32_t* status,
                                 cudaStream_t st);
cudaError_t launch_flat(const Prob& pr, const Pyr& s, const void* q, const float* pyr, char* ws,
                        int32_t* out_idx, float* out_score, int num_sms, cudaStream_t st);

}  // namespace pisa
