// leaf_tc.cu -- (placeholder while the tensor-core leaf kernel is written)
#include "pisa_common.cuh"
#include "pisa_internal.h"
namespace pisa {
cudaError_t launch_leaf_tc(const Prob& pr, const Pyr& s, const PrefillWs& w, char* ws, const void* q,
                           const void* k, int32_t* out_idx, float* out_score, int, cudaStream_t st) {
  return launch_leaf_simt(pr, s, q, k, (const int32_t*)(ws + w.kept2), out_idx, out_score, st);
}
}  // namespace pisa
