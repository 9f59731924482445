#include "pisa_common.cuh"
#include "pisa_internal.h"
namespace pisa {
cudaError_t launch_decode(const Prob&, const Pyr&, const void*, const void*, const int32_t*, float*, int32_t*,
                          int32_t*, float*, int32_t*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace pisa
