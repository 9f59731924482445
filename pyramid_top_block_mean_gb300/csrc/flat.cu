#include "pisa_common.cuh"
#include "pisa_internal.h"
namespace pisa {
cudaError_t launch_flat(const Prob&, const Pyr&, const void*, const float*, char*, int32_t*, float*, int,
                        cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace pisa
