// static_scratch.cu -- pisa_select_prefill_static: the prefill selection for
// callers that cannot allocate device memory, e.g. code running inside a
// host callback or a plug-in of a runtime that owns every device allocation
// and forbids cudaMalloc / framework allocators in its execution path.  The
// workspace lives in one fixed file-scope device array instead of caller
// memory.  The pages about the method have no counterpart for this: it is a
// deployment convenience only.
//
// The array is kStaticScratchBytes (64 MiB) on every GPU that loads this
// library, held until the process exits.  Its host-side name is only a
// stand-in: host code must use the device address from cudaGetSymbolAddress,
// fetched once per device on that device's first call (with the device
// current) and cached.
#include <mutex>

#include "pisa_common.cuh"
#include "pisa_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = (size_t)64 << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_prefill_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {nullptr};

// Device address of g_prefill_scratch on the current device (looked up once).
pisa_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PISA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_prefill_scratch) != cudaSuccess || !p) return PISA_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return PISA_OK;
}

}  // namespace

extern "C" pisa_status pisa_select_prefill_static(const pisa_params* p, const void* q, const void* k,
                                                  const float* pyramid, int32_t* out_idx, float* out_score,
                                                  void* stream) {
  const size_t need = pisa_workspace_bytes(p, PISA_MODE_PREFILL);
  if (need == 0) {
    // bad parameters, or an empty problem that needs no workspace
    return pisa_select_prefill(p, q, k, pyramid, nullptr, 0, out_idx, out_score, nullptr, stream);
  }
  if (need > kStaticScratchBytes) return PISA_ERR_WORKSPACE;
  void* ws = nullptr;
  const pisa_status rc = scratch_address(&ws);
  if (rc != PISA_OK) return rc;
  // The regular path clears the status word and the bucket counters itself;
  // everything else in the workspace is fully rewritten by every call.
  return pisa_select_prefill(p, q, k, pyramid, ws, kStaticScratchBytes, out_idx, out_score, nullptr, stream);
}

extern "C" pisa_status pisa_read_static_status(int32_t* device_code, void* stream) {
  if (!device_code) return PISA_ERR_INVALID_ARG;
  void* ws = nullptr;
  const pisa_status rc = scratch_address(&ws);
  if (rc != PISA_OK) return rc;
  // the status word is the first 256 bytes of the array, as in any workspace
  return pisa_read_device_status(ws, device_code, stream);
}
