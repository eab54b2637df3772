// lmhead_logps_fwd_noalloc: the forward with its scratch in a static device
// array instead of a caller-provided workspace, for callers that cannot
// allocate device memory (see include/lmhead.h).
#include "lmhead.h"

#include <cuda_runtime.h>

#include <mutex>

namespace {

// The forward's scratch on every GPU that loads this library.  In host code
// this name is only a stand-in for the symbol; its device address comes from
// cudaGetSymbolAddress on the device in question.
static __device__ __align__(256) unsigned char g_noalloc_scratch[LMHEAD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch on the current device; looked up once per
// device, with that device current.
lmhead_status scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return LMHEAD_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LMHEAD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return LMHEAD_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return LMHEAD_OK;
}

}  // namespace

extern "C" lmhead_status lmhead_logps_fwd_noalloc(const uint16_t* hidden, const uint16_t* weight,
                                                  const int32_t* targets,
                                                  const uint8_t* loss_mask, int64_t T, int32_t H,
                                                  int32_t V, float temperature,
                                                  int32_t chunk_size, float* logp,
                                                  float* entropy, float* lse,
                                                  lmhead_stream_t stream) {
  const size_t need = lmhead_workspace_size(LMHEAD_OP_FWD, T, H, V, chunk_size);
  if (need == 0 || T == 0) {
    // invalid sizes (reported with lmhead_logps_fwd's own codes) or no tokens
    return lmhead_logps_fwd(hidden, weight, targets, loss_mask, T, H, V, temperature, chunk_size,
                            logp, entropy, lse, nullptr, 0, stream);
  }
  if (need > LMHEAD_NOALLOC_SCRATCH_BYTES) return LMHEAD_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const lmhead_status rc = scratch_on_current_device(&scratch);
  if (rc != LMHEAD_OK) return rc;
  // The forward clears the device status word and rewrites every scratch
  // region it reads (compacted rows including their zero padding, targets,
  // partial statistics) before reading it, so nothing left by an earlier
  // call is ever used.
  return lmhead_logps_fwd(hidden, weight, targets, loss_mask, T, H, V, temperature, chunk_size,
                          logp, entropy, lse, scratch, LMHEAD_NOALLOC_SCRATCH_BYTES, stream);
}
