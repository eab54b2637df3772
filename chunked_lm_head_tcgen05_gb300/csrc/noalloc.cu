// lmhead_logps_fwd_noalloc: the forward with its scratch in a static device
// array instead of a caller-provided workspace, for callers that cannot
// allocate device memory (see include/lmhead.h).
#include "lmhead.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

namespace {

// The forward's scratch on every GPU that loads this library.  In host code
// this name is only a stand-in for the symbol; its device address comes from
// cudaGetSymbolAddress with the device (and context) in question current.
static __device__ __align__(256) unsigned char g_noalloc_scratch[LMHEAD_NOALLOC_SCRATCH_BYTES];

// The address belongs to the context the module was loaded into, so it is
// cached per (device, current context): a driver-API context made current on
// the same device, or the primary context created anew after a device reset,
// gets its own lookup.
constexpr int kMaxDevices = 64;
struct Cached {
  CUcontext ctx;
  void* ptr;
};
Cached g_scratch[kMaxDevices] = {};
std::mutex g_scratch_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of the scratch in the current context.  The first lookup in a
// context loads this file's module there if it is not loaded yet (with lazy
// module loading, CUDA's default, that is when the array's memory is taken);
// a failure, such as too little free device memory for the array, returns
// LMHEAD_ERR_CUDA.
lmhead_status scratch_in_current_context(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return LMHEAD_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LMHEAD_ERR_UNSUPPORTED;
  CtxGetCurrentFn get = ctx_get_current();
  if (!get) return LMHEAD_ERR_CUDA;
  CUcontext ctx = nullptr;   // NULL until the runtime has made a context current here
  if (get(&ctx) != CUDA_SUCCESS) return LMHEAD_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  Cached& c = g_scratch[dev];
  if (ctx == nullptr || c.ptr == nullptr || c.ctx != ctx) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();   // do not leave the failure for the caller's next check
      return LMHEAD_ERR_CUDA;
    }
    // the lookup made the device's primary context current if none was
    if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return LMHEAD_ERR_CUDA;
    c.ctx = ctx;
    c.ptr = p;
  }
  *out = c.ptr;
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
  void* scratch = nullptr;
  const lmhead_status rc = scratch_in_current_context(&scratch);
  if (rc != LMHEAD_OK) return rc;
  // lmhead_logps_fwd runs its usual checks in its usual order (sizes, pointers,
  // alignment) and then compares the workspace it needs with the array's size,
  // returning LMHEAD_ERR_WORKSPACE_TOO_SMALL before launching anything when the
  // sizes need more.  It clears the device status word and rewrites every
  // scratch region it reads (compacted rows including their zero padding,
  // targets, partial statistics) before reading it, so nothing an earlier call
  // left in the array is ever used.
  return lmhead_logps_fwd(hidden, weight, targets, loss_mask, T, H, V, temperature, chunk_size,
                          logp, entropy, lse, scratch, LMHEAD_NOALLOC_SCRATCH_BYTES, stream);
}
