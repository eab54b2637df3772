// Self-test of the bounded-wait path the GEMM kernels rely on: a CTA
// allocates TMEM, waits with the GEMMs' wait routine on an mbarrier that
// nothing ever arrives on, gives up after a short limit, records the
// timeout in the status word, frees TMEM and exits.  No fault, trap or
// unbounded spin is involved; the context stays usable afterwards.
#include "tc_gemm.cuh"

namespace lmh {
namespace {

__global__ void __launch_bounds__(64, 1) bounded_wait_selftest_kernel(int* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);   // expects one arrival that never comes
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&tmem_base), 32);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (threadIdx.x == 0) wait_bounded(smem_addr(&bar), 0, &abort_flag, status, limit_ns);
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 32);
  }
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t s) {
  bounded_wait_selftest_kernel<<<1, 64, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace lmh
