// Instantiation of the tcgen05 GEMM for the forward logits with the online
// log-sum-exp / entropy / target epilogue (A = hidden rows, B = vocabulary
// rows, both K-major).
#include "tc_gemm.cuh"

namespace lmh {

cudaError_t launch_gemm_fwd_stats(const LaunchArgs& a, int grid, bool pair, cudaStream_t s) {
  return pair ? launch_tc_gemm<EPI_FWD_STATS, false, true>(a, grid, s)
              : launch_tc_gemm<EPI_FWD_STATS, false, false>(a, grid, s);
}

}  // namespace lmh
