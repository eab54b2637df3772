// Instantiation of the tcgen05 GEMM for the forward logits GEMM with the online log-sum-exp / entropy / target epilogue (A = hidden rows, B = vocabulary rows, both K-major).
#include "tc_gemm.cuh"

namespace lmh {

cudaError_t launch_gemm_fwd_stats(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& p,
                               int grid, cudaStream_t s) {
  return launch_tc_gemm<EPI_FWD_STATS, false, false>(a, b, p, grid, s);
}

}  // namespace lmh
