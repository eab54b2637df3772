// Instantiation of the tcgen05 GEMM for the backward logit recompute with
// the dz epilogue (A = hidden rows, B = vocabulary rows, both K-major).
#include "tc_gemm.cuh"

namespace lmh {

cudaError_t launch_gemm_bwd_dz(const LaunchArgs& a, int grid, bool pair, cudaStream_t s) {
  return pair ? launch_tc_gemm<EPI_BWD_DZ, false, true>(a, grid, s)
              : launch_tc_gemm<EPI_BWD_DZ, false, false>(a, grid, s);
}

}  // namespace lmh
