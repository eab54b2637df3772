// Instantiation of the tcgen05 GEMM for the backward logit recompute with
// the dz epilogue (A = hidden rows, B = vocabulary rows, both K-major).
#include "tc_gemm.cuh"

namespace lmh {

cudaError_t launch_gemm_bwd_dz(const LaunchArgs& a, int grid, cudaStream_t s) {
  return launch_tc_gemm<EPI_BWD_DZ, false>(a, grid, s);
}

}  // namespace lmh
