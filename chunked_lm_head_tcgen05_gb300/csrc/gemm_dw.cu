// Instantiation of the tcgen05 GEMM for the d_weight GEMM dW_block = dz^T . h (A = dz read column-wise, MN-major; B = hidden rows, MN-major).
#include "tc_gemm.cuh"

namespace lmh {

cudaError_t launch_gemm_dw(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& p,
                               int grid, cudaStream_t s) {
  return launch_tc_gemm<EPI_STORE_F32, true, true>(a, b, p, grid, s);
}

}  // namespace lmh
