// Instantiation of the tcgen05 GEMM for the d_hidden GEMM dh = dz . W_block (A = dz, K-major over the vocabulary; B = W rows, MN-major).
#include "tc_gemm.cuh"

namespace lmh {

cudaError_t launch_gemm_dh(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& p,
                               int grid, cudaStream_t s) {
  return launch_tc_gemm<EPI_STORE_F32, false, true>(a, b, p, grid, s);
}

}  // namespace lmh
