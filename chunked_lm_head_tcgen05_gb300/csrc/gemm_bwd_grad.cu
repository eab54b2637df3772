// Instantiation of the tcgen05 GEMM for the two gradient contractions of a
// backward block, run in one launch:
//   problem 0: dh (+)= dz . W_block   (A = dz, K-major over the vocabulary;
//              B = W rows, MN-major; long K, so its units go first)
//   problem 1: dW_block (+)= dz^T . h  (A = dz read column-wise, MN-major;
//              B = hidden rows, MN-major)
#include "tc_gemm.cuh"

namespace lmh {

cudaError_t launch_gemm_bwd_grad(const LaunchArgs& a, int grid, bool pair, cudaStream_t s) {
  return pair ? launch_tc_gemm<EPI_STORE_F32, true, true>(a, grid, s)
              : launch_tc_gemm<EPI_STORE_F32, true, false>(a, grid, s);
}

}  // namespace lmh
