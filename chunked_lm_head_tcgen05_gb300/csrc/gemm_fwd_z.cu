// Instantiation of the tcgen05 GEMM for the forward logits of the
// single-call path: the forward statistics epilogue that also keeps the
// block's logits (fp16, relative to each tile's running maximum) for the
// backward (A = hidden rows, B = vocabulary rows, both K-major).
#include "tc_gemm.cuh"

namespace lmh {

cudaError_t launch_gemm_fwd_z(const LaunchArgs& a, int grid, bool pair, cudaStream_t s) {
  return pair ? launch_tc_gemm<EPI_FWD_Z, false, true>(a, grid, s)
              : launch_tc_gemm<EPI_FWD_Z, false, false>(a, grid, s);
}

}  // namespace lmh
