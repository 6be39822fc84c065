// Kernel instances of the MXFP4 x MXFP4 path with the MoE combine epilogue, for every token-tile width.
#include "hq_gemm_kernel.cuh"

namespace hq {

cudaError_t launch_gemm_mxfp4x_comb(const GemmArgs& a, int bt, int grid, cudaStream_t stream) {
  return launch_umma<PATH_MXFP4X, true>(a, bt, grid, stream);
}

}  // namespace hq
