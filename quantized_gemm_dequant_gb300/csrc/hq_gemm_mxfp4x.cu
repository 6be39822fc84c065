// Kernel instances of MXFP4 weights with MXFP4 activations (packed e2m1 on both operands, e8m0 block scales on both
// operands of kind::mxf4nvf4 scale_vec::2X), for every token-tile width; the combine instances are in
// hq_gemm_mxfp4x_comb.cu, compiled in parallel.
#include "hq_gemm_kernel.cuh"

namespace hq {

cudaError_t launch_gemm_mxfp4x_comb(const GemmArgs& a, int bt, int grid, cudaStream_t stream);

cudaError_t launch_gemm_mxfp4x(const GemmArgs& a, int bt, int grid, cudaStream_t stream) {
  if (a.comb) return launch_gemm_mxfp4x_comb(a, bt, grid, stream);
  return launch_umma<PATH_MXFP4X, false>(a, bt, grid, stream);
}

}  // namespace hq
