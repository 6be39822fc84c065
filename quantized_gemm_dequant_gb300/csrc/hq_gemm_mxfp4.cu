// Kernel instances of the MXFP4 path for every token-tile width (the combine instances are in
// hq_gemm_mxfp4_comb.cu, compiled in parallel).
#include "hq_gemm_kernel.cuh"

namespace hq {

cudaError_t launch_gemm_mxfp4_comb(const GemmArgs& a, int bt, int grid, cudaStream_t stream);

cudaError_t launch_gemm_mxfp4(const GemmArgs& a, int bt, int grid, cudaStream_t stream) {
  if (a.comb) return launch_gemm_mxfp4_comb(a, bt, grid, stream);
  return launch_umma<PATH_MXFP4, false>(a, bt, grid, stream);
}

}  // namespace hq
