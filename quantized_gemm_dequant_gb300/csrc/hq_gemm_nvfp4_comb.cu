// Kernel instances of the NVFP4 path with the MoE combine epilogue, for every token-tile width.
#include "hq_gemm_kernel.cuh"

namespace hq {

cudaError_t launch_gemm_nvfp4_comb(const GemmArgs& a, int bt, int grid, cudaStream_t stream) {
  return launch_umma<PATH_NVFP4, true>(a, bt, grid, stream);
}

}  // namespace hq
