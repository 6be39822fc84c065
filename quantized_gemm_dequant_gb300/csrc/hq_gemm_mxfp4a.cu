// Kernel instances of the MXFP4-weight path with MXFP8 activations (e8m0 block scales on both operands of the
// block-scaled MMA), for every token-tile width, with and without the MoE combine epilogue.
#include "hq_gemm_kernel.cuh"

namespace hq {

cudaError_t launch_gemm_mxfp4a(const GemmArgs& a, int bt, int grid, cudaStream_t stream) {
  if (a.comb) return launch_umma<PATH_MXFP4A, true>(a, bt, grid, stream);
  return launch_umma<PATH_MXFP4A, false>(a, bt, grid, stream);
}

}  // namespace hq
