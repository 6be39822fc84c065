// Instances of the register-decode kernel for the 4-bit integer formats (INT4_SYM, UINT4_ZP); see
// hq_gemm_small.cuh.
#include "hq_gemm_small.cuh"

namespace hq {

cudaError_t launch_gemm_small(const GemmArgs& a, int bt, int grid, cudaStream_t stream) {
  return launch_small_dec<DEC_INT4>(a, bt, grid, stream);
}

}  // namespace hq
