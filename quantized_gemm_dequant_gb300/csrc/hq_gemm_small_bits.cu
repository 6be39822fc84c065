// Instances of the register-decode kernel for the 1- and 3-bit weights with zero points (UINT1_ZP, UINT3_ZP); see
// hq_gemm_small.cuh.  Kept apart from hq_gemm_small_fmt.cu so that the instances compile in parallel.
#include "hq_gemm_small.cuh"

namespace hq {

cudaError_t launch_gemm_small_bits(int dec, const GemmArgs& a, int bt, int grid, cudaStream_t stream) {
  switch (dec) {
    case DEC_UINT1: return launch_small_dec<DEC_UINT1>(a, bt, grid, stream);
    case DEC_UINT3: return launch_small_dec<DEC_UINT3>(a, bt, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace hq
