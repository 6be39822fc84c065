// Instances of the register-decode kernel for the formats only it reads: MXINT4, INT8 (e0m7), FP8 E4M3 and
// UINT2 weights (UINT1 / UINT3 in hq_gemm_small_bits.cu); see hq_gemm_small.cuh.
#include "hq_gemm_small.cuh"

namespace hq {

cudaError_t launch_gemm_small_bits(int dec, const GemmArgs& a, int bt, int grid, cudaStream_t stream);

cudaError_t launch_gemm_small_fmt(int dec, const GemmArgs& a, int bt, int grid, cudaStream_t stream) {
  switch (dec) {
    case DEC_MXINT4: return launch_small_dec<DEC_MXINT4>(a, bt, grid, stream);
    case DEC_INT8: return launch_small_dec<DEC_INT8>(a, bt, grid, stream);
    case DEC_E4M3: return launch_small_dec<DEC_E4M3>(a, bt, grid, stream);
    case DEC_UINT2: return launch_small_dec<DEC_UINT2>(a, bt, grid, stream);
    case DEC_UINT1:
    case DEC_UINT3: return launch_gemm_small_bits(dec, a, bt, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace hq
