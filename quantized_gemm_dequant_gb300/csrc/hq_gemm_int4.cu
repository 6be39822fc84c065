// Kernel instances of the INT4 path for every token-tile width.
#include "hq_gemm_kernel.cuh"
#include "hq_launch.h"

namespace hq {

template <int BT>
static cudaError_t launch_bt(const GemmArgs& a, int grid, cudaStream_t stream) {
  using C = Cfg<PATH_INT4, BT>;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(hq_gemm_kernel<PATH_INT4, BT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = 1;
  }
  return launch_kernel(hq_gemm_kernel<PATH_INT4, BT>, dim3(grid), dim3(NUM_THREADS), C::SMEM_BYTES, stream, a);
}

cudaError_t launch_gemm_int4(const GemmArgs& a, int bt, int grid, cudaStream_t stream) {
  switch (bt) {
    case 16: return launch_bt<16>(a, grid, stream);
    case 32: return launch_bt<32>(a, grid, stream);
    case 64: return launch_bt<64>(a, grid, stream);
    case 128: return launch_bt<128>(a, grid, stream);
    case 256: return launch_bt<256>(a, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace hq
