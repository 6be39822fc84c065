// Activation quantization launch interface (kernels in hq_act_quant.cu).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace hq {

// Largest number of partial maxima of the NVFP4 amax pass; the workspace holds one fp32 per partial.
constexpr int ACT_AMAX_MAX_PARTS = 4096;

// bf16 x [M, K] (K % 16 == 0, 16-byte aligned) -> e4m3 [M, K] + fp32 [M] (fp8 != 0), or packed e2m1 [M, K/2] +
// ue4m3 [M, K/16] + fp32 g (NVFP4; global_amax: calibrated amax or null, then the workspace holds the partials).
cudaError_t launch_act_quant(int fp8, const void* x, int64_t M, int64_t K, const float* global_amax, void* data,
                             void* scale, float* gscale, void* workspace, cudaStream_t stream);

// Kernels one call launches (host-only).
inline int act_quant_kernels(int fp8, const float* global_amax) { return fp8 ? 1 : (global_amax ? 1 : 2); }

}  // namespace hq
