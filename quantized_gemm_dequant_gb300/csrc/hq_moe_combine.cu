// MoE layer pieces around the grouped GEMMs: the combine's final rounding and the SwiGLU between gate-up and down.
//
// The MoE speed-ups of the Humming announcement count the Gate-up and the Down GEMM of a layer ("Results: kernel
// microbenchmarks").  Between them the gated activation turns the gate and up halves of every routed row into one
// row, out = silu(gate) * up; after the Down GEMM the k routed rows of a token are summed with their top-k weights
// (the GEMM epilogue adds them into an fp32 row per token; the kernel here rounds that row to bf16).
// Memory-bound elementwise kernels: 16-byte accesses, grid-stride loops sized in multiples of the SM count,
// programmatic dependent launch.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "hq_launch.h"
#include "hq_ptx.cuh"

namespace hq {

namespace {

constexpr int EW_THREADS = 256;

__device__ __forceinline__ uint32_t bf16x2_rn(float a, float b) {  // lo = a, round to nearest even
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(b), "f"(a));
  return d;
}

// C[i] = bf16(acc[i]) for i < n (n % 4 == 0: 16-byte loads, 8-byte stores)
__global__ void __launch_bounds__(EW_THREADS) combine_round_kernel(const float* __restrict__ acc, int64_t n4,
                                                                   uint16_t* __restrict__ c) {
  pdl_trigger();
  pdl_wait();  // the sums come from the GEMM (and its split-K reduction)
  const float4* a4 = reinterpret_cast<const float4*>(acc);
  uint2* c4 = reinterpret_cast<uint2*>(c);
  for (int64_t i = (int64_t)blockIdx.x * EW_THREADS + threadIdx.x; i < n4; i += (int64_t)gridDim.x * EW_THREADS) {
    const float4 v = __ldcs(a4 + i);
    c4[i] = make_uint2(bf16x2_rn(v.x, v.y), bf16x2_rn(v.z, v.w));
  }
}

// out[r, c] = bf16(silu(g) * u), g = x[r, c], u = x[r, I + c]; silu(g) = g / (1 + exp(-g)) in fp32.  I % 8 == 0.
__global__ void __launch_bounds__(EW_THREADS) swiglu_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t I,
                                                            uint16_t* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int64_t per_row = I >> 3;
  const int64_t n8 = R * per_row;
  for (int64_t i = (int64_t)blockIdx.x * EW_THREADS + threadIdx.x; i < n8; i += (int64_t)gridDim.x * EW_THREADS) {
    // 32-bit division when it fits (the 64-bit one is a long software routine)
    const int64_t r = n8 < (int64_t(1) << 32) ? (int64_t)((uint32_t)i / (uint32_t)per_row) : i / per_row;
    const int64_t c = (i - r * per_row) << 3;
    const uint4 g = __ldcs(reinterpret_cast<const uint4*>(x + r * 2 * I + c));
    const uint4 u = __ldcs(reinterpret_cast<const uint4*>(x + r * 2 * I + I + c));
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float y[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float gv = __uint_as_float(h ? (gw[k] & 0xFFFF0000u) : (gw[k] << 16));
        const float uv = __uint_as_float(h ? (uw[k] & 0xFFFF0000u) : (uw[k] << 16));
        y[h] = __fmul_rn(__fdiv_rn(gv, __fadd_rn(1.0f, expf(-gv))), uv);
      }
      o[k] = bf16x2_rn(y[0], y[1]);
    }
    *reinterpret_cast<uint4*>(out + r * I + c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

int ew_grid(int64_t items) {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms < 1) sms = 1;
  }
  const int64_t want = (items + EW_THREADS - 1) / EW_THREADS;
  const int64_t cap = 8 * (int64_t)sms;
  return (int)(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

cudaError_t launch_combine_round(const float* acc, int64_t n, uint16_t* c, cudaStream_t stream) {
  return launch_kernel(combine_round_kernel, dim3((unsigned)ew_grid(n / 4)), dim3(EW_THREADS), 0, stream, acc, n / 4,
                       c);
}

cudaError_t launch_swiglu(const void* x, int64_t R, int64_t I, void* out, cudaStream_t stream) {
  return launch_kernel(swiglu_kernel, dim3((unsigned)ew_grid(R * (I / 8))), dim3(EW_THREADS), 0, stream,
                       (const uint16_t*)x, R, I, (uint16_t*)out);
}

}  // namespace hq
