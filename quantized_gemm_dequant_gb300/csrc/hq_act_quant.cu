// Activation quantization: bf16 activations -> the FP8 (e4m3, per-token scale) or NVFP4 operand of the GEMMs.
//
// The deployment chooses the activation type of a quantized layer ("Selecting activation types"): token-wise FP8
// feeds the W4A8 path ("End-to-end inference performance"), NVFP4 the W4A4 path ("W8A8 / W4A8 / W4A4").  The
// scales follow the format definitions with the largest magnitude of each scaled unit mapped to the format's
// largest value:
//   FP8 per token   s_t = absmax_t / 448,            code = e4m3(x / s_t)              (s_t = 0: zero codes)
//   NVFP4           g = amax / (6 * 448),            per 16 elements of a row:
//                   sb = e4m3(amax_b / (6 g)),       d = value(sb) * g,  code = e2m1(x / d)  (d = 0: zero codes)
// Conversions round to nearest even and saturate (e4m3 at 448, e2m1 at 6).  Every step is one IEEE binary32
// operation, because the codes are integer decisions taken on those results; an e2m1 zero is stored as +0, an e4m3
// zero keeps its sign.
//
// Memory-bound kernels: 16-byte loads of 8 bf16, grids in multiples of the SM count, programmatic dependent launch.
// Each division by a scale is taken as a multiplication by the scale's correctly rounded reciprocal plus one FMA
// correction, which yields the correctly rounded quotient (div_by below), so the codes are those of IEEE division.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "hq_act_quant.h"
#include "hq_launch.h"
#include "hq_ptx.cuh"

namespace hq {

namespace {

constexpr int AQ_THREADS = 256;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// two floats -> two e4m3 bytes (lo = a), round to nearest even, saturating
__device__ __forceinline__ uint32_t cvt_e4m3x2(float a, float b) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(b), "f"(a));
  return d;
}

// eight floats -> one word of eight e2m1 codes (code i in nibble i), round to nearest even, saturating; the sign
// of a zero code is kept here (see e2m1x8_clear_neg_zero)
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float (&v)[8]) {
  uint32_t d;
  asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n\t"
      "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
      : "=r"(d)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return d;
}

// -0 codes -> +0, eight at once: a nibble's magnitude m (bits 0-2) is at most 7, so m + 7 sets the nibble's bit 3
// exactly when m != 0 and never carries into the next nibble; that bit then keeps or clears the sign
__device__ __forceinline__ uint32_t e2m1x8_clear_neg_zero(uint32_t w) {
  const uint32_t s = (w & 0x77777777u) + 0x77777777u;
  return w & (s | 0x77777777u);
}

// e4m3 byte (non-negative, finite) -> float, exact
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  uint32_t h;
  asm("{\n\t.reg .b16 t;\n\tmov.b16 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h) : "h"((uint16_t)b));
  return __half2float(__ushort_as_half((uint16_t)(h & 0xFFFFu)));
}

// x / y rounded to nearest even (IEEE binary32) from yi = RN(1 / y): q = RN(x * yi) is faithful, the residual
// x - q * y is exact with one FMA, and RN(q + residual * yi) is the correctly rounded quotient (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990).  Valid
// while the residual stays a normal number: the callers use it only when the scale is at least 2^-100 (every quotient
// that can round to a nonzero code then has |x| >= 2^-110), and take the plain division otherwise.
__device__ __forceinline__ float div_by(float x, float y, float yi) {
  const float q = __fmul_rn(x, yi);
  const float r = __fmaf_rn(-q, y, x);
  return __fmaf_rn(r, yi, q);
}
constexpr float kDivMinScale = 7.8886091e-31f;  // 2^-100

// largest bf16 magnitude of 8 values (4 words), as the 16-bit pattern: finite non-negative bf16 values order like
// their bit patterns, so a SIMD unsigned max of the sign-cleared halves suffices
__device__ __forceinline__ uint32_t bf16x8_absmax_bits(const uint4& v, uint32_t m) {
  m = __vmaxu2(m, v.x & 0x7FFF7FFFu);
  m = __vmaxu2(m, v.y & 0x7FFF7FFFu);
  m = __vmaxu2(m, v.z & 0x7FFF7FFFu);
  m = __vmaxu2(m, v.w & 0x7FFF7FFFu);
  return m;
}
__device__ __forceinline__ float absmax_bits_to_f32(uint32_t m) {
  const uint32_t h = (m & 0xFFFFu) > (m >> 16) ? (m & 0xFFFFu) : (m >> 16);
  return __uint_as_float(h << 16);
}

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red is reused by consecutive calls
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.0f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// 8 bf16 -> 8 e4m3 codes of x / s
__device__ __forceinline__ uint2 quant8_e4m3(const uint4& w, float s, float si, bool fast) {
  float f[8];
  bf16x8_to_f32(w, f);
  uint32_t b[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    b[i] = fast ? cvt_e4m3x2(div_by(f[2 * i], s, si), div_by(f[2 * i + 1], s, si))
                : cvt_e4m3x2(__fdiv_rn(f[2 * i], s), __fdiv_rn(f[2 * i + 1], s));
  return make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
}

// FP8 per token: one CTA per row (grid-stride over rows).  K % 8 == 0.  Rows of at most CH * 256 chunks of 8 are
// read once and kept in registers between the absmax and the quantization (with the CTA's next row in flight);
// longer rows are read twice (the second read hits L1/L2).
template <int CH>
__global__ void __launch_bounds__(AQ_THREADS) act_quant_e4m3_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                                    uint8_t* __restrict__ q, float* __restrict__ s_out) {
  __shared__ float red[AQ_THREADS / 32];
  pdl_trigger();
  pdl_wait();
  const int64_t chunks = K >> 3;
  const bool cached = chunks <= (int64_t)CH * AQ_THREADS;
  // register-cached rows: the CTA's next row is loaded while the current one is reduced and quantized
  uint4 v[CH], nv[CH];
  auto load_row = [&](int64_t row, uint4 (&dst)[CH]) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * K);
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const int64_t c = threadIdx.x + (int64_t)j * AQ_THREADS;
      dst[j] = c < chunks ? __ldg(xr + c) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  if (cached && (int64_t)blockIdx.x < M) load_row(blockIdx.x, v);
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * K);
    const int64_t next = row + gridDim.x;
    uint32_t mb = 0;
    if (cached) {
      if (next < M) load_row(next, nv);
#pragma unroll
      for (int j = 0; j < CH; ++j) mb = bf16x8_absmax_bits(v[j], mb);
    } else {
      for (int64_t c = threadIdx.x; c < chunks; c += AQ_THREADS) mb = bf16x8_absmax_bits(__ldg(xr + c), mb);
    }
    const float amax = block_max(absmax_bits_to_f32(mb), red);
    const float s = __fdiv_rn(amax, 448.0f);
    const float si = __frcp_rn(s);
    const bool fast = s >= kDivMinScale;
    if (threadIdx.x == 0) s_out[row] = s;
    uint2* qr = reinterpret_cast<uint2*>(q + row * K);
    if (cached) {
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        const int64_t c = threadIdx.x + (int64_t)j * AQ_THREADS;
        if (c < chunks) qr[c] = s > 0.0f ? quant8_e4m3(v[j], s, si, fast) : make_uint2(0u, 0u);
        v[j] = nv[j];
      }
    } else {
      for (int64_t c = threadIdx.x; c < chunks; c += AQ_THREADS)
        qr[c] = s > 0.0f ? quant8_e4m3(__ldg(xr + c), s, si, fast) : make_uint2(0u, 0u);
    }
  }
}

// NVFP4, first pass (only without a calibrated amax): largest magnitude, one partial per CTA.
__global__ void __launch_bounds__(AQ_THREADS) act_amax_kernel(const uint16_t* __restrict__ x, int64_t n8,
                                                              float* __restrict__ partial) {
  __shared__ float red[AQ_THREADS / 32];
  pdl_trigger();
  pdl_wait();
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  uint32_t mb[4] = {0u, 0u, 0u, 0u};  // four independent chains: four loads in flight per thread
  const int64_t stride = (int64_t)gridDim.x * AQ_THREADS;
  int64_t c = (int64_t)blockIdx.x * AQ_THREADS + threadIdx.x;
  for (; c + 3 * stride < n8; c += 4 * stride) {
    const uint4 v0 = __ldg(xv + c), v1 = __ldg(xv + c + stride), v2 = __ldg(xv + c + 2 * stride),
                v3 = __ldg(xv + c + 3 * stride);
    mb[0] = bf16x8_absmax_bits(v0, mb[0]);
    mb[1] = bf16x8_absmax_bits(v1, mb[1]);
    mb[2] = bf16x8_absmax_bits(v2, mb[2]);
    mb[3] = bf16x8_absmax_bits(v3, mb[3]);
  }
  for (; c < n8; c += stride) mb[0] = bf16x8_absmax_bits(__ldg(xv + c), mb[0]);
  const uint32_t all = __vmaxu2(__vmaxu2(mb[0], mb[1]), __vmaxu2(mb[2], mb[3]));
  const float m = block_max(absmax_bits_to_f32(all), red);
  if (threadIdx.x == 0) partial[blockIdx.x] = m;
}

// 16 values of one block whose scale is d -> 16 e2m1 codes of x / d (d = 0: zero codes)
__device__ __forceinline__ uint2 quant16_e2m1(const uint4& w0, const uint4& w1, float d) {
  float f0[8], f1[8], v0[8], v1[8];
  bf16x8_to_f32(w0, f0);
  bf16x8_to_f32(w1, f1);
  if (d >= kDivMinScale) {
    const float di = __frcp_rn(d);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v0[i] = div_by(f0[i], d, di);
      v1[i] = div_by(f1[i], d, di);
    }
  } else if (d > 0.0f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v0[i] = __fdiv_rn(f0[i], d);
      v1[i] = __fdiv_rn(f1[i], d);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v0[i] = v1[i] = 0.0f;
  }
  return make_uint2(e2m1x8_clear_neg_zero(cvt_e2m1x8(v0)), e2m1x8_clear_neg_zero(cvt_e2m1x8(v1)));
}

// NVFP4 quantization: one 16-element block per thread and step, a persistent grid (the CTAs the SMs hold at once).
// K % 16 == 0.
__global__ void __launch_bounds__(AQ_THREADS) act_quant_nvfp4_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                                     const float* __restrict__ amax_in,
                                                                     const float* __restrict__ partial, int nparts,
                                                                     uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                                                     float* __restrict__ g_out) {
  __shared__ float red[AQ_THREADS / 32];
  pdl_trigger();
  pdl_wait();
  float amax;
  if (amax_in) {
    amax = *amax_in;
  } else {
    float m = 0.0f;
    for (int i = threadIdx.x; i < nparts; i += AQ_THREADS) m = fmaxf(m, partial[i]);
    amax = block_max(m, red);
  }
  const float g = __fdiv_rn(amax, 2688.0f);  // 6 * 448
  if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = g;
  const float six_g = __fmul_rn(6.0f, g);
  // amax_b / (6 g) through the reciprocal (div_by): a quotient that rounds to a nonzero e4m3 code is above 2^-10, so
  // with 6 g >= 2^-93 its residual is a multiple of 2^-149 and exact; smaller quotients give the zero code either way
  const float six_gi = __frcp_rn(six_g);
  const bool sb_fast = six_g >= 0x1p-93f;
  const int64_t nblk = M * (K >> 4);
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  uint2* qv = reinterpret_cast<uint2*>(q);
  // software-pipelined: the next block's two loads are in flight while this block is quantized
  const int64_t stride = (int64_t)gridDim.x * AQ_THREADS;
  int64_t b = (int64_t)blockIdx.x * AQ_THREADS + threadIdx.x;
  uint4 n0 = make_uint4(0u, 0u, 0u, 0u), n1 = n0;
  if (b < nblk) {
    n0 = __ldg(xv + 2 * b);
    n1 = __ldg(xv + 2 * b + 1);
  }
  for (; b < nblk; b += stride) {
    const uint4 w0 = n0, w1 = n1;
    if (b + stride < nblk) {
      n0 = __ldg(xv + 2 * (b + stride));
      n1 = __ldg(xv + 2 * (b + stride) + 1);
    }
    const float mb = absmax_bits_to_f32(bf16x8_absmax_bits(w1, bf16x8_absmax_bits(w0, 0u)));
    uint32_t sb = 0;
    float d = 0.0f;
    if (g > 0.0f) {
      sb = cvt_e4m3x2(sb_fast ? div_by(mb, six_g, six_gi) : __fdiv_rn(mb, six_g), 0.0f) & 0xFFu;
      d = __fmul_rn(e4m3_to_f32(sb), g);
    }
    qv[b] = quant16_e2m1(w0, w1, d);
    sf[b] = (uint8_t)sb;
  }
}

int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n < 1) n = 1;
  }
  return n;
}

// CTAs of a kernel that all SMs hold at once (its resident capacity)
template <typename Kernel>
int64_t resident_ctas(Kernel kernel) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, AQ_THREADS, 0) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  return (int64_t)per_sm * sm_count();
}

}  // namespace

// CTAs of the NVFP4 amax pass: one float of workspace each, at most ACT_AMAX_MAX_PARTS; no more than the SMs hold
// at once, so that every CTA reads its share in one wave.
int act_amax_grid(int64_t M, int64_t K) {
  static const int64_t resident = resident_ctas(act_amax_kernel);
  const int64_t n8 = M * (K >> 3);
  const int64_t want = (n8 + AQ_THREADS * 8 - 1) / (AQ_THREADS * 8);  // about 8 chunks per thread
  int64_t cap = resident;
  if (cap > ACT_AMAX_MAX_PARTS) cap = ACT_AMAX_MAX_PARTS;
  return (int)(want < 1 ? 1 : (want < cap ? want : cap));
}

cudaError_t launch_act_quant(int fp8, const void* x, int64_t M, int64_t K, const float* global_amax,
                             void* data, void* scale, float* gscale, void* workspace, cudaStream_t stream) {
  const int sms = sm_count();
  if (fp8) {
    const int64_t grid = M < 8 * (int64_t)sms ? M : 8 * (int64_t)sms;
    return launch_kernel(act_quant_e4m3_kernel<4>, dim3((unsigned)grid), dim3(AQ_THREADS), 0, stream,
                         (const uint16_t*)x, M, K, (uint8_t*)data, (float*)scale);
  }
  int nparts = 0;
  float* partial = reinterpret_cast<float*>(workspace);
  if (!global_amax) {
    nparts = act_amax_grid(M, K);
    cudaError_t e = launch_kernel(act_amax_kernel, dim3((unsigned)nparts), dim3(AQ_THREADS), 0, stream,
                                  (const uint16_t*)x, M * (K >> 3), partial);
    if (e != cudaSuccess) return e;
  }
  static const int64_t resident = resident_ctas(act_quant_nvfp4_kernel);
  const int64_t nblk = M * (K >> 4);
  int64_t grid = (nblk + AQ_THREADS - 1) / AQ_THREADS;
  if (grid > resident) grid = resident;
  if (grid < 1) grid = 1;
  return launch_kernel(act_quant_nvfp4_kernel, dim3((unsigned)grid), dim3(AQ_THREADS), 0, stream, (const uint16_t*)x, M,
                       K, global_amax, (const float*)partial, nparts, (uint8_t*)data, (uint8_t*)scale, gscale);
}

}  // namespace hq
