// MoE routing: group the T*topk routed rows by expert.
//
// Each block takes 1024 consecutive flat rows (t*topk + j), ranks them per
// expert in shared memory, reserves a range of each expert's row list with one
// global atomic per (block, expert) and scatters the flat row ids into it.
// The order of rows inside an expert is not fixed, which changes only which
// rows share a token tile, never a row's value.
#include <cuda_runtime.h>
#include <stdint.h>

#include "hq_launch.h"
#include "hq_ptx.cuh"

namespace hq {

constexpr int ROUTE_ROWS = 1024;
constexpr int kErrBadRouting = 6;

__global__ void __launch_bounds__(256) route_kernel(const int32_t* __restrict__ ids, int64_t rows, int E, int cap,
                                                    int* __restrict__ counts, int* __restrict__ region,
                                                    int* __restrict__ status) {
  extern __shared__ int sh[];  // hist[E], base[E]
  pdl_trigger();
  pdl_wait();  // ids may come from the previous kernel
  int* hist = sh;
  int* base = sh + E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t r0 = (int64_t)blockIdx.x * ROUTE_ROWS;
  int id[ROUTE_ROWS / 256], local[ROUTE_ROWS / 256];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < ROUTE_ROWS / 256; ++i) {
    const int64_t r = r0 + i * 256 + threadIdx.x;
    id[i] = -1;
    if (r < rows) {
      const int v = ids[r];
      if (v >= 0 && v < E) {
        id[i] = v;
        local[i] = atomicAdd(&hist[v], 1);
      } else {
        bad = true;
      }
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) base[e] = hist[e] ? atomicAdd(&counts[e], hist[e]) : 0;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < ROUTE_ROWS / 256; ++i) {
    if (id[i] < 0) continue;
    const int pos = base[id[i]] + local[i];
    if (pos < cap) region[(int64_t)id[i] * cap + pos] = (int)(r0 + i * 256 + threadIdx.x);
    else bad = true;
  }
  if (bad) atomicCAS(status, 0, kErrBadRouting);
}

cudaError_t launch_route(const int32_t* ids, int64_t rows, int E, int cap, int* counts, int* region, int* status,
                         cudaStream_t stream) {
  cudaError_t err = cudaMemsetAsync(counts, 0, sizeof(int) * (size_t)E, stream);
  if (err != cudaSuccess) return err;
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = (rows + ROUTE_ROWS - 1) / ROUTE_ROWS;
  // plain stream order after the memset above
  route_kernel<<<(unsigned)blocks, 256, 2 * E * sizeof(int), stream>>>(ids, rows, E, cap, counts, region, status);
  return cudaGetLastError();
}

}  // namespace hq

namespace hq {

// "Grouped" MoE activations: copy the routed rows into expert-contiguous order
// (rows of expert e at row_off[e] .. row_off[e] + counts[e]) so that the GEMM
// can load them with plain 2-D boxes.  Every block recomputes the expert row
// offsets from the counts (E <= 512); block 0 publishes them in row_off[0..E].
constexpr int PERMUTE_ROWS = 16;

__global__ void __launch_bounds__(256) moe_permute_kernel(const int* __restrict__ counts, const int* __restrict__ region,
                                                          int cap, int E, int topk, const uint8_t* __restrict__ src,
                                                          int row_bytes, uint8_t* __restrict__ dst,
                                                          const uint8_t* __restrict__ sf_src, int sf_bytes,
                                                          uint8_t* __restrict__ sf_dst, int* __restrict__ row_off) {
  __shared__ int off[513];
  __shared__ int src_row[PERMUTE_ROWS];
  const int tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();  // counts and region come from the routing kernel
  // exclusive scan of the clamped counts (two entries per thread)
  __shared__ int part[256];
  int c0 = 0, c1 = 0;
  if (2 * tid < E) c0 = min(max(counts[2 * tid], 0), cap);
  if (2 * tid + 1 < E) c1 = min(max(counts[2 * tid + 1], 0), cap);
  part[tid] = c0 + c1;
  __syncthreads();
  for (int o = 1; o < 256; o <<= 1) {
    const int v = tid >= o ? part[tid - o] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  const int excl = part[tid] - (c0 + c1);
  if (2 * tid < E) off[2 * tid] = excl;
  if (2 * tid + 1 < E) off[2 * tid + 1] = excl + c0;
  if (tid == 255) off[E] = part[255];
  __syncthreads();
  if (blockIdx.x == 0)
    for (int e = tid; e <= E; e += 256) row_off[e] = off[e];
  const int total = off[E];
  const int d0 = blockIdx.x * PERMUTE_ROWS;
  if (tid < PERMUTE_ROWS) {
    const int d = d0 + tid;
    int s = -1;
    if (d < total) {
      int lo = 0, hi = E;  // off[lo] <= d < off[lo + 1]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (off[mid] <= d) lo = mid;
        else hi = mid;
      }
      s = region[(int64_t)lo * cap + (d - off[lo])] / topk;
    }
    src_row[tid] = s;
  }
  __syncthreads();
  const int chunks = row_bytes / 16;
  for (int idx = tid; idx < PERMUTE_ROWS * chunks; idx += 256) {
    const int r = idx / chunks, c = idx % chunks;
    const int s = src_row[r];
    if (s < 0) continue;
    reinterpret_cast<uint4*>(dst + (int64_t)(d0 + r) * row_bytes)[c] =
        reinterpret_cast<const uint4*>(src + (int64_t)s * row_bytes)[c];
  }
  if (sf_dst) {
    const int sfc = sf_bytes / 16;
    for (int idx = tid; idx < PERMUTE_ROWS * sfc; idx += 256) {
      const int r = idx / sfc, c = idx % sfc;
      const int s = src_row[r];
      if (s < 0) continue;
      reinterpret_cast<uint4*>(sf_dst + (int64_t)(d0 + r) * sf_bytes)[c] =
          reinterpret_cast<const uint4*>(sf_src + (int64_t)s * sf_bytes)[c];
    }
  }
}

cudaError_t launch_moe_permute(const int* counts, const int* region, int cap, int E, int topk, int64_t rows,
                               const void* src, int row_bytes, void* dst, const void* sf_src, int sf_bytes, void* sf_dst,
                               int* row_off, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = (rows + PERMUTE_ROWS - 1) / PERMUTE_ROWS;
  return launch_kernel(moe_permute_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, counts, region, cap, E, topk,
                       (const uint8_t*)src, row_bytes, (uint8_t*)dst, (const uint8_t*)sf_src, sf_bytes, (uint8_t*)sf_dst,
                       row_off);
}

}  // namespace hq
