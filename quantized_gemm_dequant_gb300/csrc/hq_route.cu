// MoE routing: group the T*topk routed rows by expert.
//
// Each block takes 1024 consecutive flat rows (t*topk + j), ranks them per
// expert in shared memory, reserves a range of each expert's row list with one
// global atomic per (block, expert) and scatters the flat row ids into it.
// The order of rows inside an expert is not fixed, which changes only which
// rows share a token tile, never a row's value.
#include <cuda_runtime.h>
#include <stdint.h>

namespace hq {

constexpr int ROUTE_ROWS = 1024;
constexpr int kErrBadRouting = 6;

__global__ void __launch_bounds__(256) route_kernel(const int32_t* __restrict__ ids, int64_t rows, int E, int cap,
                                                    int* __restrict__ counts, int* __restrict__ region,
                                                    int* __restrict__ status) {
  extern __shared__ int sh[];  // hist[E], base[E]
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
  route_kernel<<<(unsigned)blocks, 256, 2 * E * sizeof(int), stream>>>(ids, rows, E, cap, counts, region, status);
  return cudaGetLastError();
}

}  // namespace hq
