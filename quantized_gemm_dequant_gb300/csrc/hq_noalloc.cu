// Dense GEMM entry point that needs no caller-provided workspace.
//
// Its scratch (device status word, Stream-K partial sums)
// lives in one file-scope device array of HQ_STATIC_SCRATCH_BYTES that every
// GPU loading this library keeps until the process exits.  The call itself
// allocates nothing.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/hq.h"

namespace {

constexpr size_t kScratchBytes = HQ_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Shared by every call on a device; holds the last call's contents.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Device address of g_scratch, looked up once per device with that device
// current (the host-side name of a __device__ array is only a stand-in and must
// never reach a kernel).  Host threads making their first call on a device at
// the same time may both look it up; they store the same address.
std::atomic<void*> g_scratch_ptr[kMaxDevices];

hq_status_t scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HQ_ERR_CUDA;
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return HQ_ERR_CUDA;
    g_scratch_ptr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return HQ_OK;
}

}  // namespace

extern "C" {

hq_status_t hq_gemm_static_scratch(const hq_format_t* fmt, const hq_act_t* A, const void* packedW, const void* bias,
                                   void* C, int64_t M, int64_t N, int64_t K, hq_stream_t stream) {
  if (!fmt || M < 0 || N < 1) return HQ_ERR_INVALID_ARG;
  if (M == 0) return HQ_OK;
  const size_t need = hq_workspace_bytes(fmt, M, 1);
  if (need == 0) return HQ_ERR_INVALID_ARG;
  if (need > kScratchBytes) return HQ_ERR_WORKSPACE;  // beyond the fixed scratch: use hq_gemm with a workspace
  void* ws = nullptr;
  const hq_status_t st = scratch_address(&ws);
  if (st != HQ_OK) return st;
  // The status word (the first 4 bytes) must start at zero.  The rest of the header (the epoch of the last
  // register-decode call and its exit count) carries over from call to call, as it does in a caller's workspace;
  // the array starts zeroed when the library's device code is loaded.
  if (cudaMemsetAsync(ws, 0, sizeof(int32_t), (cudaStream_t)stream) != cudaSuccess) return HQ_ERR_CUDA;
  return hq_gemm(fmt, A, packedW, bias, C, M, N, K, ws, kScratchBytes, stream);
}

}  // extern "C"
