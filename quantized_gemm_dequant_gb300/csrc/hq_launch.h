// Kernel launch with programmatic stream serialization (programmatic dependent launch).
//
// A kernel launched this way may be scheduled while the previous kernel of the stream is still running;
// every kernel of this library therefore executes pdl_wait() before its first access to global memory that
// a previous kernel could write (activations, routing tables, workspace, outputs).  Packed weights are
// read-only inputs: the dense GEMM kernels start copying them before the wait.  They must therefore be
// complete when the kernel before the call allows its dependents to launch; kernels that never execute
// griddepcontrol.launch_dependents (the repack kernel, ordinary kernels) allow it only when they finish.
// HQ_PDL=0 in the environment turns the attribute off (plain stream order).
#pragma once
#include <cuda_runtime.h>
#include <stdlib.h>
#include <string.h>

namespace hq {

inline bool pdl_enabled() {
  static const int on = [] {
    const char* v = getenv("HQ_PDL");
    return (v && !strcmp(v, "0")) ? 0 : 1;
  }();
  return on != 0;
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                 Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace hq
