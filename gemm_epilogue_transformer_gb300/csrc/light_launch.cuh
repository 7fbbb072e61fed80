// Launch of the auxiliary reductions with programmatic dependent launch, the
// same overlap the GEMMs use: a kernel launched here may be scheduled while
// the previous kernel on its stream is still running, so its launch latency
// and block scheduling hide behind that kernel's tail.
//
// Contract for every kernel launched through launch_light(): its first
// statement is light_kernel_enter(). That lets the next kernel on the stream
// be scheduled (it will in turn block in its own wait), then blocks until the
// previous kernel has completed and its writes are visible. Nothing is read
// or written before the wait, so the ordering on the stream is the same as
// with a plain launch; each kernel in a chain completes only after its
// predecessor has, so a later kernel also sees every earlier kernel's writes.
//
// Only the small reductions use it. The large HBM-bound kernels (the RoPE-path
// glue, the unfused element-wise kernels) keep plain launches: launched this
// way their blocks sit resident beside the previous GEMM's CTAs, and measured
// on GB300 they then ran 1-3 % slower, more than the launch latency saved.
#pragma once

#include <cuda_runtime.h>

#include "ptx.cuh"

namespace coda {

__device__ __forceinline__ void light_kernel_enter() {
  griddep_launch_dependents();
  griddep_wait();
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_light(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace coda
