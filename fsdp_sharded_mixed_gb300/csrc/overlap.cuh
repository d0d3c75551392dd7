// overlap.cuh — kernel launches that may start while the previous kernel in
// their stream is still finishing (programmatic dependent launch), and the
// device side of it. Included by the library's .cu files only.
//
// A kernel launched this way can have its blocks scheduled onto SMs as the
// previous kernel's last blocks retire, instead of after the whole grid has
// drained and the launch has been processed; it then waits, before touching
// global memory, until every kernel it may depend on has completed and its
// writes are visible. Short launches (a bucket's step, a mid-size norm pass,
// the one-thread clip coefficient between them) lose a fixed ramp and drain
// per launch, which this hides. The results do not change: nothing global is
// read or written before the wait.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace zs {

// Whether launches ask for the overlap (zs_set_launch_overlap; on by default).
bool launch_overlap();

// First thing a kernel launched by launch_kernel does before any global
// memory access: wait for the kernels it may depend on (at once when it was
// launched without the overlap), then allow the next kernel in the stream to
// be scheduled as this one's blocks retire.
__device__ __forceinline__ void overlap_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// kernel<<<grid, block, smem, stream>>>(args...), with the overlap when it is on.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = launch_overlap() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace zs
