// Programmatic dependent launch between the kernels of one forward.
//
// A kernel launched with launch_pdl may be scheduled while the previous
// kernel of its stream is still finishing: it calls pdl_wait() before it
// reads anything an earlier kernel wrote (griddepcontrol.wait returns once
// the preceding grid has completed and its memory is visible; without a
// programmatic dependency it returns at once), and pdl_trigger() to let the
// kernel after it be scheduled early.  Every kernel launched this way calls
// pdl_wait() before its first read of device data, so each kernel still
// starts its work after all earlier kernels have finished.  Only kernels
// followed by small kernels trigger early: a persistent GEMM scheduled early
// would hold its SMs idle (and keep the shared expert's GEMMs on the second
// stream off them) until its predecessor ends.
#pragma once
#include <cuda_runtime.h>

namespace moe {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline void launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace moe
