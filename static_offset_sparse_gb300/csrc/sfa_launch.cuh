// Host helper: kernel launches with programmatic stream serialization.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace sfa {

// Launch `kern` so that it may begin while the previous kernel in the stream
// finishes (programmatic dependent launch).  The kernel must call pdl_wait()
// (sfa_tma.cuh) before touching global memory; inside a stream capture the
// edge becomes a programmatic dependency of the graph.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace sfa
