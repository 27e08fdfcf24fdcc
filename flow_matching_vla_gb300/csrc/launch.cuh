// Kernel launch with the programmatic-dependent-launch attribute.
//
// Every kernel of the denoise step calls griddepcontrol.launch_dependents
// early and griddepcontrol.wait before it touches activations, so with
// ``pdl`` set the next kernel's CTAs are scheduled (and prefetch weights)
// while the current one drains.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace g3 {

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace g3
