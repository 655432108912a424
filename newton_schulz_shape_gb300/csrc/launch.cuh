// Host-side launch of the library's kernels with programmatic stream
// serialization (see griddep_wait in ptx.cuh): the next kernel's CTAs may be
// scheduled and run their set-up while this one finishes.
#pragma once

#include <cuda_runtime.h>

namespace nsk {

template <typename P>
cudaError_t launch_pdl(void (*kern)(P), dim3 grid, dim3 block, size_t smem, cudaStream_t st, const P& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace nsk
