// Host-side launch helper shared by the kernels that chain with
// programmatic dependent launch.
#pragma once

#include <cuda_runtime.h>

namespace la {

// Launch with programmatic stream serialization: the kernel may be
// dispatched while the previous one in the stream finishes; it waits in
// griddep_wait() (ptx.cuh) before touching data the previous kernels wrote.
template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, unsigned grid, unsigned block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace la
