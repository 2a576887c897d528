// Host-side launch helpers: programmatic dependent launch for kernels that
// chain in a stream, cooperative launch for grids whose CTAs hand work to
// each other.
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

// Cooperative launch: the grid is dispatched only if every CTA can be
// resident at once, so its CTAs may wait on flags other CTAs set.
template <typename Kern, typename... Args>
cudaError_t launch_coop(Kern kern, unsigned grid, unsigned block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Launch in thread-block clusters of `cluster` CTAs along x (the grid is a
// multiple of it); the CTAs of one cluster are resident together.
template <typename Kern, typename... Args>
cudaError_t launch_cluster(Kern kern, unsigned grid, unsigned cluster, unsigned block, size_t smem, cudaStream_t s,
                           Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace la
