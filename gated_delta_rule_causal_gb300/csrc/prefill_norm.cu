// Instantiations of the normalized variant's sequential chunk kernel and its
// segment summaries.
#include "prefill.h"
#include "prefill_impl.cuh"

namespace la {
namespace chunk {
namespace {

template <int DK, int DV>
cudaError_t run(const Maps& m, const Params& p, int BH, cudaStream_t s) {
    using L = Layout<kNorm, DK, DV>;
    cudaError_t e = cudaSuccess;
    if (p.nseg > 1) {
        using SL = SLayout<kNorm, DK, DV>;
        auto sk = summary_kernel<kNorm, DK, DV>;
        e = cudaFuncSetAttribute(sk, cudaFuncAttributeMaxDynamicSharedMemorySize, SL::SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        sk<<<BH * p.nsub, kThreads, SL::SMEM_ALLOC, s>>>(m.k, m.v, p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    auto kern = chunk_kernel<kNorm, DK, DV>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    kern<<<BH * p.nseg, kThreads, L::SMEM_ALLOC, s>>>(m.q, m.k, m.v, m.o, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_norm(int dk, int dv, const Maps& m, const Params& p, int BH, cudaStream_t s) {
    if (dk == 64 && dv == 64) return run<64, 64>(m, p, BH, s);
    if (dk == 64 && dv == 128) return run<64, 128>(m, p, BH, s);
    if (dk == 128 && dv == 64) return run<128, 64>(m, p, BH, s);
    if (dk == 128 && dv == 128) return run<128, 128>(m, p, BH, s);
    return cudaErrorInvalidValue;
}

}  // namespace chunk
}  // namespace la
