// Host side of the chunkwise prefill: TMA tensor maps and dispatch.
#include "prefill.h"
#include "prefill_impl.cuh"

namespace la {

namespace {

// 3-D map over a [BH, T, d] tensor with 64x64 boxes (one 128-byte swizzle
// atom wide). Rows past T read as zeros.
CUresult map_qkv(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, const void* base, int d, int T, int BH) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(d) * 2 * T};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(chunk::C), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

cudaError_t launch_chunked(const FwdArgs& a, cudaStream_t s, PFN_cuTensorMapEncodeTiled_v12000 enc, const char** what) {
    chunk::Maps m;
    *what = "cuTensorMapEncodeTiled";
    if (map_qkv(enc, &m.q, a.q, a.dk, a.T, a.BH) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (map_qkv(enc, &m.k, a.k, a.dk, a.T, a.BH) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (map_qkv(enc, &m.v, a.v, a.dv, a.T, a.BH) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (map_qkv(enc, &m.o, a.out, a.dv, a.T, a.BH) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    // The gated delta rule, its per-channel-decay form and the per-channel
    // gated variant (the delta rule's chunk algebra with T = I and W = 0) run
    // on the prep/chain kernel, whose in-chunk decay factors are taken
    // against 16-token sub-chunk references and so stay in the fp32 range.
    if (a.variant == kGdn || a.variant == kKda || a.variant == kGla) {
        *what = "chunked prefill launch";
        return chunk::launch_gdn(a, m, s);
    }
    if (a.variant == kNorm && !(a.flags & 0x2u) &&   // with or without a fixed decay
        chunk::seg_fits(a.BH, a.T, a.dk, a.dv, a.sm_count)) {
        *what = "chunked prefill launch";
        return chunk::launch_seg(a, m, s);
    }
    if (!(a.flags & 0x2u) && a.workspace && chunk::par_fits(a.BH, a.T, a.dk, a.dv, a.ws_bytes)) {
        *what = "chunked prefill launch";
        return chunk::launch_par(a, m, s);
    }
    chunk::Params p;
    p.state_in = a.state_in;
    p.state_out = a.state_out;
    p.den_out = a.den_out;
    p.T = a.T;
    p.nchunks = (a.T + chunk::C - 1) / chunk::C;
    p.flags = a.flags;
    p.status = a.status;
    // Split each sequence into segments when there are too few sequence-heads
    // to fill the GPU (one CTA per segment, one CTA per SM).
    p.nseg = 1;
    p.seg_len = p.nchunks;
    p.nsub = 0;
    p.sub_len = p.nchunks;
    p.scratch = a.workspace;
    if (a.workspace && a.BH < a.sm_count && p.nchunks >= 4) {
        int nseg = a.sm_count / a.BH;
        if (nseg > p.nchunks / 2) nseg = p.nchunks / 2;
        const size_t blk = (static_cast<size_t>(a.dk) * a.dv + a.dk) * sizeof(float);
        while (nseg > 1 && static_cast<size_t>(a.BH) * (nseg - 1) * blk > a.ws_bytes) --nseg;
        if (nseg > 1) {
            p.seg_len = (p.nchunks + nseg - 1) / nseg;
            p.nseg = (p.nchunks + p.seg_len - 1) / p.seg_len;
            // Summary runs: cut each segment before the last into m runs while
            // the runs still fit one wave of CTAs and the workspace.
            int m = 1;
            const size_t nbefore = static_cast<size_t>(a.BH) * (p.nseg - 1);
            while (p.seg_len % (2 * m) == 0 && p.seg_len / (2 * m) >= 2 &&
                   nbefore * 2 * m <= static_cast<size_t>(a.sm_count) && nbefore * 2 * m * blk <= a.ws_bytes)
                m *= 2;
            p.sub_len = p.seg_len / m;
            p.nsub = (p.nseg - 1) * m;
        }
    }
    *what = "chunked prefill launch";
    if (a.nlaunch) *a.nlaunch += (p.nseg > 1) ? 2 : 1;   // segment summaries + chunk kernel
    if (a.variant != kNorm) return cudaErrorInvalidValue;
    return chunk::launch_norm(a.dk, a.dv, m, p, a.BH, s);
}

}  // namespace la
