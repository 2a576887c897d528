// One decode step for every sequence-head: read the fp32 state once, update
// it, write it back and emit the token's output. The step is HBM-bound:
// per head it moves d_k*d_v*4 bytes in and out; everything else is small.
//
// Gated delta rule (state S [d_v, d_k], rows contiguous): for each row i
//   S~_i = g S_i,  u_i = beta (v_i - S~_i . k),  S'_i = S~_i + u_i k,
//   o_i = S'_i . q = S~_i . q + u_i (k . q)
// ("Linear Attention" concept page, gated delta rule; "Beyond attention"
// 18.2). Rows are independent, so warps take units of rows of any head.
// Each lane holds 4 consecutive columns (one 16-byte vector) of a row, and
// the two row dot products are reduced with warp shuffles. Every load of a
// unit (its state rows, and the head's q, k, v, g, beta) is issued before the
// first one is used, so a unit costs one trip to memory; the grid is sized
// to the CTAs that are resident at once, and consecutive steps chain with
// programmatic dependent launch so that one step's dispatch overlaps the
// previous step's tail.
//
// Normalized / gated variants (state S [d_k, d_v]): each row i of S is
// scaled (gla: gamma_i; norm: the head's fixed decay, 1 without one), gets
// phi(k_i) v added (z_i scaled the same way), and contributes
// phi(q_i) S'_i to the output column sums ("Linear attention and recurrent
// memory", recurrent step; "Linear attention and Hyena" 11.3). One CTA per
// head; the column sums are reduced in shared memory.
#include <cuda_bf16.h>

#include "kernels.h"
#include "launch.cuh"
#include "ptx.cuh"

namespace la {
namespace {

__device__ __forceinline__ float4 ld_stream(const float* p) {
    return __ldcs(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ void st_stream(float* p, float4 x) {
    __stcs(reinterpret_cast<float4*>(p), x);
}

template <typename IO> __device__ __forceinline__ float4 ld4(const IO* p);
template <> __device__ __forceinline__ float4 ld4<float>(const float* p) {
    return __ldg(reinterpret_cast<const float4*>(p));
}
template <> __device__ __forceinline__ float4 ld4<__nv_bfloat16>(const __nv_bfloat16* p) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
template <typename IO> __device__ __forceinline__ float ld1(const IO* p);
template <> __device__ __forceinline__ float ld1<float>(const float* p) { return __ldg(p); }
template <> __device__ __forceinline__ float ld1<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}
template <typename IO> __device__ __forceinline__ void st1(IO* p, float x);
template <> __device__ __forceinline__ void st1<float>(float* p, float x) { *p = x; }
template <> __device__ __forceinline__ void st1<__nv_bfloat16>(__nv_bfloat16* p, float x) {
    *p = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
    return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}

// Sum over the LPR consecutive lanes that hold one row.
template <int LPR>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ float elu1(float x) { return x > 0.f ? x + 1.f : __expf(x); }

// ------------------------------------------------------------ gated delta rule

constexpr int kGdnThreads = 256;
constexpr int kGdnPasses = 8;   // row passes per warp unit (loads in flight per lane)

// PC: the per-channel decay of the kda variant (gate [BH][DK]): with
// S~ = S Diag(alpha), S~ . k = S . (alpha o k) and S~ . q = S . (alpha o q).
template <int DK, typename IO, bool PC>
__global__ void __launch_bounds__(kGdnThreads) decode_gdn_kernel(FwdArgs a) {
    constexpr int LPR = DK / 4;          // lanes per row
    constexpr int RPP = 32 / LPR;        // rows per pass
    constexpr int R = RPP * kGdnPasses;  // rows per warp unit
    const int dv = a.dv;
    const int uph = (dv + R - 1) / R;    // units per head
    const long long units = static_cast<long long>(a.BH) * uph;
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR, cl = lane % LPR;
    const long long warp0 = (static_cast<long long>(blockIdx.x) * kGdnThreads + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * kGdnThreads) >> 5;
    const IO* q = static_cast<const IO*>(a.q);
    const IO* k = static_cast<const IO*>(a.k);
    const IO* v = static_cast<const IO*>(a.v);
    IO* out = static_cast<IO*>(a.out);
    const size_t ssz = static_cast<size_t>(DK) * dv;

    griddep_launch_dependents();
    griddep_wait();   // the previous step's state is complete
    for (long long u = warp0; u < units; u += nwarps) {
        const int h = static_cast<int>(u / uph);
        const int r0 = static_cast<int>(u % uph) * R;
        const float* sin = a.state_in ? a.state_in + h * ssz : nullptr;
        float* sout = a.state_out + h * ssz;
        float4 S[kGdnPasses];
        float vr[kGdnPasses];
#pragma unroll
        for (int p = 0; p < kGdnPasses; ++p) {
            const int row = r0 + p * RPP + sub;
            S[p] = (sin && row < dv) ? ld_stream(sin + static_cast<size_t>(row) * DK + 4 * cl)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int p = 0; p < kGdnPasses; ++p) {
            const int row = r0 + p * RPP + sub;
            vr[p] = row < dv ? ld1(v + static_cast<size_t>(h) * dv + row) : 0.f;
        }
        const float4 k4 = ld4(k + static_cast<size_t>(h) * DK + 4 * cl);
        const float4 q4 = ld4(q + static_cast<size_t>(h) * DK + 4 * cl);
        const float b = __ldg(a.beta + h);
        const float g = PC ? 1.f : __ldg(a.gate + h);
        const float4 al = PC ? __ldg(reinterpret_cast<const float4*>(a.gate + static_cast<size_t>(h) * DK) + cl)
                             : make_float4(1.f, 1.f, 1.f, 1.f);
        const float4 ka = make_float4(al.x * k4.x, al.y * k4.y, al.z * k4.z, al.w * k4.w);
        const float4 qa = make_float4(al.x * q4.x, al.y * q4.y, al.z * q4.z, al.w * q4.w);
        const float kq = group_sum<LPR>(dot4(k4, q4));
#pragma unroll
        for (int p = 0; p < kGdnPasses; ++p) {
            const int row = r0 + p * RPP + sub;
            const float sk = group_sum<LPR>(dot4(S[p], PC ? ka : k4));
            const float sq = group_sum<LPR>(dot4(S[p], PC ? qa : q4));
            if (row < dv) {
                const float ui = b * (vr[p] - g * sk);
                float4 n;
                n.x = g * al.x * S[p].x + ui * k4.x;
                n.y = g * al.y * S[p].y + ui * k4.y;
                n.z = g * al.z * S[p].z + ui * k4.z;
                n.w = g * al.w * S[p].w + ui * k4.w;
                st_stream(sout + static_cast<size_t>(row) * DK + 4 * cl, n);
                if (cl == 0) st1(out + static_cast<size_t>(h) * dv + row, g * sq + ui * kq);
            }
        }
    }
}

// ------------------------------------------------------------ norm / gla

constexpr int kColThreads = 256;
constexpr int kColWarps = kColThreads / 32;
constexpr int kColUnroll = 4;

template <int VAR, int DK, int DV, typename IO>
__global__ void __launch_bounds__(kColThreads) decode_cols_kernel(FwdArgs a) {
    constexpr int LPR = DV / 4;               // lanes per row
    constexpr int RPP = 32 / LPR;             // rows per warp pass
    constexpr int RSTEP = RPP * kColWarps;    // rows per CTA pass
    constexpr int NPASS = (DK + RSTEP - 1) / RSTEP;
    __shared__ float4 red[kColWarps * RPP][LPR];
    __shared__ float dred[kColWarps * RPP];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane / LPR, cl = lane % LPR;
    const int slot = warp * RPP + sub;
    const bool phi_on = !(VAR == kGla && (a.flags & 0x1u));
    const IO* q = static_cast<const IO*>(a.q);
    const IO* k = static_cast<const IO*>(a.k);
    const IO* v = static_cast<const IO*>(a.v);
    IO* out = static_cast<IO*>(a.out);
    const size_t ssz = static_cast<size_t>(DK) * DV + (VAR == kNorm ? DK : 0);

    for (int h = blockIdx.x; h < a.BH; h += gridDim.x) {
        const float4 v4 = ld4(v + static_cast<size_t>(h) * DV + 4 * cl);
        const float gnorm = (VAR == kNorm && a.gate) ? __ldg(a.gate + h) : 1.f;   // norm: fixed decay
        const float* sin = a.state_in ? a.state_in + h * ssz : nullptr;
        float* sout = a.state_out + h * ssz;
        float4 o4 = make_float4(0.f, 0.f, 0.f, 0.f);
        float den = 0.f;
#pragma unroll
        for (int p0 = 0; p0 < NPASS; p0 += kColUnroll) {
            float4 S[kColUnroll];
#pragma unroll
            for (int j = 0; j < kColUnroll; ++j) {
                const int row = (p0 + j) * RSTEP + slot;
                S[j] = (sin && p0 + j < NPASS && row < DK)
                           ? ld_stream(sin + static_cast<size_t>(row) * DV + 4 * cl)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int j = 0; j < kColUnroll; ++j) {
                const int row = (p0 + j) * RSTEP + slot;
                if (p0 + j < NPASS && row < DK) {
                    const float kr = ld1(k + static_cast<size_t>(h) * DK + row);
                    const float qr = ld1(q + static_cast<size_t>(h) * DK + row);
                    const float f = phi_on ? elu1(kr) : kr;
                    const float pr = phi_on ? elu1(qr) : qr;
                    const float gm = (VAR == kGla) ? __ldg(a.gate + static_cast<size_t>(h) * DK + row) : gnorm;
                    float4 n;
                    n.x = gm * S[j].x + f * v4.x;
                    n.y = gm * S[j].y + f * v4.y;
                    n.z = gm * S[j].z + f * v4.z;
                    n.w = gm * S[j].w + f * v4.w;
                    st_stream(sout + static_cast<size_t>(row) * DV + 4 * cl, n);
                    o4.x += pr * n.x;
                    o4.y += pr * n.y;
                    o4.z += pr * n.z;
                    o4.w += pr * n.w;
                    if (VAR == kNorm && cl == 0) {
                        const float z = gnorm * (sin ? sin[static_cast<size_t>(DK) * DV + row] : 0.f) + f;
                        sout[static_cast<size_t>(DK) * DV + row] = z;
                        den += pr * z;
                    }
                }
            }
        }
        red[slot][cl] = o4;
        if (cl == 0) dred[slot] = den;
        __syncthreads();
        if (threadIdx.x < LPR) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            float d = 0.f;
            for (int s = 0; s < kColWarps * RPP; ++s) {
                const float4 x = red[s][threadIdx.x];
                acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
                if (VAR == kNorm) d += dred[s];
            }
            const float inv = (VAR == kNorm) ? 1.f / d : 1.f;
            IO* o = out + static_cast<size_t>(h) * DV + 4 * threadIdx.x;
            st1(o + 0, acc.x * inv);
            st1(o + 1, acc.y * inv);
            st1(o + 2, acc.z * inv);
            st1(o + 3, acc.w * inv);
            if (VAR == kNorm && threadIdx.x == 0 && a.den_out) a.den_out[h] = d;
        }
        __syncthreads();
    }
}

template <int DK, typename IO, bool PC>
cudaError_t launch_gdn_dk(const FwdArgs& a, cudaStream_t s) {
    // persistent: as many CTAs as are resident at once (cached per kernel)
    static int per_sm = 0;
    if (per_sm == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_gdn_kernel<DK, IO, PC>, kGdnThreads, 0) !=
                cudaSuccess ||
            n < 1)
            n = 1;
        per_sm = n;
    }
    return launch_pdl(decode_gdn_kernel<DK, IO, PC>, static_cast<unsigned>(a.sm_count * per_sm), kGdnThreads, 0, s, a);
}

template <typename IO, bool PC>
cudaError_t launch_gdn(const FwdArgs& a, cudaStream_t s) {
    switch (a.dk) {
        case 16: return launch_gdn_dk<16, IO, PC>(a, s);
        case 32: return launch_gdn_dk<32, IO, PC>(a, s);
        case 64: return launch_gdn_dk<64, IO, PC>(a, s);
        case 128: return launch_gdn_dk<128, IO, PC>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

template <int VAR, int DK, typename IO>
cudaError_t launch_cols_dv(const FwdArgs& a, cudaStream_t s) {
    const int blocks = a.BH < a.sm_count * 8 ? a.BH : a.sm_count * 8;
    switch (a.dv) {
        case 16: decode_cols_kernel<VAR, DK, 16, IO><<<blocks, kColThreads, 0, s>>>(a); break;
        case 32: decode_cols_kernel<VAR, DK, 32, IO><<<blocks, kColThreads, 0, s>>>(a); break;
        case 64: decode_cols_kernel<VAR, DK, 64, IO><<<blocks, kColThreads, 0, s>>>(a); break;
        case 128: decode_cols_kernel<VAR, DK, 128, IO><<<blocks, kColThreads, 0, s>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <int VAR, typename IO>
cudaError_t launch_cols(const FwdArgs& a, cudaStream_t s) {
    switch (a.dk) {
        case 16: return launch_cols_dv<VAR, 16, IO>(a, s);
        case 32: return launch_cols_dv<VAR, 32, IO>(a, s);
        case 64: return launch_cols_dv<VAR, 64, IO>(a, s);
        case 128: return launch_cols_dv<VAR, 128, IO>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename IO>
cudaError_t launch_io(const FwdArgs& a, cudaStream_t s) {
    switch (a.variant) {
        case kNorm: return launch_cols<kNorm, IO>(a, s);
        case kGla: return launch_cols<kGla, IO>(a, s);
        case kGdn: return launch_gdn<IO, false>(a, s);
        case kKda: return launch_gdn<IO, true>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_decode(const FwdArgs& a, cudaStream_t s) {
    if (a.io == kFp32) return launch_io<float>(a, s);
    return launch_io<__nv_bfloat16>(a, s);
}

}  // namespace la
