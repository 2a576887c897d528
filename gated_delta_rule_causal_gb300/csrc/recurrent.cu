// Token-by-token recurrence on CUDA cores (fp32 arithmetic).
//
// This is the GPU path for fp32 io (where bf16 tensor-core operands could not
// meet a 1e-4 relative bound) and for head sizes 16 and 32. It follows the
// recurrences literally: update first, then read.
//
// One CTA per (b,h). Thread j < d_v owns one d_v index of the state in
// registers: column j of S [d_k, d_v] for the norm/gla variants, row j of
// S [d_v, d_k] for the gated delta rule (scalar or per-channel decay). Tokens
// are staged in shared memory
// kTB at a time.
#include <cuda_bf16.h>

#include "kernels.h"

namespace la {
namespace {

constexpr int kTB = 16;       // tokens staged per block
constexpr int kThreads = 128; // covers d_v <= 128

template <typename T> __device__ __forceinline__ float ld_io(const T* p, size_t i);
template <> __device__ __forceinline__ float ld_io<float>(const float* p, size_t i) { return p[i]; }
template <> __device__ __forceinline__ float ld_io<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) {
    return __bfloat162float(p[i]);
}
template <typename T> __device__ __forceinline__ void st_io(T* p, size_t i, float x);
template <> __device__ __forceinline__ void st_io<float>(float* p, size_t i, float x) { p[i] = x; }
template <> __device__ __forceinline__ void st_io<__nv_bfloat16>(__nv_bfloat16* p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

// elu(x) + 1 with alpha = 1.
__device__ __forceinline__ float elu1(float x) { return x > 0.f ? x + 1.f : expf(x); }

template <int VAR, int DK, typename IO>
__global__ void __launch_bounds__(kThreads) recurrent_kernel(FwdArgs a) {
    const int bh = blockIdx.x;
    const int tid = threadIdx.x;
    const int T = a.T, dv = a.dv;
    const bool phi_on = !(VAR == kGla && (a.flags & 0x1u));
    // norm: the fixed decay of this sequence-head (1 without one)
    const float gam = (VAR == kNorm && a.gate) ? a.gate[bh] : 1.f;

    __shared__ float sq[kTB][DK];
    __shared__ float sk[kTB][DK];
    __shared__ float sv[kTB][128];
    __shared__ float sg[kTB][(VAR == kGla || VAR == kKda) ? DK : 1];
    constexpr bool DELTA = (VAR == kGdn || VAR == kKda);   // S [d_v, d_k], delta-rule write
    __shared__ float sgs[kTB], sbs[kTB], sden[kTB];
    __shared__ float pz[kTB][DK];
    __shared__ float zsh[DK];

    const IO* q = static_cast<const IO*>(a.q) + static_cast<size_t>(bh) * T * DK;
    const IO* k = static_cast<const IO*>(a.k) + static_cast<size_t>(bh) * T * DK;
    const IO* v = static_cast<const IO*>(a.v) + static_cast<size_t>(bh) * T * dv;
    IO* out = static_cast<IO*>(a.out) + static_cast<size_t>(bh) * T * dv;

    const size_t ssz = static_cast<size_t>(DK) * dv + (VAR == kNorm ? DK : 0);
    const float* sin = a.state_in ? a.state_in + bh * ssz : nullptr;

    float s[DK];
    const bool own = tid < dv;
#pragma unroll
    for (int i = 0; i < DK; ++i) {
        float x = 0.f;
        if (own && sin) x = DELTA ? sin[static_cast<size_t>(tid) * DK + i] : sin[static_cast<size_t>(i) * dv + tid];
        s[i] = x;
    }
    if (VAR == kNorm && tid < DK) zsh[tid] = sin ? sin[static_cast<size_t>(DK) * dv + tid] : 0.f;

    for (int t0 = 0; t0 < T; t0 += kTB) {
        const int nt = min(kTB, T - t0);
        __syncthreads();
        for (int e = tid; e < nt * DK; e += kThreads) {
            const int t = e / DK, c = e % DK;
            const size_t gi = static_cast<size_t>(t0 + t) * DK + c;
            const float qv = ld_io(q, gi), kv = ld_io(k, gi);
            sq[t][c] = (!DELTA && phi_on) ? elu1(qv) : qv;
            sk[t][c] = (!DELTA && phi_on) ? elu1(kv) : kv;
            if (VAR == kGla || VAR == kKda) sg[t][c] = a.gate[(static_cast<size_t>(bh) * T + t0 + t) * DK + c];
        }
        for (int e = tid; e < nt * dv; e += kThreads) {
            const int t = e / dv, c = e % dv;
            sv[t][c] = ld_io(v, static_cast<size_t>(t0 + t) * dv + c);
        }
        if (DELTA && tid < nt) {
            if (VAR == kGdn) sgs[tid] = a.gate[static_cast<size_t>(bh) * T + t0 + tid];
            sbs[tid] = a.beta[static_cast<size_t>(bh) * T + t0 + tid];
        }
        __syncthreads();
        if (VAR == kNorm) {
            // z_t = gamma z_{t-1} + phi(k_t); den_t = phi(q_t) . z_t (update first).
            if (tid < DK) {
                float z = zsh[tid];
                for (int t = 0; t < nt; ++t) {
                    z = gam * z + sk[t][tid];
                    pz[t][tid] = sq[t][tid] * z;
                }
                zsh[tid] = z;
            }
            __syncthreads();
            if (tid < nt) {
                float d = 0.f;
                for (int i = 0; i < DK; ++i) d += pz[tid][i];
                sden[tid] = d;
                if (a.den_out) a.den_out[static_cast<size_t>(bh) * T + t0 + tid] = d;
            }
            __syncthreads();
        }
        if (own) {
            for (int t = 0; t < nt; ++t) {
                const float vj = sv[t][tid];
                float o = 0.f;
                if (VAR == kNorm) {
#pragma unroll
                    for (int i = 0; i < DK; ++i) {
                        s[i] = gam * s[i] + sk[t][i] * vj;
                        o += sq[t][i] * s[i];
                    }
                    o = o / sden[t];
                } else if (VAR == kGla) {
#pragma unroll
                    for (int i = 0; i < DK; ++i) {
                        s[i] = sg[t][i] * s[i] + sk[t][i] * vj;
                        o += sq[t][i] * s[i];
                    }
                } else {
                    const float b = sbs[t];
                    float sk_dot = 0.f;
#pragma unroll
                    for (int c = 0; c < DK; ++c) {
                        s[c] *= (VAR == kKda) ? sg[t][c] : sgs[t];   // S~ = S Diag(alpha) (kda) or g S
                        sk_dot += s[c] * sk[t][c];
                    }
                    const float u = b * (vj - sk_dot);  // beta (v - S~ k)
#pragma unroll
                    for (int c = 0; c < DK; ++c) {
                        s[c] += u * sk[t][c];           // S = S~ + u k^T
                        o += s[c] * sq[t][c];           // o = S q
                    }
                }
                st_io(out, static_cast<size_t>(t0 + t) * dv + tid, o);
            }
        }
    }
    if (a.state_out) {
        float* so = a.state_out + bh * ssz;
        if (own) {
#pragma unroll
            for (int i = 0; i < DK; ++i) {
                if (DELTA) so[static_cast<size_t>(tid) * DK + i] = s[i];
                else so[static_cast<size_t>(i) * dv + tid] = s[i];
            }
        }
        if (VAR == kNorm) {
            __syncthreads();
            if (tid < DK) so[static_cast<size_t>(DK) * dv + tid] = zsh[tid];
        }
    }
}

template <int VAR, typename IO>
cudaError_t launch_dk(const FwdArgs& a, cudaStream_t s) {
    dim3 grid(a.BH), block(kThreads);
    switch (a.dk) {
        case 16: recurrent_kernel<VAR, 16, IO><<<grid, block, 0, s>>>(a); break;
        case 32: recurrent_kernel<VAR, 32, IO><<<grid, block, 0, s>>>(a); break;
        case 64: recurrent_kernel<VAR, 64, IO><<<grid, block, 0, s>>>(a); break;
        case 128: recurrent_kernel<VAR, 128, IO><<<grid, block, 0, s>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_var(const FwdArgs& a, cudaStream_t s) {
    switch (a.variant) {
        case kNorm: return launch_dk<kNorm, IO>(a, s);
        case kGla: return launch_dk<kGla, IO>(a, s);
        case kGdn: return launch_dk<kGdn, IO>(a, s);
        case kKda: return launch_dk<kKda, IO>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_recurrent(const FwdArgs& a, cudaStream_t s) {
    if (a.io == kFp32) return launch_var<float>(a, s);
    return launch_var<__nv_bfloat16>(a, s);
}

}  // namespace la
