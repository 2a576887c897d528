// Gradients of the normalized elu+1 recurrence on CUDA cores (fp32).
//
// "Beyond — Linear attention and recurrent memory" (summarizing
// "Transformers are RNNs"): phi = elu + 1, S_t = S_{t-1} + phi(k_t) v_t^T,
// z_t = z_{t-1} + phi(k_t), o_t = S_t^T phi(q_t) / phi(q_t)^T z_t, update
// first. The pages give no gradients; by the chain rule, with
// f = phi(k), p = phi(q), num_t = S_t^T p_t, den_t = p_t . z_t:
//   dnum_t = do_t / den_t,  dden_t = -(do_t . num_t) / den_t^2
//   dp_t = S_t dnum_t + z_t dden_t
//   G_t = dS_T + sum_{tau >= t} p_tau dnum_tau^T,  g_t = dz_T + sum_{tau >= t} p_tau dden_tau
//   df_t = G_t v_t + g_t,  dv_t = G_t^T f_t,  dq = dp * phi'(q),  dk = df * phi'(k)
//   dS_0 = G_0, dz_0 = g_0.
//
// One CTA per sequence-head. Threads [0, DV) own one column j of S and of
// G (num_t, dv_t); threads [DV, DV + DK) own one row i of S and of G and z_i,
// g_i (dp_t, df_t, hence dq and dk). A forward pass brings S and z to the
// end of the sequence; the reverse pass walks tiles of kTB tokens from the
// end, recovering S_{t-1} = S_t - f_t v_t^T and z_{t-1} = z_t - f_t as it
// goes (the fp32 rounding of that subtraction grows with T). The two
// per-token scalars den_t and dden_t are block reductions, once per tile.
#include <cuda_bf16.h>

#include "kernels.h"

namespace la {
namespace {

constexpr int kTB = 16;        // tokens per tile
constexpr int kThreads = 128;  // DV column owners + DK row owners (<= 64 + 64)

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

__device__ __forceinline__ float phi(float x) { return x > 0.f ? x + 1.f : expf(x); }
__device__ __forceinline__ float dphi(float x) { return x > 0.f ? 1.f : expf(x); }

template <int DK, int DV, typename IO>
__global__ void __launch_bounds__(kThreads) norm_backward_kernel(BwdArgs a) {
    constexpr int N = DK > DV ? DK : DV;
    const int bh = blockIdx.x, tid = threadIdx.x, T = a.T;
    const bool col = tid < DV;                      // column j = tid
    const bool row = tid >= DV && tid < DV + DK;    // row i = tid - DV
    const int j = tid, i = tid - DV;
    __shared__ float sp[kTB][DK], sf[kTB][DK], sdp[kTB][DK], sdf[kTB][DK];   // phi(q), phi(k), phi'(q), phi'(k)
    __shared__ float sv[kTB][DV], sdo[kTB][DV];
    __shared__ float pz[kTB][DK], pn[kTB][DV];
    __shared__ float sden[kTB], sdden[kTB];

    const size_t qo = static_cast<size_t>(bh) * T * DK, vo = static_cast<size_t>(bh) * T * DV;
    const IO* q = static_cast<const IO*>(a.q) + qo;
    const IO* k = static_cast<const IO*>(a.k) + qo;
    const IO* v = static_cast<const IO*>(a.v) + vo;
    const IO* dout = static_cast<const IO*>(a.dout) + vo;
    IO* dq = static_cast<IO*>(a.dq) + qo;
    IO* dk = static_cast<IO*>(a.dk) + qo;
    IO* dv = static_cast<IO*>(a.dv) + vo;
    constexpr size_t SS = static_cast<size_t>(DK) * DV + DK;
    const float* sin = a.state_in ? a.state_in + bh * SS : nullptr;
    const float* dso = a.dstate_out ? a.dstate_out + bh * SS : nullptr;

    // S: column j (col) or row i (row) of the state; G likewise; z_i, g_i (row)
    float S[N], G[N];
    float z = 0.f, gz = 0.f;
#pragma unroll
    for (int e = 0; e < N; ++e) {
        float s0 = 0.f, g0 = 0.f;
        if (col && e < DK) {
            if (sin) s0 = sin[static_cast<size_t>(e) * DV + j];
            if (dso) g0 = dso[static_cast<size_t>(e) * DV + j];
        } else if (row && e < DV) {
            if (sin) s0 = sin[static_cast<size_t>(i) * DV + e];
            if (dso) g0 = dso[static_cast<size_t>(i) * DV + e];
        }
        S[e] = s0;
        G[e] = g0;
    }
    if (row) {
        if (sin) z = sin[static_cast<size_t>(DK) * DV + i];
        if (dso) gz = dso[static_cast<size_t>(DK) * DV + i];
    }

    auto load_tile = [&](int t0, int nt, bool bwd) {
        for (int e = tid; e < nt * DK; e += kThreads) {
            const int t = e / DK, c = e % DK;
            const size_t gi = static_cast<size_t>(t0 + t) * DK + c;
            const float kv = ld_io(k, gi);
            sf[t][c] = phi(kv);
            if (bwd) {
                const float qv = ld_io(q, gi);
                sp[t][c] = phi(qv);
                sdp[t][c] = dphi(qv);
                sdf[t][c] = dphi(kv);
            }
        }
        for (int e = tid; e < nt * DV; e += kThreads) {
            const int t = e / DV, c = e % DV;
            const size_t gi = static_cast<size_t>(t0 + t) * DV + c;
            sv[t][c] = ld_io(v, gi);
            if (bwd) sdo[t][c] = ld_io(dout, gi);
        }
    };

    // ---- forward to the end of the sequence
    for (int t0 = 0; t0 < T; t0 += kTB) {
        const int nt = min(kTB, T - t0);
        __syncthreads();
        load_tile(t0, nt, false);
        __syncthreads();
        for (int t = 0; t < nt; ++t) {
            if (col) {
                const float vj = sv[t][j];
#pragma unroll
                for (int e = 0; e < DK; ++e) S[e] += sf[t][e] * vj;
            } else if (row) {
                const float fi = sf[t][i];
#pragma unroll
                for (int e = 0; e < DV; ++e) S[e] += fi * sv[t][e];
                z += fi;
            }
        }
    }

    // ---- reverse, a tile at a time from the end
    const int ntile = (T + kTB - 1) / kTB;
    for (int tb = ntile - 1; tb >= 0; --tb) {
        const int t0 = tb * kTB, nt = min(kTB, T - t0);
        __syncthreads();
        load_tile(t0, nt, true);
        __syncthreads();
        // A: num_t (columns, stepping S back to the tile's start) and p_t z_t
        if (col) {
            for (int t = nt - 1; t >= 0; --t) {
                float nm[4] = {0.f, 0.f, 0.f, 0.f};   // four partial sums: shorter dependent chains
#pragma unroll
                for (int e = 0; e < DK; ++e) nm[e & 3] += sp[t][e] * S[e];
                pn[t][j] = sdo[t][j] * ((nm[0] + nm[1]) + (nm[2] + nm[3]));
                const float vj = sv[t][j];
#pragma unroll
                for (int e = 0; e < DK; ++e) S[e] -= sf[t][e] * vj;
            }
        } else if (row) {
            float zt = z;
            for (int t = nt - 1; t >= 0; --t) {
                pz[t][i] = sp[t][i] * zt;
                zt -= sf[t][i];
            }
        }
        __syncthreads();
        // B: den_t and dden_t
        if (tid < nt) {
            float d = 0.f, n = 0.f;
            for (int e = 0; e < DK; ++e) d += pz[tid][e];
            for (int e = 0; e < DV; ++e) n += pn[tid][e];
            sden[tid] = d;
            sdden[tid] = -n / (d * d);
        }
        __syncthreads();
        // C: gradients, token by token from the end of the tile
        for (int t = nt - 1; t >= 0; --t) {
            const float rden = 1.f / sden[t], dden = sdden[t];
            const size_t tt = static_cast<size_t>(t0 + t);
            if (col) {
                const float dnum = sdo[t][j] * rden;
                float dvp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int e = 0; e < DK; ++e) {
                    G[e] += sp[t][e] * dnum;
                    dvp[e & 3] += G[e] * sf[t][e];
                }
                st_io(dv, tt * DV + j, (dvp[0] + dvp[1]) + (dvp[2] + dvp[3]));
            } else if (row) {
                const float pi = sp[t][i], fi = sf[t][i];
                float dpp[4] = {0.f, 0.f, 0.f, 0.f}, dfp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int e = 0; e < DV; ++e) {
                    const float dnum = sdo[t][e] * rden;
                    dpp[e & 3] += S[e] * dnum;
                    G[e] += pi * dnum;
                    dfp[e & 3] += G[e] * sv[t][e];
                }
                gz += pi * dden;
                const float dpi = z * dden + ((dpp[0] + dpp[1]) + (dpp[2] + dpp[3]));
                const float dfi = gz + ((dfp[0] + dfp[1]) + (dfp[2] + dfp[3]));
                st_io(dq, tt * DK + i, dpi * sdp[t][i]);
                st_io(dk, tt * DK + i, dfi * sdf[t][i]);
#pragma unroll
                for (int e = 0; e < DV; ++e) S[e] -= fi * sv[t][e];
                z -= fi;
            }
        }
    }
    if (a.dstate_in) {
        float* dsi = a.dstate_in + bh * SS;
        if (col) {
#pragma unroll
            for (int e = 0; e < DK; ++e) dsi[static_cast<size_t>(e) * DV + j] = G[e];
        } else if (row) {
            dsi[static_cast<size_t>(DK) * DV + i] = gz;
        }
    }
}

template <int DK, int DV>
cudaError_t launch_dims(const BwdArgs& a, cudaStream_t s) {
    if (a.io == kBf16)
        norm_backward_kernel<DK, DV, __nv_bfloat16><<<a.BH, kThreads, 0, s>>>(a);
    else
        norm_backward_kernel<DK, DV, float><<<a.BH, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_norm_backward(const BwdArgs& a, cudaStream_t s) {
    const int dk = a.dk_dim, dv = a.dv_dim;
#define LA_BWD_CASE(K, V) \
    if (dk == K && dv == V) return launch_dims<K, V>(a, s);
    LA_BWD_CASE(16, 16) LA_BWD_CASE(16, 32) LA_BWD_CASE(16, 64)
    LA_BWD_CASE(32, 16) LA_BWD_CASE(32, 32) LA_BWD_CASE(32, 64)
    LA_BWD_CASE(64, 16) LA_BWD_CASE(64, 32) LA_BWD_CASE(64, 64)
#undef LA_BWD_CASE
    return cudaErrorInvalidValue;
}

}  // namespace la
