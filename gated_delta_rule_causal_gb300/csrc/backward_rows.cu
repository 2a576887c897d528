// Gradients of the gated delta rule (scalar or per-channel decay) on CUDA
// cores, token by token, in fp32.
//
// Forward operator ("Beyond attention" §18.2 for the scalar gate; "Linear
// attention and recurrent memory", from fixed decay to KDA, for a decay per
// key channel), S in R^{dv x dk}:
//    S~_t = S_{t-1} Diag(a_t)   (a_t = g_t 1 for the scalar gate)
//    u_t  = beta_t (v_t - S~_t k_t),   S_t = S~_t + u_t k_t^T,   o_t = S_t q_t
// The pages give no gradients. By the chain rule, with D the whole gradient
// reaching S_t (the final-state cotangent, then carried back):
//    D += do_t q_t^T,            dq_t = S_t^T do_t
//    du = D k_t,                 dv_t = beta_t du,   dbeta_t = (v_t - S~_t k_t) . du
//    dk_t = D^T u_t - beta_t S~_t^T du
//    dS~ = D - beta_t du k_t^T,  da_t = column sums of dS~ o S_{t-1} (their total for g_t)
//    D <- dS~ Diag(a_t);         dstate_in = D after token 0.
//
// Every value row of S (and of D) evolves on its own given k, a and beta, so
// the work splits by rows: one CTA per (sequence-head, block of kRows rows),
// one warp per row, each lane holding DK/32 adjacent columns. Each CTA first
// runs its rows forward and stores them at the start of every segment of
// kSeg tokens (workspace). It then walks the segments from the last: it
// reloads the segment's starting rows, recomputes the kSeg + 1 row states in
// registers, and takes the tokens in reverse. The row-local gradients (dv)
// are written directly; the sums over rows (dq, dk, the decay and beta
// gradients) go through shared memory once per token and then into fp32
// accumulators with one atomic add per column per CTA. A second kernel
// writes dq and dk in the io dtype.
//
// The per-channel gated recurrence ("Linear attention and Hyena" §11.3,
// S in R^{dk x dv}: S_t = diag(gamma_t) S_{t-1} + f_t v_t^T, o_t = S_t^T p_t
// with f = phi(k), p = phi(q)) runs through the same scheme with the key
// channels as rows: D += p_t do_t^T, dq = (S_t do_t) o phi'(q), dk = (D v_t)
// o phi'(k), dgamma = rowsums of D o S_{t-1} (all row-local), dv_t = D^T f_t
// (the one sum over rows), D <- diag(gamma_t) D.
//
// The normalized recurrence (S in R^{dk x dv} and z in R^{dk}: S_t = gamma
// S_{t-1} + f_t v_t^T, z_t = gamma z_{t-1} + f_t, gamma = 1 or one decay per
// sequence-head; o_t = S_t^T p_t / p_t.z_t) takes the key channels as rows
// too. Its two per-token factors dnum_t = do_t / den_t and
// dden_t = -(do_t.num_t) / den_t^2 = -(do_t.o_t) / den_t come from the
// outputs and normalizers of a forward call the caller runs first. Then with
// G, g the gradients reaching S_t, z_t: G += p_t dnum_t^T, g += p_t dden_t,
// dq = (S_t dnum_t + z_t dden_t) o phi'(q), dk = (G v_t + g) o phi'(k) (both
// row-local), dv_t = G^T f_t (the sum over rows), dgamma += <G, S_{t-1}> +
// <g, z_{t-1}>, then G, g <- gamma G, gamma g.
//
// This is the correctness path of these gradients (and of the normalized
// variant's wherever the chunkwise tensor-core backward does not apply): its
// cost is the token-serial walk (2 T dependent steps per row) and the
// per-token reduction, not memory bandwidth.
#include <cuda_bf16.h>

#include "kernels.h"

namespace la {
namespace {

constexpr int kRows = 16;             // value rows per CTA (one warp each)
constexpr int kSeg = 8;               // tokens per recomputed segment
constexpr int kThreads = kRows * 32;

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

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Shared memory of one CTA.
template <int DK, bool PC>
struct Smem {
    static constexpr int NV = PC ? 3 : 2;           // column sums per token: dq, dk (, da)
    static constexpr int RED = NV * DK + 2;         // + dbeta and (scalar gate) dg
    float k[kSeg][DK];
    float q[kSeg][DK];
    float a[PC ? kSeg : 1][DK];                     // per-channel decay
    float g[kSeg];                                  // scalar decay
    float b[kSeg];
    float v[kSeg][kRows];
    float dout[kSeg][kRows];
    float dv[kSeg][kRows];
    float red[2][kRows][RED];
};

template <int DK, int DV, bool PC, typename IO>
__global__ void __launch_bounds__(kThreads, 2) delta_backward_kernel(DeltaBwdArgs p) {
    constexpr int NC = DK / 32;   // columns per lane
    constexpr int NRB = DV / kRows;
    using SM = Smem<DK, PC>;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SM& sm = *reinterpret_cast<SM*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x / NRB, rb = blockIdx.x % NRB;
    const int r = rb * kRows + warp;   // this warp's value row
    const int c0 = lane * NC;          // this lane's first column
    const int T = p.T;
    const int nseg = (T + kSeg - 1) / kSeg;
    const size_t tok0 = static_cast<size_t>(bh) * T;
    const IO* q = static_cast<const IO*>(p.q);
    const IO* k = static_cast<const IO*>(p.k);
    const IO* v = static_cast<const IO*>(p.v);
    const IO* dout = static_cast<const IO*>(p.dout);
    const size_t ssz = static_cast<size_t>(DV) * DK;
    float* ck = p.ckpt + (static_cast<size_t>(bh) * nseg * DV + r) * DK + c0;   // + seg * DV * DK

    // Stage the inputs of tokens [t0, t0 + n) that every warp reads.
    auto stage = [&](int t0, int n, bool with_q) {
        for (int x = tid; x < kSeg * DK; x += kThreads) {
            const int i = x / DK, c = x % DK;
            const bool in = i < n;
            const size_t e = (tok0 + t0 + i) * DK + c;
            sm.k[i][c] = in ? ld_io(k, e) : 0.f;
            if (with_q) sm.q[i][c] = in ? ld_io(q, e) : 0.f;
            if (PC) sm.a[i][c] = in ? p.gate[e] : 1.f;
        }
        for (int x = tid; x < kSeg; x += kThreads) {
            const bool in = x < n;
            if (!PC) sm.g[x] = in ? p.gate[tok0 + t0 + x] : 1.f;
            sm.b[x] = in ? p.beta[tok0 + t0 + x] : 0.f;
        }
        for (int x = tid; x < kSeg * kRows; x += kThreads) {
            const int i = x / kRows, w = x % kRows;
            const bool in = i < n;
            const size_t e = (tok0 + t0 + i) * DV + rb * kRows + w;
            sm.v[i][w] = in ? ld_io(v, e) : 0.f;
            if (with_q) sm.dout[i][w] = in ? ld_io(dout, e) : 0.f;
        }
    };
    // One token forward on this lane's columns of row r: s <- S_t, returns
    // the error v_t - S~_t k_t (the same on every lane).
    auto step = [&](int i, float* s) -> float {
        float part = 0.f;
#pragma unroll
        for (int j = 0; j < NC; ++j) {
            s[j] *= PC ? sm.a[i][c0 + j] : sm.g[i];
            part += s[j] * sm.k[i][c0 + j];
        }
        const float err = sm.v[i][warp] - warp_sum(part);
        const float u = sm.b[i] * err;
#pragma unroll
        for (int j = 0; j < NC; ++j) s[j] += u * sm.k[i][c0 + j];
        return err;
    };

    // ---- forward: the rows at the start of every segment -------------------
    float s[NC];
#pragma unroll
    for (int j = 0; j < NC; ++j) s[j] = p.state_in ? p.state_in[bh * ssz + static_cast<size_t>(r) * DK + c0 + j] : 0.f;
    for (int sg = 0; sg < nseg; ++sg) {
        const int t0 = sg * kSeg, n = min(kSeg, T - t0);
        float* dst = ck + static_cast<size_t>(sg) * DV * DK;
#pragma unroll
        for (int j = 0; j < NC; ++j) dst[j] = s[j];
        __syncthreads();   // the previous segment's inputs are no longer read
        stage(t0, n, false);
        __syncthreads();
        for (int i = 0; i < n; ++i) step(i, s);
    }

    // ---- backward: segments from the last ---------------------------------
    float D[NC];
#pragma unroll
    for (int j = 0; j < NC; ++j) D[j] = p.dstate_out ? p.dstate_out[bh * ssz + static_cast<size_t>(r) * DK + c0 + j] : 0.f;
    int buf = 0;
    for (int sg = nseg - 1; sg >= 0; --sg) {
        const int t0 = sg * kSeg, n = min(kSeg, T - t0);
        __syncthreads();   // the previous segment's inputs and dv are no longer read
        stage(t0, n, true);
        __syncthreads();
        // the kSeg + 1 row states of the segment, and each token's error
        float st[kSeg + 1][NC];
        float err[kSeg];
        const float* src = ck + static_cast<size_t>(sg) * DV * DK;
#pragma unroll
        for (int j = 0; j < NC; ++j) st[0][j] = src[j];
#pragma unroll
        for (int i = 0; i < kSeg; ++i) {
#pragma unroll
            for (int j = 0; j < NC; ++j) st[i + 1][j] = st[i][j];
            err[i] = (i < n) ? step(i, st[i + 1]) : 0.f;
        }
#pragma unroll
        for (int i = kSeg - 1; i >= 0; --i) {
            if (i < n) {   // uniform over the CTA
                float* red = &sm.red[buf][warp][0];
                const float dor = sm.dout[i][warp], bt = sm.b[i];
                float part = 0.f;
#pragma unroll
                for (int j = 0; j < NC; ++j) {
                    D[j] += dor * sm.q[i][c0 + j];
                    red[c0 + j] = st[i + 1][j] * dor;   // dq_t = S_t^T do_t
                    part += D[j] * sm.k[i][c0 + j];
                }
                const float du = warp_sum(part);
                const float u = bt * err[i];
                float dg = 0.f;
#pragma unroll
                for (int j = 0; j < NC; ++j) {
                    const float dec = PC ? sm.a[i][c0 + j] : sm.g[i];
                    const float sd = st[i][j] * dec;                       // S~_t
                    red[DK + c0 + j] = D[j] * u - bt * sd * du;            // dk_t
                    const float dsd = D[j] - bt * du * sm.k[i][c0 + j];    // dS~
                    const float da = dsd * st[i][j];
                    if (PC) red[2 * DK + c0 + j] = da;
                    else dg += da;
                    D[j] = dsd * dec;
                }
                if (!PC) dg = warp_sum(dg);
                if (lane == 0) {
                    red[SM::NV * DK] = err[i] * du;   // dbeta_t
                    red[SM::NV * DK + 1] = dg;
                    sm.dv[i][warp] = bt * du;
                }
                __syncthreads();
                // sums over the CTA's rows, added to the totals over all rows
                const size_t t = tok0 + t0 + i;
                for (int x = tid; x < SM::RED; x += kThreads) {
                    float acc = 0.f;
#pragma unroll
                    for (int w = 0; w < kRows; ++w) acc += sm.red[buf][w][x];
                    if (x < DK) atomicAdd(p.dq_acc + t * DK + x, acc);
                    else if (x < 2 * DK) atomicAdd(p.dk_acc + t * DK + x - DK, acc);
                    else if (PC && x < 3 * DK) atomicAdd(p.dgate + t * DK + x - 2 * DK, acc);
                    else if (x == SM::NV * DK) atomicAdd(p.dbeta + t, acc);
                    else if (!PC) atomicAdd(p.dgate + t, acc);
                }
                buf ^= 1;   // the next token fills the other buffer while this one is read
            }
        }
        __syncthreads();
        IO* dvo = static_cast<IO*>(p.dv);
        for (int x = tid; x < n * kRows; x += kThreads) {
            const int i = x / kRows, w = x % kRows;
            st_io(dvo, (tok0 + t0 + i) * DV + rb * kRows + w, sm.dv[i][w]);
        }
    }
    if (p.dstate_in) {
#pragma unroll
        for (int j = 0; j < NC; ++j) p.dstate_in[bh * ssz + static_cast<size_t>(r) * DK + c0 + j] = D[j];
    }
}

// ---------------------------------------------------------------------------
// per-channel gated recurrence: rows = key channels
// ---------------------------------------------------------------------------
template <int DV>
struct SmemGla {
    float v[kSeg][DV];
    float dout[kSeg][DV];
    float f[kSeg][kRows];     // phi(k) of the CTA's channels
    float df[kSeg][kRows];    // phi'(k)
    float p[kSeg][kRows];     // phi(q)
    float dp[kSeg][kRows];    // phi'(q)
    float g[kSeg][kRows];     // gamma
    float dq[kSeg][kRows];
    float dk[kSeg][kRows];
    float dg[kSeg][kRows];
    float red[2][kRows][DV];
};

template <int DK, int DV, typename IO, bool IDPHI>
__global__ void __launch_bounds__(kThreads, 2) gla_backward_kernel(DeltaBwdArgs p) {
    constexpr int NC = DV / 32;   // value columns per lane
    constexpr int NRB = DK / kRows;
    using SM = SmemGla<DV>;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SM& sm = *reinterpret_cast<SM*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x / NRB, rb = blockIdx.x % NRB;
    const int r = rb * kRows + warp;   // this warp's key channel
    const int c0 = lane * NC;
    const int T = p.T;
    const int nseg = (T + kSeg - 1) / kSeg;
    const size_t tok0 = static_cast<size_t>(bh) * T;
    const IO* q = static_cast<const IO*>(p.q);
    const IO* k = static_cast<const IO*>(p.k);
    const IO* v = static_cast<const IO*>(p.v);
    const IO* dout = static_cast<const IO*>(p.dout);
    const size_t ssz = static_cast<size_t>(DK) * DV;
    float* ck = p.ckpt + (static_cast<size_t>(bh) * nseg * DK + r) * DV + c0;   // + seg * DK * DV

    auto stage = [&](int t0, int n, bool with_q) {
        for (int x = tid; x < kSeg * DV; x += kThreads) {
            const int i = x / DV, c = x % DV;
            const bool in = i < n;
            const size_t e = (tok0 + t0 + i) * DV + c;
            sm.v[i][c] = in ? ld_io(v, e) : 0.f;
            if (with_q) sm.dout[i][c] = in ? ld_io(dout, e) : 0.f;
        }
        for (int x = tid; x < kSeg * kRows; x += kThreads) {
            const int i = x / kRows, w = x % kRows;
            const bool in = i < n;
            const size_t e = (tok0 + t0 + i) * DK + rb * kRows + w;
            const float kk = in ? ld_io(k, e) : 0.f;
            sm.f[i][w] = in ? (IDPHI ? kk : phi(kk)) : 0.f;
            sm.df[i][w] = IDPHI ? 1.f : dphi(kk);
            sm.g[i][w] = in ? p.gate[e] : 1.f;
            if (with_q) {
                const float qq = in ? ld_io(q, e) : 0.f;
                sm.p[i][w] = in ? (IDPHI ? qq : phi(qq)) : 0.f;
                sm.dp[i][w] = IDPHI ? 1.f : dphi(qq);
            }
        }
    };
    auto step = [&](int i, float* s) {
        const float g = sm.g[i][warp], f = sm.f[i][warp];
#pragma unroll
        for (int j = 0; j < NC; ++j) s[j] = g * s[j] + f * sm.v[i][c0 + j];
    };

    // ---- forward: the rows at the start of every segment -------------------
    float s[NC];
#pragma unroll
    for (int j = 0; j < NC; ++j) s[j] = p.state_in ? p.state_in[bh * ssz + static_cast<size_t>(r) * DV + c0 + j] : 0.f;
    for (int sg = 0; sg < nseg; ++sg) {
        const int t0 = sg * kSeg, n = min(kSeg, T - t0);
        float* dst = ck + static_cast<size_t>(sg) * DK * DV;
#pragma unroll
        for (int j = 0; j < NC; ++j) dst[j] = s[j];
        __syncthreads();
        stage(t0, n, false);
        __syncthreads();
        for (int i = 0; i < n; ++i) step(i, s);
    }

    // ---- backward: segments from the last ---------------------------------
    float D[NC];
#pragma unroll
    for (int j = 0; j < NC; ++j) D[j] = p.dstate_out ? p.dstate_out[bh * ssz + static_cast<size_t>(r) * DV + c0 + j] : 0.f;
    int buf = 0;
    for (int sg = nseg - 1; sg >= 0; --sg) {
        const int t0 = sg * kSeg, n = min(kSeg, T - t0);
        __syncthreads();
        stage(t0, n, true);
        __syncthreads();
        float st[kSeg + 1][NC];
        const float* src = ck + static_cast<size_t>(sg) * DK * DV;
#pragma unroll
        for (int j = 0; j < NC; ++j) st[0][j] = src[j];
#pragma unroll
        for (int i = 0; i < kSeg; ++i) {
#pragma unroll
            for (int j = 0; j < NC; ++j) st[i + 1][j] = st[i][j];
            if (i < n) step(i, st[i + 1]);
        }
#pragma unroll
        for (int i = kSeg - 1; i >= 0; --i) {
            if (i < n) {   // uniform over the CTA
                float* red = &sm.red[buf][warp][0];
                const float pr = sm.p[i][warp], f = sm.f[i][warp];
                float a = 0.f, b = 0.f, c = 0.f;
#pragma unroll
                for (int j = 0; j < NC; ++j) {
                    const float dor = sm.dout[i][c0 + j];
                    D[j] += pr * dor;
                    a += st[i + 1][j] * dor;              // (S_t do_t) row r
                    b += D[j] * sm.v[i][c0 + j];           // (D v_t) row r
                    c += D[j] * st[i][j];                  // rowsum of D o S_{t-1}
                    red[c0 + j] = D[j] * f;                // dv_t, this row's part
                }
                a = warp_sum(a);
                b = warp_sum(b);
                c = warp_sum(c);
                if (lane == 0) {
                    sm.dq[i][warp] = a * sm.dp[i][warp];
                    sm.dk[i][warp] = b * sm.df[i][warp];
                    sm.dg[i][warp] = c;
                }
                const float g = sm.g[i][warp];
#pragma unroll
                for (int j = 0; j < NC; ++j) D[j] *= g;
                __syncthreads();
                const size_t t = tok0 + t0 + i;
                for (int x = tid; x < DV; x += kThreads) {
                    float acc = 0.f;
#pragma unroll
                    for (int w = 0; w < kRows; ++w) acc += sm.red[buf][w][x];
                    atomicAdd(p.dv_acc + t * DV + x, acc);
                }
                buf ^= 1;
            }
        }
        __syncthreads();
        IO* dqo = static_cast<IO*>(p.dq);
        IO* dko = static_cast<IO*>(p.dk);
        for (int x = tid; x < n * kRows; x += kThreads) {
            const int i = x / kRows, w = x % kRows;
            const size_t e = (tok0 + t0 + i) * DK + rb * kRows + w;
            st_io(dqo, e, sm.dq[i][w]);
            st_io(dko, e, sm.dk[i][w]);
            p.dgate[e] = sm.dg[i][w];
        }
    }
    if (p.dstate_in) {
#pragma unroll
        for (int j = 0; j < NC; ++j) p.dstate_in[bh * ssz + static_cast<size_t>(r) * DV + c0 + j] = D[j];
    }
}

// dv from its fp32 accumulator, in the io dtype.
template <typename IO>
__global__ void write_v_kernel(const float* dv_acc, IO* dv, size_t n) {
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        st_io(dv, i, dv_acc[i]);
}

template <int DK, int DV, typename IO, bool IDPHI>
cudaError_t run_gla(const DeltaBwdArgs& p, cudaStream_t s) {
    auto kern = gla_backward_kernel<DK, DV, IO, IDPHI>;
    constexpr size_t smem = sizeof(SmemGla<DV>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<p.BH * (DK / kRows), kThreads, smem, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t n = static_cast<size_t>(p.BH) * p.T * DV;
    write_v_kernel<IO><<<p.sm_count * 4, 256, 0, s>>>(p.dv_acc, static_cast<IO*>(p.dv), n);
    return cudaGetLastError();
}

template <int DK, int DV>
cudaError_t run_gla_io(const DeltaBwdArgs& p, cudaStream_t s) {
    if (p.identity_phi)
        return p.io == kBf16 ? run_gla<DK, DV, __nv_bfloat16, true>(p, s) : run_gla<DK, DV, float, true>(p, s);
    return p.io == kBf16 ? run_gla<DK, DV, __nv_bfloat16, false>(p, s) : run_gla<DK, DV, float, false>(p, s);
}

cudaError_t run_gla_dims(const DeltaBwdArgs& p, cudaStream_t s) {
    if (p.dk_dim == 64 && p.dv_dim == 64) return run_gla_io<64, 64>(p, s);
    if (p.dk_dim == 64 && p.dv_dim == 128) return run_gla_io<64, 128>(p, s);
    if (p.dk_dim == 128 && p.dv_dim == 64) return run_gla_io<128, 64>(p, s);
    if (p.dk_dim == 128 && p.dv_dim == 128) return run_gla_io<128, 128>(p, s);
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// normalized recurrence: rows = key channels, z alongside
// ---------------------------------------------------------------------------
template <int DV>
struct SmemNorm {
    float v[kSeg][DV];
    float dnum[kSeg][DV];     // do / den
    float dden[kSeg];         // -(do . o) / den
    float f[kSeg][kRows];     // phi(k) of the CTA's channels
    float df[kSeg][kRows];    // phi'(k)
    float p[kSeg][kRows];     // phi(q)
    float dp[kSeg][kRows];    // phi'(q)
    float dq[kSeg][kRows];
    float dk[kSeg][kRows];
    float gsum[kRows];        // dgamma, per row
    float red[2][kRows][DV];
};

template <int DK, int DV, typename IO, bool DECAY>
__global__ void __launch_bounds__(kThreads, 2) norm_rows_backward_kernel(DeltaBwdArgs p) {
    constexpr int NC = DV / 32;
    constexpr int NRB = DK / kRows;
    using SM = SmemNorm<DV>;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SM& sm = *reinterpret_cast<SM*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x / NRB, rb = blockIdx.x % NRB;
    const int r = rb * kRows + warp;   // this warp's key channel
    const int c0 = lane * NC;
    const int T = p.T;
    const int nseg = (T + kSeg - 1) / kSeg;
    const size_t tok0 = static_cast<size_t>(bh) * T;
    const IO* q = static_cast<const IO*>(p.q);
    const IO* k = static_cast<const IO*>(p.k);
    const IO* v = static_cast<const IO*>(p.v);
    const IO* dout = static_cast<const IO*>(p.dout);
    const IO* o = static_cast<const IO*>(p.fwd_out);
    const size_t ssz = static_cast<size_t>(DK) * DV + DK;
    const float gam = DECAY ? p.gate[bh] : 1.f;
    float* ck = p.ckpt + (static_cast<size_t>(bh) * nseg * DK + r) * DV + c0;   // + seg * DK * DV
    float* ckz = p.ckz + static_cast<size_t>(bh) * nseg * DK + r;              // + seg * DK

    auto stage = [&](int t0, int n, bool bwd) {
        for (int x = tid; x < kSeg * DV; x += kThreads) {
            const int i = x / DV, c = x % DV;
            const bool in = i < n;
            const size_t e = (tok0 + t0 + i) * DV + c;
            sm.v[i][c] = in ? ld_io(v, e) : 0.f;
            if (bwd) sm.dnum[i][c] = in ? ld_io(dout, e) / p.fwd_den[tok0 + t0 + i] : 0.f;
        }
        if (bwd) {   // warp i: dden of token i
            for (int i = warp; i < kSeg; i += kRows) {
                float d = 0.f;
                if (i < n) {
                    const size_t e = (tok0 + t0 + i) * DV;
                    for (int c = lane; c < DV; c += 32) d += ld_io(dout, e + c) * ld_io(o, e + c);
                }
                d = warp_sum(d);
                if (lane == 0) sm.dden[i] = (i < n) ? -d / p.fwd_den[tok0 + t0 + i] : 0.f;
            }
        }
        for (int x = tid; x < kSeg * kRows; x += kThreads) {
            const int i = x / kRows, w = x % kRows;
            const bool in = i < n;
            const size_t e = (tok0 + t0 + i) * DK + rb * kRows + w;
            const float kk = in ? ld_io(k, e) : 0.f;
            sm.f[i][w] = in ? phi(kk) : 0.f;
            sm.df[i][w] = dphi(kk);
            if (bwd) {
                const float qq = in ? ld_io(q, e) : 0.f;
                sm.p[i][w] = in ? phi(qq) : 0.f;
                sm.dp[i][w] = dphi(qq);
            }
        }
    };
    auto step = [&](int i, float* s, float& z) {
        const float f = sm.f[i][warp];
#pragma unroll
        for (int j = 0; j < NC; ++j) s[j] = gam * s[j] + f * sm.v[i][c0 + j];
        z = gam * z + f;
    };

    // ---- forward: the rows (and z) at the start of every segment ----------
    float s[NC];
    float z = p.state_in ? p.state_in[bh * ssz + static_cast<size_t>(DK) * DV + r] : 0.f;
#pragma unroll
    for (int j = 0; j < NC; ++j) s[j] = p.state_in ? p.state_in[bh * ssz + static_cast<size_t>(r) * DV + c0 + j] : 0.f;
    for (int sg = 0; sg < nseg; ++sg) {
        const int t0 = sg * kSeg, n = min(kSeg, T - t0);
        float* dst = ck + static_cast<size_t>(sg) * DK * DV;
#pragma unroll
        for (int j = 0; j < NC; ++j) dst[j] = s[j];
        if (lane == 0) ckz[static_cast<size_t>(sg) * DK] = z;
        __syncthreads();
        stage(t0, n, false);
        __syncthreads();
        for (int i = 0; i < n; ++i) step(i, s, z);
    }

    // ---- backward: segments from the last ---------------------------------
    float G[NC];
    float gz = p.dstate_out ? p.dstate_out[bh * ssz + static_cast<size_t>(DK) * DV + r] : 0.f;
#pragma unroll
    for (int j = 0; j < NC; ++j) G[j] = p.dstate_out ? p.dstate_out[bh * ssz + static_cast<size_t>(r) * DV + c0 + j] : 0.f;
    float gacc = 0.f;   // dgamma: this lane's part of row r's sum
    int buf = 0;
    for (int sg = nseg - 1; sg >= 0; --sg) {
        const int t0 = sg * kSeg, n = min(kSeg, T - t0);
        __syncthreads();
        stage(t0, n, true);
        __syncthreads();
        float st[kSeg + 1][NC];
        float zs[kSeg + 1];
        const float* src = ck + static_cast<size_t>(sg) * DK * DV;
#pragma unroll
        for (int j = 0; j < NC; ++j) st[0][j] = src[j];
        zs[0] = ckz[static_cast<size_t>(sg) * DK];
#pragma unroll
        for (int i = 0; i < kSeg; ++i) {
#pragma unroll
            for (int j = 0; j < NC; ++j) st[i + 1][j] = st[i][j];
            zs[i + 1] = zs[i];
            if (i < n) step(i, st[i + 1], zs[i + 1]);
        }
#pragma unroll
        for (int i = kSeg - 1; i >= 0; --i) {
            if (i < n) {   // uniform over the CTA
                float* red = &sm.red[buf][warp][0];
                const float pr = sm.p[i][warp], f = sm.f[i][warp], dd = sm.dden[i];
                gz += pr * dd;
                float a = 0.f, b = 0.f;
#pragma unroll
                for (int j = 0; j < NC; ++j) {
                    const float dn = sm.dnum[i][c0 + j];
                    G[j] += pr * dn;
                    a += st[i + 1][j] * dn;               // (S_t dnum_t) row r
                    b += G[j] * sm.v[i][c0 + j];           // (G v_t) row r
                    if (DECAY) gacc += G[j] * st[i][j];    // <G, S_{t-1}> row r
                    red[c0 + j] = G[j] * f;                // dv_t, this row's part
                }
                if (DECAY && lane == 0) gacc += gz * zs[i];   // <g, z_{t-1}> row r
                a = warp_sum(a) + zs[i + 1] * dd;
                b = warp_sum(b) + gz;
                if (lane == 0) {
                    sm.dq[i][warp] = a * sm.dp[i][warp];
                    sm.dk[i][warp] = b * sm.df[i][warp];
                }
#pragma unroll
                for (int j = 0; j < NC; ++j) G[j] *= gam;
                gz *= gam;
                __syncthreads();
                const size_t t = tok0 + t0 + i;
                for (int x = tid; x < DV; x += kThreads) {
                    float acc = 0.f;
#pragma unroll
                    for (int w = 0; w < kRows; ++w) acc += sm.red[buf][w][x];
                    atomicAdd(p.dv_acc + t * DV + x, acc);
                }
                buf ^= 1;
            }
        }
        __syncthreads();
        IO* dqo = static_cast<IO*>(p.dq);
        IO* dko = static_cast<IO*>(p.dk);
        for (int x = tid; x < n * kRows; x += kThreads) {
            const int i = x / kRows, w = x % kRows;
            const size_t e = (tok0 + t0 + i) * DK + rb * kRows + w;
            st_io(dqo, e, sm.dq[i][w]);
            st_io(dko, e, sm.dk[i][w]);
        }
    }
    if (p.dstate_in) {
#pragma unroll
        for (int j = 0; j < NC; ++j) p.dstate_in[bh * ssz + static_cast<size_t>(r) * DV + c0 + j] = G[j];
        if (lane == 0) p.dstate_in[bh * ssz + static_cast<size_t>(DK) * DV + r] = gz;
    }
    if (DECAY) {
        gacc = warp_sum(gacc);
        if (lane == 0) sm.gsum[warp] = gacc;
        __syncthreads();
        if (tid == 0) {
            float t = 0.f;
            for (int w = 0; w < kRows; ++w) t += sm.gsum[w];
            atomicAdd(p.dgate + bh, t);
        }
    }
}

template <int DK, int DV, typename IO, bool DECAY>
cudaError_t run_norm_rows(const DeltaBwdArgs& p, cudaStream_t s) {
    auto kern = norm_rows_backward_kernel<DK, DV, IO, DECAY>;
    constexpr size_t smem = sizeof(SmemNorm<DV>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<p.BH * (DK / kRows), kThreads, smem, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t n = static_cast<size_t>(p.BH) * p.T * DV;
    write_v_kernel<IO><<<p.sm_count * 4, 256, 0, s>>>(p.dv_acc, static_cast<IO*>(p.dv), n);
    return cudaGetLastError();
}

template <int DK, int DV>
cudaError_t run_norm_rows_io(const DeltaBwdArgs& p, cudaStream_t s) {
    const bool decay = p.gate != nullptr;
    if (decay)
        return p.io == kBf16 ? run_norm_rows<DK, DV, __nv_bfloat16, true>(p, s) : run_norm_rows<DK, DV, float, true>(p, s);
    return p.io == kBf16 ? run_norm_rows<DK, DV, __nv_bfloat16, false>(p, s) : run_norm_rows<DK, DV, float, false>(p, s);
}

cudaError_t run_norm_rows_dims(const DeltaBwdArgs& p, cudaStream_t s) {
    if (p.dk_dim == 64 && p.dv_dim == 64) return run_norm_rows_io<64, 64>(p, s);
    if (p.dk_dim == 64 && p.dv_dim == 128) return run_norm_rows_io<64, 128>(p, s);
    if (p.dk_dim == 128 && p.dv_dim == 64) return run_norm_rows_io<128, 64>(p, s);
    if (p.dk_dim == 128 && p.dv_dim == 128) return run_norm_rows_io<128, 128>(p, s);
    return cudaErrorInvalidValue;
}

// dq and dk from the fp32 accumulators, in the io dtype.
template <typename IO>
__global__ void write_qk_kernel(const float* dq_acc, const float* dk_acc, IO* dq, IO* dk, size_t n) {
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        st_io(dq, i, dq_acc[i]);
        st_io(dk, i, dk_acc[i]);
    }
}

template <int DK, int DV, bool PC, typename IO>
cudaError_t run(const DeltaBwdArgs& p, cudaStream_t s) {
    auto kern = delta_backward_kernel<DK, DV, PC, IO>;
    constexpr size_t smem = sizeof(Smem<DK, PC>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<p.BH * (DV / kRows), kThreads, smem, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t n = static_cast<size_t>(p.BH) * p.T * DK;
    write_qk_kernel<IO><<<p.sm_count * 4, 256, 0, s>>>(p.dq_acc, p.dk_acc, static_cast<IO*>(p.dq),
                                                        static_cast<IO*>(p.dk), n);
    return cudaGetLastError();
}

template <int DK, int DV, bool PC>
cudaError_t run_io(const DeltaBwdArgs& p, cudaStream_t s) {
    return p.io == kBf16 ? run<DK, DV, PC, __nv_bfloat16>(p, s) : run<DK, DV, PC, float>(p, s);
}

template <bool PC>
cudaError_t run_dims(const DeltaBwdArgs& p, cudaStream_t s) {
    if (p.dk_dim == 64 && p.dv_dim == 64) return run_io<64, 64, PC>(p, s);
    if (p.dk_dim == 64 && p.dv_dim == 128) return run_io<64, 128, PC>(p, s);
    if (p.dk_dim == 128 && p.dv_dim == 64) return run_io<128, 64, PC>(p, s);
    if (p.dk_dim == 128 && p.dv_dim == 128) return run_io<128, 128, PC>(p, s);
    return cudaErrorInvalidValue;
}

}  // namespace

size_t norm_rows_fwd_bytes(int BH, int T, int dv, int io) {
    const size_t o = (static_cast<size_t>(BH) * T * dv * (io == kBf16 ? 2 : 4) + 255) & ~static_cast<size_t>(255);
    const size_t den = (static_cast<size_t>(BH) * T * 4 + 255) & ~static_cast<size_t>(255);
    return o + den;
}

size_t norm_rows_bytes(int BH, int T, int dk, int dv) {
    const size_t nseg = static_cast<size_t>((T + kSeg - 1) / kSeg);
    return static_cast<size_t>(BH) * (nseg * dk * (dv + 1) + static_cast<size_t>(T) * dv) * sizeof(float);
}

size_t delta_backward_bytes(int BH, int T, int dk, int dv, bool gla) {
    const size_t nseg = static_cast<size_t>((T + kSeg - 1) / kSeg);
    const size_t acc = gla ? static_cast<size_t>(T) * dv : 2 * static_cast<size_t>(T) * dk;
    return static_cast<size_t>(BH) * (nseg * dv * dk + acc) * sizeof(float);
}

cudaError_t launch_delta_backward(const DeltaBwdArgs& args, cudaStream_t s) {
    if (!args.workspace) return cudaErrorInvalidValue;
    DeltaBwdArgs a = args;
    const size_t nseg = static_cast<size_t>((a.T + kSeg - 1) / kSeg);
    a.ckpt = a.workspace;
    if (a.norm) {   // rows and z at every segment start, then the fp32 total of dv
        a.ckz = a.ckpt + static_cast<size_t>(a.BH) * nseg * a.dk_dim * a.dv_dim;
        a.dv_acc = a.ckz + static_cast<size_t>(a.BH) * nseg * a.dk_dim;
        cudaError_t e = cudaMemsetAsync(a.dv_acc, 0, static_cast<size_t>(a.BH) * a.T * a.dv_dim * sizeof(float), s);
        if (e == cudaSuccess && a.gate && a.dgate) e = cudaMemsetAsync(a.dgate, 0, static_cast<size_t>(a.BH) * sizeof(float), s);
        if (e != cudaSuccess) return e;
        return run_norm_rows_dims(a, s);
    }
    if (a.gla) {   // rows at every segment start, then the fp32 total of dv
        a.dv_acc = a.ckpt + static_cast<size_t>(a.BH) * nseg * a.dv_dim * a.dk_dim;
        cudaError_t e = cudaMemsetAsync(a.dv_acc, 0, static_cast<size_t>(a.BH) * a.T * a.dv_dim * sizeof(float), s);
        if (e != cudaSuccess) return e;
        return run_gla_dims(a, s);
    }
    a.dq_acc = a.ckpt + static_cast<size_t>(a.BH) * nseg * a.dv_dim * a.dk_dim;
    a.dk_acc = a.dq_acc + static_cast<size_t>(a.BH) * a.T * a.dk_dim;
    // the column sums are accumulated: clear their totals first
    const size_t qk = static_cast<size_t>(a.BH) * a.T * a.dk_dim * sizeof(float);
    cudaError_t e = cudaMemsetAsync(a.dq_acc, 0, qk, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.dk_acc, 0, qk, s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(a.dgate, 0, static_cast<size_t>(a.BH) * a.T * (a.per_channel ? a.dk_dim : 1) * sizeof(float), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.dbeta, 0, static_cast<size_t>(a.BH) * a.T * sizeof(float), s);
    if (e != cudaSuccess) return e;
    return a.per_channel ? run_dims<true>(a, s) : run_dims<false>(a, s);
}

}  // namespace la
