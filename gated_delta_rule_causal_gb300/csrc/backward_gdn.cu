// Chunkwise gradients of the gated delta rule with a scalar gate (bf16 io,
// d_k = d_v = D in {64, 128}).
//
// Forward operator ("Beyond attention" §18.2, the decay applied to the state
// before the error is taken), S in R^{D x D} (value rows, key columns):
//    S_t = g_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t.
// In the WY/UT chunk form (C = 64 tokens; b_r = sum of ln g inside the chunk up
// to token r, gam_r = e^{b_r}, gam_C = e^{b_63}, lam_s = gam_C / gam_s,
// E_rs = e^{b_r - b_s}):
//    A  = strictly lower(diag(beta) E o K K^T),  Ti = (I + A)^{-1}
//    W  = Ti diag(beta gam) K,  Ut = Ti diag(beta) V,  U = Ut - W S_0^T
//    P  = lower(E o Q K^T),     O  = diag(gam) Q S_0^T + P U
//    S_C = gam_C S_0 + U^T diag(lam) K.
// The pages give no gradients; by the chain rule through these lines, with
// dS_C the gradient reaching a chunk's last state:
//    dU  = P^T dO + diag(lam) K dS_C^T,   dW = -dU S_0
//    dRv = Ti^T dU,  dRk = Ti^T dW,       dA = -(dRv Ut^T + dRk W^T)  (strictly lower)
//    dV  = diag(beta) dRv,                dP = lower(dO U^T)
//    dQ  = diag(gam) dO S_0 + (dP o E) K
//    dK  = (dP o E)^T Q + diag(lam) U dS_C + diag(beta gam) dRk + F K + F^T K,
//          F = diag(beta) (dA o E)
//    dbeta_r = dRv_r.v_r + gam_r dRk_r.k_r + sum_s (dA o E o K K^T)_rs
//    db_r    = gam_r dO_r.(S_0 q_r) + beta_r gam_r dRk_r.k_r
//              + row minus column sums of dP o P and of dA o A
//              - c_r, c_s = lam_s (U dS_C)_s.k_s,  and at the last token
//              + gam_C <dS_C, S_0> + sum_s c_s
//    dln g_t = sum_{r >= t in the chunk} db_r,   dg = dln g / g.
// Across chunks the state and its gradient follow one linear map per chunk,
// X <- gam_C X - (X A'^T) B' + C'^T D':
//    S (first chunk to last):  (A', B', C', D') = (W, lam K, Ut, lam K)
//    dS (last chunk to first): (A', B', C', D') = (K, lam W, dO, gam Q - P W).
// Every value row of X follows that map on its own, so the two chains split
// by rows.
//
// Five launches per call:
//  1. prep, one CTA per (sequence-head, chunk): gate prefix sums, K K^T and
//     Q K^T, Ti in fp32 (16x16 diagonal blocks by forward substitution, then
//     two merge levels), W, Ut and Qh = gam Q - P W; fp32 into the workspace.
//  2. the state chain, one CTA per (sequence-head, 32 value rows), walking the
//     chunks with the rows in fp32 and storing every chunk's S_0 (bf16). It
//     also forms the gate term gam_r dO_r.(S_0 q_r) from the fp32 rows (as
//     two tf32 halves): that term cancels against the others of the gate
//     gradient, and bf16 rows would cost it up to ~3% of the result.
//  3. the gradient chain, the same from the last chunk, storing every chunk's
//     dS_C (bf16) and the gradient of the initial state (fp32).
//  4. the state-dependent gradients per chunk: U, dU, dW, dQ (final), the
//     state terms of dK and of the gate gradient.
//  5. the rest per chunk: dRv, dRk, dA, dV, dK, dbeta and the gate gradient.
// Every product is a warp-level tf32 MMA (m16n8k8, fp32 accumulation) on
// shared-memory tiles; the chains prefetch the next chunk's tiles with
// asynchronous copies while they compute the current one.
//
// Tail chunks: rows past T load as zeros, with g = 1 and beta = 0, so they
// leave every real row's result unchanged; no row past T is written.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace la {
namespace gbw {

constexpr int C = 64;            // tokens per chunk
constexpr int kThreads = 256;    // eight warps
constexpr int kRows = 32;        // value rows per chain CTA
using bf16 = __nv_bfloat16;

template <int D>
struct Dims {
    static constexpr int FD = D + 4;    // fp32 row stride of a C x D tile (floats)
    static constexpr int HD = D + 8;    // bf16 row stride of a C x D or D x D tile (elements)
    static constexpr int FC = C + 4;    // fp32 row stride of a C x C tile
    static constexpr int NT = D / 32;   // n-tiles of a warp's 32 x (D/4) part of a C x D product
};

struct Params {
    const bf16* q;
    const bf16* k;
    const bf16* v;
    const bf16* dout;
    const float* gate;
    const float* beta;
    const float* state_in;
    const float* dstate_out;
    bf16* dq;
    bf16* dk;
    bf16* dv;
    float* dgate;
    float* dbeta;
    float* dstate_in;
    int BH, T, NC;
    // workspace, per (sequence-head, chunk) unit
    float* wb;     // [C]     ln-gate prefix sums
    float* wti;    // [C][C]  Ti
    float* ww;     // [C][D]  W
    float* wut;    // [C][D]  Ut
    float* wqh;    // [C][D]  Qh
    bf16* ws0;     // [D][D]  S_0
    bf16* wsc;     // [D][D]  dS_C
    float* wdu;    // [C][D]  dU
    float* wdw;    // [C][D]  dW
    float* wdk;    // [C][D]  state terms of dK
    float* wdb;    // [C]     state terms of the gate gradient
    float* wdb0;   // [C]     gam_r dO_r.(S_0 q_r), summed over the state chain's CTAs
};

__device__ __forceinline__ float bf(const bf16* p, int i) { return __bfloat162float(p[i]); }

// acc[MT][NT] (+)= sum over k in [k0, k1) of fa(m, k) fb(k, n) for the warp's
// (16 MT) x (8 NT) tile at (m0, n0); k0, k1 multiples of 8.
template <int MT, int NT, class FA, class FB>
__device__ __forceinline__ void warp_mma(float (&acc)[MT][NT][4], const FA& fa, const FB& fb, int m0, int n0, int k0,
                                         int k1) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    for (int k = k0; k < k1; k += 8) {
        uint32_t a[MT][4], b[NT][2];
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            const int m = m0 + 16 * i + g;
            a[i][0] = to_tf32(fa(m, k + t));
            a[i][1] = to_tf32(fa(m + 8, k + t));
            a[i][2] = to_tf32(fa(m, k + t + 4));
            a[i][3] = to_tf32(fa(m + 8, k + t + 4));
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const int n = n0 + 8 * j + g;
            b[j][0] = to_tf32(fb(k + t, n));
            b[j][1] = to_tf32(fb(k + t + 4, n));
        }
#pragma unroll
        for (int i = 0; i < MT; ++i)
#pragma unroll
            for (int j = 0; j < NT; ++j) mma_tf32_m16n8k8(acc[i][j], a[i], b[j]);
    }
}

template <int MT, int NT>
__device__ __forceinline__ void zero(float (&acc)[MT][NT][4]) {
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;
}

// f(row, col, value&) for every accumulator element of the warp's tile.
template <int MT, int NT, class F>
__device__ __forceinline__ void for_acc(float (&acc)[MT][NT][4], int m0, int n0, const F& f) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) f(m0 + 16 * i + g + 8 * (e >> 1), n0 + 8 * j + 2 * t + (e & 1), acc[i][j][e]);
}

// Sum of per-row partials (h[i][0]: row m0+16i+g, h[i][1]: row +8) over the
// four lanes of a quad, added to s[row] by its first lane.
template <int MT>
__device__ __forceinline__ void add_rows(float (&h)[MT][2], int m0, float* s) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float x = h[i][e];
            x += __shfl_xor_sync(0xffffffffu, x, 1);
            x += __shfl_xor_sync(0xffffffffu, x, 2);
            if (t == 0) atomicAdd(s + m0 + 16 * i + g + 8 * e, x);
        }
}

// Sum of per-column partials (h[j][0]: col n0+8j+2t, h[j][1]: +1) over the
// eight lanes sharing t, added to s[col] by the lanes with g = 0.
template <int NT>
__device__ __forceinline__ void add_cols(float (&h)[NT][2], int n0, float* s) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float x = h[j][e];
            x += __shfl_xor_sync(0xffffffffu, x, 4);
            x += __shfl_xor_sync(0xffffffffu, x, 8);
            x += __shfl_xor_sync(0xffffffffu, x, 16);
            if (g == 0) atomicAdd(s + n0 + 8 * j + 2 * t + e, x);
        }
}

// rows x (cols) tile copy, global row stride gs, shared row stride ss (both in
// elements of T), rows >= valid filled with zeros; 16-byte pieces.
template <typename T>
__device__ __forceinline__ void load_tile(T* dst, int ss, const T* src, size_t gs, int rows, int cols, int valid) {
    constexpr int E = 16 / sizeof(T);
    const int per = cols / E;
    for (int x = threadIdx.x; x < rows * per; x += blockDim.x) {
        const int r = x / per, c = (x % per) * E;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (r < valid) val = *reinterpret_cast<const uint4*>(src + r * gs + c);
        *reinterpret_cast<uint4*>(dst + r * ss + c) = val;
    }
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool full) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(full ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

template <typename T>
__device__ __forceinline__ void copy_tile_async(T* dst, int ss, const T* src, size_t gs, int rows, int cols,
                                                int valid) {
    constexpr int E = 16 / sizeof(T);
    const int per = cols / E;
    for (int x = threadIdx.x; x < rows * per; x += blockDim.x) {
        const int r = x / per, c = (x % per) * E;
        const bool in = r < valid;
        cp_async16(dst + r * ss + c, in ? src + r * gs + c : src, in);
    }
}

// Gate prefix sums of one chunk by warp 0: b (ln g summed up to each token;
// padded tokens add 0), beta (0 when padded).
__device__ __forceinline__ void gate_sums(const Params& p, size_t tok0, int n, float* vb, float* vbeta) {
    if (threadIdx.x >= 32) return;
    const int lane = threadIdx.x;
    float lo = lane < n ? logf(p.gate[tok0 + lane]) : 0.f;
    float hi = lane + 32 < n ? logf(p.gate[tok0 + lane + 32]) : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float a = __shfl_up_sync(0xffffffffu, lo, o), b = __shfl_up_sync(0xffffffffu, hi, o);
        if (lane >= o) {
            lo += a;
            hi += b;
        }
    }
    hi += __shfl_sync(0xffffffffu, lo, 31);
    vb[lane] = lo;
    vb[lane + 32] = hi;
    if (vbeta) {
        vbeta[lane] = lane < n ? p.beta[tok0 + lane] : 0.f;
        vbeta[lane + 32] = lane + 32 < n ? p.beta[tok0 + lane + 32] : 0.f;
    }
}

// ---------------------------------------------------------------------------
// 1. prep
// ---------------------------------------------------------------------------
template <int D>
struct PrepSmem {
    using Dm = Dims<D>;
    static constexpr size_t OFF_K = size_t(C) * Dm::HD * 2;
    static constexpr size_t OFF_V = OFF_K + size_t(C) * Dm::HD * 2;
    static constexpr size_t OFF_A = OFF_V + size_t(C) * Dm::HD * 2;   // K K^T -> A -> P Ti
    static constexpr size_t OFF_P = OFF_A + size_t(C) * Dm::FC * 4;
    static constexpr size_t OFF_T = OFF_P + size_t(C) * Dm::FC * 4;
    static constexpr size_t OFF_X = OFF_T + size_t(C) * Dm::FC * 4;   // 32 x 33 merge scratch
    static constexpr size_t OFF_VEC = OFF_X + 32 * 33 * 4;
    static constexpr size_t BYTES = OFF_VEC + 4 * C * 4;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 2) prep_kernel(const Params p) {
    using Dm = Dims<D>;
    using L = PrepSmem<D>;
    constexpr int FC = Dm::FC, HD = Dm::HD;
    extern __shared__ __align__(16) uint8_t smem[];
    bf16* sQ = reinterpret_cast<bf16*>(smem);
    bf16* sK = reinterpret_cast<bf16*>(smem + L::OFF_K);
    bf16* sV = reinterpret_cast<bf16*>(smem + L::OFF_V);
    float* sA = reinterpret_cast<float*>(smem + L::OFF_A);
    float* sP = reinterpret_cast<float*>(smem + L::OFF_P);
    float* sT = reinterpret_cast<float*>(smem + L::OFF_T);
    float* sX = reinterpret_cast<float*>(smem + L::OFF_X);
    float* vb = reinterpret_cast<float*>(smem + L::OFF_VEC);
    float* vbeta = vb + C;
    float* vgam = vbeta + C;
    float* vbg = vgam + C;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int unit = blockIdx.x, bh = unit / p.NC, c = unit % p.NC;
    const int n = min(C, p.T - c * C);
    const size_t tok0 = static_cast<size_t>(bh) * p.T + static_cast<size_t>(c) * C;

    load_tile(sQ, HD, p.q + tok0 * D, D, C, D, n);
    load_tile(sK, HD, p.k + tok0 * D, D, C, D, n);
    load_tile(sV, HD, p.v + tok0 * D, D, C, D, n);
    gate_sums(p, tok0, n, vb, vbeta);
    for (int x = tid; x < C * FC; x += kThreads) sT[x] = 0.f;
    __syncthreads();
    if (tid < C) {
        vgam[tid] = expf(vb[tid]);
        vbg[tid] = vbeta[tid] * vgam[tid];
    }
    // K K^T -> A, Q K^T -> P (one B fragment feeds both)
    {
        const int m0 = (warp >> 2) * 32, n0 = (warp & 3) * 16;
        float kk[2][2][4], qk[2][2][4];
        zero(kk);
        zero(qk);
        const auto fk = [&](int m, int k) { return bf(sK, m * HD + k); };
        const auto fq = [&](int m, int k) { return bf(sQ, m * HD + k); };
        const auto fkt = [&](int k, int nn) { return bf(sK, nn * HD + k); };
        warp_mma<2, 2>(kk, fk, fkt, m0, n0, 0, D);
        warp_mma<2, 2>(qk, fq, fkt, m0, n0, 0, D);
        for_acc(kk, m0, n0, [&](int r, int s, float& x) {
            sA[r * FC + s] = s < r ? vbeta[r] * expf(vb[r] - vb[s]) * x : 0.f;
        });
        for_acc(qk, m0, n0, [&](int r, int s, float& x) {
            sP[r * FC + s] = s <= r ? expf(vb[r] - vb[s]) * x : 0.f;
        });
    }
    __syncthreads();
    // Ti = (I + A)^{-1}: diagonal 16 x 16 blocks by forward substitution
    if (tid < C) {
        const int o = (tid >> 4) * 16, j = tid & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = r == j ? 1.f : 0.f;
#pragma unroll
        for (int r = 1; r < 16; ++r) {
            if (r > j) {
                float s = 0.f;
#pragma unroll
                for (int q = 0; q < r; ++q) s += sA[(o + r) * FC + o + q] * x[q];
                x[r] = -s;
            }
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sT[(o + r) * FC + o + j] = x[r];
    }
    __syncthreads();
    // merges: [T11 0; T21 T22] with T21 = -T22 A21 T11, blocks of 16 then 32
#pragma unroll 1
    for (int h = 16; h <= 32; h *= 2) {
        const int nm = C / (2 * h);   // merges at this level
        for (int x = tid; x < nm * h * h; x += kThreads) {
            const int mi = x / (h * h), r = (x / h) % h, j = x % h, o = mi * 2 * h;
            float s = 0.f;
            for (int q = j; q < h; ++q) s += sA[(o + h + r) * FC + o + q] * sT[(o + q) * FC + o + j];
            sX[mi * h * h + r * h + j] = s;   // X = A21 T11
        }
        __syncthreads();
        for (int x = tid; x < nm * h * h; x += kThreads) {
            const int mi = x / (h * h), r = (x / h) % h, j = x % h, o = mi * 2 * h;
            float s = 0.f;
            for (int q = 0; q <= r; ++q) s += sT[(o + h + r) * FC + o + h + q] * sX[mi * h * h + q * h + j];
            sT[(o + h + r) * FC + o + j] = -s;
        }
        __syncthreads();
    }
    const size_t ub = static_cast<size_t>(unit);
    // W = Ti diag(beta gam) K and Ut = Ti diag(beta) V (Ti lower: k < m0 + 32)
    {
        constexpr int NT = Dm::NT;
        const int m0 = (warp >> 2) * 32, n0 = (warp & 3) * (D / 4);
        float w[2][NT][4], u[2][NT][4];
        zero(w);
        zero(u);
        const auto fw = [&](int m, int k) { return sT[m * FC + k] * vbg[k]; };
        const auto fu = [&](int m, int k) { return sT[m * FC + k] * vbeta[k]; };
        const auto fK = [&](int k, int nn) { return bf(sK, k * HD + nn); };
        const auto fV = [&](int k, int nn) { return bf(sV, k * HD + nn); };
        warp_mma<2, NT>(w, fw, fK, m0, n0, 0, m0 + 32);
        warp_mma<2, NT>(u, fu, fV, m0, n0, 0, m0 + 32);
        float* gw = p.ww + ub * C * D;
        float* gu = p.wut + ub * C * D;
        for_acc(w, m0, n0, [&](int r, int cc, float& x) { gw[r * D + cc] = x; });
        for_acc(u, m0, n0, [&](int r, int cc, float& x) { gu[r * D + cc] = x; });
    }
    // P Ti -> sA (A is no longer read)
    {
        const int m0 = (warp >> 2) * 32, n0 = (warp & 3) * 16;
        float pt[2][2][4];
        zero(pt);
        const auto fp = [&](int m, int k) { return sP[m * FC + k]; };
        const auto ft = [&](int k, int nn) { return sT[k * FC + nn]; };
        warp_mma<2, 2>(pt, fp, ft, m0, n0, 0, m0 + 32);
        for_acc(pt, m0, n0, [&](int r, int s, float& x) { sA[r * FC + s] = x; });
    }
    __syncthreads();
    // Qh = diag(gam) Q - (P Ti) diag(beta gam) K
    {
        constexpr int NT = Dm::NT;
        const int m0 = (warp >> 2) * 32, n0 = (warp & 3) * (D / 4);
        float qh[2][NT][4];
        zero(qh);
        const auto fa = [&](int m, int k) { return sA[m * FC + k] * vbg[k]; };
        const auto fK = [&](int k, int nn) { return bf(sK, k * HD + nn); };
        warp_mma<2, NT>(qh, fa, fK, m0, n0, 0, m0 + 32);
        float* gq = p.wqh + ub * C * D;
        for_acc(qh, m0, n0, [&](int r, int cc, float& x) { gq[r * D + cc] = vgam[r] * bf(sQ, r * HD + cc) - x; });
    }
    float* gt = p.wti + ub * C * C;
    for (int x = tid; x < C * C; x += kThreads) gt[x] = sT[(x / C) * FC + x % C];
    if (tid < C) {
        p.wb[ub * C + tid] = vb[tid];
        p.wdb0[ub * C + tid] = 0.f;   // the state chain adds into it
    }
}

// ---------------------------------------------------------------------------
// 2, 3. chains over the chunks, 32 value rows per CTA
// ---------------------------------------------------------------------------
template <int D>
struct ChainSmem {
    using Dm = Dims<D>;
    static constexpr size_t F_TILE = size_t(C) * Dm::FD * 4;
    static constexpr size_t H_TILE = size_t(C) * Dm::HD * 2;
    static constexpr size_t S_TILE = size_t(C) * (kRows + 4) * 4;   // fp32 [C][R+4] or bf16 [C][R+8]
    static constexpr size_t Q_TILE = H_TILE;                         // state chain: Q, then the dO slice
    static_assert(Q_TILE + size_t(C) * (kRows + 8) * 2 <= F_TILE, "Q and the dO slice fit the Qh slot");
    static constexpr size_t STAGE = 2 * F_TILE + H_TILE + S_TILE + C * 4;
    static constexpr size_t OFF_X = 2 * STAGE;
    static constexpr size_t OFF_Z = OFF_X + size_t(kRows) * Dm::FD * 4;
    static constexpr size_t BYTES = OFF_Z + size_t(kRows) * Dm::FC * 4;
};

template <int D, bool REV>
__global__ void __launch_bounds__(kThreads, 1) chain_kernel(const Params p) {
    using Dm = Dims<D>;
    using L = ChainSmem<D>;
    constexpr int FD = Dm::FD, HD = Dm::HD, FC = Dm::FC, R = kRows;
    constexpr int SF = R + 4, SH = R + 8;   // slice strides: fp32 Ut, bf16 dO
    extern __shared__ __align__(16) uint8_t smem[];
    float* sX = reinterpret_cast<float*>(smem + L::OFF_X);
    float* sZ = reinterpret_cast<float*>(smem + L::OFF_Z);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int nrb = D / R, bh = blockIdx.x / nrb, row0 = (blockIdx.x % nrb) * R;
    __shared__ float sdb[C];   // state chain: this CTA's part of gam_r dO_r.(S_0 q_r)
    const int NC = p.NC;
    const size_t ss = static_cast<size_t>(D) * D;

    // stage layout: F0 (W), F1 (Qh, gradient chain), H (K), S (Ut or dO slice), b
    auto stage_ptr = [&](int buf, size_t off) { return smem + buf * L::STAGE + off; };
    auto issue = [&](int j, int buf) {
        const int c = REV ? NC - 1 - j : j;
        const int n = min(C, p.T - c * C);
        const size_t ub = static_cast<size_t>(bh) * NC + c;
        const size_t tok0 = static_cast<size_t>(bh) * p.T + static_cast<size_t>(c) * C;
        copy_tile_async(reinterpret_cast<float*>(stage_ptr(buf, 0)), FD, p.ww + ub * C * D, D, C, D, C);
        if (REV) {
            copy_tile_async(reinterpret_cast<float*>(stage_ptr(buf, L::F_TILE)), FD, p.wqh + ub * C * D, D, C, D, C);
            copy_tile_async(reinterpret_cast<bf16*>(stage_ptr(buf, 2 * L::F_TILE + L::H_TILE)), SH,
                            p.dout + tok0 * D + row0, D, C, R, n);
        } else {
            copy_tile_async(reinterpret_cast<float*>(stage_ptr(buf, 2 * L::F_TILE + L::H_TILE)), SF,
                            p.wut + ub * C * D + row0, D, C, R, C);
            copy_tile_async(reinterpret_cast<bf16*>(stage_ptr(buf, L::F_TILE)), HD, p.q + tok0 * D, D, C, D, n);
            copy_tile_async(reinterpret_cast<bf16*>(stage_ptr(buf, L::F_TILE + L::Q_TILE)), SH,
                            p.dout + tok0 * D + row0, D, C, R, n);
        }
        copy_tile_async(reinterpret_cast<bf16*>(stage_ptr(buf, 2 * L::F_TILE)), HD, p.k + tok0 * D, D, C, D, n);
        copy_tile_async(reinterpret_cast<float*>(stage_ptr(buf, 2 * L::F_TILE + L::H_TILE + L::S_TILE)), C,
                        p.wb + ub * C, C, 1, C, 1);
    };

    const float* x0 = REV ? p.dstate_out : p.state_in;
    for (int x = tid; x < R * D; x += kThreads) {
        const int r = x / D, cc = x % D;
        sX[r * FD + cc] = x0 ? x0[bh * ss + static_cast<size_t>(row0 + r) * D + cc] : 0.f;
    }
    issue(0, 0);
    cp_async_commit();
    if (NC > 1) issue(1, 1);
    cp_async_commit();

    bf16* gout = REV ? p.wsc : p.ws0;
    for (int j = 0; j < NC; ++j) {
        const int buf = j & 1;
        const int c = REV ? NC - 1 - j : j;
        const float* tW = reinterpret_cast<const float*>(stage_ptr(buf, 0));
        const float* tQh = reinterpret_cast<const float*>(stage_ptr(buf, L::F_TILE));
        const bf16* tK = reinterpret_cast<const bf16*>(stage_ptr(buf, 2 * L::F_TILE));
        const float* tUt = reinterpret_cast<const float*>(stage_ptr(buf, 2 * L::F_TILE + L::H_TILE));
        const bf16* tdO = reinterpret_cast<const bf16*>(stage_ptr(buf, 2 * L::F_TILE + L::H_TILE));
        const float* tb = reinterpret_cast<const float*>(stage_ptr(buf, 2 * L::F_TILE + L::H_TILE + L::S_TILE));
        cp_async_wait1();
        __syncthreads();   // this chunk's tiles and the rows' last update are visible
        {
            bf16* o = gout + (static_cast<size_t>(bh) * NC + c) * ss + static_cast<size_t>(row0) * D;
            for (int x = tid; x < R * D / 2; x += kThreads) {
                const int r = (2 * x) / D, cc = (2 * x) % D;
                *reinterpret_cast<__nv_bfloat162*>(o + r * D + cc) =
                    __floats2bfloat162_rn(sX[r * FD + cc], sX[r * FD + cc + 1]);
            }
        }
        const float bC = tb[C - 1];
        // Y = X A'^T (32 x C), Z = (Ut^T - Y) diag(lam) or -Y diag(lam)
        {
            const int n0 = warp * 8;
            float y[2][1][4];
            zero(y);
            const auto fx = [&](int m, int k) { return sX[m * FD + k]; };
            if (REV) {
                warp_mma<2, 1>(y, fx, [&](int k, int nn) { return bf(tK, nn * HD + k); }, 0, n0, 0, D);
            } else {
                warp_mma<2, 1>(y, fx, [&](int k, int nn) { return tW[nn * FD + k]; }, 0, n0, 0, D);
            }
            for_acc(y, 0, n0, [&](int m, int s, float& x) {
                const float lam = expf(bC - tb[s]);
                sZ[m * FC + s] = REV ? -x * lam : (tUt[s * SF + m] - x) * lam;
            });
            if (!REV) {
                // X Q^T with X = hi + lo (tf32 halves): fp32 accuracy; then the
                // column sums of dO^T o (X Q^T) over this CTA's rows
                const bf16* tQ = reinterpret_cast<const bf16*>(stage_ptr(buf, L::F_TILE));
                const bf16* tO = reinterpret_cast<const bf16*>(stage_ptr(buf, L::F_TILE + L::Q_TILE));
                if (tid < C) sdb[tid] = 0.f;
                float y2[2][1][4];
                zero(y2);
                const auto fqt = [&](int k, int nn) { return bf(tQ, nn * HD + k); };
                warp_mma<2, 1>(y2, fx, fqt, 0, n0, 0, D);
                warp_mma<2, 1>(y2, [&](int m, int k) {
                    const float x = sX[m * FD + k];
                    return x - __uint_as_float(to_tf32(x));
                }, fqt, 0, n0, 0, D);
                float h[1][2] = {};
                for_acc(y2, 0, n0, [&](int m, int r, float& x) { h[0][r & 1] += x * bf(tO, r * SH + m); });
                __syncthreads();   // sdb zeroed
                add_cols<1>(h, n0, sdb);
            }
        }
        __syncthreads();
        if (!REV && tid < C) atomicAdd(p.wdb0 + (static_cast<size_t>(bh) * NC + c) * C + tid, expf(tb[tid]) * sdb[tid]);
        // X <- gam_C X + Z B' (+ dO^T Qh)
        {
            constexpr int NT = D / 64;
            const int n0 = warp * (D / 8);
            float acc[2][NT][4];
            zero(acc);
            const auto fz = [&](int m, int k) { return sZ[m * FC + k]; };
            if (REV) {
                warp_mma<2, NT>(acc, fz, [&](int k, int nn) { return tW[k * FD + nn]; }, 0, n0, 0, C);
                warp_mma<2, NT>(acc, [&](int m, int k) { return bf(tdO, k * SH + m); },
                                [&](int k, int nn) { return tQh[k * FD + nn]; }, 0, n0, 0, C);
            } else {
                warp_mma<2, NT>(acc, fz, [&](int k, int nn) { return bf(tK, k * HD + nn); }, 0, n0, 0, C);
            }
            const float gC = expf(bC);
            for_acc(acc, 0, n0, [&](int m, int cc, float& x) { sX[m * FD + cc] = gC * sX[m * FD + cc] + x; });
        }
        __syncthreads();   // every warp is done with this stage
        if (j + 2 < NC) issue(j + 2, buf);
        cp_async_commit();
    }
    if (REV && p.dstate_in) {
        for (int x = tid; x < R * D; x += kThreads) {
            const int r = x / D, cc = x % D;
            p.dstate_in[bh * ss + static_cast<size_t>(row0 + r) * D + cc] = sX[r * FD + cc];
        }
    }
}

// ---------------------------------------------------------------------------
// 4. state-dependent gradients
// ---------------------------------------------------------------------------
template <int D>
struct GradASmem {
    using Dm = Dims<D>;
    static constexpr size_t H_TILE = size_t(C) * Dm::HD * 2;
    static constexpr size_t S_TILE = size_t(D) * Dm::HD * 2;
    static constexpr size_t F_TILE = size_t(C) * Dm::FD * 4;
    static constexpr size_t OFF_K = H_TILE, OFF_O = 2 * H_TILE;
    static constexpr size_t OFF_S0 = 3 * H_TILE, OFF_SC = OFF_S0 + S_TILE;
    static constexpr size_t OFF_W = OFF_SC + S_TILE, OFF_U = OFF_W + F_TILE;
    static constexpr size_t OFF_P = OFF_U + F_TILE;
    static constexpr size_t OFF_VEC = OFF_P + size_t(C) * Dm::FC * 4;
    static constexpr size_t BYTES = OFF_VEC + 4 * C * 4 + 16;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) grad_state_kernel(const Params p) {
    using Dm = Dims<D>;
    using L = GradASmem<D>;
    constexpr int FD = Dm::FD, HD = Dm::HD, FC = Dm::FC, NT = Dm::NT;
    extern __shared__ __align__(16) uint8_t smem[];
    bf16* sQ = reinterpret_cast<bf16*>(smem);
    bf16* sK = reinterpret_cast<bf16*>(smem + L::OFF_K);
    bf16* sO = reinterpret_cast<bf16*>(smem + L::OFF_O);
    bf16* sS0 = reinterpret_cast<bf16*>(smem + L::OFF_S0);
    bf16* sSC = reinterpret_cast<bf16*>(smem + L::OFF_SC);
    float* sW = reinterpret_cast<float*>(smem + L::OFF_W);   // W, then dU
    float* sU = reinterpret_cast<float*>(smem + L::OFF_U);   // Ut, then U
    float* sP = reinterpret_cast<float*>(smem + L::OFF_P);   // P, then dP o E
    float* vb = reinterpret_cast<float*>(smem + L::OFF_VEC);
    float* vgam = vb + C;
    float* vlam = vgam + C;
    float* vdb = vlam + C;
    float* vsum = vdb + C;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int unit = blockIdx.x, bh = unit / p.NC, c = unit % p.NC;
    const int n = min(C, p.T - c * C);
    const size_t tok0 = static_cast<size_t>(bh) * p.T + static_cast<size_t>(c) * C;
    const size_t ub = static_cast<size_t>(unit);

    load_tile(sQ, HD, p.q + tok0 * D, D, C, D, n);
    load_tile(sK, HD, p.k + tok0 * D, D, C, D, n);
    load_tile(sO, HD, p.dout + tok0 * D, D, C, D, n);
    load_tile(sS0, HD, p.ws0 + ub * D * D, D, D, D, D);
    load_tile(sSC, HD, p.wsc + ub * D * D, D, D, D, D);
    load_tile(sW, FD, p.ww + ub * C * D, D, C, D, C);
    load_tile(sU, FD, p.wut + ub * C * D, D, C, D, C);
    if (tid < C) {
        vb[tid] = p.wb[ub * C + tid];
        vdb[tid] = 0.f;
    }
    if (tid == 0) vsum[0] = 0.f;
    __syncthreads();
    if (tid < C) {
        vgam[tid] = expf(vb[tid]);
        vlam[tid] = expf(vb[C - 1] - vb[tid]);
    }
    __syncthreads();
    const float gC = expf(vb[C - 1]);
    const int m0 = (warp >> 2) * 32, n0c = (warp & 3) * 16, n0d = (warp & 3) * (D / 4);
    const auto fQ = [&](int m, int k) { return bf(sQ, m * HD + k); };
    const auto fO = [&](int m, int k) { return bf(sO, m * HD + k); };
    const auto fKt = [&](int k, int nn) { return bf(sK, nn * HD + k); };
    const auto fK = [&](int k, int nn) { return bf(sK, k * HD + nn); };
    const auto fS0 = [&](int k, int nn) { return bf(sS0, k * HD + nn); };
    const auto fS0t = [&](int k, int nn) { return bf(sS0, nn * HD + k); };
    const auto fSCt = [&](int k, int nn) { return bf(sSC, nn * HD + k); };
    const auto fSC = [&](int k, int nn) { return bf(sSC, k * HD + nn); };

    // P = lower(E o Q K^T); U = Ut - W S_0^T (in place); dQ <- gam dO S_0
    {
        float qk[2][2][4];
        zero(qk);
        warp_mma<2, 2>(qk, fQ, fKt, m0, n0c, 0, D);
        for_acc(qk, m0, n0c, [&](int r, int s, float& x) {
            sP[r * FC + s] = s <= r ? expf(vb[r] - vb[s]) * x : 0.f;
        });
        float ws[2][NT][4];
        zero(ws);
        warp_mma<2, NT>(ws, [&](int m, int k) { return sW[m * FD + k]; }, fS0t, m0, n0d, 0, D);
        for_acc(ws, m0, n0d, [&](int r, int i, float& x) { sU[r * FD + i] -= x; });
    }
    float dq[2][NT][4];
    zero(dq);
    warp_mma<2, NT>(dq, fO, fS0, m0, n0d, 0, D);
    for_acc(dq, m0, n0d, [&](int r, int k, float& x) { x *= vgam[r]; });
    __syncthreads();   // sP, sU complete; W no longer read
    // dU = P^T dO + diag(lam) K dS_C^T -> sW and the workspace
    {
        float du[2][NT][4];
        zero(du);
        warp_mma<2, NT>(du, [&](int m, int k) { return sP[k * FC + m]; }, [&](int k, int nn) { return fO(k, nn); },
                        m0, n0d, m0, C);
        warp_mma<2, NT>(du, [&](int m, int k) { return vlam[m] * bf(sK, m * HD + k); }, fSCt, m0, n0d, 0, D);
        float* g = p.wdu + ub * C * D;
        for_acc(du, m0, n0d, [&](int r, int i, float& x) {
            sW[r * FD + i] = x;
            g[r * D + i] = x;
        });
    }
    __syncthreads();
    // dW = -dU S_0 -> workspace; dP = lower(dO U^T) -> dP o E in place of P
    {
        float dw[2][NT][4];
        zero(dw);
        warp_mma<2, NT>(dw, [&](int m, int k) { return sW[m * FD + k]; }, fS0, m0, n0d, 0, D);
        float* g = p.wdw + ub * C * D;
        for_acc(dw, m0, n0d, [&](int r, int kk, float& x) { g[r * D + kk] = -x; });
        float dp[2][2][4];
        zero(dp);
        warp_mma<2, 2>(dp, fO, [&](int k, int nn) { return sU[nn * FD + k]; }, m0, n0c, 0, D);
        float hr[2][2] = {}, hc[2][2] = {};
        for_acc(dp, m0, n0c, [&](int r, int s, float& x) {
            float out = 0.f;
            if (s <= r) {
                const float pp = x * sP[r * FC + s];
                hr[(r - m0) >> 4][((r - m0) >> 3) & 1] += pp;
                hc[(s - n0c) >> 3][(s - n0c) & 1] -= pp;
                out = x * expf(vb[r] - vb[s]);
            }
            sP[r * FC + s] = out;
        });
        add_rows<2>(hr, m0, vdb);
        add_cols<2>(hc, n0c, vdb);
    }
    __syncthreads();   // dP o E complete
    // dQ += (dP o E) K -> global
    warp_mma<2, NT>(dq, [&](int m, int k) { return sP[m * FC + k]; }, fK, m0, n0d, 0, m0 + 32);
    {
        bf16* g = p.dq + tok0 * D;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int lane = tid & 31, r = m0 + 16 * i + (lane >> 2), cc = n0d + 8 * j + 2 * (lane & 3);
                if (r < n)
                    *reinterpret_cast<__nv_bfloat162*>(g + r * D + cc) = __floats2bfloat162_rn(dq[i][j][0], dq[i][j][1]);
                if (r + 8 < n)
                    *reinterpret_cast<__nv_bfloat162*>(g + (r + 8) * D + cc) =
                        __floats2bfloat162_rn(dq[i][j][2], dq[i][j][3]);
            }
    }
    // state terms of dK: diag(lam) U dS_C (and c_s), then + (dP o E)^T Q
    {
        float dk[2][NT][4];
        zero(dk);
        warp_mma<2, NT>(dk, [&](int m, int k) { return vlam[m] * sU[m * FD + k]; }, fSC, m0, n0d, 0, D);
        float h[2][2] = {};
        for_acc(dk, m0, n0d, [&](int r, int kk, float& x) {
            h[(r - m0) >> 4][((r - m0) >> 3) & 1] -= x * bf(sK, r * HD + kk);
        });
        float tot = 0.f;
#pragma unroll
        for (int i = 0; i < 2; ++i) tot -= h[i][0] + h[i][1];
        add_rows<2>(h, m0, vdb);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
        if ((tid & 31) == 0) atomicAdd(vdb + C - 1, tot);
        warp_mma<2, NT>(dk, [&](int m, int k) { return sP[k * FC + m]; }, fQ, m0, n0d, m0, C);
        float* g = p.wdk + ub * C * D;
        for_acc(dk, m0, n0d, [&](int r, int kk, float& x) { g[r * D + kk] = x; });
    }
    // gam_C <dS_C, S_0>
    {
        float s = 0.f;
        for (int x = tid; x < D * D; x += kThreads) {
            const int r = x / D, cc = x % D;
            s += bf(sSC, r * HD + cc) * bf(sS0, r * HD + cc);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if ((tid & 31) == 0) atomicAdd(vsum, s);
    }
    __syncthreads();
    if (tid < C) p.wdb[ub * C + tid] = vdb[tid] + p.wdb0[ub * C + tid] + (tid == C - 1 ? gC * vsum[0] : 0.f);
}

// ---------------------------------------------------------------------------
// 5. the remaining gradients
// ---------------------------------------------------------------------------
template <int D>
struct GradBSmem {
    using Dm = Dims<D>;
    static constexpr size_t CC_TILE = size_t(C) * Dm::FC * 4;
    static constexpr size_t F_TILE = size_t(C) * Dm::FD * 4;
    static constexpr size_t H_TILE = size_t(C) * Dm::HD * 2;
    static constexpr size_t OFF_A = CC_TILE;
    static constexpr size_t OFF_W = 2 * CC_TILE, OFF_UT = OFF_W + F_TILE, OFF_DU = OFF_UT + F_TILE;
    static constexpr size_t OFF_DW = OFF_DU + F_TILE, OFF_K = OFF_DW + F_TILE, OFF_V = OFF_K + H_TILE;
    static constexpr size_t OFF_VEC = OFF_V + H_TILE;
    static constexpr size_t BYTES = OFF_VEC + 5 * C * 4;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) grad_rest_kernel(const Params p) {
    using Dm = Dims<D>;
    using L = GradBSmem<D>;
    constexpr int FD = Dm::FD, HD = Dm::HD, FC = Dm::FC, NT = Dm::NT;
    extern __shared__ __align__(16) uint8_t smem[];
    float* sT = reinterpret_cast<float*>(smem);
    float* sA = reinterpret_cast<float*>(smem + L::OFF_A);    // K K^T, then F
    float* sW = reinterpret_cast<float*>(smem + L::OFF_W);
    float* sUt = reinterpret_cast<float*>(smem + L::OFF_UT);
    float* sdU = reinterpret_cast<float*>(smem + L::OFF_DU);  // dU, then dRv
    float* sdW = reinterpret_cast<float*>(smem + L::OFF_DW);  // dW, then dRk
    bf16* sK = reinterpret_cast<bf16*>(smem + L::OFF_K);
    bf16* sV = reinterpret_cast<bf16*>(smem + L::OFF_V);
    float* vb = reinterpret_cast<float*>(smem + L::OFF_VEC);
    float* vbeta = vb + C;
    float* vgam = vbeta + C;
    float* vdb = vgam + C;
    float* vdbeta = vdb + C;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int unit = blockIdx.x, bh = unit / p.NC, c = unit % p.NC;
    const int n = min(C, p.T - c * C);
    const size_t tok0 = static_cast<size_t>(bh) * p.T + static_cast<size_t>(c) * C;
    const size_t ub = static_cast<size_t>(unit);

    load_tile(sT, FC, p.wti + ub * C * C, C, C, C, C);
    load_tile(sW, FD, p.ww + ub * C * D, D, C, D, C);
    load_tile(sUt, FD, p.wut + ub * C * D, D, C, D, C);
    load_tile(sdU, FD, p.wdu + ub * C * D, D, C, D, C);
    load_tile(sdW, FD, p.wdw + ub * C * D, D, C, D, C);
    load_tile(sK, HD, p.k + tok0 * D, D, C, D, n);
    load_tile(sV, HD, p.v + tok0 * D, D, C, D, n);
    if (tid < C) {
        vb[tid] = p.wb[ub * C + tid];
        vbeta[tid] = tid < n ? p.beta[tok0 + tid] : 0.f;
        vdb[tid] = p.wdb[ub * C + tid];
        vdbeta[tid] = 0.f;
    }
    __syncthreads();
    if (tid < C) vgam[tid] = expf(vb[tid]);
    __syncthreads();
    const int m0 = (warp >> 2) * 32, n0c = (warp & 3) * 16, n0d = (warp & 3) * (D / 4);
    const auto fK = [&](int k, int nn) { return bf(sK, k * HD + nn); };
    // dRv = Ti^T dU, dRk = Ti^T dW (Ti^T upper: k >= m0); K K^T -> sA
    float rv[2][NT][4], rk[2][NT][4];
    zero(rv);
    zero(rk);
    {
        const auto ftt = [&](int m, int k) { return sT[k * FC + m]; };
        warp_mma<2, NT>(rv, ftt, [&](int k, int nn) { return sdU[k * FD + nn]; }, m0, n0d, m0, C);
        warp_mma<2, NT>(rk, ftt, [&](int k, int nn) { return sdW[k * FD + nn]; }, m0, n0d, m0, C);
        float kk[2][2][4];
        zero(kk);
        warp_mma<2, 2>(kk, [&](int m, int k) { return bf(sK, m * HD + k); },
                       [&](int k, int nn) { return bf(sK, nn * HD + k); }, m0, n0c, 0, D);
        for_acc(kk, m0, n0c, [&](int r, int s, float& x) { sA[r * FC + s] = x; });
        // dV = beta dRv; dbeta += dRv.v + gam dRk.k; db += beta gam dRk.k
        bf16* gv = p.dv + tok0 * D;
        float hb[2][2] = {}, hg[2][2] = {};
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int e2 = 0; e2 < 2; ++e2) {
                    const int lane = tid & 31, r = m0 + 16 * i + (lane >> 2) + 8 * e2;
                    const int cc = n0d + 8 * j + 2 * (lane & 3);
                    const float a0 = rv[i][j][2 * e2], a1 = rv[i][j][2 * e2 + 1];
                    const float k0 = rk[i][j][2 * e2], k1 = rk[i][j][2 * e2 + 1];
                    if (r < n) *reinterpret_cast<__nv_bfloat162*>(gv + r * D + cc) =
                        __floats2bfloat162_rn(vbeta[r] * a0, vbeta[r] * a1);
                    const float kr = k0 * bf(sK, r * HD + cc) + k1 * bf(sK, r * HD + cc + 1);
                    hb[i][e2] += a0 * bf(sV, r * HD + cc) + a1 * bf(sV, r * HD + cc + 1) + vgam[r] * kr;
                    hg[i][e2] += vbeta[r] * vgam[r] * kr;
                }
        add_rows<2>(hb, m0, vdbeta);
        add_rows<2>(hg, m0, vdb);
    }
    __syncthreads();   // dU, dW no longer read
    for_acc(rv, m0, n0d, [&](int r, int i, float& x) { sdU[r * FD + i] = x; });
    for_acc(rk, m0, n0d, [&](int r, int i, float& x) { sdW[r * FD + i] = x; });
    __syncthreads();
    // dA = -(dRv Ut^T + dRk W^T), strictly lower; F = beta dA o E in place of K K^T
    {
        float da[2][2][4];
        zero(da);
        warp_mma<2, 2>(da, [&](int m, int k) { return sdU[m * FD + k]; }, [&](int k, int nn) { return sUt[nn * FD + k]; },
                       m0, n0c, 0, D);
        warp_mma<2, 2>(da, [&](int m, int k) { return sdW[m * FD + k]; }, [&](int k, int nn) { return sW[nn * FD + k]; },
                       m0, n0c, 0, D);
        float hr[2][2] = {}, hc[2][2] = {}, hb[2][2] = {};
        for_acc(da, m0, n0c, [&](int r, int s, float& x) {
            float f = 0.f;
            if (s < r) {
                const float d = -x, e = expf(vb[r] - vb[s]), kk = sA[r * FC + s];
                const float aa = d * vbeta[r] * e * kk;
                hr[(r - m0) >> 4][((r - m0) >> 3) & 1] += aa;
                hc[(s - n0c) >> 3][(s - n0c) & 1] -= aa;
                hb[(r - m0) >> 4][((r - m0) >> 3) & 1] += d * e * kk;
                f = vbeta[r] * d * e;
            }
            sA[r * FC + s] = f;
        });
        add_rows<2>(hr, m0, vdb);
        add_cols<2>(hc, n0c, vdb);
        add_rows<2>(hb, m0, vdbeta);
    }
    __syncthreads();   // F complete
    // dK = F K + F^T K + diag(beta gam) dRk + state terms
    {
        float dk[2][NT][4];
        zero(dk);
        warp_mma<2, NT>(dk, [&](int m, int k) { return sA[m * FC + k]; }, fK, m0, n0d, 0, m0 + 32);
        warp_mma<2, NT>(dk, [&](int m, int k) { return sA[k * FC + m]; }, fK, m0, n0d, m0, C);
        const float* g1 = p.wdk + ub * C * D;
        bf16* gk = p.dk + tok0 * D;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int e2 = 0; e2 < 2; ++e2) {
                    const int lane = tid & 31, r = m0 + 16 * i + (lane >> 2) + 8 * e2;
                    const int cc = n0d + 8 * j + 2 * (lane & 3);
                    if (r < n) {
                        const float bg = vbeta[r] * vgam[r];
                        const float x0 = dk[i][j][2 * e2] + bg * sdW[r * FD + cc] + g1[r * D + cc];
                        const float x1 = dk[i][j][2 * e2 + 1] + bg * sdW[r * FD + cc + 1] + g1[r * D + cc + 1];
                        *reinterpret_cast<__nv_bfloat162*>(gk + r * D + cc) = __floats2bfloat162_rn(x0, x1);
                    }
                }
    }
    __syncthreads();
    // gate gradient: reverse prefix sums of db inside the chunk
    if (warp == 0) {
        const int lane = tid;
        float hi = vdb[lane + 32], lo = vdb[lane];
        // suffix sums: scan from the top with shuffles down
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float a = __shfl_down_sync(0xffffffffu, hi, o), b = __shfl_down_sync(0xffffffffu, lo, o);
            if (lane + o < 32) {
                hi += a;
                lo += b;
            }
        }
        lo += __shfl_sync(0xffffffffu, hi, 0);
        if (lane < n) {
            p.dgate[tok0 + lane] = lo / p.gate[tok0 + lane];
            p.dbeta[tok0 + lane] = vdbeta[lane];
        }
        if (lane + 32 < n) {
            p.dgate[tok0 + lane + 32] = hi / p.gate[tok0 + lane + 32];
            p.dbeta[tok0 + lane + 32] = vdbeta[lane + 32];
        }
    }
}

template <int D>
cudaError_t launch_all(const Params& p, cudaStream_t s) {
    const int units = p.BH * p.NC;
    cudaError_t e;
#define LA_GBW_LAUNCH(kern, grid, bytes)                                                                   \
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)); \
    if (e != cudaSuccess) return e;                                                                        \
    kern<<<grid, kThreads, bytes, s>>>(p);                                                                 \
    e = cudaGetLastError();                                                                                \
    if (e != cudaSuccess) return e;
    LA_GBW_LAUNCH(prep_kernel<D>, units, PrepSmem<D>::BYTES)
    LA_GBW_LAUNCH((chain_kernel<D, false>), p.BH * (D / kRows), ChainSmem<D>::BYTES)
    LA_GBW_LAUNCH((chain_kernel<D, true>), p.BH * (D / kRows), ChainSmem<D>::BYTES)
    LA_GBW_LAUNCH(grad_state_kernel<D>, units, GradASmem<D>::BYTES)
    LA_GBW_LAUNCH(grad_rest_kernel<D>, units, GradBSmem<D>::BYTES)
#undef LA_GBW_LAUNCH
    return cudaSuccess;
}

size_t carve(Params& p, uint8_t* base, int BH, int T, int D) {
    const int NC = (T + C - 1) / C;
    const size_t units = static_cast<size_t>(BH) * NC;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t* r = base ? base + off : nullptr;
        off += (bytes + 255) & ~static_cast<size_t>(255);
        return r;
    };
    p.wb = reinterpret_cast<float*>(take(units * C * 4));
    p.wti = reinterpret_cast<float*>(take(units * C * C * 4));
    p.ww = reinterpret_cast<float*>(take(units * C * D * 4));
    p.wut = reinterpret_cast<float*>(take(units * C * D * 4));
    p.wqh = reinterpret_cast<float*>(take(units * C * D * 4));
    p.ws0 = reinterpret_cast<bf16*>(take(units * D * D * 2));
    p.wsc = reinterpret_cast<bf16*>(take(units * D * D * 2));
    p.wdu = reinterpret_cast<float*>(take(units * C * D * 4));
    p.wdw = reinterpret_cast<float*>(take(units * C * D * 4));
    p.wdk = reinterpret_cast<float*>(take(units * C * D * 4));
    p.wdb = reinterpret_cast<float*>(take(units * C * 4));
    p.wdb0 = reinterpret_cast<float*>(take(units * C * 4));
    p.NC = NC;
    return off;
}

}  // namespace gbw

size_t gdn_chunk_backward_bytes(int BH, int T, int d) {
    gbw::Params p = {};
    return gbw::carve(p, nullptr, BH, T, d);
}

cudaError_t launch_gdn_chunk_backward(const DeltaBwdArgs& a, cudaStream_t s) {
    gbw::Params p = {};
    p.q = static_cast<const gbw::bf16*>(a.q);
    p.k = static_cast<const gbw::bf16*>(a.k);
    p.v = static_cast<const gbw::bf16*>(a.v);
    p.dout = static_cast<const gbw::bf16*>(a.dout);
    p.gate = a.gate;
    p.beta = a.beta;
    p.state_in = a.state_in;
    p.dstate_out = a.dstate_out;
    p.dq = static_cast<gbw::bf16*>(a.dq);
    p.dk = static_cast<gbw::bf16*>(a.dk);
    p.dv = static_cast<gbw::bf16*>(a.dv);
    p.dgate = a.dgate;
    p.dbeta = a.dbeta;
    p.dstate_in = a.dstate_in;
    p.BH = a.BH;
    p.T = a.T;
    gbw::carve(p, reinterpret_cast<uint8_t*>(a.workspace), a.BH, a.T, a.dk_dim);
    return a.dk_dim == 128 ? gbw::launch_all<128>(p, s) : gbw::launch_all<64>(p, s);
}

}  // namespace la
