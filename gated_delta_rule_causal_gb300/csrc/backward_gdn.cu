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
// Four launches per call:
//  1. prep, one CTA per (sequence-head, chunk): gate prefix sums, K K^T and
//     Q K^T, Ti in fp32 (16x16 diagonal blocks by forward substitution, then
//     two merge levels), W, Ut and Qh = gam Q - P W; fp32 into the workspace
//     (W, lam W, lam K and Qh, only ever MMA operands, already rounded to tf32).
//  2. both chains at once, CTAs of D/2 value rows: the state chain walks the
//     chunks with the rows in fp32 and stores every chunk's S_0 (bf16); it
//     also forms the gate term gam_r dO_r.(S_0 q_r) from the fp32 rows
//     rounded once to tf32, since that term cancels against the others of
//     the gate gradient and bf16 rows would cost it up to ~3% of the result.
//     The gradient chain walks from the last chunk, storing every chunk's
//     dS_C (bf16) and the gradient of the initial state (fp32).
//  3. the state-dependent gradients per chunk: U, dU, dW, dQ (final), the
//     state terms of dK and of the gate gradient.
//  4. the rest per chunk: dRv, dRk, dA, dV, dK, dbeta and the gate gradient.
// Every product is a warp-level tf32 MMA (m16n8k8, fp32 accumulation) on
// shared-memory tiles loaded by asynchronous copies; the chains keep their
// rows in registers and stage each chunk's tiles two chunks ahead.
//
// Tail chunks: rows past T load as zeros, with g = 1 and beta = 0, so they
// leave every real row's result unchanged; no row past T is written.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace la {
namespace gbw {

constexpr int C = 64;            // tokens per chunk
constexpr int kThreads = 256;    // eight warps (prep)
constexpr int kGradThreads = 512;   // sixteen warps (gradient kernels), each a 16-row tile:
constexpr int GMT = 1;              // m16 tiles per warp in the per-chunk products
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
    float* wb;     // [2C]    ln-gate prefix sums b, then gam = e^b
    float* wti;    // [C][C]  Ti
    float* ww;     // [C][D]  W
    float* wut;    // [C][D]  Ut
    float* wqht;   // [D][C]  Qh^T
    float* wlkt;   // [D][C]  (diag(lam) K)^T
    float* wlwt;   // [D][C]  (diag(lam) W)^T
    bf16* ws0;     // [D][D]  S_0
    bf16* wsc;     // [D][D]  dS_C
    float* wdu;    // [C][D]  dU
    float* wdw;    // [C][D]  dW
    float* wdk;    // [C][D]  state terms of dK
    float* wdb;    // [C]     state terms of the gate gradient
    float* wdb0;   // [C]     gam_r dO_r.(S_0 q_r), summed over the state chain's CTAs
};

__device__ __forceinline__ float bf(const bf16* p, int i) { return __bfloat162float(p[i]); }

// An operand value as a tf32 register: rounded to nearest, or passed as it
// is when it already fits tf32 (widened bf16, or rounded when stored).
__device__ __forceinline__ float tf32r(float x) { return __uint_as_float(to_tf32(x)); }

template <bool ROUND>
__device__ __forceinline__ uint32_t tf32_of(float x) {
    if constexpr (ROUND) return to_tf32(x);
    else return __float_as_uint(x);
}

// Operand values two k at a time (k even): fa(m, k) = {A(m, k), A(m, k + 1)},
// fb(k, n) = {B(k, n), B(k + 1, n)}. Inside an 8-wide k step lane t feeds
// k + 2t and k + 2t + 1 into the slots t and t + 4 of the m16n8k8 fragments
// (A: (g, t), (g + 8, t), (g, t + 4), (g + 8, t + 4); B: (t, g), (t + 4, g));
// A and B take the same order, so the sum is unchanged, and a row-contiguous
// operand loads its pair at once.
__device__ __forceinline__ float2 rowf(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 rowh(const bf16* p) {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}
__device__ __forceinline__ float2 colf(const float* p, int ld) { return make_float2(p[0], p[ld]); }
__device__ __forceinline__ float2 colh(const bf16* p, int ld) { return make_float2(bf(p, 0), bf(p, ld)); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return make_float2(a.x * b.x, a.y * b.y); }
__device__ __forceinline__ float2 scale2(float2 a, float s) { return make_float2(a.x * s, a.y * s); }

// acc[MT][NT] (+)= sum over k in [k0, k1) of A(m, k) B(k, n) for the warp's
// (16 MT) x (8 NT) tile at (m0, n0); k0, k1 multiples of 8. RA, RB: round the
// A, B values to tf32 (false where they already fit).
template <int MT, int NT, bool RA = true, bool RB = true, class FA, class FB>
__device__ __forceinline__ void warp_mma(float (&acc)[MT][NT][4], const FA& fa, const FB& fb, int m0, int n0, int k0,
                                         int k1) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll 4
    for (int k = k0; k < k1; k += 8) {
        uint32_t a[MT][4], b[NT][2];
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            const int m = m0 + 16 * i + g;
            const float2 lo = fa(m, k + 2 * t), hi = fa(m + 8, k + 2 * t);
            a[i][0] = tf32_of<RA>(lo.x);
            a[i][1] = tf32_of<RA>(hi.x);
            a[i][2] = tf32_of<RA>(lo.y);
            a[i][3] = tf32_of<RA>(hi.y);
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const float2 v = fb(k + 2 * t, n0 + 8 * j + g);
            b[j][0] = tf32_of<RB>(v.x);
            b[j][1] = tf32_of<RB>(v.y);
        }
#pragma unroll
        for (int i = 0; i < MT; ++i)
#pragma unroll
            for (int j = 0; j < NT; ++j) mma_tf32_m16n8k8(acc[i][j], a[i], b[j]);
    }
}

// B operand from a row-major bf16 [k][n] tile (row stride ld elements, rows
// 16-byte aligned): ldmatrix .trans of the 8 x 8 block at rows k..k+7,
// columns n..n+7 gives lane (g, t) the pair (B[k + 2t][n + g], B[k + 2t + 1][n + g])
// in one register, the lower k in the lower half: the k-pair order above.
struct BT {
    const bf16* p;
    int ld;
};

template <int NT>
__device__ __forceinline__ void ldsm_trans(uint32_t (&r)[NT], const bf16* row_addr) {
    const uint32_t a = smem_u32(row_addr);
    if constexpr (NT == 4)
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
    else if constexpr (NT == 2)
        asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(a));
    else
        asm volatile("ldmatrix.sync.aligned.m8n8.x1.trans.shared.b16 {%0}, [%1];" : "=r"(r[0]) : "r"(a));
}

template <int MT, int NT, bool RA = true, class FA>
__device__ __forceinline__ void warp_mma(float (&acc)[MT][NT][4], const FA& fa, const BT& bt, int m0, int n0, int k0,
                                         int k1) {
    static_assert(NT == 1 || NT == 2 || NT == 4, "one ldmatrix per k step");
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    // this lane's row address: block j = lane / 8 (of NT), row lane % 8
    const bf16* rp = bt.p + (lane & 7) * bt.ld + n0 + 8 * ((lane >> 3) % NT);
#pragma unroll 4
    for (int k = k0; k < k1; k += 8) {
        uint32_t a[MT][4], r[NT];
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            const int m = m0 + 16 * i + g;
            const float2 lo = fa(m, k + 2 * t), hi = fa(m + 8, k + 2 * t);
            a[i][0] = tf32_of<RA>(lo.x);
            a[i][1] = tf32_of<RA>(hi.x);
            a[i][2] = tf32_of<RA>(lo.y);
            a[i][3] = tf32_of<RA>(hi.y);
        }
        ldsm_trans<NT>(r, rp + k * bt.ld);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const uint32_t b[2] = {r[j] << 16, r[j] & 0xffff0000u};
#pragma unroll
            for (int i = 0; i < MT; ++i) mma_tf32_m16n8k8(acc[i][j], a[i], b);
        }
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

// f(row, col, value&, rs, cs) for every accumulator element of the warp's
// tile; rs (< 2 MT) and cs (< 2 NT) are the element's row and column slots in
// this lane, compile-time constants once unrolled.
template <int MT, int NT, class F>
__device__ __forceinline__ void for_acc(float (&acc)[MT][NT][4], int m0, int n0, const F& f) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                f(m0 + 16 * i + g + 8 * (e >> 1), n0 + 8 * j + 2 * t + (e & 1), acc[i][j][e], 2 * i + (e >> 1),
                  2 * j + (e & 1));
}

// Sum of per-row partials (slot rs = 2i + e: row m0 + 16i + g + 8e) over the
// four lanes of a quad, added to s[row] by its first lane.
template <int MT>
__device__ __forceinline__ void add_rows(float (&h)[2 * MT], int m0, float* s) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float x = h[2 * i + e];
            x += __shfl_xor_sync(0xffffffffu, x, 1);
            x += __shfl_xor_sync(0xffffffffu, x, 2);
            if (t == 0) atomicAdd(s + m0 + 16 * i + g + 8 * e, x);
        }
}

// Sum of per-column partials (slot cs = 2j + e: col n0 + 8j + 2t + e) over
// the eight lanes sharing t, added to s[col] by the lanes with g = 0.
template <int NT>
__device__ __forceinline__ void add_cols(float (&h)[2 * NT], int n0, float* s) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float x = h[2 * j + e];
            x += __shfl_xor_sync(0xffffffffu, x, 4);
            x += __shfl_xor_sync(0xffffffffu, x, 8);
            x += __shfl_xor_sync(0xffffffffu, x, 16);
            if (g == 0) atomicAdd(s + n0 + 8 * j + 2 * t + e, x);
        }
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool full) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(full ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// rows x COLS tile copy, global row stride gs, shared row stride ss (both in
// elements of T), rows >= valid filled with zeros; asynchronous 16-byte
// pieces (the caller commits and waits).
template <int COLS, typename T>
__device__ __forceinline__ void copy_tile_async(T* dst, int ss, const T* src, size_t gs, int rows, int valid) {
    constexpr int E = 16 / sizeof(T);
    constexpr int per = COLS / E;   // a power of two: the index split is shifts
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

    copy_tile_async<D>(sQ, HD, p.q + tok0 * D, D, C, n);
    copy_tile_async<D>(sK, HD, p.k + tok0 * D, D, C, n);
    copy_tile_async<D>(sV, HD, p.v + tok0 * D, D, C, n);
    cp_async_commit();
    gate_sums(p, tok0, n, vb, vbeta);
    for (int x = tid; x < C * FC; x += kThreads) sT[x] = 0.f;
    cp_async_wait0();
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
        const auto fk = [&](int m, int k) { return rowh(sK + m * HD + k); };
        const auto fq = [&](int m, int k) { return rowh(sQ + m * HD + k); };
        const auto fkt = [&](int k, int nn) { return rowh(sK + nn * HD + k); };
        warp_mma<2, 2, false, false>(kk, fk, fkt, m0, n0, 0, D);
        warp_mma<2, 2, false, false>(qk, fq, fkt, m0, n0, 0, D);
        for_acc(kk, m0, n0, [&](int r, int s, float& x, int rs, int cs) {
            sA[r * FC + s] = s < r ? vbeta[r] * expf(vb[r] - vb[s]) * x : 0.f;
        });
        for_acc(qk, m0, n0, [&](int r, int s, float& x, int rs, int cs) {
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
        const auto fw = [&](int m, int k) { return mul2(rowf(sT + m * FC + k), rowf(vbg + k)); };
        const auto fu = [&](int m, int k) { return mul2(rowf(sT + m * FC + k), rowf(vbeta + k)); };
        warp_mma<2, NT>(w, fw, BT{sK, HD}, m0, n0, 0, m0 + 32);
        warp_mma<2, NT>(u, fu, BT{sV, HD}, m0, n0, 0, m0 + 32);
        float* gw = p.ww + ub * C * D;
        float* gu = p.wut + ub * C * D;
        float* glw = p.wlwt + ub * C * D;
        const float bC = vb[C - 1];
        for_acc(w, m0, n0, [&](int r, int cc, float& x, int rs, int cs) {
            gw[r * D + cc] = tf32r(x);
            glw[cc * C + r] = tf32r(expf(bC - vb[r]) * x);
        });
        for_acc(u, m0, n0, [&](int r, int cc, float& x, int rs, int cs) { gu[r * D + cc] = x; });
    }
    // P Ti -> sA (A is no longer read)
    {
        const int m0 = (warp >> 2) * 32, n0 = (warp & 3) * 16;
        float pt[2][2][4];
        zero(pt);
        const auto fp = [&](int m, int k) { return rowf(sP + m * FC + k); };
        const auto ft = [&](int k, int nn) { return colf(sT + k * FC + nn, FC); };
        warp_mma<2, 2>(pt, fp, ft, m0, n0, 0, m0 + 32);
        for_acc(pt, m0, n0, [&](int r, int s, float& x, int rs, int cs) { sA[r * FC + s] = x; });
    }
    __syncthreads();
    // Qh = diag(gam) Q - (P Ti) diag(beta gam) K
    {
        constexpr int NT = Dm::NT;
        const int m0 = (warp >> 2) * 32, n0 = (warp & 3) * (D / 4);
        float qh[2][NT][4];
        zero(qh);
        const auto fa = [&](int m, int k) { return mul2(rowf(sA + m * FC + k), rowf(vbg + k)); };
        warp_mma<2, NT>(qh, fa, BT{sK, HD}, m0, n0, 0, m0 + 32);
        float* gq = p.wqht + ub * C * D;
        for_acc(qh, m0, n0, [&](int r, int cc, float& x, int rs, int cs) {
            gq[cc * C + r] = tf32r(vgam[r] * bf(sQ, r * HD + cc) - x);
        });
    }
    {
        float* gk = p.wlkt + ub * C * D;
        const float bC = vb[C - 1];
        for (int x = tid; x < C * D; x += kThreads) {
            const int d = x / C, r = x % C;
            gk[x] = tf32r(expf(bC - vb[r]) * bf(sK, r * HD + d));
        }
    }
    float* gt = p.wti + ub * C * C;
    for (int x = tid; x < C * C; x += kThreads) gt[x] = sT[(x / C) * FC + x % C];
    if (tid < C) {
        p.wb[ub * 2 * C + tid] = vb[tid];
        p.wb[ub * 2 * C + C + tid] = vgam[tid];
        p.wdb0[ub * C + tid] = 0.f;   // the state chain adds into it
    }
}

// ---------------------------------------------------------------------------
// 2, 3. both chains in one launch: one CTA per (sequence-head, direction),
//       16 value rows per warp
// ---------------------------------------------------------------------------
// Each warp holds its 16 rows of X (fp32) as MMA accumulators. In the k-pair
// order an accumulator tile (rows g, g + 8; columns 2t, 2t + 1 of each
// 8-column block) is, register for register, the A fragment of the product
// that contracts over those columns, so X and the chunk's Z = Ut^T - X W^T
// (or -X K^T) never leave the registers:
//    state chain:    Y = X W^T,  Z = Ut^T - Y,   X <- gam_C X + Z (lam K)
//    gradient chain: Y = X K^T,  Z = -Y,         X <- gam_C X + Z (lam W) + dO^T Qh
// The B operands come from double-buffered tiles (W, Q, K as stored; the
// transposed lam K, lam W and Qh written by the prep), staged two chunks
// ahead with the Ut and dO slices of the CTA's rows.

constexpr int kChainSplit = 2;   // CTAs per (sequence-head, direction), D / kChainSplit rows each

template <int D>
struct ChainSmem {
    static constexpr int RW = D / kChainSplit;   // the CTA's value rows
    static constexpr int FW = D + 8;    // fp32 [C][FW]: W (pairs along d)
    static constexpr int HD = D + 8;    // bf16 [C][HD]: Q, K (pairs along d)
    static constexpr int FT = C + 8;    // fp32 [D][FT]: (lam K)^T, (lam W)^T, Qh^T (pairs along tokens)
    static constexpr int SU = RW + 4;   // fp32 [C][SU]: the CTA's columns of Ut
    static constexpr int SO = RW + 8;   // bf16 [C][SO]: the CTA's columns of dO
    static constexpr size_t W_T = size_t(C) * FW * 4, H_T = size_t(C) * HD * 2, T_T = size_t(D) * FT * 4;
    static constexpr size_t U_T = size_t(C) * SU * 4, O_T = size_t(C) * SO * 2;
    // state chain: W, Q, (lam K)^T, Ut slice, dO slice, gam;
    // gradient chain: K, (lam W)^T, Qh^T, dO slice, gam
    static constexpr size_t FWD = W_T + H_T + T_T + U_T + O_T + C * 4;
    static constexpr size_t REV = H_T + 2 * T_T + O_T + C * 4;
    static constexpr size_t STAGE = ((FWD > REV ? FWD : REV) + 127) / 128 * 128;
    static constexpr size_t BYTES = 2 * STAGE;
    static_assert(BYTES <= 232448, "two stages fit the opt-in shared memory");
};

template <int D, bool rev>
__device__ __forceinline__ void chain_body(const Params& p, int bh, int part, uint8_t* smem) {
    using L = ChainSmem<D>;
    constexpr int FW = L::FW, HD = L::HD, FT = L::FT, NJ = D / 8;   // NJ column blocks of X
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    constexpr int RW = L::RW, SU = L::SU, SO = L::SO;
    const int rbase = part * RW, rl = 16 * warp, row0 = rbase + rl;   // the CTA's and this warp's first row
    const int NC = p.NC;
    const size_t ss = static_cast<size_t>(D) * D;

    auto stage = [&](int buf) { return smem + buf * L::STAGE; };
    auto issue = [&](int j, int buf) {
        const int c = rev ? NC - 1 - j : j;
        const int n = min(C, p.T - c * C);
        const size_t ub = static_cast<size_t>(bh) * NC + c;
        const size_t tok0 = static_cast<size_t>(bh) * p.T + static_cast<size_t>(c) * C;
        uint8_t* b = stage(buf);
        if (!rev) {
            copy_tile_async<D>(reinterpret_cast<float*>(b), FW, p.ww + ub * C * D, D, C, C);
            copy_tile_async<D>(reinterpret_cast<bf16*>(b + L::W_T), HD, p.q + tok0 * D, D, C, n);
            copy_tile_async<C>(reinterpret_cast<float*>(b + L::W_T + L::H_T), FT, p.wlkt + ub * C * D, C, D, D);
            copy_tile_async<RW>(reinterpret_cast<float*>(b + L::W_T + L::H_T + L::T_T), SU,
                                p.wut + ub * C * D + rbase, D, C, C);
            copy_tile_async<RW>(reinterpret_cast<bf16*>(b + L::W_T + L::H_T + L::T_T + L::U_T), SO,
                                p.dout + tok0 * D + rbase, D, C, n);
            copy_tile_async<C>(reinterpret_cast<float*>(b + L::FWD - C * 4), C, p.wb + ub * 2 * C + C, C, 1, 1);
        } else {
            copy_tile_async<D>(reinterpret_cast<bf16*>(b), HD, p.k + tok0 * D, D, C, n);
            copy_tile_async<C>(reinterpret_cast<float*>(b + L::H_T), FT, p.wlwt + ub * C * D, C, D, D);
            copy_tile_async<C>(reinterpret_cast<float*>(b + L::H_T + L::T_T), FT, p.wqht + ub * C * D, C, D, D);
            copy_tile_async<RW>(reinterpret_cast<bf16*>(b + L::H_T + 2 * L::T_T), SO, p.dout + tok0 * D + rbase, D, C,
                                n);
            copy_tile_async<C>(reinterpret_cast<float*>(b + L::REV - C * 4), C, p.wb + ub * 2 * C + C, C, 1, 1);
        }
    };
    float x[NJ][4];
    {
        const float* x0 = rev ? p.dstate_out : p.state_in;
#pragma unroll
        for (int jb = 0; jb < NJ; ++jb)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = row0 + g + 8 * (e >> 1), col = 8 * jb + 2 * t + (e & 1);
                x[jb][e] = x0 ? x0[bh * ss + static_cast<size_t>(row) * D + col] : 0.f;
            }
    }
    issue(0, 0);
    cp_async_commit();
    if (NC > 1) issue(1, 1);
    cp_async_commit();

    bf16* gout = rev ? p.wsc : p.ws0;
    for (int j = 0; j < NC; ++j) {
        const int buf = j & 1;
        const int c = rev ? NC - 1 - j : j;
        const uint8_t* b = stage(buf);
        const float* tgam = reinterpret_cast<const float*>(b + (rev ? L::REV : L::FWD) - C * 4);
        const float* tUs = reinterpret_cast<const float*>(b + L::W_T + L::H_T + L::T_T);
        const bf16* tOs = reinterpret_cast<const bf16*>(b + (rev ? L::H_T + 2 * L::T_T : L::W_T + L::H_T + L::T_T + L::U_T));
        // the rows entering this chunk
        {
            bf16* o = gout + (static_cast<size_t>(bh) * NC + c) * ss;
#pragma unroll
            for (int jb = 0; jb < NJ; ++jb)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    *reinterpret_cast<__nv_bfloat162*>(o + static_cast<size_t>(row0 + g + 8 * h) * D + 8 * jb + 2 * t) =
                        __floats2bfloat162_rn(x[jb][2 * h], x[jb][2 * h + 1]);
        }
        cp_async_wait1();
        __syncthreads();   // this chunk's tiles are visible
        // Y = X B1 (16 rows x C tokens); state chain also Y2 = X Q^T
        float y[8][4], y2[8][4];
#pragma unroll
        for (int jb = 0; jb < 8; ++jb)
#pragma unroll
            for (int e = 0; e < 4; ++e) y[jb][e] = y2[jb][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < NJ; ++kk) {
            const uint32_t a[4] = {to_tf32(x[kk][0]), to_tf32(x[kk][2]), to_tf32(x[kk][1]), to_tf32(x[kk][3])};
#pragma unroll
            for (int jb = 0; jb < 8; ++jb) {
                const int tok = 8 * jb + g, d = 8 * kk + 2 * t;
                if (!rev) {
                    const float2 w = rowf(reinterpret_cast<const float*>(b) + tok * FW + d);
                    const float2 qv = rowh(reinterpret_cast<const bf16*>(b + L::W_T) + tok * HD + d);
                    const uint32_t b1[2] = {__float_as_uint(w.x), __float_as_uint(w.y)};
                    const uint32_t b2[2] = {__float_as_uint(qv.x), __float_as_uint(qv.y)};
                    mma_tf32_m16n8k8(y[jb], a, b1);
                    mma_tf32_m16n8k8(y2[jb], a, b2);
                } else {
                    const float2 kv = rowh(reinterpret_cast<const bf16*>(b) + tok * HD + d);
                    const uint32_t b1[2] = {__float_as_uint(kv.x), __float_as_uint(kv.y)};
                    mma_tf32_m16n8k8(y[jb], a, b1);
                }
            }
        }
        // Z = Ut^T - Y or -Y (in place); the state chain's gate term
        // gam_r sum over rows of dO[r][row] (X Q^T)[row][r]
        if (!rev) {
            float part[8][2];
#pragma unroll
            for (int jb = 0; jb < 8; ++jb)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int tok = 8 * jb + 2 * t + e;
                    const float d0 = bf(tOs, tok * SO + rl + g), d1 = bf(tOs, tok * SO + rl + g + 8);
                    part[jb][e] = y2[jb][e] * d0 + y2[jb][2 + e] * d1;
                    y[jb][e] = tUs[tok * SU + rl + g] - y[jb][e];
                    y[jb][2 + e] = tUs[tok * SU + rl + g + 8] - y[jb][2 + e];
                }
            float* gdb = p.wdb0 + (static_cast<size_t>(bh) * NC + c) * C;
#pragma unroll
            for (int jb = 0; jb < 8; ++jb)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float v = part[jb][e];
                    v += __shfl_xor_sync(0xffffffffu, v, 4);
                    v += __shfl_xor_sync(0xffffffffu, v, 8);
                    v += __shfl_xor_sync(0xffffffffu, v, 16);
                    const int tok = 8 * jb + 2 * t + e;
                    if (g == 0) atomicAdd(gdb + tok, tgam[tok] * v);
                }
        } else {
#pragma unroll
            for (int jb = 0; jb < 8; ++jb)
#pragma unroll
                for (int e = 0; e < 4; ++e) y[jb][e] = -y[jb][e];
        }
        // X <- gam_C X + Z B2 (+ dO^T Qh)
        const float gC = tgam[C - 1];
#pragma unroll
        for (int jb = 0; jb < NJ; ++jb)
#pragma unroll
            for (int e = 0; e < 4; ++e) x[jb][e] *= gC;
        const float* tB = reinterpret_cast<const float*>(b + (rev ? L::H_T : L::W_T + L::H_T));
        const float* tQh = reinterpret_cast<const float*>(b + L::H_T + L::T_T);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {   // tokens 8 kk .. 8 kk + 7
            const uint32_t a[4] = {to_tf32(y[kk][0]), to_tf32(y[kk][2]), to_tf32(y[kk][1]), to_tf32(y[kk][3])};
            uint32_t a2[4];
            if (rev) {   // dO^T: rows g, g + 8, tokens 8 kk + 2t, +1 (bf16: already tf32)
                const float2 lo = colh(tOs + (8 * kk + 2 * t) * SO + rl + g, SO);
                const float2 hi = colh(tOs + (8 * kk + 2 * t) * SO + rl + g + 8, SO);
                a2[0] = __float_as_uint(lo.x);
                a2[1] = __float_as_uint(hi.x);
                a2[2] = __float_as_uint(lo.y);
                a2[3] = __float_as_uint(hi.y);
            }
#pragma unroll
            for (int jb = 0; jb < NJ; ++jb) {
                const float2 v = rowf(tB + (8 * jb + g) * FT + 8 * kk + 2 * t);
                const uint32_t b1[2] = {__float_as_uint(v.x), __float_as_uint(v.y)};
                mma_tf32_m16n8k8(x[jb], a, b1);
            }
            if (rev) {   // after the first pass, so that no two MMAs in a row share an accumulator
#pragma unroll
                for (int jb = 0; jb < NJ; ++jb) {
                    const float2 qv = rowf(tQh + (8 * jb + g) * FT + 8 * kk + 2 * t);
                    const uint32_t b2[2] = {__float_as_uint(qv.x), __float_as_uint(qv.y)};
                    mma_tf32_m16n8k8(x[jb], a2, b2);
                }
            }
        }
        __syncthreads();   // every warp is done with this stage
        if (j + 2 < NC) issue(j + 2, buf);
        cp_async_commit();
    }
    if (rev && p.dstate_in) {
#pragma unroll
        for (int jb = 0; jb < NJ; ++jb)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = row0 + g + 8 * (e >> 1), col = 8 * jb + 2 * t + (e & 1);
                p.dstate_in[bh * ss + static_cast<size_t>(row) * D + col] = x[jb][e];
            }
    }
}

template <int D>
__global__ void __launch_bounds__(2 * D / kChainSplit, 1) chain_kernel(const Params p) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int per_dir = p.BH * kChainSplit;
    const int i = blockIdx.x % per_dir;
    if (blockIdx.x < per_dir) chain_body<D, false>(p, i / kChainSplit, i % kChainSplit, smem);
    else chain_body<D, true>(p, i / kChainSplit, i % kChainSplit, smem);
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
__global__ void __launch_bounds__(kGradThreads, 1) grad_state_kernel(const Params p) {
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

    copy_tile_async<D>(sQ, HD, p.q + tok0 * D, D, C, n);
    copy_tile_async<D>(sK, HD, p.k + tok0 * D, D, C, n);
    copy_tile_async<D>(sO, HD, p.dout + tok0 * D, D, C, n);
    copy_tile_async<D>(sS0, HD, p.ws0 + ub * D * D, D, D, D);
    copy_tile_async<D>(sSC, HD, p.wsc + ub * D * D, D, D, D);
    copy_tile_async<D>(sW, FD, p.ww + ub * C * D, D, C, C);
    copy_tile_async<D>(sU, FD, p.wut + ub * C * D, D, C, C);
    cp_async_commit();
    if (tid < C) {
        vb[tid] = p.wb[ub * 2 * C + tid];
        vdb[tid] = 0.f;
    }
    if (tid == 0) vsum[0] = 0.f;
    cp_async_wait0();
    __syncthreads();
    if (tid < C) {
        vgam[tid] = expf(vb[tid]);
        vlam[tid] = expf(vb[C - 1] - vb[tid]);
    }
    __syncthreads();
    const float gC = expf(vb[C - 1]);
    const int m0 = (warp >> 2) * 16 * GMT, n0c = (warp & 3) * 16, n0d = (warp & 3) * (D / 4);
    const auto fQ = [&](int m, int k) { return rowh(sQ + m * HD + k); };
    const BT fQc{sQ, HD};
    const auto fO = [&](int m, int k) { return rowh(sO + m * HD + k); };
    const BT fOc{sO, HD};
    const auto fKt = [&](int k, int nn) { return rowh(sK + nn * HD + k); };
    const BT fK{sK, HD};
    const BT fS0{sS0, HD};
    const auto fS0t = [&](int k, int nn) { return rowh(sS0 + nn * HD + k); };
    const auto fSCt = [&](int k, int nn) { return rowh(sSC + nn * HD + k); };
    const BT fSC{sSC, HD};

    // P = lower(E o Q K^T); U = Ut - W S_0^T (in place); dQ <- gam dO S_0
    {
        float qk[GMT][2][4];
        zero(qk);
        warp_mma<GMT, 2, false, false>(qk, fQ, fKt, m0, n0c, 0, D);
        for_acc(qk, m0, n0c, [&](int r, int s, float& x, int rs, int cs) {
            sP[r * FC + s] = s <= r ? expf(vb[r] - vb[s]) * x : 0.f;
        });
        float ws[GMT][NT][4];
        zero(ws);
        warp_mma<GMT, NT, true, false>(ws, [&](int m, int k) { return rowf(sW + m * FD + k); }, fS0t, m0, n0d, 0, D);
        for_acc(ws, m0, n0d, [&](int r, int i, float& x, int rs, int cs) { sU[r * FD + i] -= x; });
    }
    float dq[GMT][NT][4];
    zero(dq);
    warp_mma<GMT, NT, false>(dq, fO, fS0, m0, n0d, 0, D);
    for_acc(dq, m0, n0d, [&](int r, int k, float& x, int rs, int cs) { x *= vgam[r]; });
    __syncthreads();   // sP, sU complete; W no longer read
    // dU = P^T dO + diag(lam) K dS_C^T -> sW and the workspace
    {
        float du[GMT][NT][4];
        zero(du);
        warp_mma<GMT, NT>(du, [&](int m, int k) { return colf(sP + k * FC + m, FC); }, fOc,
                        m0, n0d, m0, C);
        warp_mma<GMT, NT, true, false>(du, [&](int m, int k) { return scale2(rowh(sK + m * HD + k), vlam[m]); }, fSCt, m0,
                                     n0d, 0, D);
        float* g = p.wdu + ub * C * D;
        for_acc(du, m0, n0d, [&](int r, int i, float& x, int rs, int cs) {
            sW[r * FD + i] = x;
            g[r * D + i] = x;
        });
    }
    __syncthreads();
    // dW = -dU S_0 -> workspace; dP = lower(dO U^T) -> dP o E in place of P
    {
        float dw[GMT][NT][4];
        zero(dw);
        warp_mma<GMT, NT>(dw, [&](int m, int k) { return rowf(sW + m * FD + k); }, fS0, m0, n0d, 0, D);
        float* g = p.wdw + ub * C * D;
        for_acc(dw, m0, n0d, [&](int r, int kk, float& x, int rs, int cs) { g[r * D + kk] = -x; });
        float dp[GMT][2][4];
        zero(dp);
        warp_mma<GMT, 2, false, true>(dp, fO, [&](int k, int nn) { return rowf(sU + nn * FD + k); }, m0, n0c, 0, D);
        float hr[2 * GMT] = {}, hc[4] = {};
        for_acc(dp, m0, n0c, [&](int r, int s, float& x, int rs, int cs) {
            float out = 0.f;
            if (s <= r) {
                const float pp = x * sP[r * FC + s];
                hr[rs] += pp;
                hc[cs] -= pp;
                out = x * expf(vb[r] - vb[s]);
            }
            sP[r * FC + s] = out;
        });
        add_rows<GMT>(hr, m0, vdb);
        add_cols<2>(hc, n0c, vdb);
    }
    __syncthreads();   // dP o E complete
    // dQ += (dP o E) K -> global
    warp_mma<GMT, NT>(dq, [&](int m, int k) { return rowf(sP + m * FC + k); }, fK, m0, n0d, 0, m0 + 16 * GMT);
    {
        bf16* g = p.dq + tok0 * D;
#pragma unroll
        for (int i = 0; i < GMT; ++i)
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
        float dk[GMT][NT][4];
        zero(dk);
        warp_mma<GMT, NT>(dk, [&](int m, int k) { return scale2(rowf(sU + m * FD + k), vlam[m]); }, fSC, m0,
                                     n0d, 0, D);
        float h[2 * GMT] = {};
        for_acc(dk, m0, n0d, [&](int r, int kk, float& x, int rs, int cs) {
            h[rs] -= x * bf(sK, r * HD + kk);
        });
        float tot = 0.f;
#pragma unroll
        for (int i = 0; i < 2 * GMT; ++i) tot -= h[i];
        add_rows<GMT>(h, m0, vdb);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
        if ((tid & 31) == 0) atomicAdd(vdb + C - 1, tot);
        warp_mma<GMT, NT>(dk, [&](int m, int k) { return colf(sP + k * FC + m, FC); }, fQc, m0, n0d, m0, C);
        float* g = p.wdk + ub * C * D;
        for_acc(dk, m0, n0d, [&](int r, int kk, float& x, int rs, int cs) { g[r * D + kk] = x; });
    }
    // gam_C <dS_C, S_0>
    {
        float s = 0.f;
        for (int x = tid; x < D * D; x += kGradThreads) {
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
__global__ void __launch_bounds__(kGradThreads, 1) grad_rest_kernel(const Params p) {
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

    copy_tile_async<C>(sT, FC, p.wti + ub * C * C, C, C, C);
    copy_tile_async<D>(sW, FD, p.ww + ub * C * D, D, C, C);
    copy_tile_async<D>(sUt, FD, p.wut + ub * C * D, D, C, C);
    copy_tile_async<D>(sdU, FD, p.wdu + ub * C * D, D, C, C);
    copy_tile_async<D>(sdW, FD, p.wdw + ub * C * D, D, C, C);
    copy_tile_async<D>(sK, HD, p.k + tok0 * D, D, C, n);
    copy_tile_async<D>(sV, HD, p.v + tok0 * D, D, C, n);
    cp_async_commit();
    if (tid < C) {
        vb[tid] = p.wb[ub * 2 * C + tid];
        vbeta[tid] = tid < n ? p.beta[tok0 + tid] : 0.f;
        vdb[tid] = p.wdb[ub * C + tid];
        vdbeta[tid] = 0.f;
    }
    cp_async_wait0();
    __syncthreads();
    if (tid < C) vgam[tid] = expf(vb[tid]);
    __syncthreads();
    const int m0 = (warp >> 2) * 16 * GMT, n0c = (warp & 3) * 16, n0d = (warp & 3) * (D / 4);
    const BT fK{sK, HD};
    // dRv = Ti^T dU, dRk = Ti^T dW (Ti^T upper: k >= m0); K K^T -> sA
    float rv[GMT][NT][4], rk[GMT][NT][4];
    zero(rv);
    zero(rk);
    {
        const auto ftt = [&](int m, int k) { return colf(sT + k * FC + m, FC); };
        warp_mma<GMT, NT>(rv, ftt, [&](int k, int nn) { return colf(sdU + k * FD + nn, FD); }, m0, n0d, m0, C);
        warp_mma<GMT, NT>(rk, ftt, [&](int k, int nn) { return colf(sdW + k * FD + nn, FD); }, m0, n0d, m0, C);
        float kk[GMT][2][4];
        zero(kk);
        warp_mma<GMT, 2, false, false>(kk, [&](int m, int k) { return rowh(sK + m * HD + k); },
                                     [&](int k, int nn) { return rowh(sK + nn * HD + k); }, m0, n0c, 0, D);
        for_acc(kk, m0, n0c, [&](int r, int s, float& x, int rs, int cs) { sA[r * FC + s] = x; });
        // dV = beta dRv; dbeta += dRv.v + gam dRk.k; db += beta gam dRk.k
        bf16* gv = p.dv + tok0 * D;
        float hb[2 * GMT] = {}, hg[2 * GMT] = {};
#pragma unroll
        for (int i = 0; i < GMT; ++i)
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
                    hb[2 * i + e2] += a0 * bf(sV, r * HD + cc) + a1 * bf(sV, r * HD + cc + 1) + vgam[r] * kr;
                    hg[2 * i + e2] += vbeta[r] * vgam[r] * kr;
                }
        add_rows<GMT>(hb, m0, vdbeta);
        add_rows<GMT>(hg, m0, vdb);
    }
    __syncthreads();   // dU, dW no longer read
    for_acc(rv, m0, n0d, [&](int r, int i, float& x, int rs, int cs) { sdU[r * FD + i] = x; });
    for_acc(rk, m0, n0d, [&](int r, int i, float& x, int rs, int cs) { sdW[r * FD + i] = x; });
    __syncthreads();
    // dA = -(dRv Ut^T + dRk W^T), strictly lower; F = beta dA o E in place of K K^T
    {
        float da[GMT][2][4];
        zero(da);
        warp_mma<GMT, 2>(da, [&](int m, int k) { return rowf(sdU + m * FD + k); },
                       [&](int k, int nn) { return rowf(sUt + nn * FD + k); }, m0, n0c, 0, D);
        warp_mma<GMT, 2>(da, [&](int m, int k) { return rowf(sdW + m * FD + k); },
                       [&](int k, int nn) { return rowf(sW + nn * FD + k); }, m0, n0c, 0, D);
        float hr[2 * GMT] = {}, hc[4] = {}, hb[2 * GMT] = {};
        for_acc(da, m0, n0c, [&](int r, int s, float& x, int rs, int cs) {
            float f = 0.f;
            if (s < r) {
                const float d = -x, e = expf(vb[r] - vb[s]), kk = sA[r * FC + s];
                const float aa = d * vbeta[r] * e * kk;
                hr[rs] += aa;
                hc[cs] -= aa;
                hb[rs] += d * e * kk;
                f = vbeta[r] * d * e;
            }
            sA[r * FC + s] = f;
        });
        add_rows<GMT>(hr, m0, vdb);
        add_cols<2>(hc, n0c, vdb);
        add_rows<GMT>(hb, m0, vdbeta);
    }
    __syncthreads();   // F complete
    // dK = F K + F^T K + diag(beta gam) dRk + state terms
    {
        const float* g1 = p.wdk + ub * C * D;
        float2 pre[2][NT][2];   // state terms, loaded before the products
#pragma unroll
        for (int i = 0; i < GMT; ++i)
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int e2 = 0; e2 < 2; ++e2) {
                    const int lane = tid & 31, r = m0 + 16 * i + (lane >> 2) + 8 * e2;
                    pre[i][j][e2] = *reinterpret_cast<const float2*>(g1 + r * D + n0d + 8 * j + 2 * (lane & 3));
                }
        float dk[GMT][NT][4];
        zero(dk);
        warp_mma<GMT, NT>(dk, [&](int m, int k) { return rowf(sA + m * FC + k); }, fK, m0, n0d, 0, m0 + 16 * GMT);
        warp_mma<GMT, NT>(dk, [&](int m, int k) { return colf(sA + k * FC + m, FC); }, fK, m0, n0d, m0, C);
        bf16* gk = p.dk + tok0 * D;
#pragma unroll
        for (int i = 0; i < GMT; ++i)
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int e2 = 0; e2 < 2; ++e2) {
                    const int lane = tid & 31, r = m0 + 16 * i + (lane >> 2) + 8 * e2;
                    const int cc = n0d + 8 * j + 2 * (lane & 3);
                    if (r < n) {
                        const float bg = vbeta[r] * vgam[r];
                        const float x0 = dk[i][j][2 * e2] + bg * sdW[r * FD + cc] + pre[i][j][e2].x;
                        const float x1 = dk[i][j][2 * e2 + 1] + bg * sdW[r * FD + cc + 1] + pre[i][j][e2].y;
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
#define LA_GBW_LAUNCH(kern, grid, bytes, threads)                                                          \
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)); \
    if (e != cudaSuccess) return e;                                                                        \
    kern<<<grid, threads, bytes, s>>>(p);                                                                  \
    e = cudaGetLastError();                                                                                \
    if (e != cudaSuccess) return e;
    LA_GBW_LAUNCH(prep_kernel<D>, units, PrepSmem<D>::BYTES, kThreads)
    LA_GBW_LAUNCH(chain_kernel<D>, 2 * p.BH * kChainSplit, ChainSmem<D>::BYTES, 2 * D / kChainSplit)
    LA_GBW_LAUNCH(grad_state_kernel<D>, units, GradASmem<D>::BYTES, kGradThreads)
    LA_GBW_LAUNCH(grad_rest_kernel<D>, units, GradBSmem<D>::BYTES, kGradThreads)
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
    p.wb = reinterpret_cast<float*>(take(units * 2 * C * 4));
    p.wti = reinterpret_cast<float*>(take(units * C * C * 4));
    p.ww = reinterpret_cast<float*>(take(units * C * D * 4));
    p.wut = reinterpret_cast<float*>(take(units * C * D * 4));
    p.wqht = reinterpret_cast<float*>(take(units * C * D * 4));
    p.wlkt = reinterpret_cast<float*>(take(units * C * D * 4));
    p.wlwt = reinterpret_cast<float*>(take(units * C * D * 4));
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
