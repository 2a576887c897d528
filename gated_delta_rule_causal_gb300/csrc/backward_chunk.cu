// Chunkwise backward of the normalized elu+1 recurrence on the tcgen05
// tensor cores (d_k = d_v = 64, bf16 io, chunks of C = 64 tokens).
//
// The pages define the forward operator only ("Linear attention and
// recurrent memory", The big idea: S_t = S_{t-1} + phi(k_t) v_t^T,
// z_t = z_{t-1} + phi(k_t), o_t = phi(q_t)^T S_t / phi(q_t)^T z_t) and name
// chunked training as the reason chunkwise kernels exist. The gradients follow
// from the chain rule through that update-first recurrence. Per chunk c, with
// Q~ = phi(Q), K~ = phi(K), X_in = S_in^T and z_in the state entering the
// chunk, L the causal mask including the diagonal and P = L o Q~ K~^T:
//    num  = P V + Q~ S_in,            den  = P 1 + Q~ z_in
//    dnum = dO / den,                 dden = -rowsum(dO o num) / den^2
//    dP   = L o (dnum V^T + dden 1^T)
//    dQ~  = dP K~ + dnum S_in^T + dden z_in^T
//    dK~  = dP^T Q~ + V G^T + 1 g^T,  dV = P^T dnum + K~ G
// where G (d_k x d_v) and g are the gradients of the state and normalizer
// after the chunk: the final-state cotangent plus Q~^T dnum and Q~^T dden of
// every later chunk. dq = dQ~ o phi'(q), dk = dK~ o phi'(k), with
// phi'(x) = 1 for x > 0 and e^x otherwise, i.e. min(1, phi(x)). The initial
// state receives G and g after chunk 0 has added its own terms.
//
// Five launches, chained by programmatic dependent launch (each kernel waits
// for the previous one before reading what it wrote):
//  1-2. the forward three-phase form's chunk summaries and scan (in
//       prefill_par.cu): X_in, z_in and phi(k) operand tiles of every chunk;
//  3. bw_sum_kernel, one CTA per (head, chunk): num, den, dnum, dden and the
//     chunk's terms dG^T = dnum^T Q~ and dg = Q~^T dden;
//  4. bw_scan_kernel: G and g after every chunk, walked from the last chunk
//     to the first, and the initial state's gradient;
//  5. bw_grad_kernel, one CTA per (head, chunk): dq, dk and dv.
//
// Every product is a bf16 tcgen05 MMA with fp32 accumulation in tensor
// memory. The token and feature dimensions are 64, so the products run with
// M = 128 and only accumulator lanes 0-63 are read: the A operand's rows
// 64-127 are the next 8 KB tile of shared memory (finite data, results
// unused).
//
// Tail chunks: TMA zero-fills q, k, v and dO rows past T, and phi(k) is set
// to zero there, so padded tokens have dnum = 0 and dden = 0 and add nothing;
// their gradient rows are not stored.
#include <cuda_bf16.h>

#include "prefill.h"
#include "prefill_impl.cuh"
#include "launch.cuh"

namespace la {
namespace bwd {

using chunk::C;
using chunk::elu1;
using chunk::kmaj;
using chunk::ld_shared_bf16;
using chunk::ld_shared_v4;
using chunk::mnmaj;
using chunk::st_shared_v4;
using chunk::store_row32_bf16;

constexpr int D = 64;                  // d_k = d_v
constexpr int kThreads = 256;
constexpr uint32_t TILE = 8192;        // one [64][64] bf16 operand tile, 128-byte swizzle
constexpr uint32_t VEC = D * 4;        // one fp32 vector of 64

struct Params {
    const float* dstate_out;   // [BH][D*D + D] (S [k][v], then z), or NULL
    float* dstate_in;          // same layout, or NULL
    __nv_bfloat16* dq;         // [BH][T][D]
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    const uint8_t* xs;         // [units] X_in = S_in^T tiles [v][k]
    const float* zs;           // [units][D] z_in
    float* dG;                 // [units][v][k] fp32: dnum^T Q~ of the chunk
    float* dg;                 // [units][D]: Q~^T dden of the chunk
    uint8_t* dn;               // [units] dnum tiles [t][v]
    uint8_t* gs;               // [units] tiles of G after the chunk, [v][k]
    float* gz;                 // [units][D] g after the chunk
    float* ddn;                // [units][C] dden
    int BH, T, nch;
    unsigned flags;
    int* status;
};

// Four fp32 values of a thread's row as two bf16 pairs into global memory.
__device__ __forceinline__ void store_row32_global(__nv_bfloat16* dst, const float* x) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float* y = x + 8 * m;
        *reinterpret_cast<uint4*>(dst + 8 * m) =
            make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]), pack_bf16(y[6], y[7]));
    }
}

// Eight bf16 values of a swizzled tile row (16-byte chunk c) as floats.
__device__ __forceinline__ void load8(uint32_t tile, int row, int c, float* out) {
    const uint4 u = ld_shared_v4(tile + sw128_off(row, c));
    const float2 a = unpack_bf16(u.x), b = unpack_bf16(u.y), d = unpack_bf16(u.z), e = unpack_bf16(u.w);
    out[0] = a.x; out[1] = a.y; out[2] = b.x; out[3] = b.y;
    out[4] = d.x; out[5] = d.y; out[6] = e.x; out[7] = e.y;
}

// phi in place over the q and k tiles ([64][64] each, two 16-byte chunks
// per thread and tile); k rows at or past `nvalid` (tokens past T) become 0.
__device__ __forceinline__ void phi_tiles(uint32_t tq, uint32_t tk, int nvalid, int tid) {
#pragma unroll
    for (int i = 0; i < (2 * 64 * 8) / kThreads; ++i) {
        const int e = tid + kThreads * i;
        const bool isk = e >= 64 * 8;
        const int row = (e / 8) % 64, pc = e % 8;
        const uint32_t a = (isk ? tk : tq) + (row >> 3) * 1024 + (row & 7) * 128 + pc * 16;
        const uint4 u = ld_shared_v4(a);
        const float2 x0 = unpack_bf16(u.x), x1 = unpack_bf16(u.y), x2 = unpack_bf16(u.z), x3 = unpack_bf16(u.w);
        const float m = (isk && row >= nvalid) ? 0.f : 1.f;
        st_shared_v4(a, pack_bf16(m * elu1(x0.x), m * elu1(x0.y)), pack_bf16(m * elu1(x1.x), m * elu1(x1.y)),
                     pack_bf16(m * elu1(x2.x), m * elu1(x2.y)), pack_bf16(m * elu1(x3.x), m * elu1(x3.y)));
    }
}

__device__ __forceinline__ void publish() {
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// ---------------------------------------------------------------------------
// 3. per-chunk normalizer gradients and the chunk's state-gradient terms
// ---------------------------------------------------------------------------
struct SumL {
    static constexpr uint32_t Q = 0, K = TILE, V = 2 * TILE, XS = 3 * TILE, DO = 4 * TILE, PS = 5 * TILE,
                              DN = 6 * TILE, PAD = 7 * TILE, MISC = 8 * TILE;
    // misc: z_in, den, rowsum(dO o num), dden, dg (fp32, 64 each)
    static constexpr uint32_t BAR = MISC + 5 * VEC;
    // 67.9 KB: three CTAs (3 x 128 columns of tensor memory) share an SM
    static constexpr uint32_t SMEM = BAR + 64 + 1024;
    // dG^T reuses P's columns: P has been read out before the MMA that
    // completes num is issued
    static constexpr uint32_t COL_P = 0, COL_O = 64, COL_G = 0;
    static constexpr uint32_t TMEM_COLS = 128;
};

__global__ void __launch_bounds__(kThreads, 3) bw_sum_kernel(const __grid_constant__ CUtensorMap tmq,
                                                          const __grid_constant__ CUtensorMap tmk,
                                                          const __grid_constant__ CUtensorMap tmv,
                                                          const __grid_constant__ CUtensorMap tmdo, const Params p) {
    using L = SumL;
    griddep_launch_dependents();
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (sbase - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = 32 * (warp & 3) + lane;   // tensor-memory lane
    const int hh = warp >> 2;               // column half
    const bool rows = (warp & 3) < 2;       // lanes 0-63: the 64 token (or value) rows
    const int u = blockIdx.x;
    const int bh = u / p.nch, c = u % p.nch, t0 = c * C;
    float* sZ = reinterpret_cast<float*>(sm + L::MISC);
    float* sDen = sZ + D;
    float* sDot = sDen + D;
    float* sDden = sDot + D;
    float* sDg = sDden + D;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR);   // [0] loads, [1] MMAs, [2] test hook
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 3);
    const uint32_t aQ = sbase + L::Q, aK = sbase + L::K, aV = sbase + L::V, aXS = sbase + L::XS;
    const uint32_t aDO = sbase + L::DO, aPS = sbase + L::PS, aDN = sbase + L::DN;

    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
        tma_prefetch_desc(&tmdo);
    }
    if (tid < D) {
        sDen[tid] = 0.f;
        sDot[tid] = 0.f;
        sDg[tid] = 0.f;
    }
    // The previous kernel first, then tensor memory: a CTA never holds
    // columns while it waits on another grid, so a CTA of this grid that
    // waits in tcgen05.alloc only waits for CTAs that finish on their own.
    griddep_wait();   // the states entering every chunk are complete
    if (warp == 0) tmem_alloc(tmem_slot, L::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);

    int status_bits = 0;
    bool failed = false;
    if (p.flags & 0x100u) {   // test hook: a wait nothing will satisfy, 1 ms limit
        const bool ok = mbar_wait(&bar[2], 0, 1000000ull);
        if (__syncthreads_or(!ok)) { status_bits |= kStatusTestHook; failed = true; }
    }
    bool loading = false;
    if (!failed && tid == 0) {
        mbar_arrive_expect_tx(&bar[0], 5 * TILE + VEC);
        tma_load_3d(&tmq, &bar[0], sm + L::Q, 0, t0, bh);
        tma_load_3d(&tmk, &bar[0], sm + L::K, 0, t0, bh);
        tma_load_3d(&tmv, &bar[0], sm + L::V, 0, t0, bh);
        bulk_load(sm + L::XS, p.xs + static_cast<size_t>(u) * TILE, TILE, &bar[0]);
        tma_load_3d(&tmdo, &bar[0], sm + L::DO, 0, t0, bh);
        bulk_load(sZ, p.zs + static_cast<size_t>(u) * D, VEC, &bar[0]);
        loading = true;
    }
    int nmma = 0;   // MMA commits issued (thread 0)
    auto mma_wait = [&](uint32_t parity) {
        const bool ok = mbar_wait(&bar[1], parity, kWaitLimitNs);
        tc_fence_after();
        if (__syncthreads_or(!ok)) { status_bits |= kStatusMmaWait; failed = true; }
    };
    if (!failed) {
        const bool ok = mbar_wait(&bar[0], 0, kWaitLimitNs);
        if (__syncthreads_or(!ok)) { status_bits |= kStatusTmaWait; failed = true; }
        else loading = false;
    }
    const int nvalid = min(C, p.T - t0);
    if (!failed) {
        phi_tiles(aQ, aK, nvalid, tid);
        publish();
        // P = Q~ K~^T, O = Q~ X_in^T (tokens on the lanes)
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                mma_bf16_ss(tmem + L::COL_P, kmaj(aQ + kk * 32), kmaj(aK + kk * 32), idesc_bf16(128, 64, false, false),
                            kk > 0);
                mma_bf16_ss(tmem + L::COL_O, kmaj(aQ + kk * 32), kmaj(aXS + kk * 32), idesc_bf16(128, 64, false, false),
                            kk > 0);
            }
            mma_commit(&bar[1]);
            ++nmma;
        }
        // den_t = q~_t . z_in meanwhile (4 threads per token)
        {
            const int t = tid >> 2, q4 = tid & 3;
            float d = 0.f;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int cq = 2 * q4 + m;
                float x[8];
                load8(aQ, t, cq, x);
#pragma unroll
                for (int e = 0; e < 8; ++e) d += x[e] * sZ[8 * cq + e];
            }
            d += __shfl_xor_sync(0xffffffffu, d, 1);
            d += __shfl_xor_sync(0xffffffffu, d, 2);
            if (q4 == 0) atomicAdd(&sDen[t], d);
        }
        mma_wait(0);
    }
    if (!failed) {
        // masked scores -> bf16 P; their row sums complete den
        if (rows) {
            const int t = r;
            float x[32];
            tmem_ld32(tlane + L::COL_P + 32 * hh, x);
            tmem_ld_wait();
            float rs = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                x[i] = (32 * hh + i <= t) ? x[i] : 0.f;
                rs += x[i];
            }
            store_row32_bf16(aPS, t, 4 * hh, x);
            atomicAdd(&sDen[t], rs);
        }
        publish();
        // num = O + P V
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + L::COL_O, kmaj(aPS + kk * 32), mnmaj(aV + kk * 2048, 8192),
                            idesc_bf16(128, 64, false, true), 1);
            mma_commit(&bar[1]);
            ++nmma;
        }
        mma_wait(1);
    }
    if (!failed) {
        // dnum = dO / den as the bf16 tile, and rowsum(dO o num)
        if (rows) {
            const int t = r;
            float x[32], dn[32];
            tmem_ld32(tlane + L::COL_O + 32 * hh, x);
            tmem_ld_wait();
            const float inv = __fdividef(1.f, sDen[t]);
            float dot = 0.f;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                float g[8];
                load8(aDO, t, 4 * hh + m, g);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    dn[8 * m + e] = g[e] * inv;
                    dot += g[e] * x[8 * m + e];
                }
            }
            store_row32_bf16(aDN, t, 4 * hh, dn);
            atomicAdd(&sDot[t], dot);
        }
        publish();
        // dG^T = dnum^T Q~ (value rows on the lanes); dnum to the workspace
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + L::COL_G, mnmaj(aDN + kk * 2048, 8192), mnmaj(aQ + kk * 2048, 8192),
                            idesc_bf16(128, 64, true, true), kk > 0);
            mma_commit(&bar[1]);
            ++nmma;
            bulk_store(p.dn + static_cast<size_t>(u) * TILE, aDN, TILE);
            bulk_commit();
        }
        // dden_t = -rowsum(dO o num) / den_t^2, then dg = Q~^T dden
        if (tid < C) {
            const float inv = __fdividef(1.f, sDen[tid]);
            const float dd = -sDot[tid] * inv * inv;
            sDden[tid] = dd;
            p.ddn[static_cast<size_t>(u) * C + tid] = dd;
        }
        __syncthreads();
        {
            const int ch = tid & 63, part = tid >> 6;   // 4 parts of 16 tokens
            const uint32_t col = aQ + (ch & 7) * 2;
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int t = 16 * part + i;
                s += ld_shared_bf16(col + sw128_off(t, ch >> 3)) * sDden[t];
            }
            atomicAdd(&sDg[ch], s);
        }
        __syncthreads();
        if (tid < D) p.dg[static_cast<size_t>(u) * D + tid] = sDg[tid];
        mma_wait(2);
    }
    if (!failed && rows) {
        float* dst = p.dG + (static_cast<size_t>(u) * D + r) * D + 32 * hh;
        float x[32];
        tmem_ld32(tlane + L::COL_G + 32 * hh, x);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; i += 4) *reinterpret_cast<float4*>(dst + i) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
    }
    if (tid == 0) {
        if (loading) mbar_wait(&bar[0], 0, 100000000ull);   // let the loads land before the CTA exits
        if (failed && nmma > 0) {   // and the MMAs issued: one more commit covers them
            mma_commit(&bar[2]);
            mbar_wait(&bar[2], 0, 100000000ull);
        }
        bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
    if (status_bits && tid == 0) atomicOr(p.status, status_bits);
}

// ---------------------------------------------------------------------------
// 4. G and g after every chunk, from the last chunk to the first
// ---------------------------------------------------------------------------
constexpr int kScanThreads = 256;
constexpr int kScanBatch = 16;

// One thread per 2 key columns of one value row of G (as G^T [v][k]), and one
// per 2 channels of g.
__global__ void __launch_bounds__(kScanThreads) bw_scan_kernel(const Params p) {
    constexpr int E2 = D * D / 2, PER = E2 + D / 2;
    constexpr size_t SSZ = static_cast<size_t>(D) * D + D;
    griddep_launch_dependents();
    griddep_wait();   // every chunk's terms are complete
    const int gi = blockIdx.x * kScanThreads + threadIdx.x;
    const int bh = gi / PER, e = gi % PER;
    if (bh >= p.BH) return;
    const int nch = p.nch;
    if (e < E2) {
        const int r = e / (D / 2), col = 2 * (e % (D / 2));   // value row r, key columns col, col + 1
        float2 x = make_float2(0.f, 0.f);
        if (p.dstate_out) {   // dS_T[k][v]
            const float* so = p.dstate_out + bh * SSZ + r;
            x = make_float2(so[static_cast<size_t>(col) * D], so[static_cast<size_t>(col + 1) * D]);
        }
        const float* dG = p.dG + (static_cast<size_t>(bh) * nch * D + r) * D + col;
        uint8_t* gs = p.gs + static_cast<size_t>(bh) * nch * TILE + sw128_off(r, col / 8) + (col % 8) * 2;
        for (int c = nch - 1; c >= 0; c -= kScanBatch) {
            float2 a[kScanBatch];
#pragma unroll
            for (int i = 0; i < kScanBatch; ++i)
                if (c - i >= 0) a[i] = *reinterpret_cast<const float2*>(dG + static_cast<size_t>(c - i) * D * D);
#pragma unroll
            for (int i = 0; i < kScanBatch; ++i) {
                if (c - i >= 0) {
                    *reinterpret_cast<uint32_t*>(gs + static_cast<size_t>(c - i) * TILE) = pack_bf16(x.x, x.y);
                    x = make_float2(x.x + a[i].x, x.y + a[i].y);
                }
            }
        }
        if (p.dstate_in) {
            float* si = p.dstate_in + bh * SSZ + r;
            si[static_cast<size_t>(col) * D] = x.x;
            si[static_cast<size_t>(col + 1) * D] = x.y;
        }
    } else {
        const int ch = 2 * (e - E2);
        float2 z = make_float2(0.f, 0.f);
        if (p.dstate_out) z = *reinterpret_cast<const float2*>(p.dstate_out + bh * SSZ + static_cast<size_t>(D) * D + ch);
        for (int c = nch - 1; c >= 0; c -= kScanBatch) {
            float2 a[kScanBatch];
#pragma unroll
            for (int i = 0; i < kScanBatch; ++i)
                if (c - i >= 0) a[i] = *reinterpret_cast<const float2*>(p.dg + (static_cast<size_t>(bh) * nch + c - i) * D + ch);
#pragma unroll
            for (int i = 0; i < kScanBatch; ++i) {
                if (c - i >= 0) {
                    *reinterpret_cast<float2*>(p.gz + (static_cast<size_t>(bh) * nch + c - i) * D + ch) = z;
                    z = make_float2(z.x + a[i].x, z.y + a[i].y);
                }
            }
        }
        if (p.dstate_in) *reinterpret_cast<float2*>(p.dstate_in + bh * SSZ + static_cast<size_t>(D) * D + ch) = z;
    }
}

// ---------------------------------------------------------------------------
// 5. per-chunk input gradients
// ---------------------------------------------------------------------------
struct GradL {
    static constexpr uint32_t Q = 0, K = TILE, V = 2 * TILE, DN = 3 * TILE, XS = 4 * TILE, GS = 5 * TILE,
                              PS = 6 * TILE, DP = 7 * TILE, PAD = 8 * TILE, MISC = 9 * TILE;
    // misc: z_in, g, dden (fp32, 64 each)
    static constexpr uint32_t BAR = MISC + 3 * VEC;
    // 75.6 KB: three CTAs share an SM, two of which hold tensor memory
    // (2 x 256 columns) while the third has its tiles landing
    static constexpr uint32_t SMEM = BAR + 64 + 1024;
    static constexpr uint32_t COL_A = 0, COL_B = 64, COL_DV = 128;   // P then dQ~; dnum V^T then dK~; dV
    static constexpr uint32_t TMEM_COLS = 256;
};

__global__ void __launch_bounds__(kThreads, 3) bw_grad_kernel(const __grid_constant__ CUtensorMap tmq,
                                                           const __grid_constant__ CUtensorMap tmk,
                                                           const __grid_constant__ CUtensorMap tmv, const Params p) {
    using L = GradL;
    griddep_launch_dependents();
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (sbase - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = 32 * (warp & 3) + lane;
    const int hh = warp >> 2;
    const bool rows = (warp & 3) < 2;
    const int u = blockIdx.x;
    const int bh = u / p.nch, c = u % p.nch, t0 = c * C;
    float* sZ = reinterpret_cast<float*>(sm + L::MISC);
    float* sG = sZ + D;
    float* sDden = sG + D;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR);   // [0] loads, [1] MMAs, [2] test hook
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 3);
    const uint32_t aQ = sbase + L::Q, aK = sbase + L::K, aV = sbase + L::V, aDN = sbase + L::DN;
    const uint32_t aXS = sbase + L::XS, aGS = sbase + L::GS, aPS = sbase + L::PS, aDP = sbase + L::DP;

    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
    }
    griddep_wait();   // G and g after every chunk are complete
    // The tiles first: they need no tensor memory, so a CTA that waits in
    // tcgen05.alloc for another CTA of the SM to finish has them landing.
    bool loading = false;
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar[0], 6 * TILE + 3 * VEC);
        tma_load_3d(&tmq, &bar[0], sm + L::Q, 0, t0, bh);
        tma_load_3d(&tmk, &bar[0], sm + L::K, 0, t0, bh);
        tma_load_3d(&tmv, &bar[0], sm + L::V, 0, t0, bh);
        bulk_load(sm + L::DN, p.dn + static_cast<size_t>(u) * TILE, TILE, &bar[0]);
        bulk_load(sm + L::XS, p.xs + static_cast<size_t>(u) * TILE, TILE, &bar[0]);
        bulk_load(sm + L::GS, p.gs + static_cast<size_t>(u) * TILE, TILE, &bar[0]);
        bulk_load(sZ, p.zs + static_cast<size_t>(u) * D, VEC, &bar[0]);
        bulk_load(sG, p.gz + static_cast<size_t>(u) * D, VEC, &bar[0]);
        bulk_load(sDden, p.ddn + static_cast<size_t>(u) * C, VEC, &bar[0]);
        loading = true;
    }
    if (warp == 0) tmem_alloc(tmem_slot, L::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);

    int status_bits = 0;
    bool failed = false;
    if (p.flags & 0x100u) {   // test hook: a wait nothing will satisfy, 1 ms limit
        const bool ok = mbar_wait(&bar[2], 0, 1000000ull);
        if (__syncthreads_or(!ok)) { status_bits |= kStatusTestHook; failed = true; }
    }
    int nmma = 0;
    auto mma_wait = [&](uint32_t parity) {
        const bool ok = mbar_wait(&bar[1], parity, kWaitLimitNs);
        tc_fence_after();
        if (__syncthreads_or(!ok)) { status_bits |= kStatusMmaWait; failed = true; }
    };
    if (!failed) {
        const bool ok = mbar_wait(&bar[0], 0, kWaitLimitNs);
        if (__syncthreads_or(!ok)) { status_bits |= kStatusTmaWait; failed = true; }
        else loading = false;
    }
    constexpr uint32_t ID_KK = idesc_bf16(128, 64, false, false);
    constexpr uint32_t ID_KM = idesc_bf16(128, 64, false, true);
    constexpr uint32_t ID_MM = idesc_bf16(128, 64, true, true);
    if (!failed) {
        phi_tiles(aQ, aK, min(C, p.T - t0), tid);
        publish();
        // P = Q~ K~^T and dnum V^T (tokens on the lanes)
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                mma_bf16_ss(tmem + L::COL_A, kmaj(aQ + kk * 32), kmaj(aK + kk * 32), ID_KK, kk > 0);
                mma_bf16_ss(tmem + L::COL_B, kmaj(aDN + kk * 32), kmaj(aV + kk * 32), ID_KK, kk > 0);
            }
            mma_commit(&bar[1]);
            ++nmma;
        }
        mma_wait(0);
    }
    if (!failed) {
        // P and dP = L o (dnum V^T + dden 1^T) as bf16 tiles [t][j]
        if (rows) {
            const int t = r;
            const float dd = sDden[t];
            float x[32], y[32];
            tmem_ld32(tlane + L::COL_A + 32 * hh, x);
            tmem_ld32(tlane + L::COL_B + 32 * hh, y);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const bool in = 32 * hh + i <= t;
                x[i] = in ? x[i] : 0.f;
                y[i] = in ? y[i] + dd : 0.f;
            }
            store_row32_bf16(aPS, t, 4 * hh, x);
            store_row32_bf16(aDP, t, 4 * hh, y);
        }
        publish();
        if (tid == 0) {
            // dQ~ = dP K~ + dnum X_in (rows t)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + L::COL_A, kmaj(aDP + kk * 32), mnmaj(aK + kk * 2048, 8192), ID_KM, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + L::COL_A, kmaj(aDN + kk * 32), mnmaj(aXS + kk * 2048, 8192), ID_KM, 1);
            // dK~ = dP^T Q~ + V G^T (rows j)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + L::COL_B, mnmaj(aDP + kk * 2048, 8192), mnmaj(aQ + kk * 2048, 8192), ID_MM, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + L::COL_B, kmaj(aV + kk * 32), mnmaj(aGS + kk * 2048, 8192), ID_KM, 1);
            // dV = P^T dnum + K~ G (rows j)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + L::COL_DV, mnmaj(aPS + kk * 2048, 8192), mnmaj(aDN + kk * 2048, 8192), ID_MM, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + L::COL_DV, kmaj(aK + kk * 32), kmaj(aGS + kk * 32), ID_KK, 1);
            mma_commit(&bar[1]);
            ++nmma;
        }
        mma_wait(1);
    }
    // The tensor-memory loads are warp-collective: every lane of the row
    // warps runs them, and only the stores of rows past T are skipped.
    if (!failed && rows) {
        const int t = r;   // token row t of dq; token row j = t of dk and dv
        const bool live = t0 + t < p.T;
        const size_t row = (static_cast<size_t>(bh) * p.T + t0 + t) * D + 32 * hh;
        float x[32], f[8];
        // dq = (dQ~ + dden z_in^T) o min(1, phi(q))
        tmem_ld32(tlane + L::COL_A + 32 * hh, x);
        tmem_ld_wait();
        const float dd = sDden[t];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            load8(aQ, t, 4 * hh + m, f);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int i = 8 * m + e;
                x[i] = (x[i] + dd * sZ[32 * hh + i]) * fminf(1.f, f[e]);
            }
        }
        if (live) store_row32_global(p.dq + row, x);
        // dk = (dK~ + g^T) o min(1, phi(k))
        tmem_ld32(tlane + L::COL_B + 32 * hh, x);
        tmem_ld_wait();
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            load8(aK, t, 4 * hh + m, f);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int i = 8 * m + e;
                x[i] = (x[i] + sG[32 * hh + i]) * fminf(1.f, f[e]);
            }
        }
        if (live) store_row32_global(p.dk + row, x);
        tmem_ld32(tlane + L::COL_DV + 32 * hh, x);
        tmem_ld_wait();
        if (live) store_row32_global(p.dv + row, x);
    }
    if (tid == 0) {
        if (loading) mbar_wait(&bar[0], 0, 100000000ull);
        if (failed && nmma > 0) {
            mma_commit(&bar[2]);
            mbar_wait(&bar[2], 0, 100000000ull);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
    if (status_bits && tid == 0) atomicOr(p.status, status_bits);
}

// 3-D map over a [BH, T, 64] bf16 tensor with 64x64 boxes (one 128-byte
// swizzle atom wide); rows past T read as zeros.
CUresult map64(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, const void* base, int T, int BH) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(D) * 2 * T};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(C), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Backward workspace per unit beyond the forward phases' arrays: dnum and G
// tiles, g and dden vectors.
constexpr size_t kExtraPerUnit = 2 * TILE + 2 * VEC;

}  // namespace bwd

namespace chunk {

size_t bwd_chunk_bytes(int BH, int T) {
    const size_t units = static_cast<size_t>(BH) * ((T + C - 1) / C);
    return units * (par_state_bytes(bwd::D, bwd::D) + bwd::kExtraPerUnit);
}

cudaError_t launch_norm_backward_chunked(const BwdArgs& a, float* workspace, size_t ws_bytes, int* status,
                                         int sm_count, PFN_cuTensorMapEncodeTiled_v12000 enc, cudaStream_t s) {
    using namespace bwd;
    if (a.dk_dim != D || a.dv_dim != D || a.io != kBf16 || !workspace || bwd_chunk_bytes(a.BH, a.T) > ws_bytes)
        return cudaErrorInvalidValue;
    Maps m;
    if (map64(enc, &m.q, a.q, a.T, a.BH) != CUDA_SUCCESS || map64(enc, &m.k, a.k, a.T, a.BH) != CUDA_SUCCESS ||
        map64(enc, &m.v, a.v, a.T, a.BH) != CUDA_SUCCESS || map64(enc, &m.o, a.dout, a.T, a.BH) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // 1-2: the states entering every chunk
    FwdArgs f;
    f.q = a.q;
    f.k = a.k;
    f.v = a.v;
    f.gate = nullptr;
    f.beta = nullptr;
    f.state_in = a.state_in;
    f.out = nullptr;
    f.state_out = nullptr;
    f.den_out = nullptr;
    f.BH = a.BH;
    f.T = a.T;
    f.dk = D;
    f.dv = D;
    f.variant = kNorm;
    f.io = kBf16;
    f.flags = 0;
    f.status = status;
    f.sm_count = sm_count;
    f.workspace = workspace;
    f.ws_bytes = ws_bytes;
    f.nlaunch = nullptr;
    ParStates st;
    cudaError_t e = launch_par_states(f, m, s, &st);
    if (e != cudaSuccess) return e;
    const size_t units = static_cast<size_t>(a.BH) * st.nch;
    bwd::Params p;
    p.dstate_out = a.dstate_out;
    p.dstate_in = a.dstate_in;
    p.dq = static_cast<__nv_bfloat16*>(a.dq);
    p.dk = static_cast<__nv_bfloat16*>(a.dk);
    p.dv = static_cast<__nv_bfloat16*>(a.dv);
    p.xs = st.xs;
    p.zs = st.zs;
    p.dG = st.dx;   // the chunk summaries are dead once the scan has run
    p.dg = st.dd;
    uint8_t* w = st.end;
    p.dn = w;
    w += units * TILE;
    p.gs = w;
    w += units * TILE;
    p.gz = reinterpret_cast<float*>(w);
    w += units * VEC;
    p.ddn = reinterpret_cast<float*>(w);
    p.BH = a.BH;
    p.T = a.T;
    p.nch = st.nch;
    p.flags = a.flags;
    p.status = status;
    // 3-5
    e = cudaFuncSetAttribute(bw_sum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SumL::SMEM);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(bw_grad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GradL::SMEM);
    if (e != cudaSuccess) return e;
    e = launch_pdl(bw_sum_kernel, static_cast<unsigned>(units), kThreads, SumL::SMEM, s, m.q, m.k, m.v, m.o, p);
    if (e != cudaSuccess) return e;
    constexpr int PER = D * D / 2 + D / 2;
    const long long nthr = static_cast<long long>(a.BH) * PER;
    e = launch_pdl(bw_scan_kernel, static_cast<unsigned>((nthr + kScanThreads - 1) / kScanThreads), kScanThreads, 0, s, p);
    if (e != cudaSuccess) return e;
    return launch_pdl(bw_grad_kernel, static_cast<unsigned>(units), kThreads, GradL::SMEM, s, m.q, m.k, m.v, p);
}

}  // namespace chunk
}  // namespace la
