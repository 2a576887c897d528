// Chunkwise prefill on the tcgen05 tensor cores (sm_103a).
//
// One CTA per (b,h) sequence-head walks its sequence in chunks of C = 64
// tokens. TMA stages the q/k/v tiles (and the per-channel gate tile of the
// gated variant) of chunk c+1 while chunk c is computed. The dense products
// run as tcgen05 bf16 MMAs with fp32 accumulators in tensor memory. The fp32
// state is kept in registers (thread r owns state row r, r = value index)
// and re-published each chunk as a bf16 MMA operand in shared memory.
//
// Inside the kernel the state is always held as X [d_v rows][d_k cols]:
// X = S^T for the normalized and gated variants (S is d_k x d_v there) and
// X = S for the gated delta rule (S is d_v x d_k there). With that
// orientation every state-side product has M = 128 (value rows, padded
// when d_v = 64) and N = tokens or d_k.
//
// Chunk algebra (G_t = sum of log-gates inside the chunk up to t, Gam_t =
// exp(G_t), L = causal mask including the diagonal):
//
//  norm / gla ("Linear attention and Hyena" 11.2-11.3, secondary rescaling):
//    q~_t = phi(q_t) * Gam_t,  k~_j = phi(k_j) / Gam_j,  k^_j = phi(k_j) * Gam_C / Gam_j
//    O^T  = X_0 Q~^T + V^T (L o Q~ K~^T)^T
//    X    = diag-cols(Gam_C) X_0 + V^T K^
//    norm adds den_t = q~_t . z_0 + sum_{j<=t} q~_t . k~_j, o_t = num_t / den_t.
//
//  gated delta rule (S_t = g_t S_{t-1}(I - beta_t k_t k_t^T) + beta_t v_t k_t^T):
//    writing S_t = gam_t S_0 + sum_{j<=t} (gam_t/gam_j) u_j k_j^T gives
//    (I + A) U = diag(beta) V - diag(beta gam) K S_0^T with
//    A_tj = beta_t (gam_t/gam_j) k_t . k_j for j < t. With T = (I + A)^{-1},
//    Ut = T diag(beta) V and W = T diag(beta gam) K:
//      U^T = Ut^T - X_0 W^T
//      O^T = X_0 (diag(gam) Q)^T + U^T (M o Q K^T)^T,  M_tj = gam_t/gam_j (j <= t)
//      X   = gam_C X_0 + U^T diag(gam_C/gam) K
//    The triangular inverse T is formed in shared memory (fp32, blocked
//    forward substitution).
//
// Tail chunks (T not a multiple of 64): TMA zero-fills rows past the end.
// phi(0) = 1, so padded keys are zeroed explicitly; padded gates are 1 and
// padded betas 0, which makes padded tokens leave the state untouched.
#pragma once

#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace la {
namespace chunk {

constexpr int C = 64;          // tokens per chunk
constexpr int kThreads = 128;  // one thread per TMEM lane / state row
constexpr int kAStride = 68;   // fp32 row stride of the 64x64 solve matrix

struct Params {
    const float* gate;      // gdn: [BH, T] (gla gates travel by TMA)
    const float* beta;      // gdn: [BH, T]
    const float* state_in;  // may be NULL
    __nv_bfloat16* out;
    float* state_out;       // may be NULL
    float* den_out;         // norm, may be NULL
    int T;
    int nchunks;
    unsigned flags;
    int* status;
};

template <int VAR, int DK, int DV>
struct Layout {
    static constexpr int KA = DK / 64;  // 64-column atoms along d_k
    static constexpr int VA = DV / 64;
    // q/k tile pair: per k-atom, rows 0-63 hold block 0 and rows 64-127 block 1.
    static constexpr uint32_t QK_ATOM = 16384;
    static constexpr uint32_t QK_BYTES = KA * QK_ATOM;
    static constexpr uint32_t V_ATOM = 8192;
    static constexpr uint32_t V_BYTES = VA * V_ATOM;
    static constexpr uint32_t G_BYTES = (VAR == kGla) ? C * DK * 4 : 0;
    static constexpr uint32_t STAGE = QK_BYTES + V_BYTES + G_BYTES;
    static constexpr uint32_t TX_BYTES = 2 * KA * 8192 + V_BYTES + G_BYTES;
    static constexpr uint32_t OFF_SS = 2 * STAGE;               // bf16 state, [128 rows][DK]
    static constexpr uint32_t OFF_PS = OFF_SS + KA * 16384;     // bf16 [64 t][64 j]
    static constexpr uint32_t OFF_KH = OFF_PS + 8192;           // gla: k^ [64 j][DK]
    static constexpr uint32_t KH_BYTES = (VAR == kGla) ? KA * 8192 : 0;
    static constexpr bool GDN = (VAR == kGdn);
    static constexpr uint32_t OFF_TB1 = OFF_KH + KH_BYTES;      // gdn: T diag(beta)      [t][j]
    static constexpr uint32_t OFF_TB2 = OFF_TB1 + (GDN ? 8192 : 0);   // T diag(beta gam) [t][j]
    static constexpr uint32_t OFF_WS = OFF_TB2 + (GDN ? 8192 : 0);    // W^T [dk rows][t]
    static constexpr uint32_t OFF_US = OFF_WS + (GDN ? 16384 : 0);    // U^T [dv rows][j]
    static constexpr uint32_t OFF_AS = OFF_US + (GDN ? 16384 : 0);    // fp32 [64][68]
    static constexpr uint32_t OFF_RS = OFF_AS + (GDN ? C * kAStride * 4 : 0);  // fp32 [16][48]
    static constexpr uint32_t OFF_MISC = OFF_RS + (GDN ? 16 * 48 * 4 : 0);
    // misc: 6 arrays of 64 floats + 2 arrays of 128 floats
    static constexpr uint32_t OFF_BAR = OFF_MISC + 6 * 64 * 4 + 2 * 128 * 4;
    static constexpr uint32_t BYTES = OFF_BAR + 64;
    static constexpr uint32_t SMEM_ALLOC = BYTES + 1024;  // slack to align the base to 1024
    static constexpr uint32_t TMEM_COLS = GDN ? 512 : 256;
    // TMEM column map
    static constexpr uint32_t COL_G = 0;                 // gdn: [K;Q] K^T   | norm/gla: P
    static constexpr uint32_t COL_W = 64;                // gdn: W^T
    static constexpr uint32_t COL_U = GDN ? 128 : 0;     // gdn: U^T
    static constexpr uint32_t COL_O = GDN ? 192 : 64;    // O^T
    static constexpr uint32_t COL_S = GDN ? 256 : 128;   // Delta X
    static_assert(STAGE % 1024 == 0, "stage alignment");
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
};

__device__ __forceinline__ uint64_t kmaj(uint32_t addr) { return sdesc_sw128(addr, 16, 1024); }
__device__ __forceinline__ uint64_t mnmaj(uint32_t addr, uint32_t lbo) { return sdesc_sw128(addr, lbo, 1024); }

__device__ __forceinline__ float elu1(float x) { return x > 0.f ? x + 1.f : __expf(x); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
    return v;
}

// Store 32 fp32 values as 4 swizzled 16-byte chunks (chunks c0..c0+3) of row r.
__device__ __forceinline__ void store_row32_bf16(uint32_t tile, uint32_t r, uint32_t c0, const float* x) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float* y = x + 8 * m;
        st_shared_v4(tile + sw128_off(r, c0 + m), pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]),
                     pack_bf16(y[4], y[5]), pack_bf16(y[6], y[7]));
    }
}

template <int VAR, int DK, int DV>
__global__ void __launch_bounds__(kThreads, 1)
chunk_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
             const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmg,
             const Params p) {
    using L = Layout<VAR, DK, DV>;
    constexpr int KA = L::KA, VA = L::VA;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (sbase - raw);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x;
    const int T = p.T, nch = p.nchunks;
    const bool phi_on = !(VAR == kGla && (p.flags & 0x1u));

    float* sG = reinterpret_cast<float*>(sm + L::OFF_MISC);  // gdn: cumulative log-gate
    float* sB = sG + 64;       // gdn: beta (0 on padded tokens)
    float* sGam = sB + 64;     // gdn: exp(G_t)
    float* sBG = sGam + 64;    // gdn: beta_t exp(G_t)
    float* sKf = sBG + 64;     // gdn: exp(G_C - G_j)
    float* sDen = sKf + 64;    // norm: denominators of the chunk
    float* sGC = sDen + 64;    // gla: Gam_C per channel (128)
    float* sZ = sGC + 128;     // norm: z (128)
    uint64_t* bar_full = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
    uint64_t* bar_mma = bar_full + 2;
    uint64_t* bar_test = bar_full + 3;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_full + 4);

    const uint32_t aSS = sbase + L::OFF_SS, aPS = sbase + L::OFF_PS, aKH = sbase + L::OFF_KH;
    const uint32_t aTB1 = sbase + L::OFF_TB1, aTB2 = sbase + L::OFF_TB2;
    const uint32_t aWS = sbase + L::OFF_WS, aUS = sbase + L::OFF_US;
    float* As = reinterpret_cast<float*>(sm + L::OFF_AS);
    float* Rs = reinterpret_cast<float*>(sm + L::OFF_RS);

    if (tid == 0) {
        mbar_init(&bar_full[0], 1);
        mbar_init(&bar_full[1], 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_test, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
        if (VAR == kGla) tma_prefetch_desc(&tmg);
    }
    if (warp == 0) tmem_alloc(tmem_slot, L::TMEM_COLS);

    // ---- initial state: thread r owns row r of X (r = value index) -------------
    const int r = tid;
    const bool own = r < DV;
    const size_t ssz = static_cast<size_t>(DK) * DV + (VAR == kNorm ? DK : 0);
    const float* sin = p.state_in ? p.state_in + bh * ssz : nullptr;
    float st[DK];
#pragma unroll
    for (int c = 0; c < DK; ++c) {
        float x = 0.f;
        if (own && sin) x = (VAR == kGdn) ? sin[static_cast<size_t>(r) * DK + c] : sin[static_cast<size_t>(c) * DV + r];
        st[c] = x;
    }
#pragma unroll
    for (int b = 0; b < DK / 32; ++b)
        store_row32_bf16(aSS + (b / 2) * 16384, r, (b % 2) * 4, st + 32 * b);
    if (VAR == kNorm && tid < DK) sZ[tid] = sin ? sin[static_cast<size_t>(DK) * DV + tid] : 0.f;

    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tlane = tmem + (static_cast<uint32_t>(warp * 32) << 16);  // this warp's lanes

    int status_bits = 0;
    bool failed = false;
    if (p.flags & 0x100u) {  // test hook: a wait nothing will satisfy, 1 ms limit
        const bool ok = mbar_wait(bar_test, 0, 1000000ull);
        if (__syncthreads_or(!ok)) { status_bits |= kStatusTestHook; failed = true; }
    }

    auto issue_tma = [&](int cc, int s) {
        uint8_t* stg = sm + s * L::STAGE;
        uint64_t* bar = &bar_full[s];
        mbar_arrive_expect_tx(bar, L::TX_BYTES);
        const int y = cc * C;
#pragma unroll
        for (int a = 0; a < KA; ++a) {
            tma_load_3d(&tmq, bar, stg + a * 16384 + (VAR == kGdn ? 8192 : 0), a * 64, y, bh);
            tma_load_3d(&tmk, bar, stg + a * 16384 + (VAR == kGdn ? 0 : 8192), a * 64, y, bh);
        }
#pragma unroll
        for (int a = 0; a < VA; ++a) tma_load_3d(&tmv, bar, stg + L::QK_BYTES + a * 8192, a * 64, y, bh);
        if (VAR == kGla) tma_load_3d(&tmg, bar, stg + L::QK_BYTES + L::V_BYTES, 0, y, bh);
    };

    if (!failed && tid == 0 && nch > 0) issue_tma(0, 0);

    uint32_t mph = 0;
    // Commit the MMAs thread 0 issued, wait for them, and agree on the outcome.
    auto mma_round = [&]() -> bool {
        if (tid == 0) mma_commit(bar_mma);
        const bool ok = mbar_wait(bar_mma, mph, kWaitLimitNs);
        mph ^= 1u;
        tc_fence_after();
        if (__syncthreads_or(!ok)) { status_bits |= kStatusMmaWait; return false; }
        return true;
    };
    // Publish shared-memory writes to the tensor cores and order TMEM reads
    // before the MMAs issued after this point.
    auto publish = [&]() {
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };

    constexpr uint32_t ID_128x64_KK = idesc_bf16(128, 64, false, false);
    constexpr uint32_t ID_128x64_MK = idesc_bf16(128, 64, true, false);
    constexpr uint32_t ID_128x64_KM_NEG = idesc_bf16(128, 64, false, true, true);
    constexpr uint32_t ID_128xDK_KM = idesc_bf16(128, DK, false, true);
    constexpr uint32_t ID_128xDK_MM = idesc_bf16(128, DK, true, true);
    const uint32_t v_lbo = 8192;  // second 64-row atom of V^T (garbage rows when DV = 64)

    int c = 0;
    for (; c < nch && !failed; ++c) {
        const int s = c & 1;
        const int t0 = c * C;
        const int nvalid = min(C, T - t0);
        const uint32_t aQK = sbase + s * L::STAGE;
        const uint32_t aV = aQK + L::QK_BYTES;
        uint8_t* stg = sm + s * L::STAGE;
        if (tid == 0 && c + 1 < nch) {
            fence_proxy_async_smem();
            issue_tma(c + 1, s ^ 1);
        }
        {
            const bool ok = mbar_wait(&bar_full[s], (c >> 1) & 1, kWaitLimitNs);
            if (__syncthreads_or(!ok)) { status_bits |= kStatusTmaWait; failed = true; break; }
        }

        if constexpr (VAR == kGdn) {
            // ---- per-token gate prefix sums ------------------------------------
            if (tid < 64) {
                float g = 1.f, b = 0.f;
                if (tid < nvalid) {
                    g = p.gate[static_cast<size_t>(bh) * T + t0 + tid];
                    b = p.beta[static_cast<size_t>(bh) * T + t0 + tid];
                }
                float lg = __logf(g);
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, lg, o);
                    if (lane >= o) lg += y;
                }
                sG[tid] = lg;
                sB[tid] = b;
            }
            __syncthreads();
            if (tid >= 32 && tid < 64) sG[tid] += sG[31];
            __syncthreads();
            if (tid < 64) {
                const float G = sG[tid];
                const float gam = __expf(G);
                sGam[tid] = gam;
                sBG[tid] = sB[tid] * gam;
                sKf[tid] = __expf(sG[63] - G);
            }
            // ---- [K;Q] K^T ----------------------------------------------------
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint64_t d = kmaj(aQK + (kk / 4) * 16384 + (kk % 4) * 32);
                    mma_bf16_ss(tmem + L::COL_G, d, d, ID_128x64_KK, kk > 0);
                }
            }
            if (!mma_round()) { failed = true; break; }
            if (warp < 2) {
                // rows 0-63: A_tj = beta_t exp(G_t - G_j) k_t.k_j for j < t
                const int t = tid;
                const float Gt = sG[t], bt = sB[t];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float x[32];
                    tmem_ld32(tlane + L::COL_G + 32 * h, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        float4 o;
                        const int j = 32 * h + 4 * m;
                        o.x = (j + 0 < t) ? bt * __expf(Gt - sG[j + 0]) * x[4 * m + 0] : 0.f;
                        o.y = (j + 1 < t) ? bt * __expf(Gt - sG[j + 1]) * x[4 * m + 1] : 0.f;
                        o.z = (j + 2 < t) ? bt * __expf(Gt - sG[j + 2]) * x[4 * m + 2] : 0.f;
                        o.w = (j + 3 < t) ? bt * __expf(Gt - sG[j + 3]) * x[4 * m + 3] : 0.f;
                        *reinterpret_cast<float4*>(As + t * kAStride + j) = o;
                    }
                }
            } else {
                // rows 64-127: P_tj = exp(G_t - G_j) q_t.k_j for j <= t
                const int t = tid - 64;
                const float Gt = sG[t];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float x[32];
                    tmem_ld32(tlane + L::COL_G + 32 * h, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int j = 32 * h + i;
                        x[i] = (j <= t) ? __expf(Gt - sG[j]) * x[i] : 0.f;
                    }
                    store_row32_bf16(aPS, t, 4 * h, x);
                }
            }
            // Q' = diag(gam) Q in place (block 1); Q is no longer read by the Gram MMA.
#pragma unroll
            for (int i = 0; i < (64 * 8 * KA) / kThreads; ++i) {
                const int e = tid + kThreads * i;
                const int row = e / (8 * KA), a = (e / 8) % KA, pc = e % 8;
                const uint32_t addr = aQK + a * 16384 + 8192 + (row >> 3) * 1024 + (row & 7) * 128 + pc * 16;
                uint4 u = ld_shared_v4(addr);
                const float f = sGam[row];
                float2 x0 = unpack_bf16(u.x), x1 = unpack_bf16(u.y), x2 = unpack_bf16(u.z), x3 = unpack_bf16(u.w);
                st_shared_v4(addr, pack_bf16(x0.x * f, x0.y * f), pack_bf16(x1.x * f, x1.y * f),
                             pack_bf16(x2.x * f, x2.y * f), pack_bf16(x3.x * f, x3.y * f));
            }
            __syncthreads();
            // ---- T = (I + A)^{-1}: diagonal 16x16 blocks, one warp each ---------
            if (lane < 16) {
                const int w0 = 16 * warp, l = lane;
                float x[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float acc = (i == l) ? 1.f : 0.f;
#pragma unroll
                    for (int k = 0; k < i; ++k) acc -= As[(w0 + i) * kAStride + w0 + k] * x[k];
                    x[i] = acc;
                }
                __syncwarp(0x0000ffffu);
#pragma unroll
                for (int i = 0; i < 16; ++i) As[(w0 + i) * kAStride + w0 + l] = x[i];
            }
            __syncthreads();
            // ---- off-diagonal blocks, block row by block row --------------------
            {
                const int i = tid & 15, jg = tid >> 4;
                for (int bi = 1; bi < 4; ++bi) {
                    const int ncol = 16 * bi;
                    const float* arow = As + (16 * bi + i) * kAStride;
                    for (int m = 0; m < 2 * bi; ++m) {
                        const int j = jg + 8 * m;
                        float acc = 0.f;
                        for (int k = j; k < ncol; ++k) acc += arow[k] * As[k * kAStride + j];
                        Rs[i * 48 + j] = acc;
                    }
                    __syncthreads();
                    for (int m = 0; m < 2 * bi; ++m) {
                        const int j = jg + 8 * m;
                        float acc = 0.f;
                        for (int l = 0; l <= i; ++l) acc += arow[16 * bi + l] * Rs[l * 48 + j];
                        As[(16 * bi + i) * kAStride + j] = -acc;
                    }
                    __syncthreads();
                }
            }
            // ---- T diag(beta) and T diag(beta gam) as bf16 MMA operands ---------
            {
                const int t = tid >> 1, half = tid & 1;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int c8 = half * 4 + cc;
                    float y1[8], y2[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = 8 * c8 + e;
                        const float tv = As[t * kAStride + j];
                        y1[e] = tv * sB[j];
                        y2[e] = tv * sBG[j];
                    }
                    st_shared_v4(aTB1 + sw128_off(t, c8), pack_bf16(y1[0], y1[1]), pack_bf16(y1[2], y1[3]),
                                 pack_bf16(y1[4], y1[5]), pack_bf16(y1[6], y1[7]));
                    st_shared_v4(aTB2 + sw128_off(t, c8), pack_bf16(y2[0], y2[1]), pack_bf16(y2[2], y2[3]),
                                 pack_bf16(y2[4], y2[5]), pack_bf16(y2[6], y2[7]));
                }
            }
            publish();
            // ---- W^T = K^T (T diag(beta gam))^T, Ut^T = V^T (T diag(beta))^T ------
            if (tid == 0) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    mma_bf16_ss(tmem + L::COL_W, mnmaj(aQK + kk * 2048, 16384), kmaj(aTB2 + kk * 32),
                                ID_128x64_MK, kk > 0);
                    mma_bf16_ss(tmem + L::COL_U, mnmaj(aV + kk * 2048, v_lbo), kmaj(aTB1 + kk * 32),
                                ID_128x64_MK, kk > 0);
                }
            }
            if (!mma_round()) { failed = true; break; }
            // W^T rows (d_k index) to shared memory as the MN-major operand [dk][t]
            if (r < DK) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float x[32];
                    tmem_ld32(tlane + L::COL_W + 32 * h, x);
                    tmem_ld_wait();
                    store_row32_bf16(aWS, r, 4 * h, x);
                }
            }
            // K' = diag(gam_C / gam) K in place (block 0); its MMAs are done.
#pragma unroll
            for (int i = 0; i < (64 * 8 * KA) / kThreads; ++i) {
                const int e = tid + kThreads * i;
                const int row = e / (8 * KA), a = (e / 8) % KA, pc = e % 8;
                const uint32_t addr = aQK + a * 16384 + (row >> 3) * 1024 + (row & 7) * 128 + pc * 16;
                uint4 u = ld_shared_v4(addr);
                const float f = sKf[row];
                float2 x0 = unpack_bf16(u.x), x1 = unpack_bf16(u.y), x2 = unpack_bf16(u.z), x3 = unpack_bf16(u.w);
                st_shared_v4(addr, pack_bf16(x0.x * f, x0.y * f), pack_bf16(x1.x * f, x1.y * f),
                             pack_bf16(x2.x * f, x2.y * f), pack_bf16(x3.x * f, x3.y * f));
            }
            publish();
            // ---- U^T = Ut^T - X0 W^T ;  O^T = X0 Q'^T ----------------------------
            if (tid == 0) {
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint32_t sa = aSS + (kk / 4) * 16384 + (kk % 4) * 32;
                    mma_bf16_ss(tmem + L::COL_U, kmaj(sa), mnmaj(aWS + kk * 2048, 8192), ID_128x64_KM_NEG, 1);
                    mma_bf16_ss(tmem + L::COL_O, kmaj(sa), kmaj(aQK + 8192 + (kk / 4) * 16384 + (kk % 4) * 32),
                                ID_128x64_KK, kk > 0);
                }
            }
            if (!mma_round()) { failed = true; break; }
            {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float x[32];
                    tmem_ld32(tlane + L::COL_U + 32 * h, x);
                    tmem_ld_wait();
                    store_row32_bf16(aUS, r, 4 * h, x);
                }
            }
            publish();
            // ---- O^T += U^T P^T ;  dX = U^T K' ------------------------------------
            if (tid == 0) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    mma_bf16_ss(tmem + L::COL_O, kmaj(aUS + kk * 32), kmaj(aPS + kk * 32), ID_128x64_KK, 1);
                    mma_bf16_ss(tmem + L::COL_S, kmaj(aUS + kk * 32), mnmaj(aQK + kk * 2048, 16384),
                                ID_128xDK_KM, kk > 0);
                }
            }
            if (!mma_round()) { failed = true; break; }
            if (own) {
                const float gC = sGam[63];
#pragma unroll
                for (int b = 0; b < DK / 32; ++b) {
                    float x[32];
                    tmem_ld32(tlane + L::COL_S + 32 * b, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) st[32 * b + i] = gC * st[32 * b + i] + x[i];
                    store_row32_bf16(aSS + (b / 2) * 16384, r, (b % 2) * 4, st + 32 * b);
                }
                __nv_bfloat16* orow = p.out + (static_cast<size_t>(bh) * T + t0) * DV + r;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float x[32];
                    tmem_ld32(tlane + L::COL_O + 32 * h, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int t = 32 * h + i;
                        if (t < nvalid) orow[static_cast<size_t>(t) * DV] = __float2bfloat16_rn(x[i]);
                    }
                }
            }
            publish();
        } else {
            // ======================= normalized / gated =========================
            if constexpr (VAR == kGla) {
                // Running products Gam_t = prod_{i<=t} gamma_i per channel, in place.
                float* gt = reinterpret_cast<float*>(stg + L::QK_BYTES + L::V_BYTES);
                if (tid < DK) {
                    float G = 1.f;
                    for (int t = 0; t < C; ++t) {
                        const float g = (t < nvalid) ? gt[t * DK + tid] : 1.f;
                        G *= g;
                        gt[t * DK + tid] = G;
                    }
                    sGC[tid] = G;
                }
                __syncthreads();
            }
            // q~ (block 0), k~ (block 1), k^ (gla: its own tile) in place, 8 channels per chunk.
            {
                const float* gt = reinterpret_cast<const float*>(stg + L::QK_BYTES + L::V_BYTES);
#pragma unroll 2
                for (int i = 0; i < (64 * 8 * KA) / kThreads; ++i) {
                    const int e = tid + kThreads * i;
                    const int row = e / (8 * KA), a = (e / 8) % KA, pc = e % 8;
                    const int lc = pc ^ (row & 7);
                    const int c0 = a * 64 + lc * 8;
                    const uint32_t off = (row >> 3) * 1024 + (row & 7) * 128 + pc * 16;
                    const uint32_t qa = aQK + a * 16384 + off, ka = qa + 8192;
                    const uint4 uq = ld_shared_v4(qa), uk = ld_shared_v4(ka);
                    float q8[8], k8[8];
                    {
                        float2 t0v = unpack_bf16(uq.x), t1v = unpack_bf16(uq.y), t2v = unpack_bf16(uq.z), t3v = unpack_bf16(uq.w);
                        q8[0] = t0v.x; q8[1] = t0v.y; q8[2] = t1v.x; q8[3] = t1v.y;
                        q8[4] = t2v.x; q8[5] = t2v.y; q8[6] = t3v.x; q8[7] = t3v.y;
                        float2 u0 = unpack_bf16(uk.x), u1 = unpack_bf16(uk.y), u2 = unpack_bf16(uk.z), u3 = unpack_bf16(uk.w);
                        k8[0] = u0.x; k8[1] = u0.y; k8[2] = u1.x; k8[3] = u1.y;
                        k8[4] = u2.x; k8[5] = u2.y; k8[6] = u3.x; k8[7] = u3.y;
                    }
                    const bool valid = row < nvalid;
                    float kh[8];
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        float qq = phi_on ? elu1(q8[m]) : q8[m];
                        float kv = valid ? (phi_on ? elu1(k8[m]) : k8[m]) : 0.f;
                        if constexpr (VAR == kGla) {
                            const float G = gt[row * DK + c0 + m];
                            const float inv = __frcp_rn(G);
                            qq *= G;
                            kh[m] = kv * sGC[c0 + m] * inv;
                            kv *= inv;
                        }
                        q8[m] = qq;
                        k8[m] = kv;
                    }
                    st_shared_v4(qa, pack_bf16(q8[0], q8[1]), pack_bf16(q8[2], q8[3]), pack_bf16(q8[4], q8[5]),
                                 pack_bf16(q8[6], q8[7]));
                    st_shared_v4(ka, pack_bf16(k8[0], k8[1]), pack_bf16(k8[2], k8[3]), pack_bf16(k8[4], k8[5]),
                                 pack_bf16(k8[6], k8[7]));
                    if constexpr (VAR == kGla)
                        st_shared_v4(aKH + a * 8192 + off, pack_bf16(kh[0], kh[1]), pack_bf16(kh[2], kh[3]),
                                     pack_bf16(kh[4], kh[5]), pack_bf16(kh[6], kh[7]));
                }
            }
            publish();
            if constexpr (VAR == kNorm) {
                // den_t starts as q~_t . z_0 (z_0 = normalizer before this chunk).
                if (tid < 64) {
                    float d = 0.f;
#pragma unroll
                    for (int a = 0; a < KA; ++a)
#pragma unroll
                        for (int pc = 0; pc < 8; ++pc) {
                            const uint4 u = ld_shared_v4(aQK + a * 16384 + sw128_off(tid, pc));
                            const int c0 = a * 64 + pc * 8;
                            float2 x0 = unpack_bf16(u.x), x1 = unpack_bf16(u.y), x2 = unpack_bf16(u.z), x3 = unpack_bf16(u.w);
                            d += x0.x * sZ[c0 + 0] + x0.y * sZ[c0 + 1] + x1.x * sZ[c0 + 2] + x1.y * sZ[c0 + 3] +
                                 x2.x * sZ[c0 + 4] + x2.y * sZ[c0 + 5] + x3.x * sZ[c0 + 6] + x3.y * sZ[c0 + 7];
                        }
                    sDen[tid] = d;
                }
            }
            // ---- P = Q~ K~^T ;  O^T = X0 Q~^T ;  dX = V^T K^ ---------------------
            if (tid == 0) {
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint32_t qa = aQK + (kk / 4) * 16384 + (kk % 4) * 32;
                    mma_bf16_ss(tmem + L::COL_G, kmaj(qa), kmaj(qa + 8192), ID_128x64_KK, kk > 0);
                    mma_bf16_ss(tmem + L::COL_O, kmaj(aSS + (kk / 4) * 16384 + (kk % 4) * 32), kmaj(qa),
                                ID_128x64_KK, kk > 0);
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t bdesc = (VAR == kGla) ? mnmaj(aKH + kk * 2048, 8192)
                                                         : mnmaj(aQK + 8192 + kk * 2048, 16384);
                    mma_bf16_ss(tmem + L::COL_S, mnmaj(aV + kk * 2048, v_lbo), bdesc, ID_128xDK_MM, kk > 0);
                }
            }
            if (!mma_round()) { failed = true; break; }
            if (warp < 2) {
                // masked scores of rows t = 0..63 -> bf16 P; norm adds the row sums to den.
                const int t = tid;
                float rs = 0.f;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float x[32];
                    tmem_ld32(tlane + L::COL_G + 32 * h, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        x[i] = (32 * h + i <= t) ? x[i] : 0.f;
                        rs += x[i];
                    }
                    store_row32_bf16(aPS, t, 4 * h, x);
                }
                if (VAR == kNorm) sDen[t] += rs;
            }
            if (own) {
#pragma unroll
                for (int b = 0; b < DK / 32; ++b) {
                    float x[32];
                    tmem_ld32(tlane + L::COL_S + 32 * b, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float dec = (VAR == kGla) ? sGC[32 * b + i] : 1.f;
                        st[32 * b + i] = dec * st[32 * b + i] + x[i];
                    }
                    store_row32_bf16(aSS + (b / 2) * 16384, r, (b % 2) * 4, st + 32 * b);
                }
            }
            if (VAR == kNorm && tid < DK) {
                // z += sum_j phi(k_j) over this chunk's (valid) keys.
                const int a = tid / 64, lc = (tid % 64) / 8, e = tid % 8;
                float zs = 0.f;
                for (int j = 0; j < C; ++j) {
                    const uint32_t addr = aQK + a * 16384 + 8192 + sw128_off(j, lc) + 2 * e;
                    unsigned short hbits;
                    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(hbits) : "r"(addr));
                    zs += __bfloat162float(__ushort_as_bfloat16(hbits));
                }
                sZ[tid] += zs;
            }
            publish();
            // ---- O^T += V^T P^T ----------------------------------------------------
            if (tid == 0) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ss(tmem + L::COL_O, mnmaj(aV + kk * 2048, v_lbo), kmaj(aPS + kk * 32), ID_128x64_MK, 1);
            }
            if (!mma_round()) { failed = true; break; }
            if (own) {
                __nv_bfloat16* orow = p.out + (static_cast<size_t>(bh) * T + t0) * DV + r;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float x[32];
                    tmem_ld32(tlane + L::COL_O + 32 * h, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int t = 32 * h + i;
                        float o = x[i];
                        if (VAR == kNorm) o = o / sDen[t];
                        if (t < nvalid) orow[static_cast<size_t>(t) * DV] = __float2bfloat16_rn(o);
                    }
                }
            }
            if (VAR == kNorm && p.den_out && tid < nvalid)
                p.den_out[static_cast<size_t>(bh) * T + t0 + tid] = sDen[tid];
            publish();
        }
    }

    // ---- on failure, let an in-flight prefetch land before the CTA exits -----
    if (failed && c + 1 < nch) {
        const int s2 = (c + 1) & 1;
        mbar_wait(&bar_full[s2], ((c + 1) >> 1) & 1, 100000000ull);
    }

    // ---- final state ------------------------------------------------------------
    if (!failed && p.state_out) {
        float* so = p.state_out + bh * ssz;
        if (own) {
#pragma unroll
            for (int cc = 0; cc < DK; ++cc) {
                if (VAR == kGdn) so[static_cast<size_t>(r) * DK + cc] = st[cc];
                else so[static_cast<size_t>(cc) * DV + r] = st[cc];
            }
        }
        if (VAR == kNorm && tid < DK) so[static_cast<size_t>(DK) * DV + tid] = sZ[tid];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
    if (status_bits && tid == 0) atomicOr(p.status, status_bits);
}

}  // namespace chunk
}  // namespace la
