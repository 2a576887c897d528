// Chunkwise prefill on the tcgen05 tensor cores (sm_103a): the normalized
// variant's sequential chunk kernel and its segment summaries (the gated
// variants run on the prep/chain kernel of prefill_gdn.cu, which shares the
// helpers below). VAR is kNorm.
//
// One CTA per (b,h) sequence-head walks its sequence in chunks of C = 64
// tokens. TMA stages the q/k/v tiles of chunk c+1 while chunk c is computed. The dense products
// run as tcgen05 bf16 MMAs with fp32 accumulators in tensor memory. The
// fp32 state lives in registers and is re-published each chunk as a bf16 MMA
// operand in shared memory. Outputs leave through a shared-memory tile and a
// TMA store.
//
// Inside the kernel the state is held as X = S^T [d_v rows][d_k cols] (S is
// d_k x d_v for this variant). With that orientation the state products have M = 128 (value rows, padded when
// d_v = 64); the output products put the 64 tokens on M (rows 64-127 of
// those accumulators are unused) so each thread writes whole output rows. The 256 threads pair up on the 128
// tensor-memory lanes: thread (r, h) owns row r and the h-th half of the
// columns of whatever it reads (warp w serves lanes 32*(w%4).., h = w/4).
//
// Chunk algebra ("Linear attention and Hyena" 11.2, L = causal mask
// including the diagonal, q~ = phi(q), k~ = phi(k)):
//    O    = Q~ X_0^T + (L o Q~ K~^T) V
//    X    = X_0 + V^T K~
//    den_t = q~_t . z_0 + sum_{j<=t} q~_t . k~_j, o_t = num_t / den_t.
//
// Tail chunks (T not a multiple of 64): TMA zero-fills rows past the end.
// phi(0) = 1, so padded keys are zeroed explicitly, which makes padded
// tokens leave the state untouched; the TMA store clips rows past the end.
#pragma once

#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace la {
namespace chunk {

constexpr int C = 64;          // tokens per chunk
constexpr int kThreads = 256;  // two threads per tensor-memory lane / state row
constexpr int kAStride = 68;   // fp32 row stride of the 64x64 solve matrix

struct Params {
    const float* state_in;  // may be NULL
    float* state_out;       // may be NULL
    float* den_out;         // norm, may be NULL
    int T;
    int nchunks;
    unsigned flags;
    int* status;
    // Segments (norm / gla): the chunks of each sequence are split into nseg
    // runs of seg_len chunks, each run on its own CTA. The chunks before the
    // last segment are also cut into nsub summary runs of sub_len chunks
    // (sub_len divides seg_len). scratch holds, for every (b,h) and every
    // summary run, the state that run produces from a zero start: X [DV][DK]
    // followed by DK floats (its sum of phi(k)).
    int nseg;
    int seg_len;
    int nsub;
    int sub_len;
    float* scratch;
};

template <int VAR, int DK, int DV>
struct Layout {
    static constexpr int KA = DK / 64;  // 64-column atoms along d_k
    static constexpr int VA = DV / 64;
    // q/k tile pair: per k-atom, rows 0-63 hold block 0 and rows 64-127 block 1.
    static constexpr uint32_t QK_BYTES = KA * 16384;
    static constexpr uint32_t V_BYTES = VA * 8192;
    static constexpr uint32_t STAGE = QK_BYTES + V_BYTES;
    static constexpr uint32_t TX_BYTES = 2 * KA * 8192 + V_BYTES;
    // bf16 P [64 t][64 j]. The P V product reads it as a 128-row A operand,
    // so the 8 KB after it (rows 64-127, whose results are unused) must be
    // shared memory of this CTA: the state tile follows.
    static constexpr uint32_t OFF_PS = 2 * STAGE;
    static constexpr uint32_t OFF_SS = OFF_PS + 8192;             // bf16 state [128 rows][DK]
    static constexpr uint32_t OFF_OT = OFF_SS + KA * 16384;       // output tile [64 t][DV]
    static constexpr uint32_t OT_BYTES = VA * 8192;
    static constexpr uint32_t OFF_MISC = OFF_OT + OT_BYTES;
    static constexpr uint32_t MISC_BYTES = 3 * 128 * 4;            // den, z, this chunk's sum of phi(k)
    static constexpr uint32_t OFF_BAR = OFF_MISC + MISC_BYTES;
    static constexpr uint32_t BYTES = OFF_BAR + 64;
    static constexpr uint32_t SMEM_ALLOC = BYTES + 1024;  // slack to align the base to 1024
    // TMEM column map
    static constexpr uint32_t COL_G = 0;                 // P = Q~ K~^T [t rows][64 j]
    static constexpr uint32_t COL_O = 64;                // O [t rows][DV]
    static constexpr uint32_t COL_S = COL_O + DV;        // Delta X [dv rows][DK]
    static constexpr uint32_t TMEM_COLS = (COL_S + DK <= 256) ? 256 : 512;
    static_assert(STAGE % 1024 == 0, "stage alignment");
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
};

__device__ __forceinline__ uint64_t kmaj(uint32_t addr) { return sdesc_sw128(addr, 16, 1024); }
__device__ __forceinline__ uint64_t mnmaj(uint32_t addr, uint32_t lbo) { return sdesc_sw128(addr, lbo, 1024); }

// elu(x) + 1 with alpha = 1; exp via ex2 (x <= 0 here, so no overflow).
__device__ __forceinline__ float elu1(float x) { return x > 0.f ? x + 1.f : ex2(x * 1.4426950408889634f); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_shared_f4(uint32_t addr, float4 v) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w) : "memory");
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_shared_b16(uint32_t addr, float x) {
    const __nv_bfloat16 b = __float2bfloat16_rn(x);
    const unsigned short u = *reinterpret_cast<const unsigned short*>(&b);
    asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(u) : "memory");
}
__device__ __forceinline__ float ld_shared_bf16(uint32_t addr) {
    unsigned short h;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(addr) : "memory");
    return __bfloat162float(__ushort_as_bfloat16(h));
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

// Scale one 16-byte bf16 chunk in place by f.
__device__ __forceinline__ void scale_chunk(uint32_t addr, float f) {
    uint4 u = ld_shared_v4(addr);
    const float2 x0 = unpack_bf16(u.x), x1 = unpack_bf16(u.y), x2 = unpack_bf16(u.z), x3 = unpack_bf16(u.w);
    st_shared_v4(addr, pack_bf16(x0.x * f, x0.y * f), pack_bf16(x1.x * f, x1.y * f), pack_bf16(x2.x * f, x2.y * f),
                 pack_bf16(x3.x * f, x3.y * f));
}

template <int VAR, int DK, int DV>
__global__ void __launch_bounds__(kThreads, 1)
chunk_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
             const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo, const Params p) {
    static_assert(VAR == kNorm, "the gated variants have their own kernel");
    using L = Layout<VAR, DK, DV>;
    constexpr int KA = L::KA, VA = L::VA;
    constexpr int DKH = DK / 2;   // state columns per thread
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (sbase - raw);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = 32 * (warp & 3) + lane;   // tensor-memory lane / state row
    const int hh = warp >> 2;               // column half
    const int bh = blockIdx.x / p.nseg;
    const int seg = blockIdx.x % p.nseg;
    const int T = p.T, nch = p.nchunks;
    const int c_begin = seg * p.seg_len;
    const int nloc = min(nch, c_begin + p.seg_len) - c_begin;

    float* sDen = reinterpret_cast<float*>(sm + L::OFF_MISC);   // denominators of the chunk
    float* sZ = sDen + 128;    // z (128)
    float* sDz = sZ + 128;     // this chunk's sum of phi(k) (128)
    uint64_t* bar_full = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
    uint64_t* bar_mma = bar_full + 2;
    uint64_t* bar_test = bar_full + 3;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_full + 4);

    const uint32_t aSS = sbase + L::OFF_SS, aPS = sbase + L::OFF_PS;

    if (tid == 0) {
        mbar_init(&bar_full[0], 1);
        mbar_init(&bar_full[1], 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_test, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
        tma_prefetch_desc(&tmo);
    }
    if (warp == 0) tmem_alloc(tmem_slot, L::TMEM_COLS);

    // ---- initial state: thread (r, hh) owns X[r][hh*DK/2 .. +DK/2) ----------------
    const bool own = r < DV;
    const size_t ssz = static_cast<size_t>(DK) * DV + DK;
    const float* sin = p.state_in ? p.state_in + bh * ssz : nullptr;
    float st[DKH];
#pragma unroll
    for (int i = 0; i < DKH; ++i) {
        const int c = hh * DKH + i;
        float x = 0.f;
        if (own && sin) x = sin[static_cast<size_t>(c) * DV + r];
        st[i] = x;
    }
    // Later segments start from the states of the summary runs before them:
    // X = X + X_u.
    const size_t sblk = static_cast<size_t>(DV) * DK + DK;
    const float* sc0 = p.scratch + static_cast<size_t>(bh) * p.nsub * sblk;
    const int nprev = seg * (p.seg_len / p.sub_len);
    if (own) {
        for (int s2 = 0; s2 < nprev; ++s2) {
            const float* xs = sc0 + s2 * sblk + static_cast<size_t>(r) * DK + hh * DKH;
#pragma unroll
            for (int i = 0; i < DKH; i += 4) {
                const float4 x4 = *reinterpret_cast<const float4*>(xs + i);
                st[i + 0] += x4.x;
                st[i + 1] += x4.y;
                st[i + 2] += x4.z;
                st[i + 3] += x4.w;
            }
        }
    }
    auto publish_state = [&]() {   // bf16 copy of this thread's state columns
#pragma unroll
        for (int b = 0; b < DKH / 32; ++b) {
            const int cb = hh * DKH + 32 * b;
            store_row32_bf16(aSS + (cb / 64) * 16384, r, (cb % 64) / 8, st + 32 * b);
        }
    };
    publish_state();
    if (tid < DK) {
        float z = sin ? sin[static_cast<size_t>(DK) * DV + tid] : 0.f;
        for (int s2 = 0; s2 < nprev; ++s2) z += sc0[s2 * sblk + static_cast<size_t>(DV) * DK + tid];
        sZ[tid] = z;
    }

    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);  // this warp's lanes

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
            tma_load_3d(&tmq, bar, stg + a * 16384, a * 64, y, bh);
            tma_load_3d(&tmk, bar, stg + a * 16384 + 8192, a * 64, y, bh);
        }
#pragma unroll
        for (int a = 0; a < VA; ++a) tma_load_3d(&tmv, bar, stg + L::QK_BYTES + a * 8192, a * 64, y, bh);
    };

    if (!failed && tid == 0 && nloc > 0) issue_tma(c_begin, 0);

    uint32_t mph = 0;
    // Wait for the MMAs thread 0 committed, and agree on the outcome.
    auto mma_wait = [&]() -> bool {
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
    // Output epilogue: rows t < 64 of O (thread (t, hh) holds columns
    // [hh*DV/2, (hh+1)*DV/2)), scaled by 1/den, into the swizzled
    // [64 t][DV] tile at `ot`, then one TMA store per 64-column atom.
    auto store_output = [&](uint32_t ot, int t0) {
        if ((warp & 3) < 2) {
            const int t = r;
            const float sc = __fdividef(1.f, sDen[t]);
#pragma unroll
            for (int b = 0; b < DV / 64; ++b) {
                const int cb = hh * (DV / 2) + 32 * b;
                float x[32];
                tmem_ld32(tlane + L::COL_O + cb, x);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] *= sc;
                store_row32_bf16(ot + (cb / 64) * 8192, t, (cb % 64) / 8, x);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int a = 0; a < VA; ++a) tma_store_3d(&tmo, sm + (ot - sbase) + a * 8192, a * 64, t0, bh);
            bulk_commit();
        }
    };

    constexpr uint32_t ID_128x64_KK = idesc_bf16(128, 64, false, false);
    constexpr uint32_t ID_128xDK_MM = idesc_bf16(128, DK, true, true);
    constexpr uint32_t ID_128xDV_KK = idesc_bf16(128, DV, false, false);
    constexpr uint32_t ID_128xDV_KM = idesc_bf16(128, DV, false, true);
    const uint32_t v_lbo = 8192;  // second 64-row atom of V^T (garbage rows when DV = 64)

    int it = 0;
    for (; it < nloc && !failed; ++it) {
        const int c = c_begin + it;
        const int s = it & 1;
        const int t0 = c * C;
        const int nvalid = min(C, T - t0);
        const uint32_t aQK = sbase + s * L::STAGE;
        const uint32_t aV = aQK + L::QK_BYTES;
        uint8_t* stg = sm + s * L::STAGE;
        if (tid == 0 && it + 1 < nloc) {
            fence_proxy_async_smem();
            issue_tma(c + 1, s ^ 1);
        }
        {
            const bool ok = mbar_wait(&bar_full[s], (it >> 1) & 1, kWaitLimitNs);
            if (__syncthreads_or(!ok)) { status_bits |= kStatusTmaWait; failed = true; break; }
            tc_fence_after();
        }

        if (tid < DK) sDz[tid] = 0.f;
        // q~ (block 0), k~ (block 1) in place, 8 channels per chunk.
        {
#pragma unroll
            for (int i = 0; i < (64 * 8 * KA) / kThreads; ++i) {
                const int e = tid + kThreads * i;
                const int row = e / (8 * KA), a = (e / 8) % KA, pc = e % 8;
                const uint32_t off = (row >> 3) * 1024 + (row & 7) * 128 + pc * 16;
                const uint32_t qa = aQK + a * 16384 + off, ka = qa + 8192;
                const uint4 uq = ld_shared_v4(qa), uk = ld_shared_v4(ka);
                float q8[8], k8[8];
                {
                    const float2 a0 = unpack_bf16(uq.x), a1 = unpack_bf16(uq.y), a2 = unpack_bf16(uq.z), a3 = unpack_bf16(uq.w);
                    q8[0] = a0.x; q8[1] = a0.y; q8[2] = a1.x; q8[3] = a1.y;
                    q8[4] = a2.x; q8[5] = a2.y; q8[6] = a3.x; q8[7] = a3.y;
                    const float2 b0 = unpack_bf16(uk.x), b1 = unpack_bf16(uk.y), b2 = unpack_bf16(uk.z), b3 = unpack_bf16(uk.w);
                    k8[0] = b0.x; k8[1] = b0.y; k8[2] = b1.x; k8[3] = b1.y;
                    k8[4] = b2.x; k8[5] = b2.y; k8[6] = b3.x; k8[7] = b3.y;
                }
                const bool valid = row < nvalid;
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    q8[m] = elu1(q8[m]);
                    k8[m] = valid ? elu1(k8[m]) : 0.f;
                }
                st_shared_v4(qa, pack_bf16(q8[0], q8[1]), pack_bf16(q8[2], q8[3]), pack_bf16(q8[4], q8[5]),
                             pack_bf16(q8[6], q8[7]));
                st_shared_v4(ka, pack_bf16(k8[0], k8[1]), pack_bf16(k8[2], k8[3]), pack_bf16(k8[4], k8[5]),
                             pack_bf16(k8[6], k8[7]));
            }
        }
        publish();
        // ---- P = Q~ K~^T ;  O = Q~ X0^T ;  dX = V^T K~ -----------------------
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < DK / 16; ++kk) {
                const uint32_t qa = aQK + (kk / 4) * 16384 + (kk % 4) * 32;
                mma_bf16_ss(tmem + L::COL_G, kmaj(qa), kmaj(qa + 8192), ID_128x64_KK, kk > 0);
                mma_bf16_ss(tmem + L::COL_O, kmaj(qa), kmaj(aSS + (kk / 4) * 16384 + (kk % 4) * 32),
                            ID_128xDV_KK, kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + L::COL_S, mnmaj(aV + kk * 2048, v_lbo), mnmaj(aQK + 8192 + kk * 2048, 16384),
                            ID_128xDK_MM, kk > 0);
            mma_commit(bar_mma);
        }
        {
            // While the MMAs run: den_t = q~_t . z_0, and this chunk's sum of phi(k).
            {
                const int t = tid >> 2, q4 = tid & 3;
                float d = 0.f;
#pragma unroll
                for (int m = 0; m < KA * 2; ++m) {
                    const int cq = q4 * (KA * 2) + m;       // 8-channel group
                    const int a = cq / 8, lc = cq % 8;
                    const uint4 u = ld_shared_v4(aQK + a * 16384 + sw128_off(t, lc));
                    const float2 x0 = unpack_bf16(u.x), x1 = unpack_bf16(u.y), x2 = unpack_bf16(u.z), x3 = unpack_bf16(u.w);
                    const float* z = sZ + 8 * cq;
                    d += x0.x * z[0] + x0.y * z[1] + x1.x * z[2] + x1.y * z[3] + x2.x * z[4] + x2.y * z[5] +
                         x3.x * z[6] + x3.y * z[7];
                }
                d += __shfl_xor_sync(0xffffffffu, d, 1);
                d += __shfl_xor_sync(0xffffffffu, d, 2);
                if (q4 == 0) sDen[t] = d;
            }
            {
                constexpr int NP = kThreads / DK, RP = C / NP;
                const int ch = tid % DK, part = tid / DK;
                const uint32_t base = aQK + (ch / 64) * 16384 + 8192 + (ch % 8) * 2;
                const int lc = (ch % 64) / 8;
                float zs = 0.f;
#pragma unroll 8
                for (int j = part * RP; j < (part + 1) * RP; ++j) zs += ld_shared_bf16(base + sw128_off(j, lc));
                atomicAdd(&sDz[ch], zs);
            }
        }
        if (!mma_wait()) { failed = true; break; }
        if ((warp & 3) < 2) {
            // masked scores of rows t = 0..63 -> bf16 P; the row sums add to den.
            const int t = r;
            float x[32];
            tmem_ld32(tlane + L::COL_G + 32 * hh, x);
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
        if (own) {
#pragma unroll
            for (int b = 0; b < DKH / 32; ++b) {
                float x[32];
                tmem_ld32(tlane + L::COL_S + hh * DKH + 32 * b, x);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) st[32 * b + i] += x[i];
            }
            publish_state();
        }
        if (tid < DK) sZ[tid] += sDz[tid];
        publish();
        // ---- O += P V ----------------------------------------------------------
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + L::COL_O, kmaj(aPS + kk * 32), mnmaj(aV + kk * 2048, v_lbo), ID_128xDV_KM, 1);
            mma_commit(bar_mma);
            bulk_wait_read_all();  // the previous output store read the tile
        }
        if (p.den_out && tid < nvalid)
            p.den_out[static_cast<size_t>(bh) * T + t0 + tid] = sDen[tid];
        if (!mma_wait()) { failed = true; break; }
        store_output(sbase + L::OFF_OT, t0);
    }

    // ---- on failure, let an in-flight prefetch land before the CTA exits -----
    if (failed && it + 1 < nloc) {
        const int s2 = (it + 1) & 1;
        mbar_wait(&bar_full[s2], ((it + 1) >> 1) & 1, 100000000ull);
    }

    // ---- final state ------------------------------------------------------------
    if (!failed && p.state_out && seg == p.nseg - 1) {
        float* so = p.state_out + bh * ssz;
        if (own) {
#pragma unroll
            for (int i = 0; i < DKH; ++i) {
                const int cc = hh * DKH + i;
                so[static_cast<size_t>(cc) * DV + r] = st[i];
            }
        }
        if (tid < DK) so[static_cast<size_t>(DK) * DV + tid] = sZ[tid];
    }
    if (tid == 0) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
    if (status_bits && tid == 0) atomicOr(p.status, status_bits);
}


// ---------------------------------------------------------------------------
// Segment summaries of the normalized variant.
//
// For summary run u of sequence-head bh (the runs tile every segment but the
// last), compute the state the run's chunks produce from a zero state,
// X_s = sum_c V_c^T phi(K_c), and its sum of phi(k), and store them in
// p.scratch. Every chunk accumulates into one TMEM accumulator.
// ---------------------------------------------------------------------------
template <int VAR, int DK, int DV>
struct SLayout {
    static constexpr int KA = DK / 64;
    static constexpr int VA = DV / 64;
    static constexpr uint32_t K_BYTES = KA * 8192;
    static constexpr uint32_t V_BYTES = VA * 8192;
    static constexpr uint32_t STAGE = K_BYTES + V_BYTES;
    static constexpr uint32_t TX_BYTES = K_BYTES + V_BYTES;
    static constexpr uint32_t OFF_KH = 2 * STAGE;                  // phi(k) [64 j][DK]
    static constexpr uint32_t OFF_MISC = OFF_KH + KA * 8192;
    static constexpr uint32_t MISC_BYTES = 128 * 4;                // z
    static constexpr uint32_t OFF_BAR = OFF_MISC + MISC_BYTES;
    static constexpr uint32_t SMEM_ALLOC = OFF_BAR + 64 + 1024;
    static constexpr uint32_t TMEM_COLS = DK <= 64 ? 64 : 128;
    static_assert(STAGE % 1024 == 0, "stage alignment");
};

template <int VAR, int DK, int DV>
__global__ void __launch_bounds__(kThreads, 1)
summary_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, const Params p) {
    static_assert(VAR == kNorm, "the gated variants have their own kernel");
    using L = SLayout<VAR, DK, DV>;
    constexpr int KA = L::KA, VA = L::VA, DKH = DK / 2;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (sbase - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = 32 * (warp & 3) + lane, hh = warp >> 2;
    const int nsum = p.nsub;
    const int bh = blockIdx.x / nsum, seg = blockIdx.x % nsum;
    const int T = p.T;
    const int c_begin = seg * p.sub_len;
    const int nloc = p.sub_len;   // runs lie before the last segment, so they are full

    float* sZ = reinterpret_cast<float*>(sm + L::OFF_MISC);
    uint64_t* bar_full = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
    uint64_t* bar_mma = bar_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_full + 3);
    const uint32_t aKH = sbase + L::OFF_KH;

    if (tid == 0) {
        mbar_init(&bar_full[0], 1);
        mbar_init(&bar_full[1], 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_slot, L::TMEM_COLS);
    if (tid < DK) sZ[tid] = 0.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);

    auto issue_tma = [&](int cc, int s) {
        uint8_t* stg = sm + s * L::STAGE;
        mbar_arrive_expect_tx(&bar_full[s], L::TX_BYTES);
#pragma unroll
        for (int a = 0; a < KA; ++a) tma_load_3d(&tmk, &bar_full[s], stg + a * 8192, a * 64, cc * C, bh);
#pragma unroll
        for (int a = 0; a < VA; ++a) tma_load_3d(&tmv, &bar_full[s], stg + L::K_BYTES + a * 8192, a * 64, cc * C, bh);
    };
    if (tid == 0) issue_tma(c_begin + nloc - 1, 0);

    constexpr uint32_t ID_MM = idesc_bf16(128, DK, true, true);
    int status_bits = 0;
    bool failed = false;
    uint32_t mph = 0;
    int it = 0;
    for (; it < nloc; ++it) {
        const int c = c_begin + nloc - 1 - it;     // last chunk first
        const int s = it & 1;
        const int t0 = c * C;
        const int nvalid = min(C, T - t0);
        const uint32_t aK = sbase + s * L::STAGE, aV = aK + L::K_BYTES;
        if (tid == 0 && it + 1 < nloc) {
            fence_proxy_async_smem();
            issue_tma(c - 1, s ^ 1);   // stage s^1's MMA finished in the previous iteration
        }
        {
            const bool ok = mbar_wait(&bar_full[s], (it >> 1) & 1, kWaitLimitNs);
            if (__syncthreads_or(!ok)) { status_bits |= kStatusTmaWait; failed = true; break; }
        }
        // phi(k_j); padded rows 0.
#pragma unroll
        for (int i = 0; i < (64 * 8 * KA) / kThreads; ++i) {
            const int e = tid + kThreads * i;
            const int row = e / (8 * KA), a = (e / 8) % KA, pc = e % 8;
            const uint32_t off = a * 8192 + (row >> 3) * 1024 + (row & 7) * 128 + pc * 16;
            const uint4 uk = ld_shared_v4(aK + off);
            const float2 b0 = unpack_bf16(uk.x), b1 = unpack_bf16(uk.y), b2 = unpack_bf16(uk.z), b3 = unpack_bf16(uk.w);
            float k8[8] = {b0.x, b0.y, b1.x, b1.y, b2.x, b2.y, b3.x, b3.y};
            const bool valid = row < nvalid;
#pragma unroll
            for (int m = 0; m < 8; ++m) k8[m] = valid ? elu1(k8[m]) : 0.f;
            st_shared_v4(aKH + off, pack_bf16(k8[0], k8[1]), pack_bf16(k8[2], k8[3]), pack_bf16(k8[4], k8[5]),
                         pack_bf16(k8[6], k8[7]));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem, mnmaj(aV + kk * 2048, 8192), mnmaj(aKH + kk * 2048, 8192), ID_MM, (it > 0 || kk > 0));
            mma_commit(bar_mma);
        }
        {
            // sum of phi(k) over this chunk: each thread sums a strip of rows of one channel
            constexpr int NP = kThreads / DK, RP = C / NP;
            const int ch = tid % DK, part = tid / DK;
            const uint32_t base = aKH + (ch / 64) * 8192 + (ch % 8) * 2;
            const int lc = (ch % 64) / 8;
            float zs = 0.f;
#pragma unroll 8
            for (int j = part * RP; j < (part + 1) * RP; ++j) zs += ld_shared_bf16(base + sw128_off(j, lc));
            atomicAdd(&sZ[ch], zs);
        }
        {
            const bool ok = mbar_wait(bar_mma, mph, kWaitLimitNs);
            mph ^= 1u;
            tc_fence_after();
            if (__syncthreads_or(!ok)) { status_bits |= kStatusMmaWait; failed = true; break; }
        }
        __syncthreads();
    }
    if (failed && it + 1 < nloc) mbar_wait(&bar_full[(it + 1) & 1], ((it + 1) >> 1) & 1, 100000000ull);
    if (!failed) {
        const size_t sblk = static_cast<size_t>(DV) * DK + DK;
        float* out = p.scratch + (static_cast<size_t>(bh) * nsum + seg) * sblk;
        if (r < DV) {
#pragma unroll
            for (int b = 0; b < DKH / 32; ++b) {
                float x[32];
                tmem_ld32(tlane + hh * DKH + 32 * b, x);
                tmem_ld_wait();
                float* o = out + static_cast<size_t>(r) * DK + hh * DKH + 32 * b;
#pragma unroll
                for (int i = 0; i < 32; i += 4) *reinterpret_cast<float4*>(o + i) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
            }
        }
        if (tid < DK) out[static_cast<size_t>(DV) * DK + tid] = sZ[tid];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
    if (status_bits && tid == 0) atomicOr(p.status, status_bits);
}

}  // namespace chunk
}  // namespace la
