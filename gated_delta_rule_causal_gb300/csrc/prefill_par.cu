// Chunkwise prefill of the normalized variant (with or without a fixed decay
// per sequence-head) in three fully parallel phases, for problems whose
// per-chunk states fit in L2.
//
// The state recurrence does not depend on the outputs. With X = S^T
// [d_v][d_k] and, per chunk c of C = 64 tokens ("Linear attention and
// Hyena" §11.2):
//    dX_c = V_c^T phi(K_c),   X_c = D_c X_{c-1} + dX_c   (D_c = gamma^nvalid, 1 undecayed)
// so the work splits into
//  1. summary (per (head, chunk)): dX_c and the chunk's sum of phi(k);
//  2. scan (one thread per 2 state elements): the state entering every
//     chunk, stored as the bf16 operand tile the output phase loads as is,
//     the normalizer entering every chunk and the final state;
//  3. output (per (head, chunk)): O = Q~ X_{c-1}^T + (L o Q~ K~^T) V
//     with q~ = phi(q), k~ = phi(k), row t divided by
//     den_t = q~_t . z_{c-1} + sum_{j<=t} q~_t . k~_j.
// Phases 1 and 3 are independent over all (head, chunk) units, so the GPU
// fills even when B*H is small. They run as persistent CTAs (a few per SM,
// each looping over units with the next unit's tiles in flight) because
// dispatching one short CTA per unit costs more than the work. The three
// kernels are chained with programmatic dependent launch, so each one's
// dispatch and prologue (barriers, tensor-map prefetch) overlap the previous
// one's tail; tensor memory is allocated only after the wait on the previous
// kernel. The intermediates
// (fp32 dX, bf16 states) stay in L2 between the phases.
#include "prefill.h"
#include "prefill_impl.cuh"
#include "launch.cuh"

namespace la {
namespace par {

using chunk::C;
using chunk::elu1;
using chunk::kmaj;
using chunk::ld_shared_bf16;
using chunk::ld_shared_v4;
using chunk::mnmaj;
using chunk::st_shared_v4;
using chunk::store_row32_bf16;

struct Params {
    const float* state_in;  // S [BH][DK][DV] + z [BH][DK], or NULL
    float* state_out;       // same layout, or NULL
    float* den_out;         // [BH][T], or NULL
    float* dx;              // [BH][nch][DV][DK] fp32 chunk summaries
    float* dd;              // [BH][nch][DK]: the chunk's sum of phi(k)
    uint8_t* xs;            // [BH][nch] state entering the chunk, bf16 MMA tile (DK*DV*2 bytes)
    float* zs;              // [BH][nch][DK] normalizer entering the chunk
    uint8_t* kh;            // [BH][nch] phi(k) as the bf16 operand tile (DK*128 bytes)
    const float* gamma;     // [BH] fixed decay per sequence-head, or NULL (none)
    int BH, T, nch;
    unsigned flags;
    int* status;
};

// ---------------------------------------------------------------------------
// 1. summary (persistent CTAs: unit u = (head, chunk) for u = blockIdx.x,
//    blockIdx.x + gridDim.x, ...; the next unit's tiles load while the
//    current one is processed)
// ---------------------------------------------------------------------------
template <int VAR, int DK, int DV>
struct SumLayout {
    static constexpr int KA = DK / 64, VA = DV / 64;
    static constexpr uint32_t K_OFF = 0;                       // within a stage
    static constexpr uint32_t V_OFF = KA * 8192;
    static constexpr uint32_t STAGE = V_OFF + VA * 8192;       // multiple of 1024
    static constexpr uint32_t KH_OFF = 2 * STAGE;              // phi(k) [64 j][DK]
    static constexpr uint32_t MISC_OFF = KH_OFF + KA * 8192;   // sTot[DK], sPart[128]
    static constexpr uint32_t BAR_OFF = MISC_OFF + (DK + 128) * 4;
    static constexpr uint32_t SMEM = BAR_OFF + 64 + 1024;
    static constexpr uint32_t TX = STAGE;
    static constexpr uint32_t TMEM_COLS = DK;
};
constexpr int kSumThreads = 256;

template <int VAR, int DK, int DV>
__global__ void __launch_bounds__(kSumThreads, 3)
summary_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, const Params p) {
    static_assert(VAR == kNorm, "the gated variants have their own kernel");
    using L = SumLayout<VAR, DK, DV>;
    constexpr int KA = L::KA, VA = L::VA;
    griddep_launch_dependents();
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (sbase - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int units = p.BH * p.nch;
    float* sTot = reinterpret_cast<float*>(sm + L::MISC_OFF);   // sum of phi(k)
    float* sPart = sTot + DK;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR_OFF);   // [0,1] stages, [2] MMA, [3] test hook
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 4);
    const uint32_t aKH = sbase + L::KH_OFF;

    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
    }
    // The previous kernel first, then tensor memory: a CTA never holds
    // columns while it waits on another grid (whose CTAs may still need
    // columns of this SM to finish).
    griddep_wait();   // inputs and the workspace are free to use from here on
    if (warp == 0) tmem_alloc(tmem_slot, L::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    int status_bits = 0;
    bool failed = false;
    if (p.flags & 0x100u) {  // test hook: a wait nothing will satisfy, 1 ms limit
        const bool ok = mbar_wait(&bar[3], 0, 1000000ull);
        if (__syncthreads_or(!ok)) { status_bits |= kStatusTestHook; failed = true; }
    }
    auto issue_load = [&](int u, int s) {
        const int bh = u / p.nch, t0 = (u % p.nch) * C;
        uint8_t* stg = sm + s * L::STAGE;
        mbar_arrive_expect_tx(&bar[s], L::TX);
#pragma unroll
        for (int a = 0; a < KA; ++a) tma_load_3d(&tmk, &bar[s], stg + L::K_OFF + a * 8192, a * 64, t0, bh);
#pragma unroll
        for (int a = 0; a < VA; ++a) tma_load_3d(&tmv, &bar[s], stg + L::V_OFF + a * 8192, a * 64, t0, bh);
    };
    bool pending[2] = {false, false};
    if (!failed && tid == 0 && static_cast<int>(blockIdx.x) < units) {
        issue_load(blockIdx.x, 0);
        pending[0] = true;
    }
    int k = 0;
    for (int u = blockIdx.x; u < units && !failed; u += gridDim.x, ++k) {
        const int s = k & 1;
        const int bh = u / p.nch, c = u % p.nch;
        const int nvalid = min(C, p.T - c * C);
        const uint32_t aK = sbase + s * L::STAGE + L::K_OFF, aV = sbase + s * L::STAGE + L::V_OFF;
        if (tid == 0 && u + static_cast<int>(gridDim.x) < units) {
            issue_load(u + gridDim.x, s ^ 1);   // the previous unit is done with stage s^1
            pending[s ^ 1] = true;
        }
        if (tid == 0) bulk_wait_read_all();   // the previous phi(k) tile has left
        {
            const bool ok = mbar_wait(&bar[s], (k >> 1) & 1, kWaitLimitNs);
            if (__syncthreads_or(!ok)) { status_bits |= kStatusTmaWait; failed = true; break; }
            if (tid == 0) pending[s] = false;
        }
        // phi(k); rows past T are zero.
#pragma unroll
        for (int i = 0; i < (64 * 8 * KA) / kSumThreads; ++i) {
            const int e = tid + kSumThreads * i;
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
        // norm with a fixed decay: token j of the chunk reaches the chunk's
        // end decayed by gamma^(nvalid-1-j); the weight goes on v_j (the
        // phi(k) tile stays as the output phase reads it)
        const float lg2g = p.gamma ? lg2(__ldg(p.gamma + bh)) : 0.f;
        if (p.gamma) {
#pragma unroll
            for (int i = 0; i < (64 * 8 * VA) / kSumThreads; ++i) {
                const int e = tid + kSumThreads * i;
                const int row = e / (8 * VA), a = (e / 8) % VA, pc = e % 8;
                const uint32_t off = a * 8192 + row * 128 + pc * 16;
                const float wv = (row < nvalid) ? ex2(static_cast<float>(nvalid - 1 - row) * lg2g) : 0.f;
                const uint4 uv = ld_shared_v4(aV + off);
                const float2 c0 = unpack_bf16(uv.x), c1 = unpack_bf16(uv.y), c2 = unpack_bf16(uv.z), c3 = unpack_bf16(uv.w);
                st_shared_v4(aV + off, pack_bf16(c0.x * wv, c0.y * wv), pack_bf16(c1.x * wv, c1.y * wv),
                             pack_bf16(c2.x * wv, c2.y * wv), pack_bf16(c3.x * wv, c3.y * wv));
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // dX = V^T K^ (value rows on the lanes; rows >= d_v unused)
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem, mnmaj(aV + kk * 2048, 8192), mnmaj(aKH + kk * 2048, 8192),
                            idesc_bf16(128, DK, true, true), kk > 0);
            mma_commit(&bar[2]);
            // phi(k) for the output phase, as the operand tile it reads
            // (not kept when only the chunk states are wanted)
            if (p.kh) {
                bulk_store(p.kh + static_cast<size_t>(u) * KA * 8192, aKH, KA * 8192);
                bulk_commit();
            }
        }
        {
            // sum of phi(k) per channel, from the bf16 operand the MMA reads
            constexpr int NP = kSumThreads / DK, RP = C / NP;
            const int ch = tid % DK, part = tid / DK;
            const uint32_t base = aKH + (ch / 64) * 8192 + (ch % 8) * 2;
            const int lc = (ch % 64) / 8;
            float zs = 0.f;
            if (p.gamma) {
#pragma unroll 8
                for (int j = part * RP; j < (part + 1) * RP; ++j)
                    if (j < nvalid) zs += ex2(static_cast<float>(nvalid - 1 - j) * lg2g) * ld_shared_bf16(base + sw128_off(j, lc));
            } else {
#pragma unroll 8
                for (int j = part * RP; j < (part + 1) * RP; ++j) zs += ld_shared_bf16(base + sw128_off(j, lc));
            }
            sPart[part * DK + ch] = zs;
            __syncthreads();
            if (part == 0) {
                float z = 0.f;
#pragma unroll
                for (int q = 0; q < NP; ++q) z += sPart[q * DK + ch];
                sTot[ch] = z;
            }
        }
        {
            const bool ok = mbar_wait(&bar[2], k & 1, kWaitLimitNs);
            tc_fence_after();
            if (__syncthreads_or(!ok)) { status_bits |= kStatusMmaWait; failed = true; break; }
        }
        // thread (r, hh) stores columns [hh*DK/2, (hh+1)*DK/2) of dX row r
        const int r = 32 * (warp & 3) + lane, hh = warp >> 2;
        if (r < DV) {
            float* dst = p.dx + (static_cast<size_t>(bh) * p.nch + c) * DV * DK + static_cast<size_t>(r) * DK + hh * (DK / 2);
#pragma unroll
            for (int b = 0; b < DK / 64; ++b) {
                float x[32];
                tmem_ld32(tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + hh * (DK / 2) + 32 * b, x);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                    *reinterpret_cast<float4*>(dst + 32 * b + i) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
            }
        }
        if (tid < DK) p.dd[(static_cast<size_t>(bh) * p.nch + c) * DK + tid] = sTot[tid];
        tc_fence_before();
        __syncthreads();   // TMEM read and sTot used before the next unit overwrites them
    }
    if (failed && tid == 0) {   // let loads in flight land before the CTA exits
        for (int s2 = 0; s2 < 2; ++s2)
            if (pending[s2]) mbar_wait(&bar[s2], ((s2 == (k & 1) ? k : k + 1) >> 1) & 1, 100000000ull);
    }
    if (tid == 0) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
    if (status_bits && tid == 0) atomicOr(p.status, status_bits);
}

// ---------------------------------------------------------------------------
// 2. scan over the chunks of every head
// ---------------------------------------------------------------------------
constexpr int kScanThreads = 256;
constexpr int kScanBatch = 32;   // chunks whose loads are in flight together

// One thread per 2 state columns of one value row (and, for norm, per 2
// channels of z): a running sum over the chunks, with the loads of
// kScanBatch chunks issued before they are consumed, so that a sequence of
// up to 32 chunks costs one round trip to L2.
template <int VAR, int DK, int DV>
__global__ void __launch_bounds__(kScanThreads) scan_kernel(const Params p) {
    static_assert(VAR == kNorm, "the gated variants have their own kernel");
    constexpr int E2 = DV * DK / 2;   // column pairs of X
    constexpr int Z2 = DK / 2;        // channel pairs of z
    constexpr int PER = E2 + Z2;
    constexpr size_t SSZ = static_cast<size_t>(DK) * DV + DK;
    constexpr size_t XS_BYTES = static_cast<size_t>(DK) * DV * 2;
    griddep_launch_dependents();
    griddep_wait();   // the chunk summaries are complete
    const int gi = blockIdx.x * kScanThreads + threadIdx.x;
    const int bh = gi / PER, e = gi % PER;
    if (bh >= p.BH) return;
    const int nch = p.nch;
    // with a fixed decay: each chunk decays what enters it by gamma^nvalid
    const float lg2g = p.gamma ? lg2(__ldg(p.gamma + bh)) : 0.f;
    auto chunk_decay = [&](int c) -> float {
        return p.gamma ? ex2(static_cast<float>(min(C, p.T - c * C)) * lg2g) : 1.f;
    };
    if (e < E2) {
        const int r = e / (DK / 2), col = 2 * (e % (DK / 2));   // value row r, columns col, col+1
        float2 x = make_float2(0.f, 0.f);
        if (p.state_in) {
            const float* si = p.state_in + bh * SSZ + r;
            x = make_float2(si[static_cast<size_t>(col) * DV], si[static_cast<size_t>(col + 1) * DV]);
        }
        const float* dx = p.dx + (static_cast<size_t>(bh) * nch * DV + r) * DK + col;
        uint8_t* xs = p.xs + static_cast<size_t>(bh) * nch * XS_BYTES + (col / 64) * (DV * 128) +
                      sw128_off(r, (col % 64) / 8) + (col % 8) * 2;
        for (int c = 0; c < nch; c += kScanBatch) {
            float2 a[kScanBatch];
#pragma unroll
            for (int u = 0; u < kScanBatch; ++u)
                if (c + u < nch) a[u] = *reinterpret_cast<const float2*>(dx + static_cast<size_t>(c + u) * DV * DK);
#pragma unroll
            for (int u = 0; u < kScanBatch; ++u) {
                if (c + u < nch) {
                    *reinterpret_cast<uint32_t*>(xs + (c + u) * XS_BYTES) = pack_bf16(x.x, x.y);
                    if (p.gamma) {
                        const float dc = chunk_decay(c + u);
                        x = make_float2(dc * x.x + a[u].x, dc * x.y + a[u].y);
                    } else {
                        x = make_float2(x.x + a[u].x, x.y + a[u].y);
                    }
                }
            }
        }
        if (p.state_out) {
            float* so = p.state_out + bh * SSZ + r;
            so[static_cast<size_t>(col) * DV] = x.x;
            so[static_cast<size_t>(col + 1) * DV] = x.y;
        }
    } else {
        // the normalizer entering every chunk
        const int ch = 2 * (e - E2);
        float2 z = make_float2(0.f, 0.f);
        if (p.state_in) z = *reinterpret_cast<const float2*>(p.state_in + bh * SSZ + static_cast<size_t>(DK) * DV + ch);
        for (int c = 0; c < nch; c += kScanBatch) {
            float2 a[kScanBatch];
#pragma unroll
            for (int u = 0; u < kScanBatch; ++u)
                if (c + u < nch) a[u] = *reinterpret_cast<const float2*>(p.dd + (static_cast<size_t>(bh) * nch + c + u) * DK + ch);
#pragma unroll
            for (int u = 0; u < kScanBatch; ++u) {
                if (c + u < nch) {
                    *reinterpret_cast<float2*>(p.zs + (static_cast<size_t>(bh) * nch + c + u) * DK + ch) = z;
                    const float dc = chunk_decay(c + u);
                    z = make_float2(dc * z.x + a[u].x, dc * z.y + a[u].y);
                }
            }
        }
        if (p.state_out) *reinterpret_cast<float2*>(p.state_out + bh * SSZ + static_cast<size_t>(DK) * DV + ch) = z;
    }
}

// ---------------------------------------------------------------------------
// 3. output (persistent CTAs over the units, like the summary)
// ---------------------------------------------------------------------------
template <int VAR, int DK, int DV>
struct OutLayout {
    static constexpr int KA = DK / 64, VA = DV / 64;
    // one stage: q/k pair (per k-atom rows 0-63 q, 64-127 phi(k)), v, the
    // state entering the chunk (bf16 [DV rows][DK], KA atoms), z
    static constexpr uint32_t QK_OFF = 0;
    static constexpr uint32_t V_OFF = KA * 16384;
    static constexpr uint32_t XS_OFF = V_OFF + VA * 8192;
    static constexpr uint32_t XS_BYTES = DK * DV * 2;
    static constexpr uint32_t Z_OFF = XS_OFF + XS_BYTES;
    static constexpr uint32_t Z_BYTES = DK * 4;
    static constexpr uint32_t STAGE = ((Z_OFF + Z_BYTES) + 1023u) & ~1023u;
    static constexpr uint32_t TX = 2 * KA * 8192 + VA * 8192 + XS_BYTES + Z_BYTES;
    static constexpr uint32_t FIXED = 8192 + VA * 8192 + 64 * 4 + 64;   // P, output tile, misc, barriers
    static constexpr int NSTAGE = (2 * STAGE + FIXED + 1024 <= 232448) ? 2 : 1;
    static constexpr uint32_t PS_OFF = NSTAGE * STAGE;           // P bf16 [64 t][64 j]
    static constexpr uint32_t OT_OFF = PS_OFF + 8192;            // output tile [64 t][DV] (also rows 64-127 of the M=128 P read)
    static constexpr uint32_t MISC_OFF = OT_OFF + VA * 8192;     // sDen[64]
    static constexpr uint32_t BAR_OFF = MISC_OFF + 64 * 4;
    static constexpr uint32_t SMEM = BAR_OFF + 64 + 1024;
    static constexpr uint32_t COL_G = 0;    // P [t][64]
    static constexpr uint32_t COL_O = 64;   // O [t][DV]
    static constexpr uint32_t TMEM_COLS = (64 + DV <= 128) ? 128 : 256;
};
constexpr int kOutThreads = 256;

template <int VAR, int DK, int DV>
__global__ void __launch_bounds__(kOutThreads, 2)
output_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmv,
              const __grid_constant__ CUtensorMap tmo, const Params p) {
    static_assert(VAR == kNorm, "the gated variants have their own kernel");
    using L = OutLayout<VAR, DK, DV>;
    constexpr int KA = L::KA, VA = L::VA, NS = L::NSTAGE;
    griddep_launch_dependents();
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (sbase - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = 32 * (warp & 3) + lane;   // tensor-memory lane
    const int hh = warp >> 2;               // column half
    const int units = p.BH * p.nch;
    const int T = p.T;
    float* sDen = reinterpret_cast<float*>(sm + L::MISC_OFF);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR_OFF);   // [0,1] stages, [2] MMA, [3] test hook
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 4);
    const uint32_t aPS = sbase + L::PS_OFF, aOT = sbase + L::OT_OFF;

    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmv);
        tma_prefetch_desc(&tmo);
    }
    griddep_wait();   // the scan's start states are complete (then tensor memory, as above)
    if (warp == 0) tmem_alloc(tmem_slot, L::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);

    int status_bits = 0;
    bool failed = false;
    if (p.flags & 0x100u) {
        const bool ok = mbar_wait(&bar[3], 0, 1000000ull);
        if (__syncthreads_or(!ok)) { status_bits |= kStatusTestHook; failed = true; }
    }
    auto issue_load = [&](int u, int s) {
        const int bh = u / p.nch, t0 = (u % p.nch) * C;
        uint8_t* stg = sm + s * L::STAGE;
        mbar_arrive_expect_tx(&bar[s], L::TX);
#pragma unroll
        for (int a = 0; a < KA; ++a) {
            tma_load_3d(&tmq, &bar[s], stg + L::QK_OFF + a * 16384, a * 64, t0, bh);
            // phi(k) as the summary phase stored it
            bulk_load(stg + L::QK_OFF + a * 16384 + 8192, p.kh + (static_cast<size_t>(u) * KA + a) * 8192, 8192, &bar[s]);
        }
#pragma unroll
        for (int a = 0; a < VA; ++a) tma_load_3d(&tmv, &bar[s], stg + L::V_OFF + a * 8192, a * 64, t0, bh);
        bulk_load(stg + L::XS_OFF, p.xs + static_cast<size_t>(u) * L::XS_BYTES, L::XS_BYTES, &bar[s]);
        bulk_load(stg + L::Z_OFF, p.zs + static_cast<size_t>(u) * DK, DK * 4, &bar[s]);
    };
    bool pending[2] = {false, false};
    if (!failed && tid == 0 && static_cast<int>(blockIdx.x) < units) {
        issue_load(blockIdx.x, 0);
        pending[0] = true;
    }
    uint32_t mph = 0;
    int k = 0;
    for (int u = blockIdx.x; u < units && !failed; u += gridDim.x, ++k) {
        const int s = (NS == 2) ? (k & 1) : 0;
        const uint32_t par_full = (NS == 2) ? ((k >> 1) & 1) : (k & 1);
        const int bh = u / p.nch, c = u % p.nch;
        const float lg2g = p.gamma ? lg2(__ldg(p.gamma + bh)) : 0.f;   // log2 of the decay
        const int t0 = c * C, nvalid = min(C, T - t0);
        const uint32_t aQK = sbase + s * L::STAGE + L::QK_OFF, aV = sbase + s * L::STAGE + L::V_OFF;
        const uint32_t aXS = sbase + s * L::STAGE + L::XS_OFF;
        const float* sZ = reinterpret_cast<const float*>(sm + s * L::STAGE + L::Z_OFF);
        if (NS == 2 && tid == 0 && u + static_cast<int>(gridDim.x) < units) {
            issue_load(u + gridDim.x, s ^ 1);   // the previous unit is done with stage s^1
            pending[s ^ 1] = true;
        }
        {
            const bool ok = mbar_wait(&bar[s], par_full, kWaitLimitNs);
            if (__syncthreads_or(!ok)) { status_bits |= kStatusTmaWait; failed = true; break; }
            if (tid == 0) pending[s] = false;
        }
        // q~ = phi(q) (rows 0-63) in place, 8 channels per 16 bytes; k~ = phi(k)
        // (rows 64-127) arrived ready from the summary phase.
        {
#pragma unroll
            for (int i = 0; i < (64 * 8 * KA) / kOutThreads; ++i) {
                const int e = tid + kOutThreads * i;
                const int row = e / (8 * KA), a = (e / 8) % KA, pc = e % 8;
                const uint32_t qa = aQK + a * 16384 + (row >> 3) * 1024 + (row & 7) * 128 + pc * 16;
                const uint4 uq = ld_shared_v4(qa);
                const float2 a0 = unpack_bf16(uq.x), a1 = unpack_bf16(uq.y), a2 = unpack_bf16(uq.z),
                             a3 = unpack_bf16(uq.w);
                st_shared_v4(qa, pack_bf16(elu1(a0.x), elu1(a0.y)), pack_bf16(elu1(a1.x), elu1(a1.y)),
                             pack_bf16(elu1(a2.x), elu1(a2.y)), pack_bf16(elu1(a3.x), elu1(a3.y)));
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // P = Q~ K~^T ;  O = Q~ X_{c-1}^T  (tokens on the lanes; rows 64-127 unused)
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < DK / 16; ++kk) {
                const uint32_t qa = aQK + (kk / 4) * 16384 + (kk % 4) * 32;
                mma_bf16_ss(tmem + L::COL_G, kmaj(qa), kmaj(qa + 8192), idesc_bf16(128, 64, false, false), kk > 0);
                mma_bf16_ss(tmem + L::COL_O, kmaj(qa), kmaj(aXS + (kk / 4) * (DV * 128) + (kk % 4) * 32),
                            idesc_bf16(128, DV, false, false), kk > 0);
            }
            mma_commit(&bar[2]);
        }
        {
            // den_t = q~_t . z_{c-1} while the MMAs run (4 threads per token)
            const int t = tid >> 2, q4 = tid & 3;
            float d = 0.f;
#pragma unroll
            for (int m = 0; m < KA * 2; ++m) {
                const int cq = q4 * (KA * 2) + m;   // 8-channel group
                const int a = cq / 8, lc = cq % 8;
                const uint4 uu = ld_shared_v4(aQK + a * 16384 + sw128_off(t, lc));
                const float2 x0 = unpack_bf16(uu.x), x1 = unpack_bf16(uu.y), x2 = unpack_bf16(uu.z), x3 = unpack_bf16(uu.w);
                const float* z = sZ + 8 * cq;
                d += x0.x * z[0] + x0.y * z[1] + x1.x * z[2] + x1.y * z[3] + x2.x * z[4] + x2.y * z[5] + x3.x * z[6] +
                     x3.y * z[7];
            }
            d += __shfl_xor_sync(0xffffffffu, d, 1);
            d += __shfl_xor_sync(0xffffffffu, d, 2);
            if (q4 == 0) sDen[t] = p.gamma ? d * ex2(static_cast<float>(t + 1) * lg2g) : d;
        }
        {
            const bool ok = mbar_wait(&bar[2], mph, kWaitLimitNs);
            mph ^= 1u;
            tc_fence_after();
            if (__syncthreads_or(!ok)) { status_bits |= kStatusMmaWait; failed = true; break; }
        }
        if ((warp & 3) < 2) {
            // masked scores of rows t = 0..63 -> bf16 P; the row sums add to den.
            const int t = r;
            float x[32];
            tmem_ld32(tlane + L::COL_G + 32 * hh, x);
            tmem_ld_wait();
            float rs = 0.f;
            if (p.gamma) {
                // with a fixed decay: score (t, j) weighs gamma^(t-j), and
                // the product with the state entering the chunk gamma^(t+1)
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int j = 32 * hh + i;
                    x[i] = (j <= t) ? x[i] * ex2(static_cast<float>(t - j) * lg2g) : 0.f;
                    rs += x[i];
                }
                const float gt1 = ex2(static_cast<float>(t + 1) * lg2g);
#pragma unroll
                for (int b = 0; b < DV / 64; ++b) {
                    float y[32];
                    uint32_t u32[32];
                    tmem_ld32(tlane + L::COL_O + hh * (DV / 2) + 32 * b, y);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) u32[i] = __float_as_uint(y[i] * gt1);
                    tmem_st32(tlane + L::COL_O + hh * (DV / 2) + 32 * b, u32);
                }
                tmem_st_wait();
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    x[i] = (32 * hh + i <= t) ? x[i] : 0.f;
                    rs += x[i];
                }
            }
            store_row32_bf16(aPS, t, 4 * hh, x);
            atomicAdd(&sDen[t], rs);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // O += P V
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + L::COL_O, kmaj(aPS + kk * 32), mnmaj(aV + kk * 2048, 8192),
                            idesc_bf16(128, DV, false, true), 1);
            mma_commit(&bar[2]);
            bulk_wait_read_all();   // the previous unit's output store has left the tile
        }
        if (p.den_out && tid < nvalid) p.den_out[static_cast<size_t>(bh) * T + t0 + tid] = sDen[tid];
        {
            const bool ok = mbar_wait(&bar[2], mph, kWaitLimitNs);
            mph ^= 1u;
            tc_fence_after();
            if (__syncthreads_or(!ok)) { status_bits |= kStatusMmaWait; failed = true; break; }
        }
        // rows t < 64 of O (thread (t, hh) holds columns [hh*DV/2, (hh+1)*DV/2)),
        // divided by den, into the [64 t][DV] tile, then TMA stores.
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
                store_row32_bf16(aOT + (cb / 64) * 8192, t, (cb % 64) / 8, x);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int a = 0; a < VA; ++a) tma_store_3d(&tmo, sm + L::OT_OFF + a * 8192, a * 64, t0, bh);
            bulk_commit();
            if (NS == 1 && u + static_cast<int>(gridDim.x) < units) {
                issue_load(u + gridDim.x, 0);   // single stage: reload once this unit is done with it
                pending[0] = true;
            }
        }
    }
    if (failed && tid == 0) {   // let loads in flight land before the CTA exits
        for (int s2 = 0; s2 < NS; ++s2)
            if (pending[s2]) {
                const uint32_t par = (NS == 2) ? (((s2 == (k & 1) ? k : k + 1) >> 1) & 1) : (k & 1);
                mbar_wait(&bar[s2], par, 100000000ull);
            }
    }
    if (tid == 0) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
    if (status_bits && tid == 0) atomicOr(p.status, status_bits);
}

// CTAs of a persistent kernel that fit on one SM next to each other
// (shared memory with its 1 KB per-CTA reserve, tensor memory, threads).
int per_sm(uint32_t smem, uint32_t tmem_cols, int threads, int cap) {
    int n = static_cast<int>(233472u / (smem + 1024u));
    const int nt = static_cast<int>(512u / tmem_cols);
    const int nth = 2048 / threads;
    if (nt < n) n = nt;
    if (nth < n) n = nth;
    if (cap < n) n = cap;
    return n < 1 ? 1 : n;
}

// Phases 1 and 2 (chunk summaries, then the scan), chained by programmatic
// dependent launch; the states entering every chunk are in p.xs and p.zs
// afterwards.
template <int VAR, int DK, int DV>
cudaError_t run_states(const chunk::Maps& m, const Params& p, int sm_count, cudaStream_t s) {
    using S1 = SumLayout<VAR, DK, DV>;
    static_assert(S1::SMEM <= 232448, "shared memory budget");
    auto k1 = summary_kernel<VAR, DK, DV>;
    auto k2 = scan_kernel<VAR, DK, DV>;
    cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, S1::SMEM);
    if (e != cudaSuccess) return e;
    const int units = p.BH * p.nch;
    int g1 = sm_count * per_sm(S1::SMEM, S1::TMEM_COLS, kSumThreads, 3);
    if (g1 > units) g1 = units;
    e = launch_pdl(k1, g1, kSumThreads, S1::SMEM, s, m.k, m.v, p);
    if (e != cudaSuccess) return e;
    constexpr int PER = DV * DK / 2 + DK / 2;
    const long long threads = static_cast<long long>(p.BH) * PER;
    return launch_pdl(k2, static_cast<unsigned>((threads + kScanThreads - 1) / kScanThreads), kScanThreads, 0, s, p);
}

template <int VAR, int DK, int DV>
cudaError_t run(const chunk::Maps& m, const Params& p, int sm_count, cudaStream_t s) {
    using S3 = OutLayout<VAR, DK, DV>;
    static_assert(S3::SMEM <= 232448, "shared memory budget");
    auto k3 = output_kernel<VAR, DK, DV>;
    cudaError_t e = run_states<VAR, DK, DV>(m, p, sm_count, s);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k3, cudaFuncAttributeMaxDynamicSharedMemorySize, S3::SMEM);
    if (e != cudaSuccess) return e;
    const int units = p.BH * p.nch;
    int g3 = sm_count * per_sm(S3::SMEM, S3::TMEM_COLS, kOutThreads, 2);
    if (g3 > units) g3 = units;
    return launch_pdl(k3, g3, kOutThreads, S3::SMEM, s, m.q, m.v, m.o, p);
}

template <int VAR>
cudaError_t dispatch(int dk, int dv, const chunk::Maps& m, const Params& p, int sm_count, cudaStream_t s) {
    if (dk == 64 && dv == 64) return run<VAR, 64, 64>(m, p, sm_count, s);
    if (dk == 64 && dv == 128) return run<VAR, 64, 128>(m, p, sm_count, s);
    if (dk == 128 && dv == 64) return run<VAR, 128, 64>(m, p, sm_count, s);
    if (dk == 128 && dv == 128) return run<VAR, 128, 128>(m, p, sm_count, s);
    return cudaErrorInvalidValue;
}

}  // namespace par

namespace chunk {

size_t par_state_bytes(int dk, int dv) {
    // dX fp32 + start state bf16 + dd + zs
    return static_cast<size_t>(dk) * dv * 6 + static_cast<size_t>(dk) * 8;
}

size_t par_chunk_bytes(int dk, int dv) {
    return par_state_bytes(dk, dv) + static_cast<size_t>(dk) * 128;   // + the phi(k) tile
}

bool par_fits(int BH, int T, int dk, int dv, size_t ws_bytes) {
    const size_t nch = static_cast<size_t>((T + C - 1) / C);
    const size_t need = static_cast<size_t>(BH) * nch * par_chunk_bytes(dk, dv);
    return need <= ws_bytes && need <= kParL2Bytes;
}

namespace {

// The three-phase form's workspace: dX | dd | start states | start
// normalizers | phi(k) tiles (each a multiple of 256 bytes per unit).
par::Params carve(const FwdArgs& a, ParStates* st, bool keep_kh = true) {
    par::Params p;
    const size_t nch = static_cast<size_t>((a.T + C - 1) / C);
    const size_t units = static_cast<size_t>(a.BH) * nch;
    p.state_in = a.state_in;
    p.state_out = a.state_out;
    p.den_out = a.den_out;
    uint8_t* w = reinterpret_cast<uint8_t*>(a.workspace);
    p.dx = reinterpret_cast<float*>(w);
    w += units * a.dk * a.dv * sizeof(float);
    p.dd = reinterpret_cast<float*>(w);
    w += units * a.dk * sizeof(float);
    p.xs = w;
    w += units * a.dk * a.dv * 2;
    p.zs = reinterpret_cast<float*>(w);
    w += units * a.dk * sizeof(float);
    p.kh = keep_kh ? w : nullptr;
    if (keep_kh) w += units * a.dk * 128;
    p.gamma = a.gate;   // the normalized variant's fixed decay, or NULL
    p.BH = a.BH;
    p.T = a.T;
    p.nch = static_cast<int>(nch);
    p.flags = a.flags;
    p.status = a.status;
    if (st) {
        st->dx = p.dx;
        st->dd = p.dd;
        st->xs = p.xs;
        st->zs = p.zs;
        st->end = w;
        st->nch = p.nch;
    }
    return p;
}

}  // namespace

cudaError_t launch_par(const FwdArgs& a, const Maps& m, cudaStream_t s) {
    const par::Params p = carve(a, nullptr);
    if (a.nlaunch) *a.nlaunch += 3;   // summary, scan, output
    if (a.variant == kNorm) return par::dispatch<kNorm>(a.dk, a.dv, m, p, a.sm_count, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_par_states(const FwdArgs& a, const Maps& m, cudaStream_t s, ParStates* st) {
    const par::Params p = carve(a, st, false);
    if (a.variant != kNorm || a.gate) return cudaErrorInvalidValue;
    if (a.dk == 64 && a.dv == 64) return par::run_states<kNorm, 64, 64>(m, p, a.sm_count, s);
    return cudaErrorInvalidValue;
}

}  // namespace chunk
}  // namespace la
