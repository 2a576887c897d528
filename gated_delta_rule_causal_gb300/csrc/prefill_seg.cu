// Normalized elu+1 prefill (d_k = d_v = 64), with or without a fixed decay, in one cluster launch.
//
// "Linear attention and Hyena" §11.2-11.3: with phi = elu + 1, the state
// S_t = S_{t-1} + phi(k_t) v_t^T and z_t = z_{t-1} + phi(k_t) give
// o_t = phi(q_t)^T S_t / phi(q_t)^T z_t, and over a block of tokens the
// same outputs come from the block's causal scores plus the state that
// entered it. Here every CTA owns one segment of at most kMaxSub blocks of
// B = 128 tokens of one sequence-head. With X = S^T ([d_v][d_k]) and, per
// block j of the segment,
//   A_j = [V_j | 1]^T phi(K_j)             (rows 0..63: dX^T, rows 64..: dz)
//   P_j = L o phi(Q_j) phi(K_j)^T          (L: the causal mask)
//   O_j = phi(Q_j) [X_loc | z_loc]^T + P_j [V_j | 1]
// where X_loc, z_loc sum A_i over the segment's earlier blocks (and the
// initial state in the first segment), kept in fp32 registers. Column d_v of
// O_j is the normalizer of each token, so the quotient needs no extra pass.
// The "1" columns and rows come from a block of ones in shared memory that
// the MN-major operand descriptors reach through their leading-byte offset.
//
// The segments of one sequence-head form one thread-block cluster (at most
// kMaxSeg CTAs). Once its blocks are done, a CTA tells its predecessors that
// its stage area is free; each predecessor then copies its total (X, z) into
// that area with one distributed-shared-memory bulk copy per successor, and
// segment s sums the totals of segments 0..s-1 (the state entering it) from
// its own shared memory, then adds phi(Q_j) [X_in | z_in]^T to the outputs it
// held in tensor memory. Clusters never wait on one another, every wait is
// bounded, and a CTA that failed still sends its total, marked as invalid.
//
// With a fixed decay gamma per sequence-head (S_t = gamma S_{t-1} +
// phi(k_t) v_t^T, z likewise), every factor is a power gamma^n with n >= 0:
// score (t, i) takes gamma^(t-i); once the scores are read, phi(Q_j) rows
// take gamma^(t+1) for the state part and phi(K_j) rows gamma^(L-1-i) for
// A_j (L tokens in the block), so the state part of O_j and A_j move to the
// second batch; the running total becomes gamma^L X + A_j, a predecessor's
// total is weighted by the tokens between it and this segment, and the
// closing product of block j by gamma^(128 j).

#include "prefill.h"
#include "prefill_impl.cuh"
#include "launch.cuh"

namespace la {
namespace seg {

using chunk::elu1;
using chunk::kmaj;
using chunk::ld_shared_v4;
using chunk::mnmaj;
using chunk::st_shared_v4;
using chunk::store_row32_bf16;

constexpr int B = 128;        // tokens per block
constexpr int D = 64;         // d_k = d_v
constexpr int kMaxSub = 4;    // blocks per segment: four held outputs + scores fill tensor memory
constexpr int kMaxSeg = 6;    // segments per sequence-head (cluster size): 5 totals fit the stage area
constexpr int kWorkers = 256;             // 8 warps: conversions and tensor-memory reads
constexpr int kThreads = kWorkers + 32;   // + the warp that issues every MMA and TMA copy
constexpr int SSZ = D * D + D;   // one state: X or S plus z
constexpr uint32_t kTotBytes = SSZ * 4 + 16;   // a total as sent: [16 column groups][65 rows][4] floats, ok word

struct Params {
    const float* gamma;        // [BH] fixed decay per sequence-head in (0, 1] (decayed form only)
    const float* state_in;     // S [BH][D][D] then z [D] per head, or NULL
    float* state_out;          // same layout, or NULL
    float* den_out;            // [BH][T], or NULL
    int BH, T, nsub, nseg, per;   // blocks per head, segments (= cluster size) per head, blocks per segment
    unsigned flags;
    int* status;
};

// Shared memory (offsets from the 1024-aligned base).
struct Layout {
    static constexpr uint32_t Q = 0;                        // phi(Q_j), kMaxSub tiles [128 t][64] K-major; then the output tiles
    static constexpr uint32_t STG = Q + kMaxSub * 16384;    // 3 stages of K (phi(K) in place) and V; then the predecessors' totals
    static constexpr uint32_t STAGE = 32768;
    static constexpr int NSTAGE = 3;
    static constexpr uint32_t P = STG + NSTAGE * STAGE;     // scores bf16, 2 atoms [128 t][64 i]; then this
                                                            // segment's total as sent (kTotBytes)
    static constexpr uint32_t X = P + 32768;                // [X_loc | z_loc]^T, [80 rows][64] K-major; then [X_in | z_in]^T
    static constexpr uint32_t ONES = X + 10240;             // 16 KB of bf16 ones
    static constexpr uint32_t BAR = ONES + 16384;
    static constexpr uint32_t BYTES = BAR + 128;
    static constexpr uint32_t SMEM = BYTES + 1024;
    // tensor memory: O_j at 96 j (80 columns); the scores at COL_PA. A_j goes
    // to the next block's output columns (still free), the last one to COL_PA.
    static constexpr uint32_t COL_PA = 384;
    static constexpr uint32_t TMEM_COLS = 512;
};
static_assert(Layout::SMEM <= 232448, "shared memory budget");
static_assert(Layout::ONES > Layout::STG + (Layout::NSTAGE - 1) * Layout::STAGE + 16384, "ones block above every value tile");
static_assert(kMaxSub <= Layout::NSTAGE + 1, "a block reloads a stage at most once");
static_assert((kMaxSeg - 1) * kTotBytes <= Layout::NSTAGE * Layout::STAGE, "predecessors' totals fit the stage area");
static_assert(kTotBytes <= 32768 && kTotBytes % 16 == 0, "this CTA's total fits the score area");

// barriers
enum { kBarQ = 0, kBarLd = kMaxSub, kBarP = kMaxSub + Layout::NSTAGE, kBarO, kBarFin, kBarHook, kBarReady, kBarInbox, kBarDone, kNumBar };

template <bool DECAY>
__global__ void __launch_bounds__(kThreads, 1)
seg_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
           const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo, const Params p) {
    using L = Layout;
    constexpr int NS = L::NSTAGE;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (sbase - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool worker = tid < kWorkers;
    const bool issuer = tid == kWorkers;     // lane 0 of the last warp
    const int r = 32 * (warp & 3) + lane;    // tensor-memory lane: token, or state row
    const int hh = (warp >> 2) & 1;          // column half
    const bool rowv = worker && (warp & 3) < 2;    // state rows v = r < 64
    const bool rowz = worker && (warp & 3) == 2;   // normalizer rows (all alike); r == 64 writes
    const int bh = blockIdx.x / p.nseg, sg = static_cast<int>(cluster_ctarank());   // = blockIdx.x % nseg
    const int j0 = sg * p.per;
    const int nj = min(p.per, p.nsub - j0);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + kNumBar);
    const uint32_t aP = sbase + L::P, aX = sbase + L::X, aONES = sbase + L::ONES;
    const bool hook = (p.flags & 0x100u) != 0;   // test hook: a wait nothing will satisfy, 1 ms limit
    const float gam = DECAY ? __ldg(p.gamma + bh) : 1.f;
    const float lg = DECAY ? lg2(gam) : 0.f;   // gamma^n = ex2(n lg), n >= 0 throughout

    // loads in flight, for a clean exit after a failed wait (issuing thread): Q
    // tiles not yet waited for, and per stage the loads issued and waited for
    unsigned q_pending = 0;
    int kv_iss[NS] = {0, 0, 0}, kv_done[NS] = {0, 0, 0};
    auto load_kv = [&](int j) {
        const int t0 = (j0 + j) * B, st = j % NS;
        ++kv_iss[st];
        uint8_t* stg = sm + L::STG + st * L::STAGE;
        mbar_arrive_expect_tx(&bar[kBarLd + st], 32768);
        tma_load_3d(&tmk, &bar[kBarLd + st], stg, 0, t0, bh);
        tma_load_3d(&tmk, &bar[kBarLd + st], stg + 8192, 0, t0 + 64, bh);
        tma_load_3d(&tmv, &bar[kBarLd + st], stg + 16384, 0, t0, bh);
        tma_load_3d(&tmv, &bar[kBarLd + st], stg + 24576, 0, t0 + 64, bh);
    };
    auto load_q = [&](int j) {
        const int t0 = (j0 + j) * B;
        mbar_arrive_expect_tx(&bar[kBarQ + j], 16384);
        tma_load_3d(&tmq, &bar[kBarQ + j], sm + L::Q + j * 16384, 0, t0, bh);
        tma_load_3d(&tmq, &bar[kBarQ + j], sm + L::Q + j * 16384 + 8192, 0, t0 + 64, bh);
    };
    const int nsucc = p.nseg - 1 - sg;
    if (issuer) {   // barriers, then the first tiles on their way before anything else
        for (int i = 0; i < kNumBar; ++i)
            mbar_init(&bar[i], (i == kBarReady || i == kBarDone) && nsucc > 0 ? nsucc : 1);
        fence_mbar_init();
        if (sg > 0) mbar_arrive_expect_tx(&bar[kBarInbox], static_cast<uint32_t>(sg) * kTotBytes);
        if (!hook) {
            load_q(0);
            load_kv(0);
            for (int j = 1; j < nj && j < NS; ++j) load_kv(j);
            for (int j = 1; j < nj; ++j) load_q(j);
            q_pending = (1u << nj) - 1u;
        }
    }
    {   // ones block; the state tile starts at zero (rows past 64 stay zero)
        const uint32_t one2 = 0x3F803F80u;
        for (int i = tid; i < 16384 / 16; i += kThreads) st_shared_v4(aONES + 16 * i, one2, one2, one2, one2);
        for (int i = tid; i < 10240 / 16; i += kThreads) st_shared_v4(aX + 16 * i, 0u, 0u, 0u, 0u);
        if (issuer) {
            tma_prefetch_desc(&tmo);
        }
    }
    if (warp == 0) tmem_alloc(tmem_slot, L::TMEM_COLS);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_arrive_relaxed();   // waited for before the first access to another CTA's barriers
    const uint32_t tmem = *tmem_slot;
    const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);

    int status_bits = 0;
    bool failed = false;
    if (hook) {
        const bool ok = mbar_wait(&bar[kBarHook], 0, 1000000ull);
        if (__syncthreads_or(!ok)) { status_bits |= kStatusTestHook; failed = true; }
    }

    // running total of this thread's state row (columns hh*32..hh*32+31):
    // X rows v = r (rowv) or z (rowz); the first segment starts from state_in
    float R[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) R[i] = 0.f;
    if (sg == 0 && p.state_in && (rowv || rowz)) {
        const float* si = p.state_in + static_cast<size_t>(bh) * SSZ;
#pragma unroll
        for (int i = 0; i < 32; ++i) R[i] = rowv ? si[(hh * 32 + i) * D + r] : si[D * D + hh * 32 + i];
    }
    auto write_state_tile = [&](const float* x) {
        if (rowv) store_row32_bf16(aX, r, 4 * hh, x);
        else if (rowz && lane == 0) store_row32_bf16(aX, 64, 4 * hh, x);
    };
    auto read_a = [&](uint32_t col) {   // R += A (tensor memory rows 0..95 at `col`)
        if (rowv || rowz) {
            float a[32];
            tmem_ld32(tlane + col + hh * 32, a);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) R[i] += a[i];
        }
    };
    // phi(Q_j), phi(K_j) in place once block j has landed (workers; no CTA
    // barrier, so the conversion overlaps the issuing warp's MMA queueing);
    // key rows past T are zero (phi(0) = 1). Returns whether the wait succeeded.
    auto convert = [&](int j) -> bool {
        const bool ok = mbar_wait(&bar[kBarQ + j], 0, kWaitLimitNs) &&
                        mbar_wait(&bar[kBarLd + j % NS], (j / NS) & 1, kWaitLimitNs);
        const int nvalid = min(B, p.T - (j0 + j) * B);
        const uint32_t aQ = sbase + L::Q + j * 16384, aK = sbase + L::STG + (j % NS) * L::STAGE;
        // all eight 16-byte chunks in flight before any is converted (the
        // shared-memory accesses keep their program order)
        uint4 uq[4], uk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = tid + kWorkers * i;   // 16-byte chunk: row e / 8
            uq[i] = ld_shared_v4(aQ + 16 * e);
            uk[i] = ld_shared_v4(aK + 16 * e);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = tid + kWorkers * i;
            const float2 a0 = unpack_bf16(uq[i].x), a1 = unpack_bf16(uq[i].y), a2 = unpack_bf16(uq[i].z),
                         a3 = unpack_bf16(uq[i].w);
            st_shared_v4(aQ + 16 * e, pack_bf16(elu1(a0.x), elu1(a0.y)), pack_bf16(elu1(a1.x), elu1(a1.y)),
                         pack_bf16(elu1(a2.x), elu1(a2.y)), pack_bf16(elu1(a3.x), elu1(a3.y)));
            if ((e >> 3) < nvalid) {
                const float2 b0 = unpack_bf16(uk[i].x), b1 = unpack_bf16(uk[i].y), b2 = unpack_bf16(uk[i].z),
                             b3 = unpack_bf16(uk[i].w);
                st_shared_v4(aK + 16 * e, pack_bf16(elu1(b0.x), elu1(b0.y)), pack_bf16(elu1(b1.x), elu1(b1.y)),
                             pack_bf16(elu1(b2.x), elu1(b2.y)), pack_bf16(elu1(b3.x), elu1(b3.y)));
            } else {
                st_shared_v4(aK + 16 * e, 0u, 0u, 0u, 0u);
            }
        }
        return ok;
    };
    auto sync_mma = [&]() {   // generic smem writes and tensor-memory reads before the next MMAs
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };

    const uint32_t ID_P = idesc_bf16(128, 128, false, false);
    const uint32_t ID_O = idesc_bf16(128, 80, false, false);
    const uint32_t ID_PV = idesc_bf16(128, 80, false, true);
    const uint32_t ID_A = idesc_bf16(128, 64, true, true);
    auto issue_batch1 = [&](int j) {   // scores, the state part of O_j and (not last) A_j
        const uint32_t aQ = sbase + L::Q + j * 16384;
        const uint32_t aK = sbase + L::STG + (j % NS) * L::STAGE, aV = aK + 16384;
        const uint32_t dO = tmem + 96 * j;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ss(tmem + L::COL_PA, kmaj(aQ + kk * 32), kmaj(aK + kk * 32), ID_P, kk > 0);
        if (DECAY) {   // scores alone: the rest waits for the decayed operands
            mma_commit(&bar[kBarP]);
            return;
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_bf16_ss(dO, kmaj(aQ + kk * 32), kmaj(aX + kk * 32), ID_O, kk > 0);
        if (j + 1 < nj) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16_ss(dO + 96, mnmaj(aV + kk * 2048, aONES - aV), mnmaj(aK + kk * 2048, 8192), ID_A, kk > 0);
        }
        mma_commit(&bar[kBarP]);
    };
    auto issue_batch2 = [&](int j) {   // the score part of O_j (and the last block's A_j)
        const uint32_t aQ = sbase + L::Q + j * 16384;
        const uint32_t aK = sbase + L::STG + (j % NS) * L::STAGE, aV = aK + 16384;
        const uint32_t dO = tmem + 96 * j;
        if (DECAY) {   // decayed: the state part of O_j and A_j (into the next block's columns) too
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) mma_bf16_ss(dO, kmaj(aQ + kk * 32), kmaj(aX + kk * 32), ID_O, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ss(dO, kmaj(aP + (kk / 4) * 16384 + (kk % 4) * 32), mnmaj(aV + kk * 2048, aONES - aV), ID_PV, 1);
        if (DECAY) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16_ss(dO + 96, mnmaj(aV + kk * 2048, aONES - aV), mnmaj(aK + kk * 2048, 8192), ID_A, kk > 0);
        } else if (j + 1 == nj) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16_ss(tmem + L::COL_PA, mnmaj(aV + kk * 2048, aONES - aV), mnmaj(aK + kk * 2048, 8192), ID_A, kk > 0);
        }
        mma_commit(&bar[kBarO]);
    };
    if (!failed) {
        write_state_tile(R);
        const bool ok = !worker || convert(0);
        if (__syncthreads_or(!ok)) { status_bits |= kStatusTmaWait; failed = true; }
        if (issuer && !failed) { q_pending &= ~1u; ++kv_done[0]; }
    }
    if (!failed) {
        sync_mma();
        if (issuer) issue_batch1(0);
    }
    // Block j: while batch 1 runs, block j+1 converts; then the masked
    // scores, A_j into the running total and the next state tile; then the
    // issuer queues batch 2 of block j and batch 1 of block j+1 together.
    for (int j = 0; j < nj && !failed; ++j) {
        const bool last = j + 1 == nj;
        const bool cok = !worker || last || convert(j + 1);
        {
            // batch 1 of block j done, and with it batch 2 of block j-1
            bool ok = true;
            if (worker || (j >= 1 && j + 2 < nj)) {
                ok = mbar_wait(&bar[kBarP], j & 1, kWaitLimitNs);
                if (j > 0) ok = ok && mbar_wait(&bar[kBarO], (j - 1) & 1, kWaitLimitNs);
            }
            tc_fence_after();
            if (issuer && ok && j >= 1 && j + 2 < nj) load_kv(j + 2);   // into block j-1's stage
            if (__syncthreads_or(!cok)) { status_bits |= kStatusTmaWait; failed = true; break; }
            if (issuer && !last) { q_pending &= ~(1u << (j + 1)); ++kv_done[(j + 1) % NS]; }
            if (__syncthreads_or(!ok)) { status_bits |= kStatusMmaWait; failed = true; break; }
        }
        if (worker) {   // causal mask, bf16 scores: thread (t, hh) holds key columns hh*64..hh*64+63
            const int t = r;
            float xs[2][32];
            tmem_ld32(tlane + L::COL_PA + hh * 64, xs[0]);
            tmem_ld32(tlane + L::COL_PA + hh * 64 + 32, xs[1]);
            tmem_ld_wait();
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int i0 = hh * 64 + 32 * b;
                float* x = xs[b];
                if (DECAY) {
                    // gamma^(t-i), walking down from the diagonal (factors <= 1)
                    float f = (t >= i0 + 31) ? ex2(static_cast<float>(t - i0 - 31) * lg) : 1.f;
#pragma unroll
                    for (int i = 31; i >= 0; --i) {
                        if (i0 + i <= t) {
                            x[i] *= f;
                            f *= gam;
                        } else {
                            x[i] = 0.f;
                        }
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i0 + i > t) x[i] = 0.f;
                }
                store_row32_bf16(aP + hh * 16384, t, 4 * b, x);
            }
        }
        if (DECAY) {
            if (j > 0) {   // the state entering block j: gamma^L X + A_{j-1}
                const float gL = ex2(static_cast<float>(B) * lg);   // block j-1 was full
#pragma unroll
                for (int i = 0; i < 32; ++i) R[i] *= gL;
                read_a(96 * j);
                write_state_tile(R);
            }
            if (worker) {   // phi(Q_j) rows by gamma^(t+1), phi(K_j) rows by gamma^(L-1-i)
                const int nvalid = min(B, p.T - (j0 + j) * B);
                const uint32_t aQ = sbase + L::Q + j * 16384, aK = sbase + L::STG + (j % NS) * L::STAGE;
                uint4 uq[4], uk[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int e = tid + kWorkers * i;
                    uq[i] = ld_shared_v4(aQ + 16 * e);
                    uk[i] = ld_shared_v4(aK + 16 * e);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int e = tid + kWorkers * i, row = e >> 3;
                    const float fq = ex2(static_cast<float>(row + 1) * lg);
                    const float fk = row < nvalid ? ex2(static_cast<float>(nvalid - 1 - row) * lg) : 0.f;
                    const float2 a0 = unpack_bf16(uq[i].x), a1 = unpack_bf16(uq[i].y), a2 = unpack_bf16(uq[i].z),
                                 a3 = unpack_bf16(uq[i].w);
                    const float2 b0 = unpack_bf16(uk[i].x), b1 = unpack_bf16(uk[i].y), b2 = unpack_bf16(uk[i].z),
                                 b3 = unpack_bf16(uk[i].w);
                    st_shared_v4(aQ + 16 * e, pack_bf16(a0.x * fq, a0.y * fq), pack_bf16(a1.x * fq, a1.y * fq),
                                 pack_bf16(a2.x * fq, a2.y * fq), pack_bf16(a3.x * fq, a3.y * fq));
                    st_shared_v4(aK + 16 * e, pack_bf16(b0.x * fk, b0.y * fk), pack_bf16(b1.x * fk, b1.y * fk),
                                 pack_bf16(b2.x * fk, b2.y * fk), pack_bf16(b3.x * fk, b3.y * fk));
                }
            }
        } else if (!last) {   // the state entering block j+1
            read_a(96 * (j + 1));
            write_state_tile(R);
        }
        sync_mma();
        if (issuer) {
            issue_batch2(j);
            if (!last) issue_batch1(j + 1);
        }
    }

    // ---- the segment's total, the state entering it, and the outputs
    if (!failed) {
        const bool ok = !worker || mbar_wait(&bar[kBarO], (nj - 1) & 1, kWaitLimitNs);
        tc_fence_after();
        if (__syncthreads_or(!ok)) { status_bits |= kStatusMmaWait; failed = true; }
    }
    if (!failed) {
        if (DECAY) {
            const int nvalid = min(B, p.T - (j0 + nj - 1) * B);
            const float gL = ex2(static_cast<float>(nvalid) * lg);
#pragma unroll
            for (int i = 0; i < 32; ++i) R[i] *= gL;
            read_a(96 * nj);
        } else {
            read_a(L::COL_PA);
        }
    }
    // this CTA's total in the score area as [16 column groups][65 rows][4]
    // floats (rows 0..63 X, row 64 z; a warp's 16-byte accesses fall on
    // consecutive addresses) and whether it is valid
    const uint32_t aTOT = sbase + L::P, aIN = sbase + L::STG;
    float* tot = reinterpret_cast<float*>(sm + L::P);
    if (!failed && (rowv || (rowz && lane == 0))) {
        const int row = rowv ? r : D;
#pragma unroll
        for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(tot + ((hh * 8 + i / 4) * (D + 1) + row) * 4) =
                make_float4(R[i], R[i + 1], R[i + 2], R[i + 3]);
    }
    if (tid == 0) tot[SSZ] = failed ? 0.f : 1.f;
    fence_proxy_async_smem();   // the total, for the bulk copies
    __syncthreads();
    cluster_wait();   // every CTA of the cluster has its barriers initialized
    if (issuer) {
        // this CTA's stage area is free: the predecessors may send their totals
        for (int s2 = 0; s2 < sg; ++s2) mbar_arrive_remote(mapa_cluster(smem_u32(&bar[kBarReady]), s2));
        if (nsucc > 0) {
            if (mbar_wait(&bar[kBarReady], 0, kWaitLimitNs)) {
                for (int d = p.nseg - 1; d > sg; --d)   // the last segment, which waits on the most, first
                    bulk_push_cluster(mapa_cluster(aIN + sg * kTotBytes, d), aTOT, kTotBytes,
                                      mapa_cluster(smem_u32(&bar[kBarInbox]), d));
            } else {
                status_bits |= kStatusFlagWait;
            }
        }
    }
    float Sin[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) Sin[i] = 0.f;
    if (sg > 0) {
        // the predecessors' totals (each arrives whether or not it is valid)
        bool ok = mbar_wait(&bar[kBarInbox], 0, kWaitLimitNs);
        if (issuer)   // the predecessors' copies are done with their shared memory
            for (int s2 = 0; s2 < sg; ++s2) mbar_arrive_remote(mapa_cluster(smem_u32(&bar[kBarDone]), s2));
        if (ok && tid < sg) ok = reinterpret_cast<const float*>(sm + L::STG + tid * kTotBytes)[SSZ] != 0.f;
        if (__syncthreads_or(!ok) && !failed) { status_bits |= kStatusFlagWait; failed = true; }
        if (!failed && (rowv || rowz)) {
            const uint32_t off = aIN + (hh * 8 * (D + 1) + (rowv ? r : D)) * 16;   // z follows the D rows of X
            for (int s2 = 0; s2 < sg; ++s2) {
                // decayed: over the (sg - s2 - 1) full segments between them
                const float w = DECAY ? ex2(static_cast<float>((sg - s2 - 1) * p.per * B) * lg) : 1.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint4 u = ld_shared_v4(off + s2 * kTotBytes + i * (D + 1) * 16);
                    Sin[4 * i] += w * __uint_as_float(u.x);
                    Sin[4 * i + 1] += w * __uint_as_float(u.y);
                    Sin[4 * i + 2] += w * __uint_as_float(u.z);
                    Sin[4 * i + 3] += w * __uint_as_float(u.w);
                }
            }
            write_state_tile(Sin);   // the last batch 1 that read the tile is done
        }
        if (DECAY && !failed && worker) {   // block j's tokens are 128 j further from the segment's start
            for (int jj = 1; jj < nj; ++jj) {
                const float f = ex2(static_cast<float>(B * jj) * lg);
                for (int e = tid; e < 1024; e += kWorkers) chunk::scale_chunk(sbase + L::Q + jj * 16384 + 16 * e, f);
            }
        }
        if (!failed) {
            sync_mma();
            if (issuer) {   // O_j += phi(Q_j) [X_in | z_in]^T
                for (int jj = 0; jj < nj; ++jj)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16_ss(tmem + 96 * jj, kmaj(sbase + L::Q + jj * 16384 + kk * 32), kmaj(aX + kk * 32), ID_O, 1);
                mma_commit(&bar[kBarFin]);
            }
            const bool ok2 = !worker || mbar_wait(&bar[kBarFin], 0, kWaitLimitNs);
            tc_fence_after();
            if (__syncthreads_or(!ok2)) { status_bits |= kStatusMmaWait; failed = true; }
        }
    }
    if (!failed && sg + 1 == p.nseg && p.state_out && (rowv || (rowz && lane == 0))) {
        float* so = p.state_out + static_cast<size_t>(bh) * SSZ;
        const float gS = DECAY ? ex2(static_cast<float>(min(p.T, (j0 + nj) * B) - j0 * B) * lg) : 1.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float v = R[i] + gS * Sin[i];
            if (rowv) so[(hh * 32 + i) * D + r] = v;
            else so[D * D + hh * 32 + i] = v;
        }
    }
    if (!failed) {
        // outputs: column 64 of O_j is the normalizer; tiles where phi(Q) was
        for (int jj = 0; jj < nj && worker; ++jj) {
            const int t0 = (j0 + jj) * B;
            float x[32], dn[16];
            tmem_ld32(tlane + 96 * jj + hh * 32, x);
            tmem_ld16(tlane + 96 * jj + 64, dn);
            tmem_ld_wait();
            const float inv = __fdividef(1.f, dn[0]);
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] *= inv;
            store_row32_bf16(sbase + L::Q + jj * 16384, r, 4 * hh, x);
            if (p.den_out && hh == 0 && t0 + r < p.T) p.den_out[static_cast<size_t>(bh) * p.T + t0 + r] = dn[0];
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (issuer) {
            for (int jj = 0; jj < nj; ++jj) {
                const int t0 = (j0 + jj) * B;
                tma_store_3d(&tmo, sm + L::Q + jj * 16384, 0, t0, bh);
                if (t0 + 64 < p.T) tma_store_3d(&tmo, sm + L::Q + jj * 16384 + 8192, 0, t0 + 64, bh);
            }
            bulk_commit();
        }
    }
    if (issuer && nsucc > 0) mbar_wait(&bar[kBarDone], 0, kWaitLimitNs);   // no CTA leaves before its total arrived
    if (failed && issuer) {   // let loads and MMAs in flight finish before the CTA exits
        for (int jj = 0; jj < kMaxSub; ++jj)
            if (q_pending & (1u << jj)) mbar_wait(&bar[kBarQ + jj], 0, 100000000ull);
        for (int s2 = 0; s2 < NS; ++s2)   // at most one load per stage is outstanding
            if (kv_iss[s2] > kv_done[s2]) mbar_wait(&bar[kBarLd + s2], (kv_iss[s2] - 1) & 1, 100000000ull);
        mma_commit(&bar[kBarHook]);   // phase 0 of this barrier is never completed otherwise
        mbar_wait(&bar[kBarHook], 0, 100000000ull);
    }
    if (issuer) bulk_wait_read_all();   // the output tiles have left shared memory
    // No CTA leaves the cluster while another may still reach its shared
    // memory: a successor whose inbox wait ran out may yet arrive remotely on
    // this CTA's barriers. Every wait above is bounded, so every CTA gets here.
    cluster_arrive_release();
    cluster_wait();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
    if (status_bits && tid == 0) atomicOr(p.status, status_bits);
}

// The split of one sequence-head into segments: as many as the SMs hold side
// by side (at most kMaxSeg, one cluster), each at most kMaxSub blocks.
struct Split {
    int nsub, nseg, per;
};
bool split(int BH, int T, int sm_count, Split* out) {
    const int nsub = (T + B - 1) / B;
    int nseg = sm_count / BH;
    if (nseg < 1) nseg = 1;
    if (nseg > kMaxSeg) nseg = kMaxSeg;
    if (nseg > nsub) nseg = nsub;
    const int per = (nsub + nseg - 1) / nseg;
    if (per > kMaxSub) return false;
    out->nsub = nsub;
    out->per = per;
    out->nseg = (nsub + per - 1) / per;
    return true;
}

}  // namespace seg

namespace chunk {

bool seg_fits(int BH, int T, int dk, int dv, int sm_count) {   // with or without a fixed decay
    seg::Split sp;
    return dk == seg::D && dv == seg::D && seg::split(BH, T, sm_count, &sp);
}

cudaError_t launch_seg(const FwdArgs& a, const Maps& m, cudaStream_t s) {
    seg::Split sp;
    if (!seg::split(a.BH, a.T, a.sm_count, &sp)) return cudaErrorInvalidValue;
    seg::Params p;
    p.gamma = a.gate;   // the normalized variant's fixed decay, or NULL
    p.state_in = a.state_in;
    p.state_out = a.state_out;
    p.den_out = a.den_out;
    p.BH = a.BH;
    p.T = a.T;
    p.nsub = sp.nsub;
    p.nseg = sp.nseg;
    p.per = sp.per;
    p.flags = a.flags;
    p.status = a.status;
    auto kern = a.gate ? seg::seg_kernel<true> : seg::seg_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, seg::Layout::SMEM);
    if (e != cudaSuccess) return e;
    if (a.nlaunch) *a.nlaunch += 1;
    const unsigned grid = static_cast<unsigned>(a.BH) * sp.nseg;
    return launch_cluster(kern, grid, static_cast<unsigned>(sp.nseg), seg::kThreads, seg::Layout::SMEM, s, m.q, m.k,
                          m.v, m.o, p);
}

}  // namespace chunk
}  // namespace la
