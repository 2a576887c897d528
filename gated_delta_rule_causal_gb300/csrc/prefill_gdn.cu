// Chunkwise prefill of the gated delta rule on the tcgen05 tensor cores.
//
// Recurrence ("Beyond attention" §18.2, with the decay applied to the state
// before the error is taken): S_t = g_t S_{t-1} (I - beta_t k_t k_t^T) +
// beta_t v_t k_t^T, o_t = S_t q_t. The state is held as X = S [d_v][d_k].
//
// Chunk algebra (C = 64 tokens; G_t = sum of log2 g inside the chunk up to t,
// gam_t = 2^G_t, gam_C = gam_63). Writing S_t = gam_t S_0 +
// sum_{j<=t} (gam_t/gam_j) u_j k_j^T gives (I + A) U = diag(beta) V -
// diag(beta gam) K S_0^T with A_tj = beta_t (gam_t/gam_j) k_t.k_j (j < t).
// With T = (I + A)^{-1}, Ut = T diag(beta) V and W = T diag(beta gam) K:
//    U^T = Ut^T - X_0 W^T
//    O^T = X_0 Q^T diag(gam) + U^T P^T,       P_tj = (gam_t/gam_j) q_t.k_j (j <= t)
//    X   = gam_C X_0 + U^T diag(gam_C/gam) K
// Everything but these three lines is independent of the state.
//
// Work split. One cooperative launch per group of up to 32 sequence-heads
// runs two kinds of CTA, all resident at once:
//  * prep CTAs, in parallel over (head, chunk) units taken chunk by chunk:
//    gate prefix sums, [K;Q] K^T on the tensor cores, A and P, the
//    triangular inverse T in fp32 (16x16 diagonal blocks by forward
//    substitution, then two merge levels as warp-level tf32 MMAs), W^T and
//    Ut^T on the tensor cores. Each chunk's results ("slot": W^T, Ut^T, P as
//    bf16 MMA operands and the gate factors) go with one bulk copy to a ring
//    of R chunks per head in the workspace.
//  * chain CTAs, one per sequence-head, walking its whole sequence with the
//    fp32 state in registers: per chunk the MMAs X_0 W^T and X_0 Q^T, then
//    U^T K' and U^T P^T, and three short conversions (U, the state, the
//    output). One control warp issues every copy and MMA; eight warps
//    convert. They hand work to each other through mbarriers, so that no
//    converting thread ever waits on an issue queue.
// The two kinds hand the ring over through flags in global memory: a prep CTA
// raises a chunk's ready flag once its slot store has completed, and stores
// into a ring position only after the chain CTA has loaded the chunk R
// before it (its consumed count). Every wait on a flag is bounded, and a CTA
// that gives up raises the launch's abort word so the others stop waiting.
//
// The output is formed transposed (value rows on the 128 tensor-memory
// lanes, tokens on 64 columns) so that no product pads 64 tokens to M = 128;
// the epilogue writes it straight to global memory, two adjacent values per
// 32-bit store.
//
// Tail chunks: TMA zero-fills rows past T; padded tokens have g = 1 and
// beta = 0, which makes their rows of A, W and Ut zero, so they leave the
// state untouched; no output row past T is written.
//
// Per-channel decay (the KDA form of the rule, "Linear attention and
// recurrent memory", from fixed decay to KDA: S_t = S_{t-1} Diag(alpha_t)
// (I - beta_t k_t k_t^T) + beta_t v_t k_t^T). With Gam_t = the per-channel
// product of alpha inside the chunk up to t (a d_k vector), the same
// derivation gives
//    A_tj = beta_t (k_t o Gam_t).(k_j / Gam_j),   W = T diag(beta) (K o Gam)
//    O^T  = X_0 (Q o Gam)^T + U^T P^T,           P_tj = (q_t o Gam_t).(k_j / Gam_j)
//    X    = X_0 Diag(Gam_C) + U^T (K o Gam_C / Gam)
// A ratio Gam_t / Gam_j is never formed across a whole chunk: inside each
// 16-token sub-chunk a the factors are taken relative to a reference token
// (the 8th of the sub-chunk, cumulative log2 r_a), so the row operand
// [K;Q] o 2^(G_t - r_a) and the column operand K o 2^(r_a - G_j) of the
// pair products span at most eight tokens of decay each; columns of later
// sub-chunks b > a(j) use 2^(r_b - G_j) <= 1. Every other factor (Gam_t,
// Gam_C / Gam_t, Gam_C) is at most 1. A per-token decay below 2^-15 is
// taken as 2^-15, which keeps eight tokens of decay within 2^120: the
// factors are exact in fp32 for every decay, and the only departure from the
// recurrence is that what crosses a token of decay alpha < 2^-15 is scaled
// by 2^-15 instead of alpha. The prep CTAs write Q o Gam and K o Gam_C / Gam
// into the slot, so the chain CTAs load no q or k tiles of their own.
//
// Per-channel gated attention (GLA / RetNet family, "Linear attention and
// Hyena" 11.3: S_t = diag(gamma_t) S_{t-1} + phi(k_t) v_t^T) is the same
// per-channel chunk algebra without the delta rule: T = I, W = 0, so
// Ut = V, N_c = 0 and E_c = (phi(Q) o Gam)^T. It runs through the prep CTAs
// of the per-channel decay (no inverse) and the chain CTAs with the state
// product X_c E_c alone.
#include <atomic>

#include "prefill.h"
#include "prefill_impl.cuh"
#include "launch.cuh"

namespace la {
namespace gdn {

using chunk::C;
using chunk::elu1;
using chunk::kAStride;
using chunk::kmaj;
using chunk::ld_shared_bf16;
using chunk::ld_shared_v4;
using chunk::mnmaj;
using chunk::st_shared_v4;
using chunk::store_row32_bf16;

constexpr int kConv = 256;              // converting threads (8 warps)
constexpr int kThreads = kConv + 64;    // + a control warp and a flag warp (chain CTAs)
constexpr uint32_t kBarConv = 1;        // named barrier of the converting warps
constexpr uint32_t kBarInit = 2;        // prep CTAs: converting warps and the store warp, once
constexpr int kIssuer = 64;             // prep CTAs: the thread issuing the first MMA of a unit

__host__ __device__ constexpr uint32_t align1024(uint32_t x) { return (x + 1023u) & ~1023u; }
constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// One chunk's intermediates, byte-identical in the workspace and in shared
// memory. Tiles are bf16 with the 128-byte swizzle (1024-aligned offsets).
// The same layout serves both decays (with a scalar gate Gam_t = gam_t on
// every channel). With N_c = W^T K' and E_c = QG^T - W^T P^T the chunk's
// effect on the state and its output are affine in X_0:
//    X   = X_0 Diag(Gam_C) + Ut^T K' - X_0 N_c
//    O^T = Ut^T P^T + X_0 E_c
// so the chain needs no U^T = Ut^T - X_0 W^T of its own.
template <int DK, int DV>
struct Slot {
    static constexpr int KA = DK / 64;
    static constexpr uint32_t NC_OFF = 0;                   // -N_c [DK c][DK c']: MN-major B, KA atoms of [DK][64]
    static constexpr uint32_t E_OFF = DK * DK * 2;          // E_c  [DK c][64 t]: MN-major B
    static constexpr uint32_t U_OFF = E_OFF + DK * 128;     // Ut^T [DV][64 j]: K-major A
    static constexpr uint32_t KP_OFF = U_OFF + DV * 128;    // K' = K o Gam_C/Gam [64 j][DK]: MN-major B, KA atoms of 8 KB
    static constexpr uint32_t P_OFF = KP_OFF + KA * 8192;   // P [64 t][64 j]: K-major B
    static constexpr uint32_t TILES = P_OFF + 8192;
    static constexpr uint32_t V_OFF = TILES;                // Gam_C [DK] (fp32)
    static constexpr uint32_t BYTES = V_OFF + 512;
    // The chain loads the slot in two parts: B = [-N_c | E_c] (read by the
    // state product) and A = the rest (read by the products issued earlier).
    static constexpr uint32_t B_BYTES = U_OFF;
    static constexpr uint32_t A_BYTES = BYTES - U_OFF;
    static_assert(TILES % 1024 == 0 && BYTES % 16 == 0, "tile alignment, bulk copy sizes");
};

template <int DK, int DV>
struct ChainLayout {
    static constexpr int KA = DK / 64;
    using S = Slot<DK, DV>;
    static constexpr uint32_t STAGE = S::TILES;                 // the slot's tiles, per stage
    static constexpr uint32_t OFF_VEC = 2 * STAGE;              // the slot's vector, per stage (512 B)
    static constexpr uint32_t OFF_OT = OFF_VEC + 1024;          // output tile bf16 [64 t][DV] for the TMA store
    static constexpr uint32_t OFF_BAR = OFF_OT + DV * 128;
    static constexpr uint32_t BYTES = OFF_BAR + 256;
    // TMEM columns (lanes = value rows); buffer b = chunk & 1
    static constexpr uint32_t COL_S = 0;        // Ut^T K' - X_0 N_c   [dv][DK], two buffers 128 apart
    static constexpr uint32_t COL_O = 256;      // Ut^T P^T + X_0 E_c  [dv][64], two buffers 64 apart
    // X_c as the bf16 A operand of the state product [dv rows][DK / 2
    // columns], after buffer 0's S and O
    static constexpr uint32_t COL_A = DK + 64;
    static_assert(COL_A + DK / 2 <= 256, "the A operand fits before buffer 1");
    static constexpr uint32_t TMEM_COLS = 512;
};

template <int DK, int DV>
struct PrepLayout {
    static constexpr int KA = DK / 64;
    static constexpr int VA = DV / 64;
    using S = Slot<DK, DV>;
    static constexpr uint32_t QK_BYTES = KA * 16384;    // per k-atom: rows 0-63 k, rows 64-127 q
    static constexpr uint32_t V_BYTES = VA * 8192;
    static constexpr uint32_t STAGE = QK_BYTES + V_BYTES;
    static constexpr uint32_t TX = STAGE;
    static constexpr uint32_t OFF_TB1 = 2 * STAGE;       // T diag(beta)     bf16 [t][j]
    static constexpr uint32_t OFF_TB2 = OFF_TB1 + 8192;  // T diag(beta gam) bf16 [t][j]
    static constexpr uint32_t OFF_OUT = OFF_TB2 + 8192;  // the slot being assembled / stored
    static constexpr uint32_t OFF_AS = OFF_OUT + align1024(S::BYTES);   // fp32 [64][kAStride]
    static constexpr uint32_t OFF_RS = OFF_AS + C * kAStride * 4;       // fp32 [32][kRStride]
    // two gate buffers (units k and k + 1), each: log2 prefix, beta, beta gam, gam
    static constexpr uint32_t OFF_MISC = OFF_RS + 32 * 40 * 4;
    static constexpr uint32_t OFF_BAR = OFF_MISC + 2 * 4 * 64 * 4;
    static constexpr uint32_t BYTES = OFF_BAR + 128;
    // W^T as a bf16 K-major A operand [dk][64 j] goes over the solve matrix,
    // which is dead by then
    static constexpr uint32_t OFF_WT = OFF_AS;
    static_assert(DK * 128 <= C * kAStride * 4, "W^T fits over the solve matrix");
    static constexpr uint32_t COL_G = 0;     // [K;Q] K^T  [128][64]
    static constexpr uint32_t COL_W = 64;    // W^T        [dk][64]
    static constexpr uint32_t COL_UT = 128;  // Ut^T       [dv][64]
    static constexpr uint32_t COL_N = 192;   // -W^T K'    [dk][DK]
    static constexpr uint32_t COL_E = 320;   // W^T P^T    [dk][64]
    static constexpr uint32_t TMEM_COLS = 512;
};
constexpr int kRStride = 40;   // fp32 row stride of the merge scratch (conflict-free fragment reads)

// Prep CTA of the per-channel decay. [K;Q] is double-buffered and rescaled
// in place into the row operand; V, the fp32 gate tile and the outgoing slot
// are single-buffered (V and the gates of the next unit are loaded once the
// MMAs that read their buffer are done; the slot store of the previous unit
// has drained before the buffer is written again). The column operands of
// the four sub-chunks (16, 32, 48, 64 rows) are stacked into one 160-row
// operand, written over the gate tile and TB1, both of which are dead while
// it lives.
template <int DK, int DV>
struct PrepLayoutKda {
    static constexpr int KA = DK / 64;
    static constexpr int VA = DV / 64;
    using S = Slot<DK, DV>;
    static constexpr uint32_t QK_BYTES = KA * 16384;     // per k-atom: rows 0-63 k, rows 64-127 q
    static constexpr uint32_t OFF_V = QK_BYTES;          // V [64 t][DV]
    static constexpr uint32_t OFF_GATE = OFF_V + VA * 8192;   // alpha fp32 [64 t][DK]
    static constexpr uint32_t OFF_TB1 = OFF_GATE + DK * 256;  // T diag(beta) bf16 [t][j]
    static constexpr uint32_t OFF_B = OFF_GATE;               // column operands, over gate + TB1
    static constexpr uint32_t B_ATOM = 160 * 128;             // 160 rows of one 64-channel atom
    static constexpr uint32_t B_BYTES = B_ATOM * KA;
    static_assert(B_BYTES <= DK * 256 + 8192, "column operands fit over the gate tile and TB1");
    static constexpr uint32_t OFF_OUT = align1024(OFF_TB1 + 8192);
    static constexpr uint32_t OFF_AS = OFF_OUT + align1024(S::BYTES);   // fp32 [64][kAStride]
    static constexpr uint32_t OFF_RS = OFF_AS + C * kAStride * 4;        // fp32 [32][kRStride]
    static constexpr uint32_t OFF_BLK = OFF_RS + 32 * 40 * 4;            // log2-gate sums of 8-token blocks [8][DK]
    static constexpr uint32_t OFF_MISC = OFF_BLK + 8 * DK * 4;           // beta [64], next unit's beta [64]
    static constexpr uint32_t OFF_BAR = OFF_MISC + 2 * 64 * 4;
    static constexpr uint32_t BYTES = OFF_BAR + 128;
    // W^T as a bf16 K-major A operand goes over the solve matrix (dead by
    // then); K o Gam (the W product's operand) and Q o Gam wait in the slot
    // buffer's -N_c and E_c tiles until those are written.
    static constexpr uint32_t OFF_WT = OFF_AS;
    static_assert(DK * 128 <= C * kAStride * 4, "W^T fits over the solve matrix");
    // First row (and product column) of sub-chunk a's column operand: its
    // rows j < 16(a+1) follow the operands of the sub-chunks before it.
    static __host__ __device__ constexpr int b_row(int a) { return 8 * a * (a + 1); }
    static constexpr uint32_t COL_G = 0;     // [K;Q] B^T, 160 columns (block a at b_row(a))
    static constexpr uint32_t COL_W = 160;   // W^T    [dk][64]
    static constexpr uint32_t COL_UT = 224;  // Ut^T   [dv][64]
    static constexpr uint32_t COL_N = 288;   // -W^T K' [dk][DK]
    static constexpr uint32_t COL_E = 416;   // W^T P^T [dk][64]
    static constexpr uint32_t TMEM_COLS = 512;
};

// MODE: 0 = scalar gate (gated delta rule), 1 = per-channel decay delta rule,
// 2 = per-channel gated attention without the delta rule.
template <int DK, int DV, int MODE>
constexpr uint32_t smem_alloc() {
    constexpr uint32_t prep = MODE ? PrepLayoutKda<DK, DV>::BYTES : PrepLayout<DK, DV>::BYTES;
    constexpr uint32_t chain = ChainLayout<DK, DV>::BYTES;
    return (chain > prep ? chain : prep) + 1024;
}

struct Params {
    const float* gate;      // [BH, T]; per-channel decay: [BH, T, DK]
    const float* beta;      // [BH, T]
    const float* state_in;  // [BH, DV, DK] or NULL (zeros)
    float* state_out;       // [BH, DV, DK] or NULL
    __nv_bfloat16* out;     // [BH, T, DV]
    uint8_t* ws_slot;       // [G][R] slots: ring of the chunks of each sequence-head
    // Hand-off flags (each value = epoch | count): ready[G*R] (chunk c's
    // slot stored: c + 1), then per head consumed[G] at a stride of 16 words
    // (chunks whose slot the chain has loaded), then the abort word (= epoch
    // once a CTA of this launch gave up).
    unsigned long long* ws_flag;
    unsigned long long epoch;   // this launch's epoch, in the upper 32 bits
    int T;
    int nch;                // chunks per sequence
    int h0;                 // first sequence-head of the group
    int G;                  // sequence-heads in the group
    int R;                  // ring depth in chunks
    int n_chain;            // CTAs [0, n_chain) walk the chain, the others prepare
    unsigned flags;
    int* status;
    __device__ unsigned long long* ready(int g, int c) const { return ws_flag + static_cast<size_t>(g) * R + c % R; }
    __device__ unsigned long long* consumed(int g) const { return ws_flag + static_cast<size_t>(G) * R + 16 * g; }
    __device__ unsigned long long* abort_word() const { return ws_flag + static_cast<size_t>(G) * R + 16 * G; }
    __device__ void abort_all() const {
        *reinterpret_cast<volatile unsigned long long*>(abort_word()) = epoch;
    }
    __device__ bool wait_flag(const unsigned long long* f, unsigned long long count) const {
        return flag_wait(f, epoch | count, abort_word(), epoch);
    }
};
// Flag words the launcher reserves in front of the slots (ready, consumed, abort).
constexpr size_t flag_words(int G, int R) { return static_cast<size_t>(G) * R + 16 * (G + 1); }

__device__ __forceinline__ void st_shared_v4_u4(uint32_t addr, uint4 v) { st_shared_v4(addr, v.x, v.y, v.z, v.w); }
// Eight bf16 values scaled by f, rounded back to bf16.
__device__ __forceinline__ uint4 scale_bf16x8(uint4 u, float f) {
    const float2 a = unpack_bf16(u.x), b = unpack_bf16(u.y), c = unpack_bf16(u.z), d = unpack_bf16(u.w);
    return make_uint4(pack_bf16(a.x * f, a.y * f), pack_bf16(b.x * f, b.y * f), pack_bf16(c.x * f, c.y * f),
                      pack_bf16(d.x * f, d.y * f));
}
__device__ __forceinline__ uint32_t ld_shared_b32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_shared_b32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// ============================================================================
// chain CTA: the state-dependent part of every chunk of one sequence-head
// ============================================================================
// Per chunk c (buffer b = c & 1 of tensor memory, stage b of shared memory):
//   pre(c):   S_b = Ut^T K',  O_b = Ut^T P^T          (no state: issued early)
//   state(c): [S_b | O_b] += X_c [-N_c | E_c]           (one MMA chain, N = DK + 64)
//   converters: X_{c+1} = X_c Diag(Gam_C) + S_b (fp32 registers), stored as
//               the bf16 A operand in tensor memory (no shared-memory copy, no
//               async-proxy fence); o = O_b through the output tile.
// Only state(c) and the state update lie on the path from one chunk to the
// next.
// GLA: the per-channel gated variant without the delta rule. N_c = 0, so the
// state product is X_c E_c alone and part B of the slot is E_c; the state is
// read and written in that variant's orientation S = X^T [DK][DV].
template <int DK, int DV, bool GLA>
__device__ __forceinline__ void chain_role(const CUtensorMap* tmo, const Params& p, uint8_t* sm, uint32_t sbase) {
    using L = ChainLayout<DK, DV>;
    using S = Slot<DK, DV>;
    constexpr int DKH = DK / 2;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool control = warp == kConv / 32;
    const bool copyw = warp == kConv / 32 + 1;
    const int r = 32 * (warp & 3) + lane;   // tensor-memory lane = value row (converting warps)
    const int hh = (warp >> 2) & 1;         // column half
    const int g = blockIdx.x;
    const int bh = p.h0 + g;
    const int n = p.nch;
    const bool own = warp < kConv / 32 && r < DV;

    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
    uint64_t* bar_full = bar;        // [2] copy warp: part A of the stage's slot (and its vector) has arrived
    uint64_t* bar_fullb = bar + 13;  // [2] copy warp: part B (-N_c, E_c) has arrived
    uint64_t* bar_donea = bar + 15;  // [2] MMA: pre(c) done, part A of stage c & 1 is read
    uint64_t* bar_s = bar + 2;       // MMA: state(c) and everything before it done
    uint64_t* bar_fin = bar + 3;     // MMA: all issued MMAs done (after a failure)
    uint64_t* bar_x = bar + 4;       // converters: X_c written          (8 arrivals)
    uint64_t* bar_ep = bar + 5;      // [2] converters: chunk c's output tile written, buffer c & 1 read (8 arrivals)
    uint64_t* bar_sfree = bar + 7;   // [2] control: state(c) done, part B of stage c & 1 is read
    uint64_t* bar_ofree = bar + 9;   // copy warp: the output tile's store has read it
    uint64_t* bar_test = bar + 10;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 11);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + 12);

    if (tid == 0) {
        mbar_init(&bar_full[0], 1);
        mbar_init(&bar_full[1], 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_fin, 1);
        mbar_init(bar_x, kConv / 32);
        mbar_init(&bar_ep[0], kConv / 32);
        mbar_init(&bar_ep[1], kConv / 32);
        mbar_init(&bar_sfree[0], 1);
        mbar_init(&bar_sfree[1], 1);
        for (int i = 13; i < 17; ++i) mbar_init(&bar[i], 1);
        mbar_init(bar_ofree, 1);
        mbar_init(bar_test, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (copyw && lane == 0) tma_prefetch_desc(tmo);
    if (warp == 0) tmem_alloc(tmem_slot, L::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);

    int status_bits = 0;
    bool failed = false;
    if (p.flags & 0x100u) {  // test hook: a wait nothing will satisfy, 1 ms limit
        const bool ok = mbar_wait(bar_test, 0, 1000000ull);
        if (__syncthreads_or(!ok)) { status_bits |= kStatusTestHook; failed = true; }
    }

    const size_t ssz = static_cast<size_t>(DK) * DV;
    constexpr uint32_t ID_K = idesc_bf16(128, DK, false, true);        // Ut^T K'
    constexpr uint32_t ID_P = idesc_bf16(128, 64, false, false);       // Ut^T P^T
    constexpr uint32_t ID_X = idesc_bf16(128, DK + 64, false, true);   // X_c [-N_c | E_c]
    constexpr uint32_t ID_E = idesc_bf16(128, 64, false, true);        // X_c E_c (GLA)
    auto col_s = [](int b) { return L::COL_S + 256u * b; };             // S_b; O_b follows at + DK

    if (control) {
        // ======================= control warp (lane 0) =========================
        // Issues every MMA. Copies belong to the copy warp.
        if (lane == 0 && !failed && n > 0) {
            bool fail = false;
            auto give_up = [&](int bit) {
                fail = true;
                status_bits |= bit;
                *abort_flag = 1;
                p.abort_all();
            };
            auto wait = [&](uint64_t* b, uint32_t parity, int bit) {
                if (fail) return;
                if (!mbar_wait_or_abort(b, parity, abort_flag)) give_up(bit);
            };
            int n_s = 0;   // commits of bar_s issued: the k-th completes phase k
            auto issue_pre = [&](int c) {
                const int b = c & 1;
                const uint32_t stg = sbase + b * L::STAGE;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ss(tmem + col_s(b), kmaj(stg + S::U_OFF + kk * 32), mnmaj(stg + S::KP_OFF + kk * 2048, 8192),
                                ID_K, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ss(tmem + col_s(b) + DK, kmaj(stg + S::U_OFF + kk * 32), kmaj(stg + S::P_OFF + kk * 32),
                                ID_P, kk > 0);
                mma_commit(&bar_donea[b]);   // part A of stage b may be reloaded once these are done
            };
            auto issue_state = [&](int c) {
                const int b = c & 1;
                const uint32_t stg = sbase + b * L::STAGE;
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    if (GLA)
                        mma_bf16_ts(tmem + col_s(b) + DK, tmem + L::COL_A + 8 * kk,
                                    mnmaj(stg + S::E_OFF + kk * 2048, 8192), ID_E, true);
                    else
                        mma_bf16_ts(tmem + col_s(b), tmem + L::COL_A + 8 * kk,
                                    mnmaj(stg + S::NC_OFF + kk * 2048, DK * 128), ID_X, true);
                }
                mma_commit(bar_s);
                ++n_s;
            };
            wait(&bar_full[0], 0, kStatusTmaWait);
            if (!fail) {
                tc_fence_after();
                issue_pre(0);
            }
            for (int it = 0; it < n && !fail; ++it) {
                wait(bar_x, it & 1, kStatusMmaWait);   // X_it published, so state(it-1) was done
                if (fail) break;
                // every MMA reading stage (it-1) & 1 finished with state(it-1):
                // the copy warp may load chunk it+1 there
                if (it >= 1 && it + 1 < n) mbar_arrive(&bar_sfree[(it - 1) & 1]);
                wait(&bar_fullb[it & 1], (it >> 1) & 1, kStatusTmaWait);
                if (fail) break;
                tc_fence_after();
                issue_state(it);
                if (it + 1 < n) {
                    // buffer (it+1) & 1: its S was read before bar_x(it), its O
                    // before chunk it-1's epilogue (bar_ep[(it-1) & 1])
                    wait(&bar_full[(it + 1) & 1], ((it + 1) >> 1) & 1, kStatusTmaWait);
                    if (it >= 1) wait(&bar_ep[(it - 1) & 1], ((it - 1) >> 1) & 1, kStatusMmaWait);
                    if (fail) break;
                    tc_fence_after();
                    issue_pre(it + 1);
                }
            }
            if (fail && n_s + (n > 0 ? 1 : 0) > 0) {
                // Let every MMA issued finish before the CTA exits (bounded:
                // 100 ms): one more commit covers them all, in issue order.
                mma_commit(bar_fin);
                mbar_wait(bar_fin, 0, 100000000ull);
            }
        }
    } else if (copyw) {
        // ======================= copy warp (lane 0) ============================
        // Keeps copies and global hand-offs off the control thread. For chunk
        // c, in order: once the ring holds the chunk (its ready flag) and
        // stage c & 1 is free (bar_sfree), loads the slot (tiles into the
        // stage, the vector beside it); hands the output tile back
        // (bar_ofree) once chunk c - 2's store has read it; then, for chunk
        // c - 1, waits for its slot to arrive and publishes the consumed count,
        // waits for its output tile (bar_ep) and stores it. Each barrier waited
        // on here can only advance one more phase after a step this warp takes
        // later, so no parity wait is ever two phases behind.
        if (lane == 0 && !failed && n > 0) {
            bool fail = false;
            bool pending[2] = {false, false}, pendb[2] = {false, false};
            int load_idx[2] = {0, 0};   // chunk of the loads last issued on each stage
            auto give_up = [&](int bit) {
                fail = true;
                status_bits |= bit;
                *abort_flag = 1;
                p.abort_all();
            };
            auto wait = [&](uint64_t* b, uint32_t parity, int bit) {
                if (fail) return;
                if (!mbar_wait_or_abort(b, parity, abort_flag)) give_up(bit);
            };
            for (int c = 0; c <= n && !fail; ++c) {
                if (c < n) {
                    // the ready flag first: it is usually up long before the
                    // stage frees, so its load latency hides behind that wait
                    const int s = c & 1;
                    if (!p.wait_flag(p.ready(g, c), static_cast<unsigned long long>(c) + 1)) {
                        give_up(kStatusFlagWait);
                        break;
                    }
                    const uint8_t* src = p.ws_slot + (static_cast<size_t>(g) * p.R + c % p.R) * S::BYTES;
                    uint8_t* stg = sm + s * L::STAGE;
                    fence_proxy_async_global();
                    // part A once pre(c - 2) has read it (long done), then part B
                    // once state(c - 2) has (relayed by the control thread)
                    if (c >= 2) wait(&bar_donea[s], ((c - 2) >> 1) & 1, kStatusMmaWait);
                    if (fail) break;
                    mbar_arrive_expect_tx(&bar_full[s], S::A_BYTES);
                    bulk_load(stg + S::U_OFF, src + S::U_OFF, S::TILES - S::U_OFF, &bar_full[s]);
                    bulk_load(sm + L::OFF_VEC + s * 512, src + S::V_OFF, 512, &bar_full[s]);
                    pending[s] = true;
                    load_idx[s] = c;
                    if (c >= 2) wait(&bar_sfree[s], ((c - 2) >> 1) & 1, kStatusMmaWait);
                    if (fail) break;
                    if (GLA) {   // part B is E_c alone
                        mbar_arrive_expect_tx(&bar_fullb[s], DK * 128);
                        bulk_load(stg + S::E_OFF, src + S::E_OFF, DK * 128, &bar_fullb[s]);
                    } else {
                        mbar_arrive_expect_tx(&bar_fullb[s], S::B_BYTES);
                        bulk_load(stg, src, S::B_BYTES, &bar_fullb[s]);
                    }
                    pendb[s] = true;
                }
                // chunk c - 2's output store (the only one in flight) has long
                // read its tile: hand it back for chunk c - 1's epilogue
                if (c >= 2) {
                    bulk_wait_read_all();
                    mbar_arrive(bar_ofree);
                }
                if (c >= 1) {
                    const int c1 = c - 1, s1 = c1 & 1;
                    wait(&bar_full[s1], (c1 >> 1) & 1, kStatusTmaWait);
                    wait(&bar_fullb[s1], (c1 >> 1) & 1, kStatusTmaWait);
                    if (fail) break;
                    pending[s1] = false;
                    pendb[s1] = false;
                    // Chunks 0..c-1 are in shared memory. The wait above
                    // (acquire) orders this store after the completed copy, so
                    // a relaxed store suffices: a release would also wait for
                    // the copy just issued.
                    st_relaxed_u64(p.consumed(g), p.epoch | static_cast<unsigned long long>(c));
                    wait(&bar_ep[s1], (c1 >> 1) & 1, kStatusMmaWait);
                    if (fail) break;
                    // rows past T are clipped by the tensor map
#pragma unroll
                    for (int a = 0; a < DV / 64; ++a) tma_store_3d(tmo, sm + L::OFF_OT + a * 8192, a * 64, c1 * C, bh);
                    bulk_commit();
                }
            }
            bulk_wait_all();   // every output store has completed
            if (fail) {
                for (int s2 = 0; s2 < 2; ++s2) {
                    if (pending[s2]) mbar_wait(&bar_full[s2], (load_idx[s2] >> 1) & 1, 100000000ull);
                    if (pendb[s2]) mbar_wait(&bar_fullb[s2], (load_idx[s2] >> 1) & 1, 100000000ull);
                }
            }
        }
    } else {
        // ======================= converting warps ==============================
        // initial state: thread (r, hh) owns X[r][hh*DK/2 .. +DK/2)
        const float* sin = p.state_in ? p.state_in + bh * ssz : nullptr;
        float st[DKH];
#pragma unroll
        for (int i = 0; i < DKH; i += 4) {
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (own && sin) {
                if (GLA) {   // S[c][r]: a warp reads 32 consecutive r of each row c
                    const float* sc = sin + static_cast<size_t>(hh * DKH + i) * DV + r;
                    x = make_float4(sc[0], sc[DV], sc[2 * DV], sc[3 * DV]);
                } else {
                    x = *reinterpret_cast<const float4*>(sin + static_cast<size_t>(r) * DK + hh * DKH + i);
                }
            }
            st[i] = x.x;
            st[i + 1] = x.y;
            st[i + 2] = x.z;
            st[i + 3] = x.w;
        }
        // The bf16 state as the A operand in tensor memory: thread (r, hh)
        // writes its DK/2 values of row r as DK/4 packed columns of lane r.
        // Rows >= d_v are written once, as zeros, before the first chunk (their
        // warps own no row after that).
        auto publish_state = [&]() {
            if constexpr (DKH == 64) {
                uint32_t u[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) u[i] = pack_bf16(st[2 * i], st[2 * i + 1]);
                tmem_st32(tlane + L::COL_A + hh * 32, u);
            } else {
                static_assert(DKH == 32, "d_k in {64, 128}");
                uint32_t u[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) u[i] = pack_bf16(st[2 * i], st[2 * i + 1]);
                tmem_st16(tlane + L::COL_A + hh * 16, u);
            }
            tmem_st_wait();
        };
        auto signal_x = [&]() {   // this warp's part of X is in tensor memory
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_x);
        };
        auto signal = [&](uint64_t* b) {   // this warp's writes / TMEM reads are done
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b);
        };
        publish_state();
        signal_x();

        bool bad = failed;
        for (int it = 0; it < n && !bad; ++it) {
            const int b = it & 1;
            // ---- X_{it+1} = X_it Diag(Gam_C) + S_b, republished ------------------
            bool ok = mbar_wait_or_abort(&bar_full[b], (it >> 1) & 1, abort_flag) &&
                      mbar_wait_or_abort(bar_s, it & 1, abort_flag);
            tc_fence_after();
            // warp-uniform before the warp-collective tensor-memory loads: a
            // wait that gives up may give up in some lanes only
            ok = __all_sync(0xffffffffu, ok);
            if (ok && own) {
                const float* vec = reinterpret_cast<const float*>(sm + L::OFF_VEC + b * 512);
#pragma unroll
                for (int b2 = 0; b2 < DKH / 32; ++b2) {
                    float x[32];
                    tmem_ld32(tlane + col_s(b) + hh * DKH + 32 * b2, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        st[32 * b2 + i] = vec[hh * DKH + 32 * b2 + i] * st[32 * b2 + i] + x[i];
                }
                publish_state();
            }
            signal_x();
            bad |= !ok;
            // ---- output: o_t = O_b[:, t], through the output tile ----------------
            ok = ok && (it == 0 || mbar_wait_or_abort(bar_ofree, (it - 1) & 1, abort_flag));
            ok = __all_sync(0xffffffffu, ok);
            if (ok && own) {
                // Lane pairs (r even, r + 1) exchange values so that each
                // writes two adjacent columns of one token row of the tile in
                // one word; the copy warp stores the tile.
                const bool odd = lane & 1;
                const int col = r & ~1;
                const uint32_t aot = sbase + L::OFF_OT + (col / 64) * 8192 + (col % 8) * 2;
                const uint32_t c8 = (col % 64) / 8;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int tb = 32 * hh + 16 * q;   // first token of these 16 columns
                    float o1[16];
                    tmem_ld16(tlane + col_s(b) + DK + tb, o1);
                    tmem_ld_wait();
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        const float send = odd ? o1[2 * m] : o1[2 * m + 1];
                        const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
                        const int t = tb + 2 * m + (odd ? 1 : 0);
                        const uint32_t w = odd ? pack_bf16(recv, o1[2 * m + 1]) : pack_bf16(o1[2 * m], recv);
                        st_shared_b32(aot + sw128_off(t, c8), w);
                    }
                }
            }
            signal(&bar_ep[b]);   // also orders the tile for the TMA store
            bad |= !ok;
        }
        // ---- the final state ---------------------------------------------------
        bad = named_sync_or(kBarConv, kConv, bad);
        if (!bad) {
            float* dst = p.state_out ? p.state_out + bh * ssz : nullptr;
            if (dst && own) {
                if (GLA) {
#pragma unroll
                    for (int i = 0; i < DKH; ++i) dst[static_cast<size_t>(hh * DKH + i) * DV + r] = st[i];
                } else {
#pragma unroll
                    for (int i = 0; i < DKH; i += 4)
                        *reinterpret_cast<float4*>(dst + static_cast<size_t>(r) * DK + hh * DKH + i) =
                            make_float4(st[i], st[i + 1], st[i + 2], st[i + 3]);
                }
            }
        } else if (tid == 0) {
            if (!failed) status_bits |= kStatusMmaWait;
            *abort_flag = 1;
            p.abort_all();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
    if (status_bits && (tid == 0 || ((control || copyw) && lane == 0))) atomicOr(p.status, status_bits);
}

// ============================================================================
// prep CTA: the state-independent part of (head, chunk) units (8 warps)
// ============================================================================
__device__ __forceinline__ void sync_conv() { named_sync(kBarConv, kConv); }

// 16x8 tile of A[r0.., k..] * B[k.., n0..] over K = 8*ksteps, A and B fp32
// row-major in shared memory (strides lda, ldb), accumulated into d.
template <int KSTEPS>
__device__ __forceinline__ void tile_mma(float (&d)[4], const float* A, int lda, int r0, int ka0, const float* B,
                                         int ldb, int kb0, int n0) {
    const int lane = threadIdx.x & 31, gq = lane >> 2, cq = lane & 3;
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
        const int ka = ka0 + 8 * ks, kb = kb0 + 8 * ks;
        uint32_t a[4], b[2];
        a[0] = to_tf32(A[(r0 + gq) * lda + ka + cq]);
        a[1] = to_tf32(A[(r0 + gq + 8) * lda + ka + cq]);
        a[2] = to_tf32(A[(r0 + gq) * lda + ka + cq + 4]);
        a[3] = to_tf32(A[(r0 + gq + 8) * lda + ka + cq + 4]);
        b[0] = to_tf32(B[(kb + cq) * ldb + n0 + gq]);
        b[1] = to_tf32(B[(kb + cq + 4) * ldb + n0 + gq]);
        mma_tf32_m16n8k8(d, a, b);
    }
}
// Store s * d (a 16x8 tile) to M[r0.., n0..] (fp32 row-major, stride ld).
__device__ __forceinline__ void tile_store(float* M, int ld, int r0, int n0, const float (&d)[4], float s) {
    const int lane = threadIdx.x & 31, gq = lane >> 2, cq = lane & 3;
    *reinterpret_cast<float2*>(M + (r0 + gq) * ld + n0 + 2 * cq) = make_float2(s * d[0], s * d[1]);
    *reinterpret_cast<float2*>(M + (r0 + gq + 8) * ld + n0 + 2 * cq) = make_float2(s * d[2], s * d[3]);
}

// T = (I + A)^{-1} in place, A strictly lower triangular in As (fp32
// [64][kAStride]); Rs is scratch. Run by the eight converting warps; every
// step ends at their named barrier.
__device__ __forceinline__ void invert_unit_lower(float* As, float* Rs, int warp, int lane) {
    // ---- T = (I + A)^{-1}: diagonal 16x16 blocks by forward substitution ------
    if (warp < 4 && lane < 16) {
        const int w0 = 16 * warp, l = lane;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float* arow = As + (w0 + i) * kAStride + w0;
            float a0 = (i == l) ? 1.f : 0.f, a1 = 0.f;
#pragma unroll
            for (int kq = 0; kq + 1 < i; kq += 2) {
                a0 -= arow[kq] * x[kq];
                a1 -= arow[kq + 1] * x[kq + 1];
            }
            if (i & 1) a0 -= arow[i - 1] * x[i - 1];
            x[i] = a0 + a1;
        }
        __syncwarp(0x0000ffffu);
#pragma unroll
        for (int i = 0; i < 16; ++i) As[(w0 + i) * kAStride + w0 + l] = x[i];
    }
    sync_conv();
    // ---- merge level 1 (warps 0-3, one 16x8 tile each):
    //      T_10 = -T_11 (A_10 T_00), T_32 = -T_33 (A_32 T_22)
    {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        const int m = warp >> 1, nt = warp & 1;
        const int rb = 16 + 32 * m, cb = 32 * m;
        float* X = Rs + warp * 16 * 8;   // 16x8, stride 8
        if (warp < 4) {
            tile_mma<2>(d, As, kAStride, rb, cb, As, kAStride, cb, cb + 8 * nt);
            tile_store(X, 8, 0, 0, d, 1.f);
        }
        sync_conv();   // every read of A_10 / A_32 precedes the overwrite below
        if (warp < 4) {
            float e[4] = {0.f, 0.f, 0.f, 0.f};
            tile_mma<2>(e, As, kAStride, rb, rb, X, 8, 0, 0);
            tile_store(As, kAStride, rb, cb + 8 * nt, e, -1.f);
        }
        sync_conv();
    }
    // ---- merge level 2 (8 warps, one 16x8 tile each):
    //      T[32:64, 0:32] = -T_B (A[32:64, 0:32] T_A)
    {
        const int mt = warp >> 2, nt = warp & 3;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        tile_mma<4>(d, As, kAStride, 32 + 16 * mt, 0, As, kAStride, 0, 8 * nt);
        tile_store(Rs, kRStride, 16 * mt, 8 * nt, d, 1.f);
        sync_conv();
        float e[4] = {0.f, 0.f, 0.f, 0.f};
        tile_mma<4>(e, As, kAStride, 32 + 16 * mt, 32, Rs, kRStride, 0, 8 * nt);
        tile_store(As, kAStride, 32 + 16 * mt, 8 * nt, e, -1.f);
        sync_conv();
    }
}

// Row r of -N_c from tensor memory (columns hh*DK/2 ..) into the slot's
// MN-major tile: the 64-column atom of column c' at c' / 64, DK rows each.
template <int DK>
__device__ __forceinline__ void store_neg_nc(uint32_t tcol, int hh, uint32_t aNC, int r) {
#pragma unroll
    for (int b2 = 0; b2 < DK / 64; ++b2) {
        float x[32];
        const int col = hh * (DK / 2) + 32 * b2;
        tmem_ld32(tcol + col, x);
        tmem_ld_wait();
        store_row32_bf16(aNC + (col / 64) * (DK * 128), r, (col % 64) / 8, x);
    }
}

// Store warp of a prep CTA (lane 0 of warp 8). For each unit of the CTA, in
// order: waits until the converting warps have assembled its slot
// (slot_full), waits until the chain has loaded the chunk R before it from
// the same ring position, stores the slot, hands the buffer back
// (slot_free) once the copy has read it, and raises the chunk's ready flag
// once the copy has completed. Keeps every global hand-off off the
// converting warps.
template <uint32_t BYTES>
__device__ __forceinline__ void store_loop(const Params& p, uint64_t* slot_full, uint64_t* slot_free,
                                           const uint8_t* out, volatile int* abort_smem, int& status_bits) {
    const int pid = blockIdx.x - p.n_chain, np = gridDim.x - p.n_chain, nunits = p.G * p.nch;
    for (int k = 0;; ++k) {
        const int u = pid + k * np;
        if (u >= nunits) break;
        if (!mbar_wait_or_abort(slot_full, k & 1, abort_smem)) {
            if (!*abort_smem) status_bits |= kStatusFlagWait;   // else the converting warps recorded it
            break;
        }
        const int g = u % p.G, c = u / p.G;
        if (c >= p.R && !p.wait_flag(p.consumed(g), static_cast<unsigned long long>(c - p.R) + 1)) {
            status_bits |= kStatusFlagWait;
            *abort_smem = 1;
            p.abort_all();
            break;
        }
        uint8_t* dst = p.ws_slot + (static_cast<size_t>(g) * p.R + c % p.R) * BYTES;
        bulk_store(dst, smem_u32(out), BYTES);
        bulk_commit();
        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        mbar_arrive(slot_free);
        bulk_wait_all();
        fence_proxy_async_global();
        st_release_u64(p.ready(g, c), p.epoch | (static_cast<unsigned long long>(c) + 1));
    }
    bulk_wait_all();
}

// Gate preparation of one unit by the whole store warp (scalar decay): lane l
// takes tokens 2l and 2l + 1 and writes, into gate buffer gb ([4][64] floats),
// the cumulative log2 gate G_t, beta_t (0 on padded tokens), beta_t gam_t
// and gam_t = 2^G_t; then every lane arrives on gates_full (32 arrivals).
__device__ __forceinline__ void prepare_gates(const Params& p, int u, float* gb, uint64_t* gates_full) {
    const int lane = threadIdx.x & 31;
    const int bh = p.h0 + u % p.G;
    const int t0 = (u / p.G) * C + 2 * lane;
    const size_t base = static_cast<size_t>(bh) * p.T;
    float g0 = 1.f, g1 = 1.f, b0 = 0.f, b1 = 0.f;
    if (t0 < p.T) { g0 = __ldg(p.gate + base + t0); b0 = __ldg(p.beta + base + t0); }
    if (t0 + 1 < p.T) { g1 = __ldg(p.gate + base + t0 + 1); b1 = __ldg(p.beta + base + t0 + 1); }
    const float l0 = lg2(g0), l1 = lg2(g1);
    float sum = l0 + l1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, sum, o);
        if (lane >= o) sum += y;
    }
    const float G0 = sum - l1, G1 = sum;   // inclusive prefix at tokens 2l, 2l + 1
    const float gam0 = ex2(G0), gam1 = ex2(G1);
    *reinterpret_cast<float2*>(gb + 2 * lane) = make_float2(G0, G1);
    *reinterpret_cast<float2*>(gb + 64 + 2 * lane) = make_float2(b0, b1);
    *reinterpret_cast<float2*>(gb + 128 + 2 * lane) = make_float2(b0 * gam0, b1 * gam1);
    *reinterpret_cast<float2*>(gb + 192 + 2 * lane) = make_float2(gam0, gam1);
    mbar_arrive(gates_full);   // release: this lane's writes precede the waiters' reads
}

// Store warp of a scalar-decay prep CTA (all 32 lanes): prepares the gates of
// the CTA's first unit, then per unit k prepares unit k + 1's gates (into the
// buffer unit k - 1 used, free since its slot was assembled) and stores unit
// k's slot (lane 0, as store_loop does).
template <uint32_t BYTES>
__device__ __forceinline__ void store_gate_loop(const Params& p, uint64_t* slot_full, uint64_t* slot_free,
                                                uint64_t* gates_full, float* gbuf, const uint8_t* out,
                                                volatile int* abort_smem, int& status_bits) {
    const int lane = threadIdx.x & 31;
    const int pid = blockIdx.x - p.n_chain, np = gridDim.x - p.n_chain, nunits = p.G * p.nch;
    if (pid < nunits) prepare_gates(p, pid, gbuf, &gates_full[0]);
    for (int k = 0;; ++k) {
        const int u = pid + k * np;
        if (u >= nunits) break;
        if (u + np < nunits) prepare_gates(p, u + np, gbuf + ((k + 1) & 1) * 256, &gates_full[(k + 1) & 1]);
        bool stop = false;
        if (lane == 0) {
            if (!mbar_wait_or_abort(slot_full, k & 1, abort_smem)) {
                if (!*abort_smem) status_bits |= kStatusFlagWait;   // else the converting warps recorded it
                stop = true;
            }
            const int g = u % p.G, c = u / p.G;
            if (!stop && c >= p.R && !p.wait_flag(p.consumed(g), static_cast<unsigned long long>(c - p.R) + 1)) {
                status_bits |= kStatusFlagWait;
                *abort_smem = 1;
                p.abort_all();
                stop = true;
            }
            if (!stop) {
                uint8_t* dst = p.ws_slot + (static_cast<size_t>(g) * p.R + c % p.R) * BYTES;
                bulk_store(dst, smem_u32(out), BYTES);
                bulk_commit();
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                mbar_arrive(slot_free);
                bulk_wait_all();
                fence_proxy_async_global();
                st_release_u64(p.ready(g, c), p.epoch | (static_cast<unsigned long long>(c) + 1));
            }
        }
        if (__shfl_sync(0xffffffffu, stop ? 1 : 0, 0)) break;
    }
    if (lane == 0) bulk_wait_all();
}

template <int DK, int DV>
__device__ __forceinline__ void prep_role(const CUtensorMap* tmq, const CUtensorMap* tmk, const CUtensorMap* tmv,
                                          const Params& p, uint8_t* sm, uint32_t sbase) {
    using L = PrepLayout<DK, DV>;
    using S = Slot<DK, DV>;
    constexpr int KA = L::KA, VA = L::VA;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = 32 * (warp & 3) + lane;
    const int hh = warp >> 2;
    const int pid = blockIdx.x - p.n_chain;
    const int np = gridDim.x - p.n_chain;
    const int nunits = p.G * p.nch;
    const int T = p.T;

    float* As = reinterpret_cast<float*>(sm + L::OFF_AS);
    float* Rs = reinterpret_cast<float*>(sm + L::OFF_RS);
    // gate buffer of unit k: gbuf + (k & 1) * 256 = cumulative log2 gate,
    // beta (0 on padded tokens), beta_t gam_t, gam_t (64 each), written by
    // the store warp a unit ahead
    float* gbuf = reinterpret_cast<float*>(sm + L::OFF_MISC);
    uint64_t* bar_full = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
    uint64_t* bar_m = bar_full + 2;
    uint64_t* bar_test = bar_full + 3;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_full + 4);
    uint64_t* slot_full = bar_full + 5;   // converting warps: the slot buffer is assembled
    uint64_t* slot_free = bar_full + 6;   // store warp: the slot buffer was read by its store
    volatile int* abort_smem = reinterpret_cast<volatile int*>(bar_full + 7);
    uint64_t* gates_full = bar_full + 8;  // [2] store warp: a unit's gate buffer is written (32 arrivals)
    uint64_t* drain = bar_full + 10;      // after a failure: the MMAs of both issuing threads are done
    const uint32_t aTB1 = sbase + L::OFF_TB1, aTB2 = sbase + L::OFF_TB2;

    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(&bar_full[i], 1);
        for (int i = 5; i < 7; ++i) mbar_init(&bar_full[i], 1);
        mbar_init(&gates_full[0], 32);
        mbar_init(&gates_full[1], 32);
        mbar_init(drain, 2);
        *abort_smem = 0;
        fence_mbar_init();
        tma_prefetch_desc(tmq);
        tma_prefetch_desc(tmk);
        tma_prefetch_desc(tmv);
    }
    if (warp == 0) tmem_alloc(tmem_slot, L::TMEM_COLS);
    tc_fence_before();
    named_sync(kBarInit, kConv + 32);
    tc_fence_after();
    if (warp == kConv / 32) {
        int sbits = 0;
        if (!(p.flags & 0x100u))
            store_gate_loop<S::BYTES>(p, slot_full, slot_free, gates_full, gbuf, sm + L::OFF_OUT, abort_smem, sbits);
        if (sbits && lane == 0) atomicOr(p.status, sbits);
        return;
    }
    const uint32_t tmem = *tmem_slot;
    const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);

    auto wait_all = [&](uint64_t* b, uint32_t parity) -> bool {
        const bool ok = mbar_wait(b, parity, kWaitLimitNs);
        tc_fence_after();
        return !named_sync_or(kBarConv, kConv, !ok);
    };
    // the same, also giving up when the store warp has given up
    auto wait_all_abort = [&](uint64_t* b, uint32_t parity) -> bool {
        const bool ok = mbar_wait_or_abort(b, parity, abort_smem);
        return !named_sync_or(kBarConv, kConv, !ok);
    };
    auto publish = [&]() {
        fence_proxy_async_smem();
        tc_fence_before();
        sync_conv();
        tc_fence_after();
    };

    int status_bits = 0;
    bool failed = false;
    if (p.flags & 0x100u) {
        const bool ok = mbar_wait(bar_test, 0, 1000000ull);
        if (named_sync_or(kBarConv, kConv, !ok)) { status_bits |= kStatusTestHook; failed = true; }
    }

    // unit u -> (head g = u % G, chunk u / G): the units go chunk by chunk
    auto unit_g = [&](int u) { return u % p.G; };
    auto unit_i = [&](int u) { return u / p.G; };
    bool pending[2] = {false, false};
    auto issue_load = [&](int u, int s) {
        const int bh = p.h0 + unit_g(u);
        const int y = unit_i(u) * C;
        uint8_t* stg = sm + s * L::STAGE;
        mbar_arrive_expect_tx(&bar_full[s], L::TX);
#pragma unroll
        for (int a = 0; a < KA; ++a) {
            tma_load_3d(tmk, &bar_full[s], stg + a * 16384, a * 64, y, bh);
            tma_load_3d(tmq, &bar_full[s], stg + a * 16384 + 8192, a * 64, y, bh);
        }
#pragma unroll
        for (int a = 0; a < VA; ++a) tma_load_3d(tmv, &bar_full[s], stg + L::QK_BYTES + a * 8192, a * 64, y, bh);
        pending[s] = true;
    };
    // gate and beta of a unit, one token per thread (threads 0-63), copied
    // asynchronously into shared memory a unit ahead (padded tokens: 1 and 0)
    constexpr uint32_t ID_G = idesc_bf16(128, 64, false, false);   // [K;Q] K^T
    constexpr uint32_t ID_WU = idesc_bf16(128, 64, true, false);   // K^T TB2^T, V^T TB1^T
    constexpr uint32_t ID_NEG_N = idesc_bf16(128, DK, false, true, true);   // -(W^T K')
    constexpr uint32_t ID_EP = idesc_bf16(128, 64, false, false);            // W^T P^T

    if (!failed && tid == 0 && pid < nunits) issue_load(pid, 0);
    uint32_t mph = 0;
    int k = 0;
    for (; !failed; ++k) {
        const int u = pid + k * np;
        if (u >= nunits) break;
        const int s = k & 1;
        const int un = u + np;
        const uint32_t stg = sbase + s * L::STAGE;
        const uint32_t aOut = sbase + L::OFF_OUT;
        float* oVec = reinterpret_cast<float*>(sm + L::OFF_OUT + S::V_OFF);   // gam_C per channel
        const float* sG2 = gbuf + (k & 1) * 256;   // cumulative log2 gate (from the store warp)
        const float* sB = sG2 + 64;                // beta (0 on padded tokens)
        const float* sBG = sB + 64;                // beta_t gam_t
        const float* sGam = sBG + 64;              // gam_t
        uint32_t pw[16];   // this thread's row of P (rows 64-127), bf16 pairs
        if (tid == 0 && un < nunits) {
            fence_proxy_async_smem();
            issue_load(un, s ^ 1);   // stage s^1's MMAs finished with the previous unit
        }
        if (!wait_all(&bar_full[s], (k >> 1) & 1)) { status_bits |= kStatusTmaWait; failed = true; break; }
        if (tid == 0) pending[s] = false;
        // [K;Q] K^T
        if (tid == kIssuer) {
#pragma unroll
            for (int kk = 0; kk < DK / 16; ++kk) {
                const uint64_t d = kmaj(stg + (kk / 4) * 16384 + (kk % 4) * 32);
                mma_bf16_ss(tmem + L::COL_G, d, d, ID_G, kk > 0);
            }
            mma_commit(bar_m);
        }
        // the unit's gates, prepared by the store warp meanwhile
        if (!wait_all_abort(&gates_full[k & 1], (k >> 1) & 1)) { status_bits |= kStatusFlagWait; failed = true; break; }
        if (!wait_all(bar_m, mph)) { status_bits |= kStatusMmaWait; failed = true; break; }
        mph ^= 1u;
        if ((warp & 3) < 2) {
            // rows 0-63: A_tj = beta_t 2^(G_t - G_j) k_t.k_j for j < t
            const int t = r;
            const float Gt = sG2[t], bt = sB[t];
            float x[32];
            tmem_ld32(tlane + L::COL_G + 32 * hh, x);
            tmem_ld_wait();
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int j = 32 * hh + 4 * m;
                float4 o;
                o.x = (j + 0 < t) ? bt * ex2(Gt - sG2[j + 0]) * x[4 * m + 0] : 0.f;
                o.y = (j + 1 < t) ? bt * ex2(Gt - sG2[j + 1]) * x[4 * m + 1] : 0.f;
                o.z = (j + 2 < t) ? bt * ex2(Gt - sG2[j + 2]) * x[4 * m + 2] : 0.f;
                o.w = (j + 3 < t) ? bt * ex2(Gt - sG2[j + 3]) * x[4 * m + 3] : 0.f;
                *reinterpret_cast<float4*>(As + t * kAStride + j) = o;
            }
        } else {
            // rows 64-127: P_tj = 2^(G_t - G_j) q_t.k_j for j <= t, held as bf16
            // pairs until the slot buffer is free
            const int t = r - 64;
            const float Gt = sG2[t];
            float x[32];
            tmem_ld32(tlane + L::COL_G + 32 * hh, x);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int j = 32 * hh + 2 * i;
                pw[i] = pack_bf16((j <= t) ? ex2(Gt - sG2[j]) * x[2 * i] : 0.f,
                                  (j + 1 <= t) ? ex2(Gt - sG2[j + 1]) * x[2 * i + 1] : 0.f);
            }
        }
        sync_conv();
        invert_unit_lower(As, Rs, warp, lane);
        // ---- T diag(beta) and T diag(beta gam) as bf16 MMA operands --------------
        {
            const int t = tid >> 2, q4 = tid & 3;
            const float* trow = As + t * kAStride + 16 * q4;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const float4 t0 = *reinterpret_cast<const float4*>(trow + 8 * cc);
                const float4 t1 = *reinterpret_cast<const float4*>(trow + 8 * cc + 4);
                const float4 b0 = *reinterpret_cast<const float4*>(sB + 16 * q4 + 8 * cc);
                const float4 b1 = *reinterpret_cast<const float4*>(sB + 16 * q4 + 8 * cc + 4);
                const float4 c0 = *reinterpret_cast<const float4*>(sBG + 16 * q4 + 8 * cc);
                const float4 c1 = *reinterpret_cast<const float4*>(sBG + 16 * q4 + 8 * cc + 4);
                const int c8 = 2 * q4 + cc;
                st_shared_v4(aTB1 + sw128_off(t, c8), pack_bf16(t0.x * b0.x, t0.y * b0.y), pack_bf16(t0.z * b0.z, t0.w * b0.w),
                             pack_bf16(t1.x * b1.x, t1.y * b1.y), pack_bf16(t1.z * b1.z, t1.w * b1.w));
                st_shared_v4(aTB2 + sw128_off(t, c8), pack_bf16(t0.x * c0.x, t0.y * c0.y), pack_bf16(t0.z * c0.z, t0.w * c0.w),
                             pack_bf16(t1.x * c1.x, t1.y * c1.y), pack_bf16(t1.z * c1.z, t1.w * c1.w));
            }
        }
        publish();
        // ---- W^T = K^T (T diag(beta gam))^T, Ut^T = V^T (T diag(beta))^T, issued
        //      before the slot buffer is free; its stores below overlap them ----------
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                mma_bf16_ss(tmem + L::COL_W, mnmaj(stg + kk * 2048, 16384), kmaj(aTB2 + kk * 32), ID_WU, kk > 0);
                mma_bf16_ss(tmem + L::COL_UT, mnmaj(stg + L::QK_BYTES + kk * 2048, 8192), kmaj(aTB1 + kk * 32),
                            ID_WU, kk > 0);
            }
            mma_commit(bar_m);
        }
        // the slot buffer is written from here on: the previous unit's store has
        // long read it
        if (k >= 1 && !wait_all_abort(slot_free, (k - 1) & 1)) { status_bits |= kStatusFlagWait; failed = true; break; }
        if ((warp & 3) >= 2) {
#pragma unroll
            for (int m = 0; m < 4; ++m)
                st_shared_v4(aOut + S::P_OFF + sw128_off(r - 64, 4 * hh + m), pw[4 * m], pw[4 * m + 1], pw[4 * m + 2],
                             pw[4 * m + 3]);
        }
        if (tid < DK) oVec[tid] = ex2(sG2[63]);
        // ---- K' = K o Gam_C/Gam = diag(gam_C/gam) K: thread (t, part) scales
        //      DK/4 channels of row t ------------------------------------------------
        {
            const int t = tid >> 2, part = tid & 3;
            const float fk = ex2(sG2[63] - sG2[t]);
#pragma unroll
            for (int i = 0; i < DK / 32; ++i) {
                const int cidx = part * (DK / 32) + i;   // 16-byte chunk of the row
                const int a = cidx / 8, c8 = cidx % 8;
                const uint32_t ro = sw128_off(t, c8);
                st_shared_v4_u4(aOut + S::KP_OFF + a * 8192 + ro, scale_bf16x8(ld_shared_v4(stg + a * 16384 + ro), fk));
            }
        }
        if (!wait_all(bar_m, mph)) { status_bits |= kStatusMmaWait; failed = true; break; }
        mph ^= 1u;
        // W^T as the bf16 A operand of the two products below
        if (r < DK) {
            float x[32];
            tmem_ld32(tlane + L::COL_W + 32 * hh, x);
            tmem_ld_wait();
            store_row32_bf16(sbase + L::OFF_WT, r, 4 * hh, x);
        }
        publish();
        // ---- -N_c = -(W^T K') and W^T P^T; Ut^T into the slot meanwhile -------------
        if (tid == 0) {
            const uint32_t aWT = sbase + L::OFF_WT;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + L::COL_N, kmaj(aWT + kk * 32), mnmaj(aOut + S::KP_OFF + kk * 2048, 8192), ID_NEG_N,
                            kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + L::COL_E, kmaj(aWT + kk * 32), kmaj(aOut + S::P_OFF + kk * 32), ID_EP, kk > 0);
            mma_commit(bar_m);
        }
        if (r < DV) {
            float x[32];
            tmem_ld32(tlane + L::COL_UT + 32 * hh, x);
            tmem_ld_wait();
            store_row32_bf16(aOut + S::U_OFF, r, 4 * hh, x);
        }
        if (!wait_all(bar_m, mph)) { status_bits |= kStatusMmaWait; failed = true; break; }
        mph ^= 1u;
        if (r < DK) {
            store_neg_nc<DK>(tlane + L::COL_N, hh, aOut + S::NC_OFF, r);
            // E_c[r][t] = gam_t q_t[r] - (W^T P^T)[r][t]; q from the stage
            float x[32];
            tmem_ld32(tlane + L::COL_E + 32 * hh, x);
            tmem_ld_wait();
            const uint32_t aq = stg + (r / 64) * 16384 + (r % 8) * 2;
            const uint32_t c8 = (r % 64) / 8;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int t = 32 * hh + i;
                x[i] = sGam[t] * ld_shared_bf16(aq + sw128_off(64 + t, c8)) - x[i];
            }
            store_row32_bf16(aOut + S::E_OFF, r, 4 * hh, x);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        sync_conv();
        if (tid == 0) mbar_arrive(&slot_full[0]);   // to the store warp
    }

    if (failed && tid == 0) {
        for (int s2 = 0; s2 < 2; ++s2)
            if (pending[s2]) mbar_wait(&bar_full[s2], ((s2 == (k & 1) ? k : k + 1) >> 1) & 1, 100000000ull);
    }
    if (failed && tid == 0) {
        *abort_smem = 1;
        p.abort_all();
    }
    // after a failure, MMAs of the last unit may still be in flight: the two
    // issuing threads commit them to one barrier and it completes before the
    // tensor memory is released (bounded: 100 ms)
    if (failed && (tid == 0 || tid == kIssuer)) mma_commit(drain);
    if (failed && tid == 0) mbar_wait(drain, 0, 100000000ull);
    tc_fence_before();
    sync_conv();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
    if (status_bits && tid == 0) atomicOr(p.status, status_bits);
}

// ============================================================================
// prep CTA of the per-channel decay (8 warps)
// ============================================================================
// Per-token log2 decays are floored here, so that the factors of the
// 16-token sub-chunk references (at most eight tokens of decay each) stay
// inside the fp32 exponent range.
constexpr float kLog2DecayFloor = -15.f;
// Exponent kept inside the fp32 range (a guard: with the floor above no
// factor reaches it).
__device__ __forceinline__ float ex2c(float x) { return ex2(fminf(fmaxf(x, -126.f), 126.f)); }

// GLA: the per-channel gated variant without the delta rule (no beta, T = I,
// W = 0). q and k pass through the feature map phi (elu + 1, or the identity
// under the flag) first; the unit then needs only P, Ut^T = V^T, K' and
// E_c = (phi(Q) o Gam)^T, no inverse and no product after P.
template <int DK, int DV, bool GLA>
__device__ __forceinline__ void prep_role_kda(const CUtensorMap* tmq, const CUtensorMap* tmk, const CUtensorMap* tmv,
                                              const Params& p, uint8_t* sm, uint32_t sbase) {
    using L = PrepLayoutKda<DK, DV>;
    using S = Slot<DK, DV>;
    constexpr int KA = L::KA, VA = L::VA;
    constexpr int NCP = DK / 2;          // channel pairs
    constexpr int NSEG = kConv / NCP;    // token segments of the element pass
    constexpr int SL = C / NSEG;         // 16 tokens (d_k 128) or 8 (d_k 64)
    static_assert(SL == 8 || SL == 16, "a segment is one or two 8-token blocks of one sub-chunk");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = 32 * (warp & 3) + lane;
    const int hh = warp >> 2;
    const int pid = blockIdx.x - p.n_chain;
    const int np = gridDim.x - p.n_chain;
    const int nunits = p.G * p.nch;
    const int T = p.T;
    const bool phi_on = GLA && !(p.flags & 0x1u);   // the GLA feature map elu + 1 unless disabled
    // element pass: thread (cp, seg) owns channels c0, c0 + 1 of tokens
    // [seg*SL, seg*SL + SL), all inside sub-chunk sa
    const int cp = tid % NCP, seg = tid / NCP;
    const int c0 = 2 * cp;
    const int ka = c0 / 64;
    const uint32_t ch = (c0 % 64) / 8, bo = (c0 % 8) * 2;
    const int sa = seg * SL / 16;
    const int blk0 = seg * SL / 8;       // first 8-token block of the segment

    float* As = reinterpret_cast<float*>(sm + L::OFF_AS);
    float* Rs = reinterpret_cast<float*>(sm + L::OFF_RS);
    float* sBlk = reinterpret_cast<float*>(sm + L::OFF_BLK);   // log2-gate sum of each 8-token block [8][DK]
    float* sB = reinterpret_cast<float*>(sm + L::OFF_MISC);    // beta (0 on padded tokens)
    float* sBin = sB + 64;                                      // next unit's beta, copied ahead
    const float* sGate = reinterpret_cast<const float*>(sm + L::OFF_GATE);
    uint8_t* outp = sm + L::OFF_OUT;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
    uint64_t* bar_qk = bar;       // k and q of a unit
    uint64_t* bar_v = bar + 2;    // v of a unit
    uint64_t* bar_g = bar + 3;    // gate tile of a unit
    uint64_t* bar_m = bar + 4;    // MMAs
    uint64_t* bar_test = bar + 5;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 6);
    uint64_t* slot_full = bar + 7;   // converting warps: the slot buffer is assembled
    uint64_t* slot_free = bar + 8;   // store warp: the slot buffer was read by its store
    volatile int* abort_smem = reinterpret_cast<volatile int*>(bar + 9);
    const uint32_t aTB1 = sbase + L::OFF_TB1, aOut = sbase + L::OFF_OUT, aV = sbase + L::OFF_V;

    if (tid == 0) {
        for (int i = 0; i < 6; ++i) mbar_init(&bar[i], 1);
        mbar_init(slot_full, 1);
        mbar_init(slot_free, 1);
        *abort_smem = 0;
        fence_mbar_init();
        tma_prefetch_desc(tmq);
        tma_prefetch_desc(tmk);
        tma_prefetch_desc(tmv);
    }
    if (warp == 0) tmem_alloc(tmem_slot, L::TMEM_COLS);
    tc_fence_before();
    named_sync(kBarInit, kConv + 32);
    tc_fence_after();
    if (warp == kConv / 32) {
        int sbits = 0;
        if (lane == 0 && !(p.flags & 0x100u))
            store_loop<S::BYTES>(p, slot_full, slot_free, sm + L::OFF_OUT, abort_smem, sbits);
        if (sbits) atomicOr(p.status, sbits);
        return;
    }
    const uint32_t tmem = *tmem_slot;
    const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);

    auto wait_all = [&](uint64_t* b, uint32_t parity) -> bool {
        const bool ok = mbar_wait(b, parity, kWaitLimitNs);
        tc_fence_after();
        return !named_sync_or(kBarConv, kConv, !ok);
    };
    // the same, also giving up when the store warp has given up
    auto wait_all_abort = [&](uint64_t* b, uint32_t parity) -> bool {
        const bool ok = mbar_wait_or_abort(b, parity, abort_smem);
        return !named_sync_or(kBarConv, kConv, !ok);
    };
    auto publish = [&]() {
        fence_proxy_async_smem();
        tc_fence_before();
        sync_conv();
        tc_fence_after();
    };

    int status_bits = 0;
    bool failed = false;
    if (p.flags & 0x100u) {
        const bool ok = mbar_wait(bar_test, 0, 1000000ull);
        if (named_sync_or(kBarConv, kConv, !ok)) { status_bits |= kStatusTestHook; failed = true; }
    }

    auto unit_g = [&](int u) { return u % p.G; };   // as in the scalar-gate role
    auto unit_i = [&](int u) { return u / p.G; };
    // Copies in flight (thread 0): the single k/q, V and gate buffers (one
    // load at a time each, the n-th completing phase n).
    int qk_issued = 0, qk_done = 0, v_issued = 0, v_done = 0, g_issued = 0, g_done = 0;
    auto issue_qk = [&](int u) {
        const int bh = p.h0 + unit_g(u);
        const int y = unit_i(u) * C;
        mbar_arrive_expect_tx(bar_qk, L::QK_BYTES);
#pragma unroll
        for (int a = 0; a < KA; ++a) {
            tma_load_3d(tmk, bar_qk, sm + a * 16384, a * 64, y, bh);
            tma_load_3d(tmq, bar_qk, sm + a * 16384 + 8192, a * 64, y, bh);
        }
        ++qk_issued;
    };
    auto issue_v = [&](int u) {
        const int bh = p.h0 + unit_g(u);
        const int y = unit_i(u) * C;
        mbar_arrive_expect_tx(bar_v, VA * 8192);
#pragma unroll
        for (int a = 0; a < VA; ++a) tma_load_3d(tmv, bar_v, sm + L::OFF_V + a * 8192, a * 64, y, bh);
        ++v_issued;
    };
    // the gate rows of a chunk are contiguous: one bulk copy of the valid rows
    auto issue_g = [&](int u) {
        const int bh = p.h0 + unit_g(u);
        const int y = unit_i(u) * C;
        const int rows = T - y < C ? T - y : C;
        const uint32_t bytes = static_cast<uint32_t>(rows) * DK * 4;
        mbar_arrive_expect_tx(bar_g, bytes);
        bulk_load(sm + L::OFF_GATE, p.gate + (static_cast<size_t>(bh) * T + y) * DK, bytes, bar_g);
        ++g_issued;
    };
    auto load_b = [&](int u) {   // asynchronously, one token per thread (threads 0-63)
        if (!GLA && u < nunits && tid < 64) {
            const int bh = p.h0 + unit_g(u);
            const int t = unit_i(u) * C + tid;
            if (t < T) {
                cp_async4(smem_u32(sBin + tid), p.beta + static_cast<size_t>(bh) * T + t);
                cp_async_commit();
            } else {
                sBin[tid] = 0.f;
            }
        }
    };

    constexpr uint32_t ID_WU = idesc_bf16(128, 64, true, false);   // (K o Gam)^T TB1^T, V^T TB1^T
    constexpr uint32_t ID_NEG_N = idesc_bf16(128, DK, false, true, true);   // -(W^T K')
    constexpr uint32_t ID_EP = idesc_bf16(128, 64, false, false);            // W^T P^T

    load_b(pid);
    if (!failed && tid == 0 && pid < nunits) {
        issue_qk(pid);
        issue_v(pid);
        issue_g(pid);
    }
    uint32_t mph = 0;
    int k = 0;
    for (; !failed; ++k) {
        const int u = pid + k * np;
        if (u >= nunits) break;
        const int un = u + np;
        const uint32_t stg = sbase;   // [K;Q], rescaled in place into the row operand
        const int nvalid = T - unit_i(u) * C;   // tokens of the unit inside the sequence
        // ---- log2 gates: prefix sums inside each segment, 8-token block sums -----
        if (!wait_all(bar_g, k & 1)) { status_bits |= kStatusTmaWait; failed = true; break; }
        if (tid == 0) ++g_done;
        float lp0[SL], lp1[SL];
        {
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int i = 0; i < SL; ++i) {
                const int t = seg * SL + i;
                float2 g = make_float2(1.f, 1.f);
                if (t < nvalid) g = *reinterpret_cast<const float2*>(sGate + t * DK + c0);
                // A decay below 2^-15 acts as 2^-15 (kLog2DecayFloor): eight
                // tokens of decay then span at most 2^120, so every factor
                // below is exact in fp32; what crosses such a token is still
                // scaled down by 2^-15 or more.
                a0 += fmaxf(lg2(g.x), kLog2DecayFloor);
                a1 += fmaxf(lg2(g.y), kLog2DecayFloor);
                lp0[i] = a0;
                lp1[i] = a1;
            }
            *reinterpret_cast<float2*>(sBlk + blk0 * DK + c0) = make_float2(lp0[7], lp1[7]);
            if (SL == 16)
                *reinterpret_cast<float2*>(sBlk + (blk0 + 1) * DK + c0) =
                    make_float2(lp0[SL - 1] - lp0[7], lp1[SL - 1] - lp1[7]);
        }
        if (!GLA && tid < 64) {
            cp_async_wait();   // this thread's own copy
            sB[tid] = sBin[tid];
        }
        load_b(un);
        sync_conv();
        // ---- cumulative log2 at the 8-token block ends Bc[b]: the segment offset,
        //      the sub-chunk references r_a = Bc[2a] (its 8th token), its start
        //      S_a = Bc[2a-1] and end E_a = Bc[2a+1], G_C = Bc[7] ----------------------
        float off0 = 0.f, off1 = 0.f, rr0[4], rr1[4], GC0, GC1;
        float Sa0 = 0.f, Sa1 = 0.f, Ea0 = 0.f, Ea1 = 0.f;
        {
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const float2 x = *reinterpret_cast<const float2*>(sBlk + b * DK + c0);
                s0 += x.x;
                s1 += x.y;
                if (b + 1 == blk0) { off0 = s0; off1 = s1; }
                if ((b & 1) == 0) { rr0[b / 2] = s0; rr1[b / 2] = s1; }
                if (b + 1 == 2 * sa) { Sa0 = s0; Sa1 = s1; }
                if (b == 2 * sa + 1) { Ea0 = s0; Ea1 = s1; }
            }
            GC0 = s0;
            GC1 = s1;
        }
        float ra0 = rr0[0], ra1 = rr1[0];
#pragma unroll
        for (int a = 1; a < 4; ++a)
            if (a == sa) { ra0 = rr0[a]; ra1 = rr1[a]; }
        // Per-channel factors, every exponent <= 0: the columns of a later
        // sub-chunk b are k f 2^(r_b - E_a) with f = 2^(E_a - G) per element,
        // taken up to the reference token as 2^(r_a - G) 2^(E_a - r_a) and
        // directly after it: each product joins two factors <= 1, so an
        // underflow only hides values that are themselves negligible.
        const float cF0 = ex2(Ea0 - ra0), cF1 = ex2(Ea1 - ra1);
        float cB0[4], cB1[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            cB0[b] = b > sa ? ex2(rr0[b] - Ea0) : 0.f;
            cB1[b] = b > sa ? ex2(rr1[b] - Ea1) : 0.f;
        }
        if (!wait_all(bar_qk, k & 1)) { status_bits |= kStatusTmaWait; failed = true; break; }
        if (tid == 0) ++qk_done;
        // ---- element pass over the thread's tokens and channel pair:
        //      [K;Q] o 2^(G - r_a) in place (row operand), K o 2^(r_a - G) (own
        //      column operand), K o 2^(r_b - G) (columns of later sub-chunks b) ----
        {
            const uint32_t aKQ = stg + ka * 16384;
            const uint32_t aB = sbase + L::OFF_B + ka * L::B_ATOM;
            const int ref = 16 * sa + 7;
#pragma unroll
            for (int i = 0; i < SL; ++i) {
                const int t = seg * SL + i;
                const uint32_t ro = sw128_off(t, ch) + bo;   // in [64][DK] tiles of 8 KB atoms
                const uint32_t ak = aKQ + ro;
                const uint32_t aq = aKQ + sw128_off(64 + t, ch) + bo;
                float2 kv = unpack_bf16(ld_shared_b32(ak));
                float2 qv = unpack_bf16(ld_shared_b32(aq));
                if (GLA) {
                    if (phi_on) {
                        kv = make_float2(elu1(kv.x), elu1(kv.y));
                        qv = make_float2(elu1(qv.x), elu1(qv.y));
                    }
                    if (t >= nvalid) kv = make_float2(0.f, 0.f);   // phi(0) = 1: padded keys write nothing
                }
                const float G0 = off0 + lp0[i], G1 = off1 + lp1[i];
                const float e10 = ex2c(G0 - ra0), e11 = ex2c(G1 - ra1);
                const float e20 = ex2c(ra0 - G0), e21 = ex2c(ra1 - G1);
                float f0, f1;
                if (t <= ref) {
                    f0 = e20 * cF0;
                    f1 = e21 * cF1;
                } else {
                    f0 = ex2(Ea0 - G0);
                    f1 = ex2(Ea1 - G1);
                }
                st_shared_b32(ak, pack_bf16(kv.x * e10, kv.y * e11));
                st_shared_b32(aq, pack_bf16(qv.x * e10, qv.y * e11));
                const float kf0 = kv.x * f0, kf1 = kv.y * f1;
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const uint32_t ab = aB + sw128_off(L::b_row(b) + t, ch) + bo;
                    if (b == sa) st_shared_b32(ab, pack_bf16(kv.x * e20, kv.y * e21));
                    if (b > sa) st_shared_b32(ab, pack_bf16(kf0 * cB0[b], kf1 * cB1[b]));
                }
            }
        }
        publish();
        // ---- [K;Q] B^T on the tensor cores: the four column operands stacked
        //      into one N = 160 product; the slot pass below reads the same
        //      operands meanwhile --------------------------------------------------------
        if (tid == 0) {
            constexpr uint32_t idg = idesc_bf16(128, 160, false, false);
#pragma unroll
            for (int kk = 0; kk < DK / 16; ++kk)
                mma_bf16_ss(tmem + L::COL_G, kmaj(stg + (kk / 4) * 16384 + (kk % 4) * 32),
                            kmaj(sbase + L::OFF_B + (kk / 4) * L::B_ATOM + (kk % 4) * 32), idg, kk > 0);
            mma_commit(bar_m);
        }
        // the slot buffer is written from here on: the previous unit's store has read it
        if (k >= 1 && !wait_all_abort(slot_free, (k - 1) & 1)) { status_bits |= kStatusFlagWait; failed = true; break; }
        // ---- slot pass: K o Gam and Q o Gam are the row operand times 2^r_a, and
        //      K o Gam_C/Gam is the last sub-chunk's column operand (k 2^(r_3 - G),
        //      all 64 rows) times 2^(G_C - r_3). Each joins a factor <= 1 to one
        //      within eight tokens of decay of 1, so every value stays in range
        //      (or is negligible where a factor underflows). K o Gam and Q o Gam
        //      wait in the -N_c and E_c tiles until those are written. ----------------
        {
            // r_a, r_3 and G_C again from the block sums (fewer live registers)
            float ra0s = 0.f, ra1s = 0.f, r30 = 0.f, r31 = 0.f, gc0 = 0.f, gc1 = 0.f;
            {
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    const float2 x = *reinterpret_cast<const float2*>(sBlk + b * DK + c0);
                    s0 += x.x;
                    s1 += x.y;
                    if (b == 2 * sa) { ra0s = s0; ra1s = s1; }
                    if (b == 6) { r30 = s0; r31 = s1; }
                }
                gc0 = s0;
                gc1 = s1;
            }
            const float ca0 = ex2(ra0s), ca1 = ex2(ra1s);
            const float cz0 = ex2(gc0 - r30), cz1 = ex2(gc1 - r31);
            const uint32_t aKQ = stg + ka * 16384;
            const uint32_t aB3 = sbase + L::OFF_B + ka * L::B_ATOM;
#pragma unroll
            for (int i = 0; i < SL; ++i) {
                const int t = seg * SL + i;
                const uint32_t ro = sw128_off(t, ch) + bo;
                const float2 rk = unpack_bf16(ld_shared_b32(aKQ + ro));
                const float2 rq = unpack_bf16(ld_shared_b32(aKQ + sw128_off(64 + t, ch) + bo));
                const float2 b3 = unpack_bf16(ld_shared_b32(aB3 + sw128_off(L::b_row(3) + t, ch) + bo));
                st_shared_b32(aOut + S::NC_OFF + ka * 8192 + ro, pack_bf16(rk.x * ca0, rk.y * ca1));
                st_shared_b32(aOut + S::E_OFF + ka * 8192 + ro, pack_bf16(rq.x * ca0, rq.y * ca1));
                st_shared_b32(aOut + S::KP_OFF + ka * 8192 + ro, pack_bf16(b3.x * cz0, b3.y * cz1));
            }
            if (seg == 0) *reinterpret_cast<float2*>(outp + S::V_OFF + c0 * 4) = make_float2(ex2(gc0), ex2(gc1));
        }
        // the pair products are done, and the slot pass has read the stage and
        // the column operands (the barrier inside)
        if (!wait_all(bar_m, mph)) { status_bits |= kStatusMmaWait; failed = true; break; }
        mph ^= 1u;
        if (tid == 0 && un < nunits) {
            fence_proxy_async_smem();
            issue_g(un);    // into the gate tile, under the column operands
            issue_qk(un);   // into the stage
        }
        // ---- A (rows 0-63) and P (rows 64-127). A warp's lanes 0-15 and 16-31
        //      lie in consecutive sub-chunks a0, a0 + 1: it reads both products and
        //      each lane keeps its own. --------------------------------------------
        {
            const int a0 = 2 * (warp & 1);
            float x[32];
            {
                float y[32];
                tmem_ld32(tlane + L::COL_G + L::b_row(a0) + 32 * hh, x);
                tmem_ld32(tlane + L::COL_G + L::b_row(a0 + 1) + 32 * hh, y);
                tmem_ld_wait();
                const bool hi = lane >= 16;
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] = hi ? y[i] : x[i];
            }
            if ((warp & 3) < 2) {
                if (!GLA) {   // (no A without the delta rule)
                    // A_tj = beta_t (k_t o Gam_t).(k_j / Gam_j) for j < t
                    const int t = r;
                    const float bt = sB[t];
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        const int j = 32 * hh + 4 * m;
                        float4 o;
                        o.x = (j + 0 < t) ? bt * x[4 * m + 0] : 0.f;
                        o.y = (j + 1 < t) ? bt * x[4 * m + 1] : 0.f;
                        o.z = (j + 2 < t) ? bt * x[4 * m + 2] : 0.f;
                        o.w = (j + 3 < t) ? bt * x[4 * m + 3] : 0.f;
                        *reinterpret_cast<float4*>(As + t * kAStride + j) = o;
                    }
                }
            } else {
                // P_tj = (q_t o Gam_t).(k_j / Gam_j) for j <= t
                const int t = r - 64;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int j = 32 * hh + i;
                    x[i] = (j <= t) ? x[i] : 0.f;
                }
                store_row32_bf16(aOut + S::P_OFF, t, 4 * hh, x);
            }
        }
        if constexpr (GLA) {
            // ---- Ut^T = V^T and E_c = (phi(Q) o Gam)^T, both by transposing in
            //      shared memory: thread (r, hh) gathers column r of 32 tokens --------
            if (!wait_all(bar_v, k & 1)) { status_bits |= kStatusTmaWait; failed = true; break; }
            if (tid == 0) ++v_done;
            float qg[32], vt[32];
            if (r < DK) {
                const uint32_t aq = aOut + S::E_OFF + (r / 64) * 8192 + (r % 8) * 2;
                const uint32_t c8 = (r % 64) / 8;
#pragma unroll
                for (int i = 0; i < 32; ++i) qg[i] = ld_shared_bf16(aq + sw128_off(32 * hh + i, c8));
            }
            if (r < DV) {
                const uint32_t av = aV + (r / 64) * 8192 + (r % 8) * 2;
                const uint32_t c8 = (r % 64) / 8;
#pragma unroll
                for (int i = 0; i < 32; ++i) vt[i] = ld_shared_bf16(av + sw128_off(32 * hh + i, c8));
            }
            sync_conv();   // Q o Gam and V are read
            if (tid == 0 && un < nunits) {
                fence_proxy_async_smem();
                issue_v(un);
            }
            if (r < DK) store_row32_bf16(aOut + S::E_OFF, r, 4 * hh, qg);
            if (r < DV) store_row32_bf16(aOut + S::U_OFF, r, 4 * hh, vt);
            fence_proxy_async_smem();
            tc_fence_before();
            sync_conv();
            if (tid == 0) mbar_arrive(&slot_full[0]);   // to the store warp
            continue;
        }
        sync_conv();
        invert_unit_lower(As, Rs, warp, lane);
        // ---- T diag(beta) as a bf16 MMA operand -----------------------------------
        {
            const int t = tid >> 2, q4 = tid & 3;
            const float* trow = As + t * kAStride + 16 * q4;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const float4 t0 = *reinterpret_cast<const float4*>(trow + 8 * cc);
                const float4 t1 = *reinterpret_cast<const float4*>(trow + 8 * cc + 4);
                const float4 b0 = *reinterpret_cast<const float4*>(sB + 16 * q4 + 8 * cc);
                const float4 b1 = *reinterpret_cast<const float4*>(sB + 16 * q4 + 8 * cc + 4);
                st_shared_v4(aTB1 + sw128_off(t, 2 * q4 + cc), pack_bf16(t0.x * b0.x, t0.y * b0.y),
                             pack_bf16(t0.z * b0.z, t0.w * b0.w), pack_bf16(t1.x * b1.x, t1.y * b1.y),
                             pack_bf16(t1.z * b1.z, t1.w * b1.w));
            }
        }
        if (!wait_all(bar_v, k & 1)) { status_bits |= kStatusTmaWait; failed = true; break; }
        if (tid == 0) ++v_done;
        publish();
        // ---- W^T = (K o Gam)^T (T diag(beta))^T, Ut^T = V^T (T diag(beta))^T ---------
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + L::COL_W, mnmaj(aOut + S::NC_OFF + kk * 2048, 8192), kmaj(aTB1 + kk * 32), ID_WU,
                            kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + L::COL_UT, mnmaj(aV + kk * 2048, 8192), kmaj(aTB1 + kk * 32), ID_WU, kk > 0);
            mma_commit(bar_m);
        }
        if (!wait_all(bar_m, mph)) { status_bits |= kStatusMmaWait; failed = true; break; }
        mph ^= 1u;
        if (tid == 0 && un < nunits) {
            fence_proxy_async_smem();
            issue_v(un);
        }
        // W^T as the bf16 A operand of the two products below; Q o Gam (column
        // r, this thread's tokens) read before its tile is overwritten by E_c
        float qg[32];
        if (r < DK) {
            float x[32];
            tmem_ld32(tlane + L::COL_W + 32 * hh, x);
            tmem_ld_wait();
            store_row32_bf16(sbase + L::OFF_WT, r, 4 * hh, x);
            const uint32_t aq = aOut + S::E_OFF + (r / 64) * 8192 + (r % 8) * 2;
            const uint32_t c8 = (r % 64) / 8;
#pragma unroll
            for (int i = 0; i < 32; ++i) qg[i] = ld_shared_bf16(aq + sw128_off(32 * hh + i, c8));
        }
        publish();
        // ---- -N_c = -(W^T K') and W^T P^T ------------------------------------------
        if (tid == 0) {
            const uint32_t aWT = sbase + L::OFF_WT;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + L::COL_N, kmaj(aWT + kk * 32), mnmaj(aOut + S::KP_OFF + kk * 2048, 8192), ID_NEG_N,
                            kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + L::COL_E, kmaj(aWT + kk * 32), kmaj(aOut + S::P_OFF + kk * 32), ID_EP, kk > 0);
            mma_commit(bar_m);
        }
        if (r < DV) {   // Ut^T into the slot while the products run
            float x[32];
            tmem_ld32(tlane + L::COL_UT + 32 * hh, x);
            tmem_ld_wait();
            store_row32_bf16(aOut + S::U_OFF, r, 4 * hh, x);
        }
        if (!wait_all(bar_m, mph)) { status_bits |= kStatusMmaWait; failed = true; break; }
        mph ^= 1u;
        if (r < DK) {
            store_neg_nc<DK>(tlane + L::COL_N, hh, aOut + S::NC_OFF, r);   // over K o Gam, read by now
            float x[32];
            tmem_ld32(tlane + L::COL_E + 32 * hh, x);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] = qg[i] - x[i];
            store_row32_bf16(aOut + S::E_OFF, r, 4 * hh, x);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        sync_conv();
        if (tid == 0) mbar_arrive(&slot_full[0]);   // to the store warp
    }

    if (failed && tid == 0) {
        if (qk_issued > qk_done) mbar_wait(bar_qk, (qk_issued - 1) & 1, 100000000ull);
        if (v_issued > v_done) mbar_wait(bar_v, (v_issued - 1) & 1, 100000000ull);
        if (g_issued > g_done) mbar_wait(bar_g, (g_issued - 1) & 1, 100000000ull);
    }
    if (failed && tid == 0) {
        *abort_smem = 1;
        p.abort_all();
    }
    tc_fence_before();
    sync_conv();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
    if (status_bits && tid == 0) atomicOr(p.status, status_bits);
}

template <int DK, int DV, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
gdn_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
           const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (sbase - raw);
    if (static_cast<int>(blockIdx.x) < p.n_chain) {
        chain_role<DK, DV, MODE == 2>(&tmo, p, sm, sbase);
    } else {
        if (threadIdx.x >= kConv + 32) return;   // the prep role: eight converting warps and a store warp
        if constexpr (MODE != 0)
            prep_role_kda<DK, DV, MODE == 2>(&tmq, &tmk, &tmv, p, sm, sbase);
        else
            prep_role<DK, DV>(&tmq, &tmk, &tmv, p, sm, sbase);
    }
}

// Every launch takes a fresh epoch (the upper half of each flag value), so a
// flag of an earlier launch is never mistaken for one of this launch.
std::atomic<unsigned> g_epoch{0};

template <int DK, int DV, int MODE>
cudaError_t run(const chunk::Maps& m, const FwdArgs& a, int G, int R, cudaStream_t s) {
    constexpr uint32_t smem = smem_alloc<DK, DV, MODE>();
    static_assert(smem <= 232448, "shared memory budget");
    auto kern = gdn_kernel<DK, DV, MODE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int nch = (a.T + C - 1) / C;
    Params p;
    p.gate = a.gate;
    p.beta = a.beta;
    p.state_in = a.state_in;
    p.state_out = a.state_out;
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.ws_flag = reinterpret_cast<unsigned long long*>(a.workspace);
    p.ws_slot = reinterpret_cast<uint8_t*>(a.workspace) + align_up(flag_words(G, R) * 8, 1024);
    p.T = a.T;
    p.nch = nch;
    p.R = R;
    p.flags = a.flags;
    p.status = a.status;
    // One cooperative launch per group of sequence-heads: every CTA is
    // resident, so the chain and prep CTAs may wait on each other's flags.
    for (int h0 = 0; h0 < a.BH; h0 += G) {
        p.h0 = h0;
        p.G = a.BH - h0 < G ? a.BH - h0 : G;
        p.n_chain = p.G;
        p.epoch = static_cast<unsigned long long>(g_epoch.fetch_add(1) + 1) << 32;
        // The workspace is shared with the other variants' scratch: clear the
        // flag words so that no stale value reads as raised.
        e = cudaMemsetAsync(p.ws_flag, 0, flag_words(G, R) * 8, s);
        if (e != cudaSuccess) return e;
        const int units = p.G * nch;
        int n_prep = a.sm_count - p.n_chain;
        if (n_prep > units) n_prep = units;
        if (n_prep < 1) return cudaErrorInvalidConfiguration;
        e = launch_coop(kern, static_cast<unsigned>(p.n_chain + n_prep), kThreads, smem, s, m.q, m.k, m.v, m.o, p);
        if (e != cudaSuccess) return e;
        if (a.nlaunch) ++*a.nlaunch;
    }
    return cudaSuccess;
}

}  // namespace gdn

namespace chunk {

size_t gdn_slot_bytes(int dk, int dv) {
    return 2 * static_cast<size_t>(dk) * dk + static_cast<size_t>(2 * dk + dv) * 128 + 8192 + 512;
}

int gdn_group(int BH) { return BH < kGdnMaxGroup ? BH : kGdnMaxGroup; }

// Flag words, then a ring of R chunks per sequence-head of a group of G.
static size_t ring_bytes(int G, int R, int dk, int dv) {
    return gdn::align_up(gdn::flag_words(G, R) * 8, 1024) + static_cast<size_t>(G) * R * gdn_slot_bytes(dk, dv);
}

size_t gdn_workspace_bytes(int BH, int dk, int dv, int W) { return ring_bytes(gdn_group(BH), 2 * W, dk, dv); }

cudaError_t launch_gdn(const FwdArgs& a, const Maps& m, cudaStream_t s) {
    const int G = gdn_group(a.BH);
    const int mode = a.variant == kKda ? 1 : a.variant == kGla ? 2 : 0;
    const int nch = (a.T + C - 1) / C;
    // the deepest ring (up to 2 kGdnWindow chunks, no deeper than the
    // sequence) that the workspace holds
    int R = 2 * kGdnWindow;
    if (R > nch) R = nch < 2 ? 2 : nch;
    while (R > 2 && ring_bytes(G, R, a.dk, a.dv) > a.ws_bytes) --R;
    if (!a.workspace || ring_bytes(G, R, a.dk, a.dv) > a.ws_bytes) return cudaErrorInvalidValue;
    if (mode == 2) {
        if (a.dk == 64 && a.dv == 64) return gdn::run<64, 64, 2>(m, a, G, R, s);
        if (a.dk == 64 && a.dv == 128) return gdn::run<64, 128, 2>(m, a, G, R, s);
        if (a.dk == 128 && a.dv == 64) return gdn::run<128, 64, 2>(m, a, G, R, s);
        if (a.dk == 128 && a.dv == 128) return gdn::run<128, 128, 2>(m, a, G, R, s);
        return cudaErrorInvalidValue;
    }
    if (mode == 1) {
        if (a.dk == 64 && a.dv == 64) return gdn::run<64, 64, 1>(m, a, G, R, s);
        if (a.dk == 64 && a.dv == 128) return gdn::run<64, 128, 1>(m, a, G, R, s);
        if (a.dk == 128 && a.dv == 64) return gdn::run<128, 64, 1>(m, a, G, R, s);
        if (a.dk == 128 && a.dv == 128) return gdn::run<128, 128, 1>(m, a, G, R, s);
        return cudaErrorInvalidValue;
    }
    if (a.dk == 64 && a.dv == 64) return gdn::run<64, 64, 0>(m, a, G, R, s);
    if (a.dk == 64 && a.dv == 128) return gdn::run<64, 128, 0>(m, a, G, R, s);
    if (a.dk == 128 && a.dv == 64) return gdn::run<128, 64, 0>(m, a, G, R, s);
    if (a.dk == 128 && a.dv == 128) return gdn::run<128, 128, 0>(m, a, G, R, s);
    return cudaErrorInvalidValue;
}

}  // namespace chunk
}  // namespace la
