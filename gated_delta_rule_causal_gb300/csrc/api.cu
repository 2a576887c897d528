// C ABI of the library (declared in include/la.h): argument validation,
// kernel selection and the device status word.
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/la.h"
#include "kernels.h"
#include "prefill.h"

struct la_handle {
    la_config cfg;
    int sm_count;
    int* d_status;  // device status word (bounded-wait failures)
    float* d_ws;    // workspace of the chunked prefill
    size_t ws_bytes;
    PFN_cuTensorMapEncodeTiled_v12000 encode;
    std::string last_error;
    int last_launches;  // kernels enqueued by the last successful call
    // la_forward_host: device staging for two groups of sequence-heads, the
    // copy-in / compute / copy-out streams and the events that chain them
    // (all created on first use)
    uint8_t* d_stage;
    size_t stage_bytes;
    cudaStream_t s_in, s_comp, s_out;
    cudaEvent_t ev_start, ev_done, ev_in[2], ev_comp[2], ev_out[2];
    bool host_ready;
    // la_backward_gated: checkpoints and accumulators (allocated on first
    // use, grown when a call needs more)
    float* d_bws;
    size_t bws_bytes;
};

namespace {

// la_forward_host: how a call crosses the host link. Below kLargeCall bytes
// per call: two groups of sequence-heads (best of 1, 2, 4, 8 on the
// normalized B4 H8 T2048 call) moved by copy kernels. From there on, by the
// copy engines, which need no SM (the chunkwise kernels of the gated
// variants fill each SM's shared memory, so copy kernels could not run
// beside them):
// - the sequence in kTimeSegments segments of every head (strided 2-D
//   copies), the state handed from one segment's kernels to the next in
//   device memory. Every launch keeps every head, so a segment's kernels take
//   ~1/kTimeSegments of the call's, where a group of heads would still walk
//   the whole sequence (gated delta B2 H16 T8192: 1.26 ms per call with 4
//   segments, 1.27 with 8, 1.40 with 16; 1.43 with 4 head groups);
// - LA_GLA alone in kHostGroupsLarge groups of heads: its calls run two
//   launches of 32 heads per segment, and time segments measured slower
//   (B4 H16 T4096: 1.91 ms with 4 groups, 2.02 with 4 segments).
constexpr int kHostGroupsSmall = 2;
constexpr int kHostGroupsLarge = 4;
constexpr int kTimeSegments = 4;
constexpr size_t kLargeCall = size_t(64) << 20;
constexpr int kCopyCtas = 64;    // CTAs of one gather / scatter over the host link

// Up to six contiguous byte ranges copied by one launch: the inputs of a
// group of sequence-heads from mapped page-locked host memory into the
// staging, or its results back. One launch instead of one copy per tensor
// (each copy costs several microseconds of fixed time); the host link, not
// the launch, bounds the rate. 16-byte accesses where both ends and the
// length allow, else 4-byte, else bytes.
struct CopySeg {
    const uint8_t* src;
    uint8_t* dst;
    size_t bytes;
};
struct CopyJob {
    CopySeg seg[6];
    int n;
};

__global__ void __launch_bounds__(256) copy_segments_kernel(const CopyJob job) {
    const size_t tid = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
    const size_t nthr = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (int s = 0; s < job.n; ++s) {
        const CopySeg g = job.seg[s];
        const uintptr_t al = reinterpret_cast<uintptr_t>(g.src) | reinterpret_cast<uintptr_t>(g.dst) | g.bytes;
        if ((al & 15) == 0) {
            const uint4* a = reinterpret_cast<const uint4*>(g.src);
            uint4* b = reinterpret_cast<uint4*>(g.dst);
            const size_t n = g.bytes / 16;
            size_t i = tid;
            for (; i + 3 * nthr < n; i += 4 * nthr) {   // four loads in flight per thread
                const uint4 x0 = a[i], x1 = a[i + nthr], x2 = a[i + 2 * nthr], x3 = a[i + 3 * nthr];
                b[i] = x0;
                b[i + nthr] = x1;
                b[i + 2 * nthr] = x2;
                b[i + 3 * nthr] = x3;
            }
            for (; i < n; i += nthr) b[i] = a[i];
        } else if ((al & 3) == 0) {
            const uint32_t* a = reinterpret_cast<const uint32_t*>(g.src);
            uint32_t* b = reinterpret_cast<uint32_t*>(g.dst);
            for (size_t i = tid; i < g.bytes / 4; i += nthr) b[i] = a[i];
        } else {
            for (size_t i = tid; i < g.bytes; i += nthr) g.dst[i] = g.src[i];
        }
    }
}

// The device address of page-locked host memory (its own address under
// unified addressing), or NULL when the GPU cannot address it directly.
const uint8_t* mapped(const void* p) {
    if (!p) return nullptr;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (at.type != cudaMemoryTypeHost || !at.devicePointer) return nullptr;
    return static_cast<const uint8_t*>(at.devicePointer);
}

int fail(la_handle* h, int code, const std::string& msg) {
    if (h) h->last_error = msg;
    return code;
}

int cuda_fail(la_handle* h, cudaError_t e, const char* what) {
    return fail(h, LA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

bool supported_d(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Make the handle's device current for the duration of a call.
struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) return;
        ok = (prev == dev) || (cudaSetDevice(dev) == cudaSuccess);
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

bool valid_variant(int v) {
    return v == LA_NORM_ELU1 || v == LA_GLA || v == LA_GDN || v == LA_NORM_DECAY || v == LA_KDA;
}

size_t state_elems(const la_config& c, int variant) {
    return static_cast<size_t>(c.d_k) * c.d_v + ((variant == LA_NORM_ELU1 || variant == LA_NORM_DECAY) ? c.d_k : 0);
}

int check_common(la_handle* h, const void* q, const void* k, const void* v, const float* gate,
                 const float* beta, const float* state_in, const void* out, const float* state_out,
                 const float* den_out, int variant) {
    if (!valid_variant(variant))
        return fail(h, LA_ERR_INVALID_ARG, "variant must be LA_NORM_ELU1, LA_GLA, LA_GDN, LA_NORM_DECAY or LA_KDA");
    if (!q || !k || !v || !out) return fail(h, LA_ERR_INVALID_ARG, "q, k, v and out are required");
    if (variant != LA_NORM_ELU1 && !gate)
        return fail(h, LA_ERR_INVALID_ARG, "gate is required for LA_GLA, LA_GDN, LA_NORM_DECAY and LA_KDA");
    if ((variant == LA_GDN || variant == LA_KDA) && !beta)
        return fail(h, LA_ERR_INVALID_ARG, "beta is required for LA_GDN and LA_KDA");
    if (variant != LA_NORM_ELU1 && variant != LA_NORM_DECAY && den_out)
        return fail(h, LA_ERR_INVALID_ARG, "den_out is only defined for LA_NORM_ELU1 and LA_NORM_DECAY");
    const void* ptrs[] = {q, k, v, gate, beta, state_in, out, state_out, den_out};
    const char* names[] = {"q", "k", "v", "gate", "beta", "state_in", "out", "state_out", "den_out"};
    for (int i = 0; i < 9; ++i)
        if (ptrs[i] && !aligned16(ptrs[i]))
            return fail(h, LA_ERR_MISALIGNED, std::string(names[i]) + " is not 16-byte aligned");
    return LA_OK;
}

la::FwdArgs make_args(la_handle* h, const void* q, const void* k, const void* v, const float* gate,
                      const float* beta, const float* state_in, void* out, float* state_out, float* den_out,
                      int variant, int T) {
    la::FwdArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.gate = gate;
    a.beta = beta;
    a.state_in = state_in;
    a.out = out;
    a.state_out = state_out;
    a.den_out = den_out;
    a.BH = h->cfg.B * h->cfg.H;
    a.T = T;
    a.dk = h->cfg.d_k;
    a.dv = h->cfg.d_v;
    // LA_NORM_DECAY runs as the normalized variant with a per-(b,h) decay in
    // `gate`; plain LA_NORM_ELU1 carries no gate.
    a.variant = (variant == LA_NORM_DECAY) ? la::kNorm : (variant == LA_KDA) ? la::kKda : variant;
    if (variant == LA_NORM_ELU1) a.gate = nullptr;
    a.io = h->cfg.io == LA_FP32 ? la::kFp32 : la::kBf16;
    a.flags = h->cfg.flags;
    a.status = h->d_status;
    a.sm_count = h->sm_count;
    a.workspace = h->d_ws;
    a.ws_bytes = h->ws_bytes;
    a.nlaunch = &h->last_launches;
    return a;
}

// Enqueue the kernels of one prefill whose arguments were validated: the
// chunkwise tensor-core form when the configuration allows it, else the
// recurrent kernel. Adds the launches to h->last_launches.
int enqueue_forward(la_handle* h, la::FwdArgs& a, int variant, int chunk, cudaStream_t s) {
    const la_config& c = h->cfg;
    const bool tc_ok = c.io == LA_BF16 && (c.d_k == 64 || c.d_k == 128) && (c.d_v == 64 || c.d_v == 128);
    // the decayed normalized variant runs chunkwise only in the single-launch
    // or the three-phase form
    const bool chunked = tc_ok && chunk != 1 &&
                         (variant != LA_NORM_DECAY ||
                          (!(c.flags & LA_FLAG_SEQUENTIAL_CHUNKS) &&
                           (la::chunk::seg_fits(a.BH, a.T, c.d_k, c.d_v, h->sm_count) ||
                            la::chunk::par_fits(a.BH, a.T, c.d_k, c.d_v, h->ws_bytes))));
    cudaError_t e;
    if (chunked) {
        const char* what = "";
        e = la::launch_chunked(a, s, h->encode, &what);
        if (e != cudaSuccess) return cuda_fail(h, e, what);
    } else {
        e = la::launch_recurrent(a, s);
        if (e != cudaSuccess) return cuda_fail(h, e, "recurrent kernel launch");
        h->last_launches += 1;
    }
    return LA_OK;
}

// la_forward_host for a large call: the sequence in segments of Ts tokens
// (a multiple of the 64-token chunk) for all sequence-heads at once. Per
// segment s, staging half b = s & 1: s_in copies the segment's slices of q,
// k, v, gate and beta in (one strided copy each: BH rows of len tokens), s_comp
// runs the prefill of len tokens from the state the previous segment left
// (device buffer (s - 1) & 1; the caller's state_in is staged into buffer 1
// for segment 0) into buffer s & 1, s_out copies the outputs (and den) out.
// A half is refilled two segments later, after its kernels and its
// copy-out. The final state leaves after the last segment.
int host_time_split(la_handle* h, const void* q, const void* k, const void* v, const float* gate,
                    const float* beta, const float* state_in, void* out, float* state_out, float* den_out,
                    int variant, int T, int chunk) {
    const la_config& c = h->cfg;
    const int BH = c.B * c.H;
    const size_t io = (c.io == LA_BF16) ? 2 : 4;
    const size_t ss = state_elems(c, variant);
    const bool per_token_gate = variant == LA_GLA || variant == LA_KDA || variant == LA_GDN;
    const size_t gate_row = (variant == LA_GLA || variant == LA_KDA) ? c.d_k * 4 : 4;   // bytes per token
    int Ts = (T + kTimeSegments - 1) / kTimeSegments;
    Ts = (Ts + 63) / 64 * 64;
    const int nseg = (T + Ts - 1) / Ts;
    // bytes per token of every sequence-head: q, k, v, gate, beta, out, den
    const size_t row[7] = {c.d_k * io, c.d_k * io, c.d_v * io, (gate && per_token_gate) ? gate_row : 0,
                           beta ? 4 : 0, c.d_v * io, den_out ? 4 : 0};
    size_t off[7], half = 0;
    for (int i = 0; i < 7; ++i) {
        off[i] = half;
        half += (static_cast<size_t>(BH) * Ts * row[i] + 255) & ~static_cast<size_t>(255);
    }
    const size_t sbytes = (static_cast<size_t>(BH) * ss * 4 + 255) & ~static_cast<size_t>(255);
    const size_t hgate = (variant == LA_NORM_DECAY && gate) ? ((BH * 4 + 255) & ~static_cast<size_t>(255)) : 0;
    const size_t need = 2 * half + 2 * sbytes + hgate;
    cudaError_t e;
    if (need > h->stage_bytes) {
        if (h->d_stage) {   // grow the staging (frees the old one after the work that used it)
            cudaStreamSynchronize(h->s_in);
            cudaStreamSynchronize(h->s_comp);
            cudaStreamSynchronize(h->s_out);
            cudaFree(h->d_stage);
            h->d_stage = nullptr;
            h->stage_bytes = 0;
        }
        e = cudaMalloc(&h->d_stage, need);
        if (e != cudaSuccess) return cuda_fail(h, e, "staging allocation");
        h->stage_bytes = need;
    }
    uint8_t* sbuf[2] = {h->d_stage + 2 * half, h->d_stage + 2 * half + sbytes};
    float* dgate_head = reinterpret_cast<float*>(h->d_stage + 2 * half + 2 * sbytes);
    // segment 0 reads the state from buffer 1; the per-head decay once
    e = cudaSuccess;
    if (state_in) e = cudaMemcpyAsync(sbuf[1], state_in, static_cast<size_t>(BH) * ss * 4, cudaMemcpyHostToDevice, h->s_in);
    if (e == cudaSuccess && hgate)
        e = cudaMemcpyAsync(dgate_head, gate, static_cast<size_t>(BH) * 4, cudaMemcpyHostToDevice, h->s_in);
    if (e != cudaSuccess) return cuda_fail(h, e, "staging copy-in");
    const void* src[5] = {q, k, v, per_token_gate ? gate : nullptr, beta};
    for (int sg = 0; sg < nseg; ++sg) {
        const int b = sg & 1;
        const int t0 = sg * Ts;
        const int len = (T - t0 < Ts) ? T - t0 : Ts;
        uint8_t* st = h->d_stage + b * half;
        if (sg >= 2) e = cudaStreamWaitEvent(h->s_in, h->ev_comp[b], 0);
        for (int i = 0; i < 5 && e == cudaSuccess; ++i)
            if (src[i] && row[i])
                e = cudaMemcpy2DAsync(st + off[i], len * row[i], static_cast<const uint8_t*>(src[i]) + t0 * row[i],
                                      static_cast<size_t>(T) * row[i], len * row[i], BH, cudaMemcpyHostToDevice,
                                      h->s_in);
        if (e == cudaSuccess) e = cudaEventRecord(h->ev_in[b], h->s_in);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h->s_comp, h->ev_in[b], 0);
        if (e == cudaSuccess && sg >= 2) e = cudaStreamWaitEvent(h->s_comp, h->ev_out[b], 0);
        if (e != cudaSuccess) return cuda_fail(h, e, "staging copy-in");
        const float* g_arg = !gate ? nullptr : per_token_gate ? reinterpret_cast<const float*>(st + off[3])
                           : (variant == LA_NORM_DECAY) ? dgate_head : nullptr;
        const float* sin = (sg == 0 && !state_in) ? nullptr : reinterpret_cast<const float*>(sbuf[(sg + 1) & 1]);
        la::FwdArgs a = make_args(h, st + off[0], st + off[1], st + off[2], g_arg,
                                  beta ? reinterpret_cast<const float*>(st + off[4]) : nullptr, sin, st + off[5],
                                  reinterpret_cast<float*>(sbuf[b]), den_out ? reinterpret_cast<float*>(st + off[6]) : nullptr,
                                  variant, len);
        int rc = enqueue_forward(h, a, variant, chunk, h->s_comp);
        if (rc != LA_OK) return rc;
        e = cudaEventRecord(h->ev_comp[b], h->s_comp);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h->s_out, h->ev_comp[b], 0);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(static_cast<uint8_t*>(out) + t0 * row[5], static_cast<size_t>(T) * row[5], st + off[5],
                                  len * row[5], len * row[5], BH, cudaMemcpyDeviceToHost, h->s_out);
        if (e == cudaSuccess && den_out)
            e = cudaMemcpy2DAsync(reinterpret_cast<uint8_t*>(den_out) + t0 * row[6], static_cast<size_t>(T) * row[6],
                                  st + off[6], len * row[6], len * row[6], BH, cudaMemcpyDeviceToHost, h->s_out);
        if (e == cudaSuccess) e = cudaEventRecord(h->ev_out[b], h->s_out);
        if (e != cudaSuccess) return cuda_fail(h, e, "staging copy-out");
    }
    // s_out follows the last segment's kernels: the final state leaves now
    if (state_out) {
        e = cudaMemcpyAsync(state_out, sbuf[(nseg - 1) & 1], static_cast<size_t>(BH) * ss * 4, cudaMemcpyDeviceToHost,
                            h->s_out);
        if (e != cudaSuccess) return cuda_fail(h, e, "state copy-out");
    }
    return LA_OK;
}

// Grow the handle's backward workspace to `need` bytes (frees the old one
// after the work that used it).
int grow_bws(la_handle* h, size_t need) {
    if (need <= h->bws_bytes) return LA_OK;
    if (h->d_bws) {
        cudaFree(h->d_bws);   // waits for the work that used it
        h->d_bws = nullptr;
        h->bws_bytes = 0;
    }
    const cudaError_t e = cudaMalloc(&h->d_bws, need);
    if (e != cudaSuccess) return cuda_fail(h, e, "backward workspace allocation");
    h->bws_bytes = need;
    return LA_OK;
}

// Gradients of the normalized variant (gamma NULL) or of its fixed-decay form
// on the row-split CUDA-core kernel (d_k, d_v in {64, 128}): the forward
// first, its outputs and normalizers into the backward workspace, then the
// token-serial rows. Arguments validated by the caller.
int norm_rows_backward(la_handle* h, const void* q, const void* k, const void* v, const float* gamma,
                       const float* state_in, const void* dout, const float* dstate_out, void* dq, void* dk,
                       void* dv, float* dgamma, float* dstate_in, int variant, int T, cudaStream_t s) {
    const la_config& c = h->cfg;
    const int BH = c.B * c.H;
    const int io = c.io == LA_FP32 ? la::kFp32 : la::kBf16;
    const size_t fwd = la::norm_rows_fwd_bytes(BH, T, c.d_v, io);
    const size_t o_bytes = (static_cast<size_t>(BH) * T * c.d_v * (io == la::kBf16 ? 2 : 4) + 255) & ~static_cast<size_t>(255);
    int rc = grow_bws(h, fwd + la::norm_rows_bytes(BH, T, c.d_k, c.d_v));
    if (rc != LA_OK) return rc;
    uint8_t* ws = reinterpret_cast<uint8_t*>(h->d_bws);
    float* den = reinterpret_cast<float*>(ws + o_bytes);
    la::FwdArgs f = make_args(h, q, k, v, gamma, nullptr, state_in, ws, nullptr, den, variant, T);
    rc = enqueue_forward(h, f, variant, 0, s);
    if (rc != LA_OK) return rc;
    la::DeltaBwdArgs a = {};
    a.q = q;
    a.k = k;
    a.v = v;
    a.gate = gamma;
    a.state_in = state_in;
    a.dout = dout;
    a.dstate_out = dstate_out;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.dgate = dgamma;
    a.dstate_in = dstate_in;
    a.BH = BH;
    a.T = T;
    a.dk_dim = c.d_k;
    a.dv_dim = c.d_v;
    a.io = io;
    a.norm = true;
    a.fwd_out = ws;
    a.fwd_den = den;
    a.sm_count = h->sm_count;
    a.workspace = reinterpret_cast<float*>(ws + fwd);
    const cudaError_t e = la::launch_delta_backward(a, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "normalized backward launch");
    h->last_launches += 2;   // the row kernel and the dv conversion, after the forward's
    return LA_OK;
}

}  // namespace

extern "C" {

int la_version(void) { return 100; }

int la_create(const la_config* cfg, la_handle** out) {
    if (!cfg || !out) return LA_ERR_INVALID_ARG;
    *out = nullptr;
    if (cfg->B < 1 || cfg->H < 1) return LA_ERR_INVALID_ARG;
    if (cfg->io != LA_BF16 && cfg->io != LA_FP32) return LA_ERR_INVALID_ARG;
    if (!supported_d(cfg->d_k) || !supported_d(cfg->d_v)) return LA_ERR_UNSUPPORTED;
    if (static_cast<long long>(cfg->B) * cfg->H > (1LL << 30)) return LA_ERR_UNSUPPORTED;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
        cudaGetLastError();
        return LA_ERR_CUDA;
    }
    if (cfg->device < 0 || cfg->device >= ndev) return LA_ERR_INVALID_ARG;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, cfg->device) != cudaSuccess) return LA_ERR_CUDA;
    if (!(prop.major == 10 && prop.minor == 3)) return LA_ERR_UNSUPPORTED;  // built for sm_103a only

    la_handle* h = new (std::nothrow) la_handle();
    if (!h) return LA_ERR_CUDA;
    h->cfg = *cfg;
    h->sm_count = prop.multiProcessorCount;
    h->d_status = nullptr;
    h->d_ws = nullptr;
    h->ws_bytes = 0;
    h->encode = nullptr;
    h->last_launches = 0;
    h->d_stage = nullptr;
    h->stage_bytes = 0;
    h->host_ready = false;
    h->d_bws = nullptr;
    h->bws_bytes = 0;
    DeviceGuard g(cfg->device);
    if (!g.ok) { delete h; return LA_ERR_CUDA; }
    if (cudaMalloc(&h->d_status, sizeof(int)) != cudaSuccess || cudaMemset(h->d_status, 0, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        if (h->d_status) cudaFree(h->d_status);
        delete h;
        return LA_ERR_CUDA;
    }
    // Fixed workspace. Normalized / gated: one state block (S plus a d_k
    // vector) per SM, enough for every segment split the chunked prefill
    // chooses (B*H*(segments-1) stays below the SM count). Gated delta rule on
    // the tensor-core path: the states of one group of sequence-heads and two
    // windows of per-chunk intermediates.
    h->ws_bytes = static_cast<size_t>(h->sm_count) * (static_cast<size_t>(cfg->d_k) * cfg->d_v + cfg->d_k) * sizeof(float);
    const bool tc_shape = cfg->io == LA_BF16 && (cfg->d_k == 64 || cfg->d_k == 128) && (cfg->d_v == 64 || cfg->d_v == 128);
    if (tc_shape) {
        const size_t gdn = la::chunk::gdn_workspace_bytes(cfg->B * cfg->H, cfg->d_k, cfg->d_v, la::chunk::kGdnWindow);
        if (gdn > h->ws_bytes) h->ws_bytes = gdn;
        // three-phase normalized / gated prefill: per-chunk states of up to
        // 128 chunks (T = 8192) per sequence-head, capped at the L2 budget
        size_t par = static_cast<size_t>(cfg->B) * cfg->H * 128 * la::chunk::par_chunk_bytes(cfg->d_k, cfg->d_v);
        if (par > la::chunk::kParL2Bytes) par = la::chunk::kParL2Bytes;
        if (par > h->ws_bytes) h->ws_bytes = par;
    }
    if (cudaMalloc(&h->d_ws, h->ws_bytes) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(h->d_status);
        delete h;
        return LA_ERR_CUDA;
    }
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
        cudaGetLastError();
        cudaFree(h->d_ws);
        cudaFree(h->d_status);
        delete h;
        return LA_ERR_CUDA;
    }
    h->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    *out = h;
    return LA_OK;
}

void la_destroy(la_handle* h) {
    if (!h) return;
    {
        DeviceGuard g(h->cfg.device);
        if (h->host_ready) {
            cudaStreamSynchronize(h->s_in);
            cudaStreamSynchronize(h->s_comp);
            cudaStreamSynchronize(h->s_out);
            cudaStreamDestroy(h->s_in);
            cudaStreamDestroy(h->s_comp);
            cudaStreamDestroy(h->s_out);
            for (cudaEvent_t e : {h->ev_start, h->ev_done, h->ev_in[0], h->ev_in[1], h->ev_comp[0], h->ev_comp[1],
                                  h->ev_out[0], h->ev_out[1]})
                cudaEventDestroy(e);
        }
        if (h->d_stage) cudaFree(h->d_stage);
        if (h->d_bws) cudaFree(h->d_bws);
        if (h->d_status) cudaFree(h->d_status);
        if (h->d_ws) cudaFree(h->d_ws);
    }
    delete h;
}

const char* la_last_error(const la_handle* h) { return h ? h->last_error.c_str() : "null handle"; }

int la_forward(la_handle* h, const void* q, const void* k, const void* v, const float* gate, const float* beta,
               const float* state_in, void* out, float* state_out, float* den_out, int variant, int T, int chunk,
               void* cuda_stream) {
    if (!h) return LA_ERR_INVALID_ARG;
    h->last_error.clear();
    h->last_launches = 0;
    if (T < 0) return fail(h, LA_ERR_INVALID_ARG, "T must be >= 0");
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const la_config& c = h->cfg;
    if (T == 0) {
        if (!valid_variant(variant))
            return fail(h, LA_ERR_INVALID_ARG, "variant must be LA_NORM_ELU1, LA_GLA, LA_GDN, LA_NORM_DECAY or LA_KDA");
        if (state_out && !aligned16(state_out)) return fail(h, LA_ERR_MISALIGNED, "state_out is not 16-byte aligned");
        if (!state_out || state_out == state_in) return LA_OK;
        DeviceGuard g(c.device);
        const size_t bytes = state_elems(c, variant) * sizeof(float) * c.B * c.H;
        cudaError_t e = state_in ? cudaMemcpyAsync(state_out, state_in, bytes, cudaMemcpyDeviceToDevice, s)
                                 : cudaMemsetAsync(state_out, 0, bytes, s);
        return e == cudaSuccess ? LA_OK : cuda_fail(h, e, "state copy");
    }
    int rc = check_common(h, q, k, v, gate, beta, state_in, out, state_out, den_out, variant);
    if (rc != LA_OK) return rc;
    if (chunk != 0 && chunk != 1 && chunk != 64)
        return fail(h, LA_ERR_UNSUPPORTED, "chunk must be 0 (default), 1 (recurrent) or 64");
    const bool tc_ok = c.io == LA_BF16 && (c.d_k == 64 || c.d_k == 128) && (c.d_v == 64 || c.d_v == 128);
    if (chunk == 64 && !tc_ok)
        return fail(h, LA_ERR_UNSUPPORTED, "chunk 64 needs bf16 io and d_k, d_v in {64, 128}");
    if (static_cast<long long>(T) * (c.d_k > c.d_v ? c.d_k : c.d_v) > (1LL << 31) - 1)
        return fail(h, LA_ERR_UNSUPPORTED, "T * d exceeds 2^31 - 1");
    DeviceGuard g(c.device);
    if (!g.ok) return fail(h, LA_ERR_CUDA, "cannot select the handle's device");
    la::FwdArgs a = make_args(h, q, k, v, gate, beta, state_in, out, state_out, den_out, variant, T);
    return enqueue_forward(h, a, variant, chunk, s);
}

int la_forward_host(la_handle* h, const void* q, const void* k, const void* v, const float* gate, const float* beta,
                    const float* state_in, void* out, float* state_out, float* den_out, int variant, int T, int chunk,
                    void* cuda_stream) {
    if (!h) return LA_ERR_INVALID_ARG;
    h->last_error.clear();
    h->last_launches = 0;
    if (T < 1) return fail(h, LA_ERR_INVALID_ARG, "T must be >= 1");
    int rc = check_common(h, q, k, v, gate, beta, state_in, out, state_out, den_out, variant);
    if (rc != LA_OK) return rc;
    if (chunk != 0 && chunk != 1 && chunk != 64)
        return fail(h, LA_ERR_UNSUPPORTED, "chunk must be 0 (default), 1 (recurrent) or 64");
    const la_config& c = h->cfg;
    const bool tc_ok = c.io == LA_BF16 && (c.d_k == 64 || c.d_k == 128) && (c.d_v == 64 || c.d_v == 128);
    if (chunk == 64 && !tc_ok)
        return fail(h, LA_ERR_UNSUPPORTED, "chunk 64 needs bf16 io and d_k, d_v in {64, 128}");
    if (static_cast<long long>(T) * (c.d_k > c.d_v ? c.d_k : c.d_v) > (1LL << 31) - 1)
        return fail(h, LA_ERR_UNSUPPORTED, "T * d exceeds 2^31 - 1");
    DeviceGuard g(c.device);
    if (!g.ok) return fail(h, LA_ERR_CUDA, "cannot select the handle's device");
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    cudaError_t e;
    if (!h->host_ready) {
        e = cudaStreamCreateWithFlags(&h->s_in, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->s_comp, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->s_out, cudaStreamNonBlocking);
        cudaEvent_t* evs[] = {&h->ev_start, &h->ev_done, &h->ev_in[0], &h->ev_in[1], &h->ev_comp[0], &h->ev_comp[1],
                              &h->ev_out[0], &h->ev_out[1]};
        for (cudaEvent_t* ev : evs)
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(h, e, "stream / event creation");
        h->host_ready = true;
    }

    // Sequence-heads in groups; per group the bytes of every staged tensor,
    // each slice 256-byte aligned.
    const int BH = c.B * c.H;
    const size_t io = (c.io == LA_BF16) ? 2 : 4;
    const size_t ss = state_elems(c, variant);
    const size_t tok = static_cast<size_t>(T);
    const size_t gate_per_head = (variant == LA_GLA || variant == LA_KDA) ? tok * c.d_k : (variant == LA_GDN) ? tok
                               : (variant == LA_NORM_DECAY) ? 1 : 0;
    const size_t per_head[9] = {
        tok * c.d_k * io, tok * c.d_k * io, tok * c.d_v * io,                    // q, k, v
        gate ? gate_per_head * 4 : 0, beta ? tok * 4 : 0, state_in ? ss * 4 : 0,  // gate, beta, state_in
        tok * c.d_v * io, state_out ? ss * 4 : 0, den_out ? tok * 4 : 0};         // out, state_out, den_out
    size_t call_bytes = 0;
    for (int i = 0; i < 9; ++i) call_bytes += per_head[i] * BH;
    const bool large = call_bytes >= kLargeCall;
    if (large && variant != LA_GLA) {
        e = cudaEventRecord(h->ev_start, s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h->s_in, h->ev_start, 0);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h->s_comp, h->ev_start, 0);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h->s_out, h->ev_start, 0);
        if (e != cudaSuccess) return cuda_fail(h, e, "stream ordering");
        rc = host_time_split(h, q, k, v, gate, beta, state_in, out, state_out, den_out, variant, T, chunk);
        if (rc != LA_OK) return rc;
        e = cudaEventRecord(h->ev_done, h->s_out);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, h->ev_done, 0);
        if (e != cudaSuccess) return cuda_fail(h, e, "stream ordering");
        return LA_OK;
    }
    const int want = large ? kHostGroupsLarge : kHostGroupsSmall;
    const int G0 = BH < want ? BH : want;
    const int gbh = (BH + G0 - 1) / G0;
    const int G = (BH + gbh - 1) / gbh;
    size_t off[9], buf = 0;
    for (int i = 0; i < 9; ++i) {
        off[i] = buf;
        buf += (per_head[i] * gbh + 255) & ~static_cast<size_t>(255);
    }
    if (2 * buf > h->stage_bytes) {
        // grow the staging (frees the old one after the work that used it)
        if (h->d_stage) {
            cudaStreamSynchronize(h->s_in);
            cudaStreamSynchronize(h->s_comp);
            cudaStreamSynchronize(h->s_out);
            cudaFree(h->d_stage);
            h->d_stage = nullptr;
            h->stage_bytes = 0;
        }
        e = cudaMalloc(&h->d_stage, 2 * buf);
        if (e != cudaSuccess) return cuda_fail(h, e, "staging allocation");
        h->stage_bytes = 2 * buf;
    }
    const void* src[6] = {q, k, v, gate, beta, state_in};
    void* dst[3] = {out, state_out, den_out};
    // copy kernels for a small call when the GPU can address every host
    // buffer, else the copy engines
    const uint8_t* msrc[6];
    uint8_t* mdst[3];
    bool by_kernel = !large;
    for (int i = 0; i < 6; ++i) {
        msrc[i] = mapped(src[i]);
        if (src[i] && !msrc[i]) by_kernel = false;
    }
    for (int i = 0; i < 3; ++i) {
        mdst[i] = const_cast<uint8_t*>(mapped(dst[i]));
        if (dst[i] && !mdst[i]) by_kernel = false;
    }

    // copy-in, compute and copy-out of group i overlap those of its
    // neighbours; each staging half b is reused two groups later, after its
    // kernels (copy-in waits) and its copy-out (compute waits) are done
    e = cudaEventRecord(h->ev_start, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->s_in, h->ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->s_comp, h->ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->s_out, h->ev_start, 0);
    if (e != cudaSuccess) return cuda_fail(h, e, "stream ordering");
    for (int gi = 0; gi < G; ++gi) {
        const int b = gi & 1;
        const int h0 = gi * gbh;
        const int nh = (BH - h0 < gbh) ? BH - h0 : gbh;
        uint8_t* st = h->d_stage + b * buf;
        if (gi >= 2) e = cudaStreamWaitEvent(h->s_in, h->ev_comp[b], 0);
        if (by_kernel && e == cudaSuccess) {
            CopyJob job{};
            for (int i = 0; i < 6; ++i)
                if (src[i] && per_head[i]) job.seg[job.n++] = {msrc[i] + per_head[i] * h0, st + off[i], per_head[i] * nh};
            copy_segments_kernel<<<kCopyCtas, 256, 0, h->s_in>>>(job);
            e = cudaGetLastError();
            ++h->last_launches;
        } else {
            for (int i = 0; i < 6 && e == cudaSuccess; ++i)
                if (src[i] && per_head[i])
                    e = cudaMemcpyAsync(st + off[i], static_cast<const uint8_t*>(src[i]) + per_head[i] * h0,
                                        per_head[i] * nh, cudaMemcpyHostToDevice, h->s_in);
        }
        if (e == cudaSuccess) e = cudaEventRecord(h->ev_in[b], h->s_in);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h->s_comp, h->ev_in[b], 0);
        if (e == cudaSuccess && gi >= 2) e = cudaStreamWaitEvent(h->s_comp, h->ev_out[b], 0);
        if (e != cudaSuccess) return cuda_fail(h, e, "staging copy-in");
        la::FwdArgs a = make_args(h, st + off[0], st + off[1], st + off[2],
                                  gate ? reinterpret_cast<const float*>(st + off[3]) : nullptr,
                                  beta ? reinterpret_cast<const float*>(st + off[4]) : nullptr,
                                  state_in ? reinterpret_cast<const float*>(st + off[5]) : nullptr, st + off[6],
                                  state_out ? reinterpret_cast<float*>(st + off[7]) : nullptr,
                                  den_out ? reinterpret_cast<float*>(st + off[8]) : nullptr, variant, T);
        a.BH = nh;
        rc = enqueue_forward(h, a, variant, chunk, h->s_comp);
        if (rc != LA_OK) return rc;
        e = cudaEventRecord(h->ev_comp[b], h->s_comp);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h->s_out, h->ev_comp[b], 0);
        if (by_kernel && e == cudaSuccess) {
            CopyJob job{};
            for (int i = 0; i < 3; ++i)
                if (dst[i] && per_head[6 + i])
                    job.seg[job.n++] = {st + off[6 + i], mdst[i] + per_head[6 + i] * h0, per_head[6 + i] * nh};
            copy_segments_kernel<<<kCopyCtas, 256, 0, h->s_out>>>(job);
            e = cudaGetLastError();
            ++h->last_launches;
        } else {
            for (int i = 0; i < 3 && e == cudaSuccess; ++i)
                if (dst[i] && per_head[6 + i])
                    e = cudaMemcpyAsync(static_cast<uint8_t*>(dst[i]) + per_head[6 + i] * h0, st + off[6 + i],
                                        per_head[6 + i] * nh, cudaMemcpyDeviceToHost, h->s_out);
        }
        if (e == cudaSuccess) e = cudaEventRecord(h->ev_out[b], h->s_out);
        if (e != cudaSuccess) return cuda_fail(h, e, "staging copy-out");
    }
    e = cudaEventRecord(h->ev_done, h->s_out);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, h->ev_done, 0);
    if (e != cudaSuccess) return cuda_fail(h, e, "stream ordering");
    return LA_OK;
}

int la_decode_step(la_handle* h, const void* q, const void* k, const void* v, const float* gate, const float* beta,
                   const float* state_in, void* out, float* state_out, float* den_out, int variant,
                   void* cuda_stream) {
    if (!h) return LA_ERR_INVALID_ARG;
    h->last_error.clear();
    h->last_launches = 0;
    int rc = check_common(h, q, k, v, gate, beta, state_in, out, state_out, den_out, variant);
    if (rc != LA_OK) return rc;
    if (!state_out) return fail(h, LA_ERR_INVALID_ARG, "state_out is required for a decode step");
    DeviceGuard g(h->cfg.device);
    if (!g.ok) return fail(h, LA_ERR_CUDA, "cannot select the handle's device");
    la::FwdArgs a = make_args(h, q, k, v, gate, beta, state_in, out, state_out, den_out, variant, 1);
    cudaError_t e = la::launch_decode(a, static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return cuda_fail(h, e, "decode kernel launch");
    h->last_launches = 1;
    return LA_OK;
}

int la_backward(la_handle* h, const void* q, const void* k, const void* v, const float* state_in, const void* dout,
                const float* dstate_out, void* dq, void* dk, void* dv, float* dstate_in, int variant, int T,
                void* cuda_stream) {
    if (!h) return LA_ERR_INVALID_ARG;
    h->last_error.clear();
    h->last_launches = 0;
    if (variant != LA_NORM_ELU1) return fail(h, LA_ERR_UNSUPPORTED, "la_backward supports LA_NORM_ELU1 only");
    if (T < 1) return fail(h, LA_ERR_INVALID_ARG, "T must be >= 1");
    if (!q || !k || !v || !dout || !dq || !dk || !dv)
        return fail(h, LA_ERR_INVALID_ARG, "q, k, v, dout, dq, dk and dv are required");
    const la_config& c = h->cfg;
    const bool small_d = (c.d_k == 16 || c.d_k == 32 || c.d_k == 64) && (c.d_v == 16 || c.d_v == 32 || c.d_v == 64);
    const bool rows_d = (c.d_k == 64 || c.d_k == 128) && (c.d_v == 64 || c.d_v == 128);
    if (!small_d && !rows_d)
        return fail(h, LA_ERR_UNSUPPORTED, "la_backward supports d_k, d_v in {16, 32, 64} or in {64, 128}");
    if (static_cast<long long>(T) * (c.d_k > c.d_v ? c.d_k : c.d_v) > (1LL << 31) - 1)
        return fail(h, LA_ERR_UNSUPPORTED, "T * d exceeds 2^31 - 1");
    const void* ptrs[] = {q, k, v, state_in, dout, dstate_out, dq, dk, dv, dstate_in};
    const char* names[] = {"q", "k", "v", "state_in", "dout", "dstate_out", "dq", "dk", "dv", "dstate_in"};
    for (int i = 0; i < 10; ++i)
        if (ptrs[i] && !aligned16(ptrs[i]))
            return fail(h, LA_ERR_MISALIGNED, std::string(names[i]) + " is not 16-byte aligned");
    DeviceGuard g(c.device);
    if (!g.ok) return fail(h, LA_ERR_CUDA, "cannot select the handle's device");
    la::BwdArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.state_in = state_in;
    a.dout = dout;
    a.dstate_out = dstate_out;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.dstate_in = dstate_in;
    a.BH = c.B * c.H;
    a.T = T;
    a.dk_dim = c.d_k;
    a.dv_dim = c.d_v;
    a.io = c.io == LA_FP32 ? la::kFp32 : la::kBf16;
    a.flags = c.flags;
    // The chunkwise tensor-core backward where the shape allows it and the
    // per-chunk states of at least one sequence-head fit the workspace: the
    // sequence-heads run in groups whose states fit it, one five-launch chain
    // per group. Otherwise the token-serial kernel.
    const size_t per_head = la::chunk::bwd_chunk_bytes(1, T);
    if (c.io == LA_BF16 && c.d_k == 64 && c.d_v == 64 && h->d_ws && per_head <= h->ws_bytes) {
        const int most = static_cast<int>(std::min<size_t>(h->ws_bytes / per_head, static_cast<size_t>(a.BH)));
        const int ngroups = (a.BH + most - 1) / most;
        const int group = (a.BH + ngroups - 1) / ngroups;   // groups of even size
        const size_t ss = static_cast<size_t>(c.d_k) * c.d_v + c.d_k;   // floats per state
        const size_t row = static_cast<size_t>(T) * 64 * 2;            // bytes of one head's q (= k, v, dout)
        auto off = [](const void* p, size_t bytes) -> const void* {
            return p ? static_cast<const uint8_t*>(p) + bytes : nullptr;
        };
        int launches = 0;
        for (int h0 = 0; h0 < a.BH; h0 += group) {
            la::BwdArgs g = a;
            g.BH = std::min(group, a.BH - h0);
            const size_t hb = static_cast<size_t>(h0) * row;
            const size_t sb = static_cast<size_t>(h0) * ss * sizeof(float);
            g.q = off(q, hb);
            g.k = off(k, hb);
            g.v = off(v, hb);
            g.dout = off(dout, hb);
            g.dq = const_cast<void*>(off(dq, hb));
            g.dk = const_cast<void*>(off(dk, hb));
            g.dv = const_cast<void*>(off(dv, hb));
            g.state_in = static_cast<const float*>(off(state_in, sb));
            g.dstate_out = static_cast<const float*>(off(dstate_out, sb));
            g.dstate_in = static_cast<float*>(const_cast<void*>(off(dstate_in, sb)));
            const cudaError_t e = la::chunk::launch_norm_backward_chunked(
                g, h->d_ws, h->ws_bytes, h->d_status, h->sm_count, h->encode, static_cast<cudaStream_t>(cuda_stream));
            if (e != cudaSuccess) return cuda_fail(h, e, "chunkwise backward launch");
            launches += 5;
        }
        h->last_launches = launches;
        return LA_OK;
    }
    // d_k, d_v in {64, 128}: the row-split kernel after a forward (it keeps
    // checkpoints, so its rounding does not grow with T); smaller heads: the
    // one-CTA-per-head kernel
    if (rows_d)
        return norm_rows_backward(h, q, k, v, nullptr, state_in, dout, dstate_out, dq, dk, dv, nullptr, dstate_in,
                                  LA_NORM_ELU1, T, static_cast<cudaStream_t>(cuda_stream));
    const cudaError_t e = la::launch_norm_backward(a, static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return cuda_fail(h, e, "backward kernel launch");
    h->last_launches = 1;
    return LA_OK;
}

int la_backward_gated(la_handle* h, const void* q, const void* k, const void* v, const float* gate, const float* beta,
                      const float* state_in, const void* dout, const float* dstate_out, void* dq, void* dk, void* dv,
                      float* dgate, float* dbeta, float* dstate_in, int variant, int T, void* cuda_stream) {
    if (!h) return LA_ERR_INVALID_ARG;
    h->last_error.clear();
    h->last_launches = 0;
    if (variant != LA_GDN && variant != LA_KDA && variant != LA_GLA && variant != LA_NORM_DECAY)
        return fail(h, LA_ERR_UNSUPPORTED, "la_backward_gated supports LA_GDN, LA_KDA, LA_GLA and LA_NORM_DECAY");
    if (T < 1) return fail(h, LA_ERR_INVALID_ARG, "T must be >= 1");
    const bool gla = variant == LA_GLA || variant == LA_NORM_DECAY;   // no beta
    if (!q || !k || !v || !gate || !dout || !dq || !dk || !dv || !dgate)
        return fail(h, LA_ERR_INVALID_ARG, "q, k, v, gate, dout, dq, dk, dv and dgate are required");
    if (!gla && (!beta || !dbeta)) return fail(h, LA_ERR_INVALID_ARG, "beta and dbeta are required");
    const la_config& c = h->cfg;
    if (!((c.d_k == 64 || c.d_k == 128) && (c.d_v == 64 || c.d_v == 128)))
        return fail(h, LA_ERR_UNSUPPORTED, "la_backward_gated supports d_k, d_v in {64, 128}");
    if (static_cast<long long>(T) * (c.d_k > c.d_v ? c.d_k : c.d_v) > (1LL << 31) - 1)
        return fail(h, LA_ERR_UNSUPPORTED, "T * d exceeds 2^31 - 1");
    const void* ptrs[] = {q, k, v, gate, beta, state_in, dout, dstate_out, dq, dk, dv, dgate, dbeta, dstate_in};
    const char* names[] = {"q", "k", "v", "gate", "beta", "state_in", "dout", "dstate_out", "dq", "dk", "dv",
                           "dgate", "dbeta", "dstate_in"};
    for (int i = 0; i < 14; ++i)
        if (ptrs[i] && !aligned16(ptrs[i]))
            return fail(h, LA_ERR_MISALIGNED, std::string(names[i]) + " is not 16-byte aligned");
    DeviceGuard g(c.device);
    if (!g.ok) return fail(h, LA_ERR_CUDA, "cannot select the handle's device");
    if (variant == LA_NORM_DECAY)
        return norm_rows_backward(h, q, k, v, gate, state_in, dout, dstate_out, dq, dk, dv, dgate, dstate_in,
                                  LA_NORM_DECAY, T, static_cast<cudaStream_t>(cuda_stream));
    const int BH = c.B * c.H;
    // the scalar-gate rule in bf16 with square heads: chunkwise kernels
    const bool chunked = variant == LA_GDN && c.io == LA_BF16 && c.d_k == c.d_v;
    const int grc = grow_bws(h, chunked ? la::gdn_chunk_backward_bytes(BH, T, c.d_k)
                                        : la::delta_backward_bytes(BH, T, c.d_k, c.d_v, gla));
    if (grc != LA_OK) return grc;
    la::DeltaBwdArgs a = {};
    a.q = q;
    a.k = k;
    a.v = v;
    a.gate = gate;
    a.beta = beta;
    a.state_in = state_in;
    a.dout = dout;
    a.dstate_out = dstate_out;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.dgate = dgate;
    a.dbeta = dbeta;
    a.dstate_in = dstate_in;
    a.BH = BH;
    a.T = T;
    a.dk_dim = c.d_k;
    a.dv_dim = c.d_v;
    a.io = c.io == LA_FP32 ? la::kFp32 : la::kBf16;
    a.per_channel = variant != LA_GDN;
    a.gla = gla;
    a.identity_phi = gla && (c.flags & LA_FLAG_IDENTITY_PHI);
    a.dq_acc = a.dk_acc = a.dv_acc = nullptr;
    if (gla) {
        a.beta = nullptr;
        a.dbeta = nullptr;
    }
    a.sm_count = h->sm_count;
    a.workspace = h->d_bws;
    if (chunked) {
        const cudaError_t e = la::launch_gdn_chunk_backward(a, static_cast<cudaStream_t>(cuda_stream));
        if (e != cudaSuccess) return cuda_fail(h, e, "gated backward launch");
        h->last_launches = 4;   // prep, both chunk chains in one launch, the two gradient kernels
        return LA_OK;
    }
    const cudaError_t e = la::launch_delta_backward(a, static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return cuda_fail(h, e, "gated backward launch");
    h->last_launches = 2;   // the token-serial kernel and the dq / dk conversion
    return LA_OK;
}

int la_last_launches(const la_handle* h) { return h ? h->last_launches : 0; }

int la_status(la_handle* h, void* cuda_stream) {
    if (!h) return LA_ERR_INVALID_ARG;
    DeviceGuard g(h->cfg.device);
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(h, e, "stream synchronize");
    int word = 0;
    e = cudaMemcpy(&word, h->d_status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(h, e, "status read");
    if (word != 0) {
        e = cudaMemset(h->d_status, 0, sizeof(int));
        if (e != cudaSuccess) return cuda_fail(h, e, "status clear");
        char buf[160];
        std::snprintf(buf, sizeof(buf), "a bounded device wait expired (status bits 0x%x: 1=TMA, 2=MMA, 4=test hook, 8=hand-off flag)", word);
        return fail(h, LA_ERR_TIMEOUT, buf);
    }
    return LA_OK;
}

}  // extern "C"
