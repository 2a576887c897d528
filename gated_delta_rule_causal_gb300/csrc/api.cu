// C ABI of the library (declared in include/la.h): argument validation,
// kernel selection and the device status word.
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
};

namespace {

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

bool valid_variant(int v) { return v == LA_NORM_ELU1 || v == LA_GLA || v == LA_GDN || v == LA_NORM_DECAY; }

size_t state_elems(const la_config& c, int variant) {
    return static_cast<size_t>(c.d_k) * c.d_v + ((variant == LA_NORM_ELU1 || variant == LA_NORM_DECAY) ? c.d_k : 0);
}

int check_common(la_handle* h, const void* q, const void* k, const void* v, const float* gate,
                 const float* beta, const float* state_in, const void* out, const float* state_out,
                 const float* den_out, int variant) {
    if (!valid_variant(variant))
        return fail(h, LA_ERR_INVALID_ARG, "variant must be LA_NORM_ELU1, LA_GLA, LA_GDN or LA_NORM_DECAY");
    if (!q || !k || !v || !out) return fail(h, LA_ERR_INVALID_ARG, "q, k, v and out are required");
    if (variant != LA_NORM_ELU1 && !gate)
        return fail(h, LA_ERR_INVALID_ARG, "gate is required for LA_GLA, LA_GDN and LA_NORM_DECAY");
    if (variant == LA_GDN && !beta) return fail(h, LA_ERR_INVALID_ARG, "beta is required for LA_GDN");
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
    a.variant = (variant == LA_NORM_DECAY) ? la::kNorm : variant;
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
            return fail(h, LA_ERR_INVALID_ARG, "variant must be LA_NORM_ELU1, LA_GLA, LA_GDN or LA_NORM_DECAY");
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
    cudaError_t e;
    // the decayed normalized variant runs chunkwise only in the three-phase form
    const bool chunked = tc_ok && chunk != 1 &&
                         (variant != LA_NORM_DECAY ||
                          (!(c.flags & LA_FLAG_SEQUENTIAL_CHUNKS) &&
                           la::chunk::par_fits(a.BH, T, c.d_k, c.d_v, h->ws_bytes)));
    if (chunked) {
        const char* what = "";
        e = la::launch_chunked(a, s, h->encode, &what);
        if (e != cudaSuccess) return cuda_fail(h, e, what);
    } else {
        e = la::launch_recurrent(a, s);
        if (e != cudaSuccess) return cuda_fail(h, e, "recurrent kernel launch");
        h->last_launches = 1;
    }
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
        std::snprintf(buf, sizeof(buf), "a bounded device wait expired (status bits 0x%x: 1=TMA, 2=MMA, 4=test hook)", word);
        return fail(h, LA_ERR_TIMEOUT, buf);
    }
    return LA_OK;
}

}  // extern "C"
