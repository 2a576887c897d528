// la_forward_noalloc: the chunked tensor-core prefill without any device
// allocation by the library.
//
// Some callers cannot let a library call cudaMalloc: code that runs inside a
// host framework owning all device memory (an inference server, a plugin
// host with its own pool), or latency-critical loops that forbid allocation
// after start-up. la_create allocates (the status word and the segment
// workspace), so this entry point takes the configuration directly and uses
// a scratch array that lives in the library's own device image instead.
//
// The scratch is one file-scope array of kScratchBytes per GPU that loads the
// library; it stays allocated until the process exits. Its first 256 bytes
// hold the status word the kernels set when a bounded wait expires
// (la_noalloc_status reads and clears it); the rest
// holds segment summaries (normalized / gated), which the summary kernel fully
// writes before the chunk kernel reads them, or the gated delta rule's states
// and per-chunk slots, each written by one launch before the next reads it,
// so nothing else needs clearing between calls.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/la.h"
#include "kernels.h"
#include "prefill.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB per device
constexpr size_t kStatusBytes = 256;                // status word, padded

// In host code this name is only a stand-in for the device array; the device
// address comes from cudaGetSymbolAddress (per device, with it current).
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// First call on a device: resolve the scratch address, clear the status word,
// fetch the SM count and the tensor-map encoder. Returns 0 or an LA_ERR_*.
int setup(int dev, void** addr, int* sms) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return LA_ERR_CUDA;
        }
        if (cudaMemset(p, 0, kStatusBytes) != cudaSuccess) {
            cudaGetLastError();
            return LA_ERR_CUDA;
        }
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return LA_ERR_CUDA;
        }
        g_sms[dev] = n;
        g_addr[dev] = p;
    }
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn) {
            cudaGetLastError();
            return LA_ERR_CUDA;
        }
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *addr = g_addr[dev];
    *sms = g_sms[dev];
    return LA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Scratch the chunked prefill needs for this shape: the segment summaries the
// normalized / gated launcher picks (mirrors it), or the least the gated
// delta rule's launcher accepts (it sizes its windows to the scratch).
size_t scratch_needed(int variant, int BH, int T, int dk, int dv, int sms) {
    const int nch = (T + 63) / 64;
    // the gated delta rule, and the gated variant when the three-phase form
    // does not fit: the least ring the prep/chain launcher accepts
    if (variant == LA_GDN || variant == LA_GLA) return la::chunk::gdn_workspace_bytes(BH, dk, dv, 1);
    if (BH >= sms || nch < 4) return 0;
    int nseg = sms / BH;
    if (nseg > nch / 2) nseg = nch / 2;
    if (nseg <= 1) return 0;
    const int seg_len = (nch + nseg - 1) / nseg;
    nseg = (nch + seg_len - 1) / seg_len;
    return static_cast<size_t>(BH) * (nseg - 1) * (static_cast<size_t>(dk) * dv + dk) * sizeof(float);
}

}  // namespace

extern "C" int la_forward_noalloc(const la_config* cfg, const void* q, const void* k, const void* v,
                                  const float* gate, const float* beta, const float* state_in, void* out,
                                  float* state_out, float* den_out, int variant, int T, void* cuda_stream) {
    if (!cfg) return LA_ERR_INVALID_ARG;
    if (cfg->B < 1 || cfg->H < 1 || T < 1) return LA_ERR_INVALID_ARG;
    if (variant != LA_NORM_ELU1 && variant != LA_GLA && variant != LA_GDN) return LA_ERR_INVALID_ARG;
    if (cfg->io != LA_BF16) return LA_ERR_UNSUPPORTED;
    if (!((cfg->d_k == 64 || cfg->d_k == 128) && (cfg->d_v == 64 || cfg->d_v == 128))) return LA_ERR_UNSUPPORTED;
    if (!q || !k || !v || !out) return LA_ERR_INVALID_ARG;
    if (variant != LA_NORM_ELU1 && !gate) return LA_ERR_INVALID_ARG;
    if (variant == LA_GDN && !beta) return LA_ERR_INVALID_ARG;
    if (variant != LA_NORM_ELU1 && den_out) return LA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, gate, beta, state_in, out, state_out, den_out};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return LA_ERR_MISALIGNED;
    if (static_cast<long long>(cfg->B) * cfg->H > (1LL << 30)) return LA_ERR_UNSUPPORTED;
    if (static_cast<long long>(T) * (cfg->d_k > cfg->d_v ? cfg->d_k : cfg->d_v) > (1LL << 31) - 1)
        return LA_ERR_UNSUPPORTED;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return LA_ERR_CUDA;
    }
    if (dev != cfg->device) return LA_ERR_INVALID_ARG;  // the caller makes cfg->device current
    void* base = nullptr;
    int sms = 0;
    const int rc = setup(dev, &base, &sms);
    if (rc != LA_OK) return rc;

    const int BH = cfg->B * cfg->H;
    if (scratch_needed(variant, BH, T, cfg->d_k, cfg->d_v, sms) > kScratchBytes - kStatusBytes)
        return LA_ERR_UNSUPPORTED;  // the shape needs more scratch than the static array holds

    la::FwdArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    // Plain LA_NORM_ELU1 carries no gate, as in la_forward: the normalized
    // kernels read a non-NULL gate as a per-(b,h) decay.
    a.gate = (variant == LA_NORM_ELU1) ? nullptr : gate;
    a.beta = beta;
    a.state_in = state_in;
    a.out = out;
    a.state_out = state_out;
    a.den_out = den_out;
    a.BH = BH;
    a.T = T;
    a.dk = cfg->d_k;
    a.dv = cfg->d_v;
    a.variant = variant;
    a.io = la::kBf16;
    a.flags = cfg->flags;
    a.status = static_cast<int*>(base);
    a.sm_count = sms;
    a.workspace = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + kStatusBytes);
    a.ws_bytes = kScratchBytes - kStatusBytes;
    a.nlaunch = nullptr;
    const char* what = "";
    if (la::launch_chunked(a, static_cast<cudaStream_t>(cuda_stream), g_encode, &what) != cudaSuccess) {
        cudaGetLastError();
        return LA_ERR_CUDA;
    }
    return LA_OK;
}

extern "C" int la_noalloc_status(int device, void* cuda_stream) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return LA_ERR_CUDA;
    }
    if (dev != device) return LA_ERR_INVALID_ARG;  // the caller makes `device` current
    void* base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        base = g_addr[dev];
    }
    if (!base) return LA_OK;  // no call has run on this device: nothing can have failed
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) {
        cudaGetLastError();
        return LA_ERR_CUDA;
    }
    int word = 0;
    if (cudaMemcpy(&word, base, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return LA_ERR_CUDA;
    }
    if (word == 0) return LA_OK;
    if (cudaMemset(base, 0, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return LA_ERR_CUDA;
    }
    return LA_ERR_TIMEOUT;
}
