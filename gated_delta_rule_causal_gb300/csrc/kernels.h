// Internal interface between the C ABI (api.cu) and the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

namespace la {

enum Variant : int { kNorm = 0, kGla = 1, kGdn = 2, kKda = 3 };   // kKda: gated delta rule, per-channel decay
enum Io : int { kBf16 = 0, kFp32 = 1 };

// Everything a launch needs. Pointers are device pointers owned by the caller.
struct FwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* gate;
    const float* beta;
    const float* state_in;
    void* out;
    float* state_out;
    float* den_out;
    int BH;          // batch * heads
    int T;           // tokens per sequence (1 for decode)
    int dk, dv;
    int variant;     // Variant
    int io;          // Io
    unsigned flags;  // LA_FLAG_*
    int* status;     // device status word
    int sm_count;
    float* workspace;  // scratch for segment summaries (may be NULL)
    size_t ws_bytes;
    int* nlaunch;      // if not NULL, incremented by the number of kernels enqueued
};

// Token-by-token recurrence on CUDA cores; any supported head size, fp32 or
// bf16 io. One CTA per sequence-head.
cudaError_t launch_recurrent(const FwdArgs& a, cudaStream_t s);

// One decode step for every sequence-head; streams the fp32 state.
cudaError_t launch_decode(const FwdArgs& a, cudaStream_t s);

// Chunkwise tensor-core prefill (tcgen05, TMA); bf16 io, d_k, d_v in {64,128}.
// Returns cudaSuccess or the first CUDA error; `what` names the failing step.
cudaError_t launch_chunked(const FwdArgs& a, cudaStream_t s, PFN_cuTensorMapEncodeTiled_v12000 encode,
                           const char** what);

// Gradients of the normalized elu+1 recurrence (see backward.cu).
struct BwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* state_in;    // NULL: zero initial state
    const void* dout;         // gradient of the outputs [BH][T][dv]
    const float* dstate_out;  // gradient of the final state (S then z), or NULL
    void* dq;
    void* dk;
    void* dv;
    float* dstate_in;         // gradient of the initial state, or NULL
    int BH, T, dk_dim, dv_dim;
    int io;                   // Io
    unsigned flags = 0;       // LA_FLAG_* (the test hook)
};

// Gradients of the gated delta rule, scalar (gate [BH][T]) or per-channel
// (gate [BH][T][dk]) decay, state S [dv][dk] per sequence-head; or of the
// per-channel gated recurrence (gla: gate [BH][T][dk], no beta, state S
// [dk][dv]). Pointers are device pointers; dgate, dbeta and the accumulators
// are overwritten.
struct DeltaBwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* gate;
    const float* beta;
    const float* state_in;     // NULL: zero initial state
    const void* dout;
    const float* dstate_out;   // NULL: no gradient on the final state
    void* dq;
    void* dk;
    void* dv;
    float* dgate;
    float* dbeta;
    float* dstate_in;          // NULL: not wanted
    int BH, T, dk_dim, dv_dim;
    int io;                    // Io
    bool per_channel;
    bool gla;                  // per-channel gated recurrence (no beta; rows = key channels)
    bool norm;                 // normalized recurrence (rows = key channels; gate: one decay per
                               // sequence-head or NULL; dgate [BH] or NULL)
    bool identity_phi;         // gla without the feature map
    const void* fwd_out;       // norm: the forward's outputs [BH][T][dv] (io dtype)
    const float* fwd_den;      // norm: the forward's normalizers [BH][T]
    int sm_count;
    float* workspace;          // delta_backward_bytes(BH, T, dk, dv) bytes
    // carved from the workspace by the launch: rows at every segment start,
    // fp32 totals of dq and dk
    float* ckpt;
    float* dq_acc;
    float* dk_acc;
    float* dv_acc;             // gla, norm: fp32 total of dv
    float* ckz;                // norm: z at every segment start
};

// Workspace bytes launch_delta_backward needs (checkpoints + accumulators;
// norm: the caller places the forward's outputs and normalizers first, see
// norm_rows_fwd_bytes).
size_t delta_backward_bytes(int BH, int T, int dk, int dv, bool gla);
size_t norm_rows_bytes(int BH, int T, int dk, int dv);
size_t norm_rows_fwd_bytes(int BH, int T, int dv, int io);
// Token-serial CUDA-core kernel, rows split over CTAs (see backward_rows.cu);
// d_k, d_v in {64, 128}.
cudaError_t launch_delta_backward(const DeltaBwdArgs& a, cudaStream_t s);

// Chunkwise gradients of the scalar-gate delta rule (see backward_gdn.cu):
// bf16 io, dk_dim = dv_dim = 64 or 128, no per-channel decay. Four launches;
// the workspace holds gdn_chunk_backward_bytes(BH, T, d) bytes.
size_t gdn_chunk_backward_bytes(int BH, int T, int d);
cudaError_t launch_gdn_chunk_backward(const DeltaBwdArgs& a, cudaStream_t s);

// One CTA per sequence-head on CUDA cores; d_k, d_v in {16, 32, 64}.
cudaError_t launch_norm_backward(const BwdArgs& a, cudaStream_t s);

}  // namespace la
