// Host-side entry points of the chunkwise prefill, one per variant (each
// instantiated in its own translation unit so they compile in parallel).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "kernels.h"

namespace la {
namespace chunk {

struct Maps {
    CUtensorMap q, k, v, o;
};

struct Params;

// Normalized variant: the sequential chunk kernel (with segment summaries).
cudaError_t launch_norm(int dk, int dv, const Maps& m, const Params& p, int BH, cudaStream_t s);

// Gated delta rule (scalar or per-channel decay) and per-channel gated
// attention (the same kernel with T = I and W = 0): one cooperative
// launch per group of at most kGdnMaxGroup sequence-heads, in which prep CTAs
// feed a ring of per-chunk slots to one chain CTA per head; the workspace
// holds the hand-off flags and the ring (2 kGdnWindow chunks per head at
// most, as deep as the workspace allows).
constexpr int kGdnMaxGroup = 32;   // chain CTAs per launch
constexpr int kGdnWindow = 4;      // half the deepest ring, in chunks (8: a deeper ring spills L2)
size_t gdn_slot_bytes(int dk, int dv);
int gdn_group(int BH);
// Workspace for a ring of 2W chunks (W >= 1 is the least the launcher accepts).
size_t gdn_workspace_bytes(int BH, int dk, int dv, int W);
cudaError_t launch_gdn(const FwdArgs& a, const Maps& m, cudaStream_t s);

// Normalized, d_k = d_v = 64, no decay: one launch in which each CTA runs a
// segment of up to four 128-token blocks of one sequence-head, and the
// segments of a sequence-head (a thread-block cluster of at most 6) pass
// their totals through distributed shared memory. Fits when every
// sequence-head splits into such segments; needs no workspace.
bool seg_fits(int BH, int T, int dk, int dv, int sm_count);
cudaError_t launch_seg(const FwdArgs& a, const Maps& m, cudaStream_t s);

// Normalized: three fully parallel phases (chunk
// summaries, a scan over the chunks, outputs) when the per-chunk states of
// the whole problem fit in the workspace and comfortably in L2.
constexpr size_t kParL2Bytes = size_t(48) << 20;
size_t par_chunk_bytes(int dk, int dv);
size_t par_state_bytes(int dk, int dv);   // the same without the phi(k) tile
bool par_fits(int BH, int T, int dk, int dv, size_t ws_bytes);
cudaError_t launch_par(const FwdArgs& a, const Maps& m, cudaStream_t s);

// The first two phases alone (undecayed, d_k = d_v = 64), for the chunkwise
// backward: per chunk, the state entering it (bf16 [d_v][d_k] operand tile
// in xs, z in zs); dx and dd hold the chunk summaries and are free
// afterwards. phi(k) tiles are not kept. `end` is the first byte of the
// workspace past these arrays.
struct ParStates {
    float* dx;
    float* dd;
    uint8_t* xs;
    float* zs;
    uint8_t* end;
    int nch;
};
cudaError_t launch_par_states(const FwdArgs& a, const Maps& m, cudaStream_t s, ParStates* st);

// Chunkwise backward of the normalized variant (d_k = d_v = 64, bf16 io):
// workspace it needs, and the launch (five kernels: the two state phases
// above, then per-chunk normalizer gradients, the reverse scan of the state
// gradient, and the per-chunk input gradients).
size_t bwd_chunk_bytes(int BH, int T);
cudaError_t launch_norm_backward_chunked(const BwdArgs& a, float* workspace, size_t ws_bytes, int* status,
                                         int sm_count, PFN_cuTensorMapEncodeTiled_v12000 enc, cudaStream_t s);

}  // namespace chunk
}  // namespace la
