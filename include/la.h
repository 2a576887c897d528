/*
 * la.h - C ABI of the causal linear-attention operator with a fixed matrix
 * state, for NVIDIA GB300 (sm_103a).
 *
 * The operator runs a sequence of tokens through a recurrent matrix state,
 * one independent recurrence per (batch, head). Five variants:
 *
 *   LA_NORM_ELU1  normalized kernel attention, phi(x) = elu(x) + 1:
 *                   S_t = S_{t-1} + phi(k_t) v_t^T,   z_t = z_{t-1} + phi(k_t),
 *                   o_t = phi(q_t)^T S_t / phi(q_t)^T z_t.
 *                 ("Linear Attention" concept page, normalized kernel
 *                 formulation; "Linear attention and recurrent memory", The
 *                 big idea; "Linear attention and Hyena", section 11.2.)
 *   LA_NORM_DECAY LA_NORM_ELU1 with a fixed decay per sequence-head,
 *                 gamma in (0, 1], on the state and the normalizer alike:
 *                   S_t = gamma S_{t-1} + phi(k_t) v_t^T,  z_t = gamma z_{t-1} + phi(k_t).
 *                 ("Linear attention and recurrent memory", Fixed decay
 *                 versus an input-dependent gate.)
 *   LA_GLA        per-channel gated attention (GLA / RetNet family):
 *                   S_t = diag(gamma_t) S_{t-1} + phi(k_t) v_t^T,  o_t = S_t^T phi(q_t),
 *                 gamma_t in (0,1]^{d_k}. ("Linear attention and Hyena",
 *                 section 11.3 and Exercise 11.5.)
 *   LA_GDN        gated delta rule, S in R^{d_v x d_k}, unit-length keys:
 *                   S_t = g_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *                   o_t = S_t q_t.
 *                 ("Beyond attention", section 18.2; "Linear Attention"
 *                 concept page, gated delta rule.)
 *   LA_KDA        LA_GDN with a per-channel (diagonal) decay on the key channels:
 *                   S_t = S_{t-1} Diag(alpha_t) (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *                 alpha_t in (0,1]^{d_k}. ("Linear attention and recurrent
 *                 memory", From fixed decay to KDA's gated delta write.)
 *
 * Decays of LA_GLA and LA_KDA below 2^-15 act as 2^-15 in the chunkwise
 * kernel (16-token sub-chunk references keep every factor exact in fp32
 * down to there): what crosses such a token is scaled by 2^-15 instead of
 * the decay, a departure of at most 2^-15 of the quantity crossing it. The
 * recurrent kernel (chunk 1) uses every decay as given.
 *
 * Every variant updates first and then reads, so token t attends to itself.
 *
 * LAYOUTS. Every tensor is contiguous and row-major. BH = B*H and (b,h) is
 * the index b*H + h.
 *   q, k       [B, H, T, d_k]   io dtype
 *   v, out     [B, H, T, d_v]   io dtype
 *   gate       LA_NORM_ELU1: unused (pass NULL)
 *              LA_NORM_DECAY: [B, H] fp32, gamma in (0, 1], one per sequence-head
 *              LA_GLA: [B, H, T, d_k] fp32, gamma in (0, 1]
 *              LA_GDN: [B, H, T] fp32, g in (0, 1]
 *              LA_KDA: [B, H, T, d_k] fp32, alpha in (0, 1]
 *   beta       LA_GDN, LA_KDA: [B, H, T] fp32 in [0, 1]; NULL otherwise
 *   state      fp32, one block per (b,h):
 *              LA_NORM_ELU1, LA_NORM_DECAY: S [d_k, d_v] immediately followed by z [d_k]
 *              LA_GLA:       S [d_k, d_v]
 *              LA_GDN, LA_KDA: S [d_v, d_k]
 *   den_out    LA_NORM_ELU1, LA_NORM_DECAY, optional: [B, H, T] fp32
 *              denominators phi(q_t)^T z_t.
 * For la_decode_step, drop the T axis: q,k [B,H,d_k], v,out [B,H,d_v],
 * gate [B,H,d_k] (gla, kda) or [B,H] (gdn, norm with decay), beta [B,H].
 *
 * Keys of LA_GDN and LA_KDA are assumed to have unit L2 norm; the library does not
 * normalize them. No scale is applied to q.
 *
 * OWNERSHIP. The caller owns every buffer. Pointers to q, k, v, gate, beta,
 * state and out are CUDA device pointers (device memory, or managed memory
 * resident on the device). The library never frees or retains them after a
 * call returns. la_create allocates the handle, one device status word and a
 * fixed workspace; la_destroy frees all three. The chunked prefill uses the
 * workspace
 *   - LA_NORM_ELU1: for the per-chunk states of the three-phase form (up to
 *     128 chunks per sequence-head, at most 48 MB; a call whose states do
 *     not fit takes the sequential kernel instead) and for segment summaries
 *     when B*H is too small to fill the GPU ((SM count) x (d_k*d_v + d_k)
 *     floats);
 *   - LA_GDN, LA_KDA, LA_GLA: for the hand-off flags and a ring of up to 8
 *     chunks of per-chunk intermediates for each of a group of
 *     G = min(B*H, 32) sequence-heads: G*8*(2*d_k*d_k + 256*d_k + 128*d_v
 *     + 8704) bytes plus a few KB, 22.7 MB at G = 32, d_k = d_v = 128 (a
 *     smaller workspace only makes the ring shallower).
 * The largest of these is allocated when the configuration can take the
 * tensor-core path (bf16, d_k, d_v in {64, 128}). Calls that overlap on the
 * GPU through the same handle (different streams) would share that
 * workspace: serialize them.
 *
 * EXECUTION. Calls are asynchronous on the given CUDA stream (NULL = the
 * legacy default stream) and never synchronize the device, except
 * la_status. A handle serves one host thread at a time.
 *
 * ERRORS. Every entry point returns 0 (LA_OK) or a positive LA_ERR_* code,
 * and validates all arguments before anything is launched, so a rejected
 * call never touches the GPU. la_last_error(h) returns the text of the
 * last failure on h. Nothing is printed and no exception crosses the ABI.
 * Device-side failures (a bounded wait that expired) are recorded in the
 * device status word and reported by la_status.
 */
#ifndef LA_H
#define LA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct la_handle la_handle;

typedef enum { LA_NORM_ELU1 = 0, LA_GLA = 1, LA_GDN = 2, LA_NORM_DECAY = 3, LA_KDA = 4 } la_variant;

/* dtype of q, k, v and out. State, gates and beta are always fp32. */
typedef enum { LA_BF16 = 0, LA_FP32 = 1 } la_dtype;

enum {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = 1,  /* NULL handle or required pointer, bad enum, negative size */
    LA_ERR_UNSUPPORTED = 2,  /* head size or chunk size outside the supported set, wrong GPU */
    LA_ERR_MISALIGNED = 3,   /* a tensor pointer is not 16-byte aligned */
    LA_ERR_CUDA = 4,         /* a CUDA runtime call failed; see la_last_error */
    LA_ERR_TIMEOUT = 5       /* a bounded wait inside a kernel expired (la_status) */
};

/* la_config.flags */
#define LA_FLAG_IDENTITY_PHI 0x1u   /* LA_GLA without the feature map (phi = identity) */
#define LA_FLAG_SEQUENTIAL_CHUNKS 0x2u /* LA_NORM_ELU1 chunked prefill: always walk the
                                          chunks of a sequence-head in order (split into segments
                                          when B*H is small) instead of the three-phase parallel
                                          form the library picks when the per-chunk states fit
                                          its workspace; results agree within rounding */
#define LA_FLAG_TEST_TIMEOUT 0x100u /* test hook: the chunked prefill kernel waits once on a
                                       barrier nothing signals, with a 1 ms limit, then
                                       records LA_ERR_TIMEOUT in the status word and exits */

typedef struct {
    int B;          /* batch, >= 1 */
    int H;          /* heads, >= 1 */
    int d_k;        /* key/query size: 16, 32, 64 or 128 */
    int d_v;        /* value size: 16, 32, 64 or 128 */
    la_dtype io;    /* dtype of q, k, v, out */
    unsigned flags; /* LA_FLAG_* */
    int device;     /* CUDA device ordinal the handle is bound to */
} la_config;

/* Create a handle bound to cfg->device. Checks that the device is an
 * sm_103 GPU (LA_ERR_UNSUPPORTED otherwise). */
int la_create(const la_config* cfg, la_handle** out);

/*
 * Prefill: run T tokens of every (b,h) sequence from state_in and write the
 * outputs and the final state.
 *   state_in  NULL means S_0 = 0 (and z_0 = 0).
 *   state_out NULL means the final state is not written. It may alias
 *             state_in.
 *   T         tokens per sequence, >= 0. T = 0 writes no output and copies
 *             state_in (or zeros) to state_out.
 *   chunk     0 = default (64). 1 = token-by-token recurrent kernel. 64 =
 *             chunkwise tensor-core kernel (bf16 io, d_k and d_v in {64, 128}).
 *             fp32 io and head sizes 16/32 always use the recurrent kernel.
 *             LA_NORM_ELU1 and LA_NORM_DECAY with d_k = d_v = 64 compute
 *             their chunkwise form in blocks of 128 tokens, in one launch,
 *             when each sequence-head splits into at most
 *             min(6, SM count / (B*H)) segments (one segment when B*H > SM
 *             count) of at most 4 blocks each; the segments of a
 *             sequence-head form one thread-block cluster. Otherwise they
 *             take the forms described under the workspace below. LA_GDN,
 *             LA_KDA and LA_GLA run one cooperative launch per group of up
 *             to 32 sequence-heads.
 *             Other values: LA_ERR_UNSUPPORTED.
 *   den_out   optional, LA_NORM_ELU1 and LA_NORM_DECAY only.
 * Every pointer must be 16-byte aligned (LA_ERR_MISALIGNED otherwise).
 * LA_NORM_DECAY runs chunkwise in the single-launch form (d_k = d_v = 64,
 * as above) or the three-phase form; a call that fits neither runs the
 * recurrent kernel.
 */
int la_forward(la_handle* h, const void* q, const void* k, const void* v,
               const float* gate, const float* beta, const float* state_in,
               void* out, float* state_out, float* den_out,
               int variant, int T, int chunk, void* cuda_stream);

/*
 * Prefill from host memory: the same operation and arguments as la_forward,
 * but q, k, v, gate, beta, state_in, out, state_out and den_out are host
 * pointers (page-locked memory, cudaHostAlloc or cudaHostRegister, for the
 * copies to run asynchronously). The library splits the call into pieces
 * and, on three streams of its own, copies piece i + 1 in, runs the kernels
 * of piece i and copies piece i - 1 out at the same time. A call that moves
 * less than 64 MiB over the host link runs as up to 2 groups of
 * sequence-heads and, when the GPU can address every buffer (page-locked
 * memory under unified addressing), one copy kernel per group and direction
 * moves the data; otherwise the copy engine does, one copy per tensor. A
 * call of 64 MiB or more is moved by the copy engines, which leave every SM
 * to the kernels: split along the sequence into 4 segments of every
 * sequence-head (multiples of 64 tokens, one strided copy per tensor and
 * segment, the state handed from segment to segment in device memory), or,
 * for LA_GLA, into up to 4 groups of sequence-heads. la_last_launches counts
 * the copy kernels too. Staging for two
 * groups lives in device memory that the handle allocates on
 * first use and grows when a call needs more (la_destroy frees it). The call
 * is ordered after the work already enqueued on cuda_stream, and the work
 * enqueued on cuda_stream after it waits for its last copy-out; the host
 * buffers must stay valid until then. T >= 1. Calls through one handle must
 * not overlap (they share the staging and the workspace).
 */
int la_forward_host(la_handle* h, const void* q, const void* k, const void* v,
                    const float* gate, const float* beta, const float* state_in,
                    void* out, float* state_out, float* den_out,
                    int variant, int T, int chunk, void* cuda_stream);

/*
 * One decode step: advance every (b,h) state by one token and write its
 * output. state_out may equal state_in, which updates the state in place.
 * state_in NULL means a zero state. state_out must not be NULL.
 * den_out is optional ([B,H] fp32, LA_NORM_ELU1 and LA_NORM_DECAY only).
 */
int la_decode_step(la_handle* h, const void* q, const void* k, const void* v,
                   const float* gate, const float* beta, const float* state_in,
                   void* out, float* state_out, float* den_out,
                   int variant, void* cuda_stream);

/*
 * Prefill without any device allocation by the library (no handle).
 *
 * The pages describe no counterpart of this call; it exists for callers that
 * cannot let a library call cudaMalloc: code running under a host framework
 * that owns all device memory (an inference server or plugin host with its
 * own pool), or a latency-critical loop that forbids allocation after
 * start-up. la_create allocates, so this entry point takes the configuration
 * directly and computes exactly what la_forward computes with the chunkwise
 * tensor-core kernel (chunk 64; bf16 io; d_k, d_v in {64, 128}; all three
 * variants). Arguments, layouts and results are those of la_forward.
 *
 * Scratch: a file-scope device array of 16 MiB in the library's own image,
 * held on every GPU that loads the library until the process exits. It holds
 * the segment summaries of the normalized and per-channel gated variants and
 * a status word for expired device waits, which this call does not read
 * (it returns before its kernels run): la_noalloc_status reports it. A shape
 * whose summaries would not fit returns LA_ERR_UNSUPPORTED; on a GB300 every
 * supported shape fits. Every call shares the array: calls that overlap on
 * the GPU (different streams, or other host threads) race on it and must be
 * serialized by the caller.
 *
 * Set-up: the first call on a device, with cfg->device current, resolves the
 * array's device address, clears the status word and loads the tensor-map
 * encoder; make that first call before any stream capture. cfg->device must
 * be the current device (LA_ERR_INVALID_ARG otherwise).
 */
int la_forward_noalloc(const la_config* cfg, const void* q, const void* k, const void* v,
                       const float* gate, const float* beta, const float* state_in,
                       void* out, float* state_out, float* den_out,
                       int variant, int T, void* cuda_stream);

/* The status of la_forward_noalloc calls on `device` (which must be the
 * current device): synchronize cuda_stream, then read and clear the status
 * word in the static scratch. Returns LA_OK, LA_ERR_TIMEOUT if one of those
 * calls' kernels recorded an expired bounded wait since the word was last
 * cleared (its outputs are then not valid), LA_ERR_INVALID_ARG or
 * LA_ERR_CUDA. Allocates nothing. The word is shared by every such call on
 * the device, whatever the stream. */
int la_noalloc_status(int device, void* cuda_stream);

/* Synchronize cuda_stream, then read and clear the device status word.
 * Returns LA_OK, LA_ERR_TIMEOUT if a kernel recorded an expired wait since
 * the last call, or LA_ERR_CUDA. */
int la_status(la_handle* h, void* cuda_stream);

/* Destroy a handle (NULL is allowed). */
void la_destroy(la_handle* h);

/* Text of the last failure on h ("" if none). Valid until the next call on h. */
const char* la_last_error(const la_handle* h);

/*
 * Backward of the prefill (LA_NORM_ELU1 only; d_k, d_v both in {16, 32, 64}
 * or both in {64, 128}; bf16 or fp32 io; the fixed-decay form's gradients
 * are in la_backward_gated). Given the same q, k, v, state_in as a forward call and the
 * gradients of its outputs (dout [B,H,T,d_v], io dtype) and, optionally, of
 * its final state (dstate_out, fp32, S then z as above; NULL means zero),
 * writes the gradients dq, dk [B,H,T,d_k], dv [B,H,T,d_v] (io dtype) and,
 * if dstate_in is not NULL, the gradient of the initial state (fp32, same
 * layout). The pages give the forward operator only; the gradients follow
 * from the chain rule through the update-first recurrence (phi'(x) = 1 for
 * x > 0, e^x otherwise).
 * bf16 io with d_k = d_v = 64: the chunkwise tensor-core form (chunks of 64
 * tokens), five kernels per group of sequence-heads whose per-chunk states
 * fit the handle's workspace (about 41 KB per chunk of each sequence-head):
 * the states entering every chunk, per-chunk normalizer gradients, a reverse
 * scan of the state gradient, and the per-chunk input gradients. Other
 * shapes with d_k, d_v in {64, 128} (fp32 io, d = 128, or a single
 * sequence-head whose chunk states exceed the workspace): a forward call
 * (its outputs and normalizers into the backward workspace), then the
 * token-serial row kernel of la_backward_gated (key channels as rows,
 * checkpoints every 8 tokens). d_k, d_v in {16, 32}: one CUDA-core kernel
 * per sequence-head that runs the recurrence forward to the final state,
 * then backward, recovering earlier states by subtracting each token's
 * update, so its fp32 rounding grows with T. la_last_launches tells which
 * ran (a multiple of 5; the forward's launches + 2; or 1). An expired
 * bounded wait in the chunkwise kernels is reported by la_status.
 * Errors as for la_forward: LA_ERR_UNSUPPORTED for another variant or head
 * size, LA_ERR_INVALID_ARG, LA_ERR_MISALIGNED, LA_ERR_CUDA.
 */
int la_backward(la_handle* h, const void* q, const void* k, const void* v,
                const float* state_in, const void* dout, const float* dstate_out,
                void* dq, void* dk, void* dv, float* dstate_in,
                int variant, int T, void* cuda_stream);

/*
 * Backward of the prefill of the gated delta rule (LA_GDN), of its
 * per-channel-decay form (LA_KDA), of the per-channel gated variant (LA_GLA)
 * and of the normalized variant with a fixed decay per sequence-head
 * (LA_NORM_DECAY: gate [B,H], dgate [B,H], state S then z as in la_forward;
 * a forward call runs first, as for la_backward's larger heads); d_k, d_v in
 * {64, 128}; bf16 or fp32 io.
 * Given the forward call's q, k, v, gate, beta and state_in (same layouts as
 * la_forward: gate [B,H,T] for LA_GDN, [B,H,T,d_k] for LA_KDA and LA_GLA; beta
 * [B,H,T]; state_in [B,H,d_v*d_k] fp32 or NULL for zero), the gradient of
 * its outputs (dout [B,H,T,d_v], io dtype) and optionally of its final state
 * (dstate_out, fp32, same layout as the state; NULL means zero), writes dq,
 * dk [B,H,T,d_k] and dv [B,H,T,d_v] (io dtype), dgate (fp32, the gate's
 * shape), dbeta [B,H,T] (fp32) and, if dstate_in is not NULL, the gradient
 * of the initial state (fp32). The pages give the forward operator only; the
 * gradients follow from the chain rule through the decay-first delta rule
 * (S~ = S Diag(a), u = beta (v - S~ k), S = S~ + u k^T, o = S q) and, for
 * LA_GLA, through S_t = diag(gamma_t) S_{t-1} + phi(k_t) v_t^T,
 * o_t = S_t^T phi(q_t) (phi = elu + 1, the identity under
 * LA_FLAG_IDENTITY_PHI). LA_GLA and LA_NORM_DECAY take no beta: beta and
 * dbeta may be NULL and are ignored; LA_GLA's state_in, dstate_out and
 * dstate_in are [B,H,d_k*d_v] (S [d_k][d_v]).
 * LA_GDN with bf16 io and d_k = d_v (64 or 128): the chunkwise form (chunks
 * of 64 tokens), four launches: a per-chunk prep (the UT inverse of the
 * chunk and its W, Ut and gam Q - P W), one launch walking both chunk chains
 * (the state forward, its gradient backward, value rows split over CTAs),
 * and two per-chunk gradient kernels; every product is a tf32 MMA with fp32
 * accumulation. Its workspace is 4 * B*H * ceil(T/64) * (8*64*d + 64*64 +
 * 4*64) + 2 * B*H * ceil(T/64) * 2*d*d bytes (d = d_k, each part rounded up
 * to 256 bytes); la_last_launches reports 4. The gate gradient's per-chunk
 * terms are added by several CTAs in fp32, so its last bits may vary from
 * run to run.
 * Every other case: a token-serial CUDA-core kernel: the state's value rows
 * (LA_GLA: its key channels) are split over CTAs of 16 rows, run forward
 * with checkpoints every 8 tokens, then walked back segment by segment; sums
 * over rows are accumulated in fp32 (the order of those additions varies
 * from run to run, so the last bits of dq, dk, dgate and dbeta, or of
 * LA_GLA's dv, may too). Its workspace (4 * B*H * (ceil(T/8) * d_v*d_k +
 * 2*T*d_k) bytes; LA_GLA: T*d_v in place of 2*T*d_k) and the chunkwise one
 * are allocated by the handle on first use and grown when a call needs more
 * (la_destroy frees it). la_last_launches reports 2 (plus memsets of the
 * accumulated outputs, not counted; LA_NORM_DECAY: the forward's launches
 * plus 2).
 * Errors: LA_ERR_UNSUPPORTED for another variant or head size,
 * LA_ERR_INVALID_ARG (T < 1, a required pointer NULL), LA_ERR_MISALIGNED,
 * LA_ERR_CUDA.
 */
int la_backward_gated(la_handle* h, const void* q, const void* k, const void* v,
                      const float* gate, const float* beta, const float* state_in,
                      const void* dout, const float* dstate_out,
                      void* dq, void* dk, void* dv, float* dgate, float* dbeta, float* dstate_in,
                      int variant, int T, void* cuda_stream);

/* Number of CUDA kernels the last successful la_forward / la_decode_step /
 * la_backward on h enqueued (0 after a failed or a T = 0 call, or for a NULL
 * handle). A diagnostic: which algorithm the library picked shows in this
 * count (1: the recurrent kernel or a decode step; 1 or 2: the chunk kernel,
 * with segment summaries when B*H is small; 3: the three-phase parallel form;
 * LA_GDN, LA_KDA and LA_GLA: one per group of 32 sequence-heads; la_backward:
 * 5 per head group for the chunkwise form, 1 for the token-serial kernel;
 * la_backward_gated: 4 for the chunkwise form, 2 for the token-serial one,
 * the forward's + 2 for LA_NORM_DECAY). */
int la_last_launches(const la_handle* h);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int la_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LA_H */
