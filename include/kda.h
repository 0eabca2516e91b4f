/*
 * kda.h -- C ABI of the Kimi Delta Attention (KDA) operator for NVIDIA GB300
 * (sm_103a).
 *
 * KDA is the gated delta-rule recurrence with one retention value per key
 * channel.  Per head, with a state S of d_k x d_v numbers (row i = key
 * channel i):
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 *     alpha_t = exp(g_t),     o_t = S_t^T q_t   (read after the update)
 *
 * Sources (page title -- section):
 *   "Kimi K3 Architecture Explained" -- Step 3 "Forgetting, Channel by
 *       Channel" (the recurrence, rows = key channels) and "Inside a KDA Layer".
 *   "From GPT-2 to Kimi K3, from first principles" -- Chapter 5 (the four
 *       verbs retain/erase/write/read; g = gmin*sigmoid(z), gmin = -5) and
 *       Chapter 6 (chunked prefill vs. fused-recurrent single-token decode).
 *   "An infra-oriented diagram of Kimi K3" -- KDA card (96 heads, 128 x 128
 *       state, width-4 depthwise causal conv, Swish, L2Norm, scaled-sigmoid
 *       decay, sigmoid beta) and the packed-token note (cumulative sequence
 *       offsets delimit documents).
 *
 * Conventions shared by every entry point
 *   - All tensor arguments are DEVICE pointers owned by the caller; the
 *     library never allocates, frees or keeps them.  Tensors are dense,
 *     row-major and 16-byte aligned, except beta / z_beta ([T, H] fp32,
 *     read element by element), which need only 4-byte alignment.
 *   - Layouts:  q, k, g   [T, H, d_k]      v, out  [T, H, d_v]
 *               beta      [T, H]           states  [N, H, d_k, d_v] fp32
 *               cu_seqlens [N + 1] int32: document n owns tokens
 *               cu_seqlens[n] .. cu_seqlens[n+1]-1; cu_seqlens[0] = 0 and
 *               cu_seqlens[N] = T.  Documents never see each other: state
 *               and conv history restart at every document.
 *   - q/k/v (and out) are fp32 or bf16 (kda_dims.qkv_dtype); g, beta and
 *     every state are fp32.  Arithmetic is fp32 on CUDA cores or bf16
 *     operands with fp32 accumulation on the tensor cores.
 *   - Supported head sizes: d_k = d_v in {16, 32, 64, 128}; anything else
 *     returns KDA_ERR_UNSUPPORTED.  The tensor-core prefill serves
 *     d = 128 with bf16 inputs; the other shapes use the CUDA-core path.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *     is asynchronous: the returned status covers argument checks and the
 *     kernel launches only.  Invalid arguments return an error and launch
 *     nothing.  Errors found on the device go to the workspace status word
 *     (kda_get_device_status).
 *   - kda_last_error() returns a thread-local message for the last failure.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID = 1,      /* bad pointer, size, alignment or layout      */
    KDA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (head size, dtype) */
    KDA_ERR_CUDA = 3,         /* a CUDA runtime call failed                   */
    KDA_ERR_TIMEOUT = 4,      /* a device-side wait gave up (status word)     */
    KDA_ERR_DEVICE = 5        /* the device flagged bad input (status word)   */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/* Device status word values (kda_get_device_status). */
#define KDA_DEVICE_OK 0
#define KDA_DEVICE_BAD_OFFSETS 1  /* cu_seqlens not 0..T and non-decreasing */
#define KDA_DEVICE_TIMEOUT 2      /* a bounded device-side wait ran out      */
#define KDA_DEVICE_RANGE 3        /* a value the tensor-core prefill keeps in fp16 operands (v, the
                                     state, the pseudo-values) reached 65504 in magnitude: the
                                     results of that call are not valid                          */
#define KDA_DEVICE_BAD_SNAPSHOT 4 /* a snapshot offset outside (0, T], out of order, or neither a
                                     multiple of KDA_SNAPSHOT_ALIGN into its document nor its end */

/* Prefix snapshots are taken every multiple of this many tokens into a document. */
#define KDA_SNAPSHOT_ALIGN 64

typedef struct {
    int32_t H;          /* heads                                   */
    int32_t d_k;        /* key/query channels per head             */
    int32_t d_v;        /* value channels per head (= d_k)         */
    int32_t qkv_dtype;  /* kda_dtype of q, k, v and of out         */
} kda_dims;

/*
 * Bytes of device workspace kda_prefill takes for T packed tokens in N
 * documents: 256 for the device status word and, when N > 1, N int32 (rounded
 * up to 256 bytes) for the order in which the documents get their CTAs,
 * longest first.  The caller allocates it, 256-byte aligned, and may reuse it
 * across calls that do not overlap on the GPU.
 */
KDA_API size_t kda_prefill_workspace_size(kda_dims dims, int64_t T, int32_t N);

/*
 * Multi-token prefill of N packed documents ("chunk" mode of "From GPT-2 to
 * Kimi K3", Chapter 6; the recurrence of "Kimi K3 Architecture Explained",
 * Step 3).
 *   q, k     [T, H, d_k]  qkv_dtype; q and k are expected L2-normalised
 *   v        [T, H, d_v]  qkv_dtype
 *   g        [T, H, d_k]  fp32 log-decay (alpha = exp(g)), normally in (-5, 0)
 *   beta     [T, H]       fp32 write strength
 *   init_state [N, H, d_k, d_v] fp32 or NULL (zero state)
 *   cu_seqlens [N + 1] int32 device offsets, or NULL when N == 1 (one
 *              document of T tokens)
 *   out      [T, H, d_v]  qkv_dtype, written for every token
 *   final_state [N, H, d_k, d_v] fp32 or NULL; may alias init_state
 *   workspace  kda_prefill_workspace_size() bytes (at least 256); its status
 *              word is cleared by this call and set if the device finds
 *              cu_seqlens invalid (then out and final_state are
 *              unspecified).  With room for the order, a first small kernel
 *              sorts the documents by length and the longest start first; a
 *              256-byte workspace runs them in document order.  The results
 *              are the same either way.
 * g is used as given; the tensor-core path relies on g >= -5 per token (the
 * bounded gate) to keep its 16-token rescaling factors inside fp32 range.
 * The tensor-core path (bf16, d = 128) keeps v, the state and the
 * pseudo-values in fp16 operands: a magnitude of 65504 or more (or a NaN)
 * there sets KDA_DEVICE_RANGE in the status word, and the results of that
 * call are then not valid.  Outputs match the exact recurrence per element
 * within 2e-2 of their RMS plus their own bf16 rounding; final states within
 * 2e-2 of their RMS.
 * T = 0 is allowed (final_state = init_state).
 */
KDA_API kda_status kda_prefill(const void *q, const void *k, const void *v,
                       const float *g, const float *beta,
                       const float *init_state, const int32_t *cu_seqlens,
                       int32_t N, int64_t T, kda_dims dims, void *out,
                       float *final_state, void *workspace,
                       size_t workspace_bytes, void *stream);

/*
 * kda_prefill that also keeps prefix snapshots: the state at given token
 * boundaries, so that a later request sharing that prefix can resume from it
 * ("From GPT-2 to Kimi K3, from first principles", Chapter 14: KDA states
 * stored sparsely at fixed token boundaries and restored to resume prefill).
 * Arguments and results as kda_prefill, plus:
 *   snapshot_offsets [n_snapshots] int32 device, strictly increasing token
 *              offsets into the packed T tokens.  Offset p names the
 *              document with bos < p <= eos (its cu_seqlens bounds) and the
 *              state after that document's tokens [bos, p): each p must be a
 *              multiple of KDA_SNAPSHOT_ALIGN (64) tokens into its document,
 *              or that document's end.
 *   n_snapshots  >= 0; 0 makes the call kda_prefill
 *   snapshots  [n_snapshots, H, d_k, d_v] fp32 device, written (state i in
 *              final_state's layout); caller-owned
 * Resuming: kda_prefill of the document's tokens [p, eos) with init_state =
 * snapshots[i] gives the same outputs and final state as the full run, up
 * to rounding.  Offsets that break the rules set KDA_DEVICE_BAD_SNAPSHOT in
 * the workspace's status word (read it with kda_get_device_status); the
 * snapshots are then unspecified, the outputs and final states are not
 * affected.  Errors as kda_prefill, and KDA_ERR_INVALID for n_snapshots < 0
 * or a missing snapshot_offsets / snapshots pointer.
 */
KDA_API kda_status kda_prefill_snapshots(const void *q, const void *k, const void *v,
                                         const float *g, const float *beta,
                                         const float *init_state, const int32_t *cu_seqlens,
                                         int32_t N, int64_t T, kda_dims dims, void *out,
                                         float *final_state, const int32_t *snapshot_offsets,
                                         int32_t n_snapshots, float *snapshots, void *workspace,
                                         size_t workspace_bytes, void *stream);

/*
 * Bytes of device workspace kda_prologue_prefill needs (0 for invalid
 * arguments): the status word, two segment-sized sets of q, k, v, g, beta and
 * the running [H, d_k, d_v] fp32 state.
 */
KDA_API size_t kda_prologue_prefill_workspace_size(kda_dims dims, int64_t T, int64_t segment_tokens);

/*
 * The KDA input path and recurrence of ONE document from the raw projections
 * ("An infra-oriented diagram of Kimi K3", KDA card: ShortConv, Swish, L2Norm,
 * the scaled-sigmoid decay and the sigmoid beta; then the chunked prefill of
 * "From GPT-2 to Kimi K3", Chapter 6), segment by segment: the prologue of
 * the next segment overlaps the prefill of the current one, and the fp32
 * state is carried across segments.  Equal (up to rounding) to kda_prologue
 * followed by kda_prefill, without T-sized intermediates.
 *   q_raw, k_raw, v_raw [T, H, d]  qkv_dtype;  conv_w [3, H*d, 4] fp32
 *   z_g [T, H, d_k] fp32;  z_beta [T, H] fp32   (both required)
 *   init_state, final_state [H, d_k, d_v] fp32 or NULL; final_state may alias
 *   segment_tokens  tokens per segment (rounded up to a multiple of 64)
 *   out [T, H, d_v] qkv_dtype
 *   workspace  kda_prologue_prefill_workspace_size() bytes, 256-byte aligned;
 *              its first word is the device status word
 *   stream           the caller's stream: the prefills run on it, and it
 *                    holds the end of the whole call (results ready in its
 *                    order)
 *   prologue_stream  the caller's second stream for the prologues, which
 *                    start after the work already queued on `stream`; give
 *                    it a lower priority than `stream` so that the prefill's
 *                    serial chain is not held back.  The same stream as
 *                    `stream` runs the segments one after another (no
 *                    overlap, same results).
 * Both streams belong to the caller.  The call creates five CUDA events to
 * order the two streams and destroys them before it returns (CUDA releases
 * an event once the work it tracks is done); the library keeps no stream,
 * event or memory from the call.  Calls that share a workspace must not
 * overlap on the GPU.
 */
KDA_API kda_status kda_prologue_prefill(const void *q_raw, const void *k_raw, const void *v_raw,
                                        const float *conv_w, const float *z_g, const float *z_beta,
                                        const float *init_state, int64_t T, kda_dims dims,
                                        int64_t segment_tokens, void *out, float *final_state,
                                        void *workspace, size_t workspace_bytes, void *stream,
                                        void *prologue_stream);

/*
 * Bytes of device workspace kda_prefill_segmented needs (0 for invalid
 * arguments).  It holds the status word, the segment offsets, a zero value
 * tile, five [segments, H, d_k, d_v] fp32 state sets and one [T, H, d_v]
 * output tile.
 */
KDA_API size_t kda_prefill_segmented_workspace_size(kda_dims dims, int64_t T, int32_t num_segments);

/*
 * Prefill of ONE document of T tokens split into num_segments segments that
 * run as independent documents (for long documents whose heads alone cannot
 * fill the GPU).  Over a segment the state evolves affinely, S_out = P S_in +
 * R, and such maps compose by (P2, R2) o (P1, R1) = (P2 P1, P2 R1 + R2)
 * ("From GPT-2 to Kimi K3, from first principles", Chapter 6, context
 * parallelism).  R comes from a prefill from zero with v, P from a prefill
 * from the identity with v = 0, a scan joins the segments, and a prefill from
 * each segment's incoming state with v = 0 gives the outputs that state adds.
 * The result equals kda_prefill of the document (up to rounding) at three
 * times its arithmetic.
 *   q, k, g  [T, H, d_k];  v, out [T, H, d_v];  beta [T, H]  (as kda_prefill)
 *   init_state, final_state [H, d_k, d_v] fp32 or NULL; final_state may alias
 *   num_segments >= 1; segments are whole 64-token chunks, the last may be
 *   shorter, and fewer segments than asked are used when T is short
 *   workspace  kda_prefill_segmented_workspace_size() bytes, 256-byte
 *              aligned; its first word is the device status word
 */
KDA_API kda_status kda_prefill_segmented(const void *q, const void *k, const void *v,
                                         const float *g, const float *beta,
                                         const float *init_state, int64_t T, kda_dims dims,
                                         int32_t num_segments, void *out, float *final_state,
                                         void *workspace, size_t workspace_bytes, void *stream);

/*
 * One decode step for N independent sequences, one token each
 * ("fused_recurrent" mode of "From GPT-2 to Kimi K3", Chapter 6).  Reads
 * every fp32 state once and writes it back in place.
 *   q, k [N, H, d_k]; v, out [N, H, d_v]  qkv_dtype
 *   g    [N, H, d_k] fp32;  beta [N, H] fp32
 *   state [N, H, d_k, d_v] fp32, updated in place
 * Equivalent to kda_prefill with N one-token documents.
 */
KDA_API kda_status kda_decode_step(const void *q, const void *k, const void *v,
                           const float *g, const float *beta, float *state,
                           void *out, int32_t N, kda_dims dims, void *stream);

/*
 * The KDA input path of the infra diagram's KDA card, fused into one pass
 * per tensor:
 *   q, k, v = Swish(ShortConv_4(raw))   (depthwise, causal, no bias, zero
 *                                        history at each document start;
 *                                        tap 3 multiplies the current token)
 *   q, k   /= sqrt(sum over the head's d channels of x^2 + 1e-6)
 *   g      = -5 * sigmoid(z_g)          ("From GPT-2 to Kimi K3", Chapter 5)
 *   beta   = sigmoid(z_beta)
 *   q_raw, k_raw, v_raw [T, H, d] qkv_dtype;  conv_w [3, H*d, 4] fp32
 *   (filters of q, k, v; channel h*d + c);  z_g [T, H, d] fp32 or NULL;
 *   z_beta [T, H] fp32 or NULL (the matching output is then not written);
 *   cu_seqlens [N + 1] int32 device offsets or NULL when N == 1.
 *   Outputs q, k, v [T, H, d] qkv_dtype; g [T, H, d] fp32; beta [T, H] fp32.
 * Offsets are clamped to [0, T] on the device, so bad offsets cannot cause
 * out-of-range accesses; the results are then unspecified.
 */
KDA_API kda_status kda_prologue(const void *q_raw, const void *k_raw,
                        const void *v_raw, const float *conv_w,
                        const float *z_g, const float *z_beta,
                        const int32_t *cu_seqlens, int32_t N, int64_t T,
                        kda_dims dims, void *q, void *k, void *v, float *g,
                        float *beta, void *stream);

/*
 * One decode step with the ShortConv cache ("From GPT-2 to Kimi K3",
 * Chapter 5: the width-4 convolution "is a short local preprocessor whose
 * state must also be cached during decoding").  Per sequence and head: the
 * prologue of kda_prologue (conv over the cached window, Swish, L2 norm of
 * q and k, the two gates) on this token's raw projections, then the update
 * of kda_decode_step, in one kernel.
 *   q_raw, k_raw, v_raw [N, H, d] qkv_dtype (this token's raw projections)
 *   conv_w [3, H*d, 4] fp32 (as kda_prologue)
 *   conv_state [N, 3, 3, H, d] qkv_dtype: the raw inputs of the previous three
 *       tokens (index 0 = t-3 ... 2 = t-1; then q, k, v), zero for a new
 *       sequence; shifted in place (this token becomes index 2)
 *   z_g [N, H, d] fp32, z_beta [N, H] fp32 (gate logits)
 *   state [N, H, d, d] fp32 in place;  out [N, H, d] qkv_dtype
 * Equivalent to kda_prologue + kda_prefill over each sequence's whole history.
 */
KDA_API kda_status kda_decode_step_conv(const void *q_raw, const void *k_raw, const void *v_raw,
                                        const float *conv_w, void *conv_state, const float *z_g,
                                        const float *z_beta, float *state, void *out,
                                        int32_t N, kda_dims dims, void *stream);

/*
 * Multi-token verify with a rollback point, for speculative decoding ("From
 * GPT-2 to Kimi K3", Chapter 14: accepted draft updates are replayed on
 * chip; cached KDA states are read-only snapshots and a hit works on a
 * private copy).  Each of N sequences runs its K draft tokens from
 * state_in, which is not modified; every draft output is written, and
 * state_out receives the state after the first accept[n] tokens.
 *   q, k, g [N*K, H, d] (row n*K + t is draft t of sequence n); v, out
 *   likewise; beta [N*K, H]; state_in, state_out [N, H, d, d] fp32 (must not
 *   alias); accept [N] int32 device, clamped to 0..K.
 * N * K * H and 2 * N * H must not exceed 2^31 - 1 (KDA_ERR_INVALID).
 */
KDA_API kda_status kda_decode_verify(const void *q, const void *k, const void *v, const float *g,
                                     const float *beta, const float *state_in,
                                     const int32_t *accept, int32_t N, int32_t K, kda_dims dims,
                                     void *out, float *state_out, void *stream);

/*
 * Head-wise RMSNorm and the full-rank output gate that follow the
 * recurrent read ("From GPT-2 to Kimi K3", Chapter 5 "A third gate: control
 * what leaves the module"; infra diagram KDA card "Head RMSNorm + gate"):
 *   y = o / sqrt(mean over the head's d channels of o^2 + eps) * w * sigmoid(z)
 *   o, z, y [T, H, d] qkv_dtype (z = the gate logits W_g x);  w [d] fp32 or
 *   NULL (ones), shared by all heads.  y may alias o.
 */
KDA_API kda_status kda_output_gate(const void *o, const void *z, const float *weight, int64_t T,
                                   kda_dims dims, float eps, void *y, void *stream);

/*
 * Diagnostic of the bounded device-side waits (the method's sources have no
 * counterpart).
 * Every wait of the tensor-core prefill gives up after a time limit,
 * records KDA_DEVICE_TIMEOUT in the workspace status word and lets its CTA
 * leave, instead of hanging.  This call launches one CTA that waits on a
 * shared-memory barrier nothing arrives on, with the same wait and a limit
 * of limit_ns (0 .. 1e9); afterwards kda_get_device_status reports
 * KDA_ERR_TIMEOUT.  Clears the status word first; never faults.
 */
KDA_API kda_status kda_selftest_wait(int64_t limit_ns, void *workspace, size_t workspace_bytes,
                                     void *stream);

/*
 * Waits for `stream`, then copies the workspace status word (one of the
 * KDA_DEVICE_* values) to *status_out.  Returns KDA_ERR_DEVICE /
 * KDA_ERR_TIMEOUT when the word is set, KDA_OK when it is clear.
 */
KDA_API kda_status kda_get_device_status(const void *workspace, int32_t *status_out,
                                 void *stream);

/* Thread-local text of the last error of this thread ("" if none). */
KDA_API const char *kda_last_error(void);

/*
 * kda_prefill for callers that cannot allocate device memory: code embedded
 * in an engine that owns every byte of device memory, or a serving loop that
 * must not allocate once it has started, has no way to provide kda_prefill's
 * workspace.  The method's sources have no counterpart to this entry point;
 * it is a deployment convenience, not part of KDA.
 * Same arguments and results as kda_prefill, minus the workspace: the
 * library keeps a fixed 64 KiB scratch array in device memory per GPU
 * (held until the process exits) and passes it as the workspace.  Up to
 * 16,320 documents the array also holds their longest-first order; larger
 * batches run in document order, with the same results.
 *   status_out  device int32 or NULL; receives the device status word
 *               (KDA_DEVICE_*) of this call, in stream order.
 * The first call in each CUDA context looks the array's address up and,
 * under CUDA's lazy module loading, loads the library's modules (the array
 * and the prefill kernels) into the context, which takes device memory: make
 * that first call at start-up, before any stream capture.  Later calls in the
 * same context allocate nothing: no cudaMalloc or cudaFree, no allocating
 * library routine.  The address is cached per context ID, so a context
 * created after cudaDeviceReset (which destroys the old context's copy of
 * the array) does its own first-call lookup again.  Calls share the array:
 * calls that overlap on the GPU race.
 */
KDA_API kda_status kda_prefill_noalloc(const void *q, const void *k, const void *v,
                                       const float *g, const float *beta,
                                       const float *init_state, const int32_t *cu_seqlens,
                                       int32_t N, int64_t T, kda_dims dims, void *out,
                                       float *final_state, int32_t *status_out, void *stream);

/*
 * Number of CUDA kernels this library has queued in this process since it
 * was loaded (all threads, all devices).  Runtime memsets/copies are not
 * counted.  Lets a caller check how many kernels a timed region launched.
 */
KDA_API uint64_t kda_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
