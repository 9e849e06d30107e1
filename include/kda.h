/*
 * kda.h -- C ABI of libkda.so, the GB300 (sm_103a) Kimi Delta Attention forward.
 *
 * KDA is a gated delta-rule linear-attention recurrence with per-channel decay
 * (the K3 text backbone's KDA layers; "kimi-k3-mlx" review, sections "The A_log
 * shape mismatch ..." and "Attention is 93 layers ..."; "ISEEKYAN/k3" README,
 * which names the chunked KDA forward and a recurrent path as the operator's
 * compute paths).  Per sequence n and head h, over the tokens t of the sequence:
 *
 *     S <- Diag(exp(g_t)) S                              (row c = key channel c)
 *     S <- S - beta_t k_t (k_t^T S) + beta_t k_t v_t^T
 *     o_t = scale * S^T q_t
 *
 * S is a K x V fp32 matrix.  The gate g is a log-decay in [-5, 0] (the K3
 * gate_lower_bound is -5.0).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer is a DEVICE pointer owned by the caller, and so is
 *    every workspace: the library allocates no memory.  kda_chunk_fwd,
 *    kda_chunk_fwd_fused and kda_recurrent_bwd take a caller-owned device
 *    workspace of at least the size their *_workspace_size query returns
 *    (16-byte aligned; the call owns it until its stream work completes, and
 *    nothing in it needs to be initialised); a smaller one returns
 *    KDA_ERR_WORKSPACE before anything is enqueued.  kda_chunk_fwd_noalloc
 *    keeps its workspace in a fixed array inside the library instead.  Calls
 *    from different host threads are safe.
 *  - status: those three entry points also take an optional caller-owned
 *    device int32 status word (4-byte aligned, or NULL).  The call sets it to
 *    KDA_OK on its stream; a kernel that cannot complete sets it to an error
 *    (KDA_ERR_TIMEOUT: a bounded device-side wait gave up; KDA_ERR_RANGE: the
 *    backward skipped a sequence whose offsets are malformed).  The caller
 *    reads it after the stream work completes, as for kda_check_range; the
 *    call's return value only covers what the host can check.
 *  - Layouts are row-major and token-major, as the K3 gate tensor (B, T, 96, 128):
 *        q, k, g [B, T, H, K]    v [B, T, H, V]    beta [B, T, H]
 *        o [B, T, H, V]          states [N, H, K, V] (V contiguous, fp32)
 *  - in_dtype selects the element type of q, k, v, g, beta (KDA_BF16 or
 *    KDA_F32); o_dtype that of o.  States are always fp32.
 *  - Supported head sizes: K, V in {64, 128}.  Anything else returns
 *    KDA_ERR_UNSUPPORTED; nothing falls back to another implementation.
 *  - q, k, v, g, o and the state tensors must be 16-byte aligned; beta and
 *    cu_seqlens need only the alignment of their element type.
 *  - stream is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Work is enqueued asynchronously; the call returns before the
 *    GPU finishes.
 *  - Errors found on the host return before anything is enqueued, so no
 *    output is touched.  A failed launch returns KDA_ERR_CUDA.
 *  - g outside [-5, 0] is a precondition violation: results are then
 *    unspecified (the in-chunk decay products are only kept in range by the
 *    bound), but no memory outside the given tensors is accessed.
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
    KDA_ERR_INVALID_ARG = 1, /* null pointer, negative size, misalignment, inconsistent B/N */
    KDA_ERR_UNSUPPORTED = 2, /* head size or dtype outside the supported set */
    KDA_ERR_WORKSPACE = 3,   /* workspace smaller than the call needs (see the *_workspace_size queries) */
    KDA_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
    KDA_ERR_RANGE = 5,       /* an input lies outside its documented range (device status word) */
    KDA_ERR_TIMEOUT = 6      /* a bounded device-side wait gave up (device status word) */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/* Human-readable name of a status code (static storage, never NULL). */
KDA_API const char *kda_status_string(kda_status status);

/* Version of this ABI; bumped on any incompatible change. */
KDA_API int kda_abi_version(void);

/*
 * kda_chunk_fwd_workspace_size -- device workspace bytes that kda_chunk_fwd
 * (and kda_chunk_fwd_fused) needs for these sizes; packed = 1 when cu_seqlens
 * will be given.  For bf16 inputs with K = V = 128 (the tensor-core path):
 *
 *     ceil(4 * hdr / 1024) * 1024 + max_chunks * H * 147968 bytes,
 *     max_chunks = B * ceil(T / 64)          (packed = 0; hdr = 0)
 *     max_chunks = ceil(T / 64) + N           (packed = 1; hdr = 2 N + 1 + max_chunks)
 *
 * (a slot per 64-token chunk and head holding the chunk-local results as the
 * state kernel's MMA operands, written by the first kernel and read by the
 * second), and 0 when N * H = 0.  Every other path (fp32 inputs, K or V = 64)
 * needs none: 0.  Invalid sizes also give 0; the entry point validates them.
 */
KDA_API size_t kda_chunk_fwd_workspace_size(kda_dtype in_dtype, int B, int T, int H, int K, int V, int N,
                                            int packed);

/*
 * kda_chunk_fwd -- chunked prefill.
 *
 * Computes the recurrence above for N independent sequences with a chunked
 * (64-token) algorithm: in-chunk gated products A = K K^T and P = Q K^T with
 * cumulative per-channel decay, a UT transform of the decayed keys, and the
 * state carried from chunk to chunk (tensor-core path: a chunk-local kernel
 * over all chunks at once, then one state chain per sequence and head with the
 * state in tensor memory).  Results equal the token-by-token recurrence up to
 * rounding.
 *
 *  q, k, g, v, beta   inputs as laid out above, element type in_dtype.
 *  scale              read-out scale; scale <= 0 selects K^-0.5.
 *  initial_state      [N, H, K, V] fp32 state before the first token of each
 *                     sequence, or NULL for zeros.  Read only.
 *  cu_seqlens         NULL: B sequences of T tokens each (N must equal B).
 *                     Non-NULL: device int32 [N+1] offsets of N sequences packed
 *                     along the token axis of a B == 1 batch; cu_seqlens[0] = 0,
 *                     non-decreasing, cu_seqlens[N] = T.  The kernel clamps
 *                     offsets into [0, T] and treats a decreasing pair as an
 *                     empty sequence, so malformed offsets never cause an
 *                     out-of-bounds access (but leave tokens unwritten).
 *  B, T, H, K, V, N   sizes; T = 0 or N = 0 is valid (nothing but the final
 *                     state is written).
 *  o                  [B, T, H, V] output, element type o_dtype.
 *  final_state        [N, H, K, V] fp32 state after each sequence's last token,
 *                     or NULL to skip.  May alias initial_state exactly (the
 *                     state is then updated in place); no other overlap is
 *                     allowed.
 *  workspace          device memory of workspace_bytes >= the size
 *                     kda_chunk_fwd_workspace_size returns (16-byte aligned;
 *                     may be NULL when that size is 0).  Calls whose stream
 *                     work overlaps must not share a workspace.
 *  status             optional device status word (see the conventions):
 *                     KDA_ERR_TIMEOUT if a bounded wait inside the kernels gave
 *                     up, in which case o and final_state are unspecified.
 */
KDA_API kda_status kda_chunk_fwd(const void *q, const void *k, const void *v, const void *g,
                         const void *beta, kda_dtype in_dtype, float scale,
                         const float *initial_state, const int32_t *cu_seqlens,
                         int B, int T, int H, int K, int V, int N,
                         void *o, kda_dtype o_dtype, float *final_state,
                         void *workspace, size_t workspace_bytes, int32_t *status, void *stream);

/*
 * kda_chunk_fwd_noalloc -- kda_chunk_fwd without any memory allocation.
 *
 * (The paper has no counterpart: this is a deployment variant of the entry
 * point above.)  Some callers cannot let a library allocate device memory in
 * the middle of their work: a serving process that reserved all free HBM for
 * its own state pool at start-up, or a runtime whose memory is managed by a
 * custom allocator that the library does not know about.  kda_chunk_fwd takes
 * a workspace that someone has to allocate.  This entry point computes
 * exactly what kda_chunk_fwd computes, with the same arguments minus the
 * workspace and status word, but keeps its workspace in one fixed 64 MiB
 * device array that every GPU loading libkda.so holds until the process
 * exits; it calls no allocation routine.  The caller still passes all inputs
 * and outputs.  A device-side wait that gives up is not reported (there is no
 * status word); o and final_state are then unspecified.
 *
 *  - Supported: in_dtype KDA_BF16 with K = V = 128 (the tensor-core path);
 *    anything else returns KDA_ERR_UNSUPPORTED.
 *  - The workspace needed is what kda_chunk_fwd_workspace_size returns:
 *    147968 bytes per (chunk, head) slot, with ceil(T / 64) * B slots per head
 *    without cu_seqlens and ceil(T / 64) + N with it (plus 4 * (2 N + 1 +
 *    slots per head) bytes, rounded up to 1 KiB, of chunk bookkeeping).  A
 *    call needing more than 64 MiB returns KDA_ERR_WORKSPACE before anything
 *    is enqueued (e.g. H = 96: T <= 256 for one sequence; H = 8: T <= 3584).
 *  - The first call made on a device looks up the array's device address (a
 *    CUDA runtime call); make that first call before any stream capture.
 *  - Every call shares the one array and leaves its last contents there;
 *    nothing in it needs to start at zero (each call writes every byte it
 *    reads).  Calls whose GPU work overlaps (different streams without
 *    ordering between them) race on the array and give wrong results.
 */
KDA_API kda_status kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const void *g,
                                 const void *beta, kda_dtype in_dtype, float scale,
                                 const float *initial_state, const int32_t *cu_seqlens,
                                 int B, int T, int H, int K, int V, int N,
                                 void *o, kda_dtype o_dtype, float *final_state, void *stream);

/*
 * kda_chunk_fwd_fused -- chunked prefill with the input prologue fused into
 * the tile loads ("kimi-k3-mlx" review, section "Attention is 93 layers ...":
 * short convolution of kernel size 4 on q, k and v, per-channel forget gate
 * with gate_lower_bound; section "The A_log shape mismatch ...": A_log has K
 * entries shared by all heads, dt_bias has H*K entries).  Per token:
 *
 *     q = l2norm(conv4(q_raw; conv_q)),  k = l2norm(conv4(k_raw; conv_k)),
 *     v = conv4(v_raw; conv_v),
 *     g[t,h,c] = max(lower_bound, -exp(A_log[c]) * softplus(gate_x[t,h,c] + dt_bias[h*K+c]))
 *
 * conv4 is causal and depthwise: y[t,ch] = sum_{j=0..3} w[ch][j] * x[t-3+j, ch],
 * with zero history before the first token of each sequence (tap 3 multiplies
 * the current token); conv_act = 0 for none, 1 for SiLU after the convolution.
 * l2norm(x) = x / sqrt(sum_c x_c^2 + l2_eps) over the K channels of one head.
 *
 *  q_raw, k_raw, gate_x [B, T, H, K], v_raw [B, T, H, V], beta [B, T, H]:
 *                     element type in_dtype.
 *  conv_q, conv_k     fp32 [H*K][4];  conv_v fp32 [H*V][4]  (channel = h*D + c).
 *  A_log fp32 [K];  dt_bias fp32 [H*K].
 *  Everything else as for kda_chunk_fwd, including the workspace (the same
 *  kda_chunk_fwd_workspace_size) and the status word.
 */
KDA_API kda_status kda_chunk_fwd_fused(const void *q_raw, const void *k_raw, const void *v_raw,
                               const void *gate_x, const void *beta, kda_dtype in_dtype,
                               const float *conv_q, const float *conv_k, const float *conv_v,
                               int conv_act, const float *A_log, const float *dt_bias,
                               float lower_bound, float l2_eps, float scale,
                               const float *initial_state, const int32_t *cu_seqlens,
                               int B, int T, int H, int K, int V, int N,
                               void *o, kda_dtype o_dtype, float *final_state,
                               void *workspace, size_t workspace_bytes, int32_t *status, void *stream);

/*
 * kda_trace_events -- timing hook for the tensor-core prefill.
 *
 * (The pages have no counterpart: instrumentation.)  The tensor-core prefill
 * runs as two kernels, the chunk-local one and the state chain.  The next
 * kda_chunk_fwd, kda_chunk_fwd_fused or kda_chunk_fwd_noalloc call made by the
 * calling host thread records these CUDA events (cudaEvent_t passed as void*;
 * any may be NULL) on its stream: begin before its first kernel, split after
 * the chunk-local kernel, end after its last kernel.  That call consumes the
 * setting; a call that takes the CUDA-core path records nothing and clears it
 * too.  The events belong to the caller.
 */
KDA_API void kda_trace_events(void *begin, void *split, void *end);

/*
 * kda_set_wait_limit -- testing hook: how many times a bounded device-side
 * wait of the tensor-core prefill polls before it gives up (0 restores the
 * default, about a second).  Process-wide; read when a call launches its
 * kernels.  With kda_inject_wait_timeout it makes a wait give up quickly, so
 * that the status word's KDA_ERR_TIMEOUT path can be exercised without a
 * fault: the kernels then skip the rest of their work, drain the copies and
 * MMAs in flight, and exit normally.  (The pages have no counterpart: failure
 * detection.)
 */
KDA_API void kda_set_wait_limit(uint32_t iterations);

/*
 * kda_inject_wait_timeout -- testing hook: the next kda_chunk_fwd,
 * kda_chunk_fwd_fused, kda_chunk_fwd_noalloc or kda_chunk_bwd call made by the
 * calling host thread on the tensor-core path makes the first wait of one of its
 * kernels (kernel = 1: the chunk-local kernel, in every CTA; 2: the state
 * kernel's MMA issuer, in every CTA; 3: the chunked backward's chain kernel, 4:
 * its chunk kernel, in every CTA) a wait on an mbarrier that nothing arrives on.  That
 * wait runs out after the kda_set_wait_limit polls, records KDA_ERR_TIMEOUT in
 * the call's status word and the kernels take their give-up path (no fault, no
 * trap).  The call consumes the setting; another kernel value clears it.
 * (The pages have no counterpart: failure detection.)
 */
KDA_API void kda_inject_wait_timeout(int kernel);

/*
 * kda_recurrent_step -- one decode token for each of N sequences.
 *
 * Applies one step of the recurrence to the fp32 state in place, streaming it
 * through HBM once (read, update, write):
 *
 *     a = S_old^T (k * exp(g)),  b = S_old^T (q * exp(g))
 *     delta = beta (v - a),      o = scale (b + (q . k) delta)
 *     S_new = Diag(exp(g)) S_old + k delta^T
 *
 * which equals decay, delta update and read-out of the recurrence above.
 *
 *  q, k, g [N, H, K], v [N, H, V], beta [N, H]: element type in_dtype.
 *  state   [N, H, K, V] fp32, read and written in place.
 *  o       [N, H, V], element type o_dtype.
 */
KDA_API kda_status kda_recurrent_step(const void *q, const void *k, const void *v, const void *g,
                              const void *beta, kda_dtype in_dtype, float scale, float *state,
                              int N, int H, int K, int V, void *o, kda_dtype o_dtype,
                              void *stream);

/*
 * kda_output_gate -- the layer's output gate on o ("kimi-k3-mlx" review,
 * section "Attention is 93 layers ...": KDA carries a full-rank output gate;
 * "NeMo AutoModel draft_kimi_k3", module description: K3's norms are RMS norms
 * with the variance in fp32 and its output gates are sigmoid gates).  Per
 * (token, head) row of V values:
 *
 *     out = o / sqrt(mean(o^2) + eps) * weight * sigmoid(gate)
 *
 *  o       [B, T, H, V] fp32 (the output of kda_chunk_fwd / kda_recurrent_step),
 *          device, 16-byte aligned.
 *  gate    [B, T, H, V], element type gate_dtype (the gate projection), device,
 *          16-byte aligned.
 *  weight  [V] fp32 shared by all heads, device, 16-byte aligned; NULL means ones.
 *  eps     >= 0 (finite).
 *  out     [B, T, H, V], element type out_dtype, device, 16-byte aligned.  It may
 *          be o itself when out_dtype is KDA_F32 (in place); any other overlap
 *          with o or gate is invalid.
 *
 * Sizes: B, T >= 0, H > 0, V in {64, 128}.  Returns KDA_ERR_INVALID_ARG for
 * null or misaligned pointers (with B*T > 0), negative sizes, a negative or
 * non-finite eps, or a bf16 out aliasing o; KDA_ERR_UNSUPPORTED for another V
 * or dtype.  Nothing is launched when a check fails.  Stream-ordered on
 * `stream`.
 */
KDA_API kda_status kda_output_gate(const float *o, const void *gate, kda_dtype gate_dtype,
                           const float *weight, float eps, int B, int T, int H, int V,
                           void *out, kda_dtype out_dtype, void *stream);

/*
 * kda_gate_proj -- the projections that produce kda_chunk_fwd_fused's gate_x
 * and beta from the layer input ("kimi-k3-mlx" review, section "Attention is
 * 93 layers ...": a low-rank forget gate through f_a and f_b; section "The
 * A_log shape mismatch ...": b_proj is [96, H] with H = 7168 the model width).
 * Per token t (a row of x):
 *
 *     y_t      = f_a x_t                   (fp32, not rounded to bf16)
 *     gate_x_t = f_b y_t
 *     beta_t   = 1 / (1 + exp(-(b_proj x_t)))
 *
 * Both GEMMs run on the tensor cores with fp32 accumulation; y is carried into
 * the second as a bf16 pair (hi + lo) so that its rounding does not reach
 * gate_x.  The first GEMM is split along D into up to 8 ranges whose fp32
 * partial sums are added in a fixed order, so results do not depend on
 * scheduling.  The pages give no rank for f_a/f_b; R = 128 (the head size) is
 * the model's, R = 64 is also accepted.
 *
 *  x       [B, T, D] bf16, device.
 *  f_a     [R, D] bf16;  f_b [HK, R] bf16;  b_proj [NH, D] bf16; device.
 *  gate_x  [B, T, HK] bf16 out, device (HK = H * K: kda_chunk_fwd_fused's
 *          gate_x [B, T, H, K]).
 *  beta    [B, T, NH] bf16 out, device (NH = H: kda_chunk_fwd_fused's beta).
 *  dtype   KDA_BF16 (anything else: KDA_ERR_UNSUPPORTED).
 *  workspace   device, 16-byte aligned, at least kda_gate_proj_workspace_size
 *          bytes: y as bf16 hi and lo (4 R bytes per token) and the fp32 partial
 *          sums of [f_a x | b_proj x] (4 S (R + NH) bytes per token, S the number of
 *          ranges: min(8, D / 64, max(1, 128 / ceil(B T / 128))), made exact so that
 *          none is empty); owned by the caller and in use until the call's work on
 *          `stream` has completed.  0 for invalid sizes.
 *  status  optional device int32 (4-byte aligned): set to KDA_OK on the stream,
 *          then to KDA_ERR_TIMEOUT if a bounded wait inside a kernel gave up
 *          (the outputs are then incomplete).
 *
 * Sizes: B, T >= 0 with B * T < 2^31; D > 0 a multiple of 64; R in {64, 128};
 * NH > 0 a multiple of 16 with R + NH <= 256; HK > 0 a multiple of 256.
 * Every pointer 16-byte aligned.  Returns KDA_ERR_INVALID_ARG for null or
 * misaligned pointers (with B * T > 0), negative sizes or outputs that overlap
 * an input, the workspace or each other; KDA_ERR_UNSUPPORTED for sizes outside
 * the set above; KDA_ERR_WORKSPACE for a workspace that is too small.  Nothing
 * is launched when a check fails.  Stream-ordered on `stream`.
 */
KDA_API size_t kda_gate_proj_workspace_size(int B, int T, int D, int R, int NH);
KDA_API kda_status kda_gate_proj(const void *x, const void *f_a, const void *f_b, const void *b_proj,
                                 kda_dtype dtype, int B, int T, int D, int R, int HK, int NH,
                                 void *gate_x, void *beta, void *workspace, size_t workspace_bytes,
                                 int32_t *status, void *stream);

/*
 * kda_state_compose -- one step of the prefix over segment transitions, for
 * context-parallel prefill (the sequence split into consecutive segments, one
 * per rank).  The recurrence is affine in the state: over a segment,
 * S_end = M S_start + S_zero, with M = prod_t (I - beta_t k_t k_t^T) Diag(e^{g_t})
 * (later tokens on the left; kda_chunk_fwd with v = 0 and initial state I gives
 * M as its final state) and S_zero the segment's final state from a zero start.
 * This call evaluates, for every head h,
 *
 *     out[h] = M[h] S[h] + A[h]        (K x K times K x V, fp32)
 *
 *  M    [H, K, K] fp32, device;  S, A, out  [H, K, V] fp32, device; all 16-byte
 *       aligned.  A may be NULL (zero) or equal to out (accumulate in place);
 *       out must not overlap M or S.
 *  K, V in {64, 128}, H >= 0.
 *
 * Returns KDA_ERR_INVALID_ARG for null or misaligned pointers or a forbidden
 * overlap, KDA_ERR_UNSUPPORTED for another K or V; nothing is launched then.
 * Stream-ordered on `stream`.
 */
KDA_API kda_status kda_state_compose(const float *M, const float *S, const float *A, float *out,
                             int H, int K, int V, void *stream);

/*
 * kda_check_range -- debug check of an input's documented range, e.g. the
 * prefill's precondition that every log decay g lies in [-5, 0] (the K3
 * gate_lower_bound, "kimi-k3-mlx" review, "Attention is 93 layers ...").
 *
 *  x       count elements of dtype, device.
 *  status  caller-owned device int32: set to KDA_OK on the stream, then to
 *          KDA_ERR_RANGE by the check if any element lies outside [lo, hi] or is
 *          NaN.  The caller reads it after the stream work completes.
 *
 * Returns KDA_ERR_INVALID_ARG for a null x (count > 0), a null or misaligned
 * (4-byte) status, a negative count or lo > hi; KDA_ERR_UNSUPPORTED for another
 * dtype.  Stream-ordered and asynchronous: the call's own return value says
 * nothing about the data.
 */
KDA_API kda_status kda_check_range(const void *x, kda_dtype dtype, int64_t count, float lo, float hi,
                           int32_t *status, void *stream);

/*
 * kda_recurrent_bwd -- gradients of  L = <dO, o> + <dS_T, S_T>  through the
 * recurrence above (the backward of kda_chunk_fwd), for training.  Per token,
 * with S' = Diag(e^{g_t}) S_{t-1}, a = S'^T k_t, delta = beta_t (v_t - a):
 *
 *     dq_t = scale S_t dO_t,  ddelta = dS^T k_t,  dv_t = beta_t ddelta,
 *     dbeta_t = ddelta . (v_t - a),  dk_t = dS delta + S' da  (da = -beta_t ddelta),
 *     dg_t[c] = sum_x (dS + k_t da^T)[c, x] S'[c, x],
 *     dS_{t-1} = Diag(e^{g_t}) (dS + k_t da^T),  after dS += scale q_t dO_t^T,
 *
 * run token by token on the CUDA cores in fp32, one CTA per (sequence, head),
 * with the state recomputed from checkpoints every 64 tokens.
 *
 *  q, k, v, g, beta, in_dtype, scale, initial_state, cu_seqlens, B, T, H, K, V, N:
 *          as kda_chunk_fwd.
 *  dO      [B, T, H, V] fp32, device.  dS_T [N, H, K, V] fp32 or NULL (zero).
 *  dq, dk, dg [B, T, H, K], dv [B, T, H, V], dbeta [B, T, H]: fp32 outputs, device.
 *  dS0     [N, H, K, V] fp32 or NULL (not written).
 *
 * The caller passes a device workspace of at least
 * kda_recurrent_bwd_workspace_size bytes (16-byte aligned):
 * 4 * K * V * (max_blocks * H + 64 * N * H) with max_blocks = B * ceil(T / 64),
 * or ceil(T / 64) + N with cu_seqlens (state checkpoints every 64 tokens, and
 * 64 recomputed states per chain); KDA_ERR_WORKSPACE before anything is
 * enqueued if it is smaller.  status: optional device word, KDA_ERR_RANGE if
 * a sequence was skipped because malformed (overlapping) offsets would need
 * more checkpoints than the workspace holds; its gradients are then NaN, and
 * rows it shares with another sequence are unspecified.  Alignment and error
 * rules as kda_chunk_fwd; dbeta needs 4-byte alignment.
 */
KDA_API size_t kda_recurrent_bwd_workspace_size(kda_dtype in_dtype, int B, int T, int H, int K, int V, int N,
                                                int packed);

KDA_API kda_status kda_recurrent_bwd(const void *q, const void *k, const void *v, const void *g,
                             const void *beta, kda_dtype in_dtype, float scale,
                             const float *initial_state, const int32_t *cu_seqlens, int B, int T,
                             int H, int K, int V, int N, const float *dO, const float *dS_T,
                             float *dq, float *dk, float *dv, float *dg, float *dbeta, float *dS0,
                             void *workspace, size_t workspace_bytes, int32_t *status, void *stream);

/*
 * kda_chunk_bwd -- the same gradients (of L = <dO, o> + <dS_T, S_T>), chunk by
 * chunk (the backward of the chunked form in "ISEEKYAN/k3" README's chunked KDA
 * forward; the per-channel decay of "kimi-k3-mlx" review, "The A_log shape
 * mismatch ...").  For bf16 inputs with K = V = 128 it runs the tensor-core
 * prefill once more, keeping the state that enters every 64-token chunk and the
 * chunk's operands (W, q e^G, k e^{G_C - G}, P, U~, e^{G_C}), then carries the
 * state gradient backwards chunk by chunk,
 *
 *     dU = scale P^T dO + Kb dS',   dS = scale (q e^G)^T dO + Diag(e^{G_C}) dS' - W^T dU,
 *
 * and forms every chunk's dq, dk, dv, dg, dbeta in parallel from (S, U, dU, dS',
 * dO) and the chunk's A and T.  The products of both steps run on the tensor cores
 * (operands split hi + lo into bf16, three MMA terms, fp32 accumulation); the
 * elementwise passes in fp32 on the CUDA cores.  Other dtypes and head sizes take
 * kda_recurrent_bwd.
 *
 * Arguments, outputs and rules as kda_recurrent_bwd.  The caller passes a device
 * workspace of at least kda_chunk_bwd_workspace_size bytes (16-byte aligned): for
 * the chunked path kda_chunk_fwd_workspace_size + 2 B T H V (o, bf16), each rounded
 * up to 256 bytes, + 4 slots (K V + 2 * 64 * 64 + 64 V + K V + 64 V) with slots =
 * max_chunks * H (the entering state, A and T, U, dS' and dU of every chunk) + a
 * scratch of 152 * 638976 bytes (one area per CTA of the gradient kernel); for the
 * other sizes kda_recurrent_bwd_workspace_size.  status: optional device word,
 * KDA_ERR_TIMEOUT if a bounded wait of the forward's kernels, of the backward chain
 * or of the gradient kernel gave up (the kernels then drain their work in flight
 * and return; the gradients are unspecified), KDA_ERR_RANGE as kda_recurrent_bwd
 * on the other sizes.
 */
KDA_API size_t kda_chunk_bwd_workspace_size(kda_dtype in_dtype, int B, int T, int H, int K, int V, int N,
                                            int packed);
KDA_API kda_status kda_chunk_bwd(const void *q, const void *k, const void *v, const void *g,
                                 const void *beta, kda_dtype in_dtype, float scale,
                                 const float *initial_state, const int32_t *cu_seqlens,
                                 int B, int T, int H, int K, int V, int N, const float *dO,
                                 const float *dS_T, float *dq, float *dk, float *dv, float *dg,
                                 float *dbeta, float *dS0, void *workspace, size_t workspace_bytes,
                                 int32_t *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
