/*
 * kda.h - C ABI of libkda.so: Kimi Delta Attention (KDA) on one NVIDIA GB300
 * (sm_103a).
 *
 * The method, per head with d_k = d_v = 128 and per token t, in order
 * ("Kimi K3 · KDA layer", OpenModelAtlas, KDA equation list; "Kimi K3:
 * Architecture and SGLang Day-0 Support", section "Math details: how KDA
 * gates and rewrites the same S"):
 *
 *     S  <- Diag(alpha_t) S                       decay, row j scaled by alpha_t[j]
 *     S  <- S + beta_t k_t (v_t - S^T k_t)^T      delta-rule write
 *     o~_t = scale * S^T q_t                      readout of the updated state
 *
 * with alpha_t = exp(log_alpha_t).  The state S is d_k x d_v fp32, row j =
 * key channel j, column c = value channel c.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library never allocates, frees or retains them beyond the call.
 *   - Every tensor pointer must be 16-byte aligned, except per-row scalars
 *     (beta, beta_logit, A, cu_seqlens), which need only their element's
 *     alignment.  Tensors are dense and row-major.  Token tensors are
 *     token-major [t][h][i] with i (the 128 channels) contiguous; states are
 *     [n][h][j][c].
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Calls are asynchronous on that stream.
 *   - Argument errors are detected on the host before any launch and return
 *     KDA_ERR_INVALID_ARGUMENT (or KDA_ERR_UNSUPPORTED / KDA_ERR_WORKSPACE);
 *     nothing is written in that case.  A failed launch returns KDA_ERR_CUDA.
 *   - Kernels never trap.  A device-side check or a bounded wait that gives
 *     up records a code in a device status word; kda_get_device_status reads
 *     and clears it.
 *   - Contents are not validated on the host (values of cu_seqlens, the
 *     range of log_alpha): those are the caller's contract.
 *   - The library holds no mutable host state; calls are thread-safe.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_HEAD_DIM 128 /* d_k = d_v, fixed */

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARGUMENT = 1, /* null/misaligned pointer, bad size or dtype */
    KDA_ERR_UNSUPPORTED = 2,      /* a valid request this build does not implement */
    KDA_ERR_WORKSPACE = 3,        /* workspace missing or smaller than required */
    KDA_ERR_CUDA = 4,             /* a CUDA runtime call or launch failed */
    KDA_ERR_DEVICE_TIMEOUT = 5,   /* a kernel's bounded wait gave up */
    KDA_ERR_DEVICE_CHECK = 6      /* a kernel's self-check failed */
} kda_status;

typedef enum {
    KDA_BF16 = 0, /* bfloat16, round-to-nearest-even on output */
    KDA_FP32 = 1
} kda_dtype;

/* Human-readable name of a status code (static storage, never NULL). */
const char *kda_status_string(kda_status status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int32_t kda_version(void);

/*
 * Bytes of scratch that kda_prefill needs for these sizes (0 = none; the
 * workspace pointer may then be NULL).
 */
size_t kda_prefill_workspace_size(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                                  kda_dtype in_dtype);

/*
 * kda_prefill - the recurrence over packed variable-length sequences.
 *
 * Computes, for every sequence n (tokens [cu_seqlens[n], cu_seqlens[n+1]))
 * and head h, the token-by-token recurrence above starting from S0[n][h]
 * (zeros when S0 is NULL), writes o~ for every token, and the state after
 * the sequence's last token to S_final[n][h] (skipped when S_final is NULL).
 * Implemented chunk-wise (parallel inside a chunk, recurrent across chunks:
 * "Kimi K3's Architecture: Kimi Delta Attention, Attention Residuals, and
 * 896 Experts", section "Channel-wise decay, and the floor K3 puts under
 * it"), which is an exact rewrite of the recurrence up to rounding.
 *
 *   in_dtype     element type of q, k, v (KDA_BF16 or KDA_FP32)
 *   out_dtype    element type of o
 *   num_seqs     N >= 1
 *   total_tokens T >= 0, must equal cu_seqlens[N]
 *   num_heads    H >= 1
 *   q, k         [T][H][128] in_dtype; expected unit-norm per head
 *   v            [T][H][128] in_dtype
 *   log_alpha    [T][H][128] fp32, each in [-5, 0] (the pages' decay floor
 *                g_min = -5; values below it are outside the contract)
 *   beta         [T][H] fp32 write strength
 *   S0           [N][H][128][128] fp32, or NULL for zero initial states
 *   cu_seqlens   [N+1] int32 (device): 0 = cu[0] <= cu[1] <= ... <= cu[N] = T
 *   scale        readout scale, 1/sqrt(128) in the pages
 *   o            [T][H][128] out_dtype
 *   S_final      [N][H][128][128] fp32 or NULL; may alias S0 exactly (in-place
 *                resume); partial overlap is not allowed
 *   workspace    device scratch of at least kda_prefill_workspace_size() bytes
 *
 * A zero-length sequence writes no output and S_final[n] = S0[n] (or zeros).
 * Results do not depend on how sequences are packed: a sequence gives the
 * same bits alone or packed with others, in any order.
 */
kda_status kda_prefill(kda_dtype in_dtype, kda_dtype out_dtype, int32_t num_seqs,
                       int32_t total_tokens, int32_t num_heads, const void *q, const void *k,
                       const void *v, const float *log_alpha, const float *beta,
                       const float *S0, const int32_t *cu_seqlens, float scale, void *o,
                       float *S_final, void *workspace, size_t workspace_bytes, void *stream);

/*
 * kda_prefill_with_checkpoints - kda_prefill that also leaves read-only state
 * snapshots at fixed token intervals, the states a prefix cache keeps for later
 * requests that share the prefix ("Kimi K3: Architecture and SGLang Day-0
 * Support", section "RadixAttention: prefix caching for KDA state": a cached
 * KDA state is a read-only checkpoint that a request copies into its own slot
 * before it writes).
 *
 * For sequence n, snapshot i (i = 0, 1, ...) is the state after the sequence's
 * first (i + 1) * ckpt_every tokens, written to
 * ckpt_states[ckpt_base[n] + i][h][128][128] (fp32, row = key channel) for
 * every i < ckpt_base[n + 1] - ckpt_base[n] whose token count lies inside the
 * sequence; the caller sizes ckpt_base[n + 1] - ckpt_base[n] (at most
 * floor(len_n / ckpt_every) snapshots are written; slots beyond are left as
 * they are).  A snapshot equals, to rounding, the S_final of a kda_prefill
 * over that prefix alone.
 *
 *   ckpt_every   0 (no snapshots: identical to kda_prefill) or a positive
 *                multiple of 32, the tensor-core kernel's chunk length
 *   ckpt_base    [N+1] int32 (device), non-decreasing snapshot offsets;
 *                read only when ckpt_every > 0
 *   ckpt_states  [ckpt_base[N]][H][128][128] fp32 (device, 16-byte aligned);
 *                must not overlap any other argument
 *   (all other arguments as kda_prefill)
 * Errors: as kda_prefill; KDA_ERR_INVALID_ARGUMENT also for a ckpt_every that
 * is negative or not a multiple of 32, or null/misaligned ckpt_base/ckpt_states
 * when ckpt_every > 0.
 */
kda_status kda_prefill_with_checkpoints(kda_dtype in_dtype, kda_dtype out_dtype, int32_t num_seqs,
                                        int32_t total_tokens, int32_t num_heads, const void *q,
                                        const void *k, const void *v, const float *log_alpha,
                                        const float *beta, const float *S0,
                                        const int32_t *cu_seqlens, float scale, void *o,
                                        float *S_final, void *workspace, size_t workspace_bytes,
                                        int32_t ckpt_every, const int32_t *ckpt_base,
                                        float *ckpt_states, void *stream);

/*
 * kda_prefill_head_decay - kda_prefill_with_checkpoints for the Gated DeltaNet
 * case: one decay per (token, head) shared by all 128 key channels, i.e.
 * Diag(alpha_t) = alpha_t I ("Kimi K3's Architecture: Kimi Delta Attention,
 * Attention Residuals, and 896 Experts", section "Channel-wise decay, and the
 * floor K3 puts under it": Gated DeltaNet keeps one decay value per head, KDA
 * one per key channel).  The same kernels run it; only the decay is read as a
 * scalar and broadcast.
 *
 *   log_alpha    [T][H] fp32 (4-byte aligned), each in [-5, 0] as for kda_prefill
 *   (all other arguments, checkpoints included, as kda_prefill_with_checkpoints)
 */
kda_status kda_prefill_head_decay(kda_dtype in_dtype, kda_dtype out_dtype, int32_t num_seqs,
                                  int32_t total_tokens, int32_t num_heads, const void *q,
                                  const void *k, const void *v, const float *log_alpha,
                                  const float *beta, const float *S0, const int32_t *cu_seqlens,
                                  float scale, void *o, float *S_final, void *workspace,
                                  size_t workspace_bytes, int32_t ckpt_every,
                                  const int32_t *ckpt_base, float *ckpt_states, void *stream);

/*
 * kda_prefill_unbounded_decay - kda_prefill for decays without the floor: any
 * log_alpha <= 0, -inf included (alpha = 0 clears the state).  Below the floor
 * of -5 the chunk's reciprocal decays overflow, which is why Kimi Linear's
 * unbounded gate needed a position-pair fallback inside each chunk ("Kimi K3's
 * Architecture: Kimi Delta Attention, Attention Residuals, and 896 Experts",
 * section "Channel-wise decay, and the floor K3 puts under it").  Here bf16
 * inputs run the tensor-core kernel chunk by chunk: a 32-token chunk whose decay
 * factors all lie within the range the floor would guarantee (about e^{+-80}
 * around the chunk's middle) takes the tensor-core form, any other chunk runs
 * token by token on the state inside the same kernel, exact for any decay.
 * fp32 inputs run the token-by-token kernel, which has no reciprocal and is
 * exact up to fp32 rounding.  Arguments, layouts and errors as kda_prefill.
 */
kda_status kda_prefill_unbounded_decay(kda_dtype in_dtype, kda_dtype out_dtype, int32_t num_seqs,
                                       int32_t total_tokens, int32_t num_heads, const void *q,
                                       const void *k, const void *v, const float *log_alpha,
                                       const float *beta, const float *S0,
                                       const int32_t *cu_seqlens, float scale, void *o,
                                       float *S_final, void *workspace, size_t workspace_bytes,
                                       void *stream);

/*
 * kda_decode_step - one token per request, state updated in place.
 *
 * One step of the recurrence for each (request b, head h): "each step reads
 * and writes only S" ("Kimi K3: Architecture and SGLang Day-0 Support",
 * section "Attention mechanisms in detail: linear attention").  The state is
 * streamed through HBM exactly once (one read, one write).
 *
 *   batch       B >= 1 requests
 *   q, k, v     [B][H][128] in_dtype
 *   log_alpha   [B][H][128] fp32 (may be -inf: alpha = 0 resets the state)
 *   beta        [B][H] fp32
 *   S_inout     [B][H][128][128] fp32, read then overwritten
 *   o           [B][H][128] out_dtype
 */
kda_status kda_decode_step(kda_dtype in_dtype, kda_dtype out_dtype, int32_t batch,
                           int32_t num_heads, const void *q, const void *k, const void *v,
                           const float *log_alpha, const float *beta, float *S_inout,
                           float scale, void *o, void *stream);

/*
 * kda_decode_step_head_decay - kda_decode_step with one decay per (request,
 * head): log_alpha is [B][H] fp32 (4-byte aligned), broadcast over the 128 key
 * channels (the Gated DeltaNet case, as kda_prefill_head_decay).
 */
kda_status kda_decode_step_head_decay(kda_dtype in_dtype, kda_dtype out_dtype, int32_t batch,
                                      int32_t num_heads, const void *q, const void *k,
                                      const void *v, const float *log_alpha, const float *beta,
                                      float *S_inout, float scale, void *o, void *stream);

/*
 * kda_frontend - inputs of the recurrence from the pre-convolution
 * projections ("Kimi K3 · KDA layer", KDA equation list; "Inside Kimi K3:
 * How KDA, AttnRes, and 896 Experts Work", section "Short convolutions give
 * KDA local order before recurrence"):
 *
 *   x^c_t   = SiLU( sum_{j=0..3} w_j * x^p_{t-j} )   x in {q, k, v}, per channel
 *   q^, k^  = x^c / sqrt(sum x^c^2 + l2_eps)          per head, 128 channels
 *   log_alpha = -5 * sigmoid( e^{A_h} (z + b) )
 *   beta      = sigmoid(beta_logit)
 *
 * Tokens before the start of their own sequence count as zero.  Tap j = 0
 * multiplies the current token.
 *
 *   qp, kp, vp  [T][H][128] bf16
 *   conv_w      [3][H*128][4] fp32 (stream q/k/v, channel h*128+i, tap j)
 *   z           [T][H][128] bf16
 *   A           [H] fp32
 *   b           [H][128] fp32, or NULL for zeros
 *   beta_logit  [T][H] bf16
 *   out_dtype   element type of q_hat, k_hat, v_out
 *   q_hat, k_hat, v_out  [T][H][128] out_dtype
 *   log_alpha   [T][H][128] fp32;  beta [T][H] fp32
 */
kda_status kda_frontend(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                        const void *qp, const void *kp, const void *vp, const float *conv_w,
                        const void *z, const float *A, const float *b, const void *beta_logit,
                        const int32_t *cu_seqlens, float l2_eps, kda_dtype out_dtype,
                        void *q_hat, void *k_hat, void *v_out, float *log_alpha, float *beta,
                        void *stream);

/*
 * kda_frontend_unbounded_decay - kda_frontend with Kimi Linear's decay gate,
 * log_alpha = -e^{A_h} softplus(z + b), in (-inf, 0) (same section as
 * kda_prefill_unbounded_decay), instead of K3's -5 sigmoid(e^{A_h}(z + b)).
 * Everything else, arguments and errors included, as kda_frontend.  Its
 * log_alpha may lie below -5: feed it to kda_prefill_unbounded_decay.
 */
kda_status kda_frontend_unbounded_decay(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                                        const void *qp, const void *kp, const void *vp,
                                        const float *conv_w, const void *z, const float *A,
                                        const float *b, const void *beta_logit,
                                        const int32_t *cu_seqlens, float l2_eps,
                                        kda_dtype out_dtype, void *q_hat, void *k_hat,
                                        void *v_out, float *log_alpha, float *beta, void *stream);

/*
 * kda_output_gate - o^g = sigmoid(g) * RMSNorm(o~) per head over its 128
 * channels, RMSNorm(x) = x / sqrt(mean(x^2) + eps), unit weight ("Kimi K3 ·
 * KDA layer", KDA equation list).
 *
 *   num_rows   T*H rows of 128 channels
 *   o_tilde    [rows][128] in_dtype;  g [rows][128] bf16;  out [rows][128] out_dtype
 */
kda_status kda_output_gate(int64_t num_rows, kda_dtype in_dtype, const void *o_tilde,
                           const void *g, float eps, kda_dtype out_dtype, void *out,
                           void *stream);

/*
 * Bytes of device scratch kda_layer_core needs for these sizes.
 */
size_t kda_layer_core_workspace_size(int32_t num_seqs, int32_t total_tokens, int32_t num_heads);

/*
 * kda_layer_core - one KDA layer core over packed variable-length sequences:
 * front end, recurrence and output gate ("Kimi K3 · KDA layer", KDA equation
 * list), i.e. kda_frontend -> kda_prefill -> kda_output_gate on `stream`.
 *
 * All intermediates (q^, k^, v, log_alpha, beta, o~) stay fp32: with the
 * front end's short-convolution smoothing, consecutive keys are close to
 * parallel and the recurrence is ill-conditioned, so rounding q^, k^, v to
 * bf16 between the stages moves the output by several percent.  The
 * intermediates live in `workspace`, which must hold
 * kda_layer_core_workspace_size() bytes; nothing is allocated.
 *
 *   qp, kp, vp, z [T][H][128] bf16; conv_w [3][H*128][4] fp32; A [H] fp32;
 *   b [H][128] fp32 or NULL; beta_logit [T][H] bf16; g [T][H][128] bf16;
 *   cu_seqlens [N+1] int32 (device); S0 [N][H][128][128] fp32 or NULL;
 *   o_gated [T][H][128] out_dtype; S_final [N][H][128][128] fp32 or NULL.
 */
kda_status kda_layer_core(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                          const void *qp, const void *kp, const void *vp, const float *conv_w,
                          const void *z, const float *A, const float *b, const void *beta_logit,
                          const void *g, const int32_t *cu_seqlens, const float *S0, float scale,
                          float l2_eps, float rms_eps, kda_dtype out_dtype, void *o_gated,
                          float *S_final, void *workspace, size_t workspace_bytes, void *stream);

/*
 * kda_layer_core_unbounded_decay - kda_layer_core with Kimi Linear's unbounded
 * decay gate (kda_frontend_unbounded_decay -> kda_prefill_unbounded_decay ->
 * kda_output_gate through the same workspace, fp32 intermediates).  Arguments,
 * workspace size and errors as kda_layer_core.
 */
kda_status kda_layer_core_unbounded_decay(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                                          const void *qp, const void *kp, const void *vp,
                                          const float *conv_w, const void *z, const float *A,
                                          const float *b, const void *beta_logit, const void *g,
                                          const int32_t *cu_seqlens, const float *S0, float scale,
                                          float l2_eps, float rms_eps, kda_dtype out_dtype,
                                          void *o_gated, float *S_final, void *workspace,
                                          size_t workspace_bytes, void *stream);

/*
 * kda_layer_core_noalloc - kda_layer_core without a caller-provided workspace.
 *
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory themselves, for example a plugin inside a host
 * application that owns every device allocation and hands out no scratch, or a
 * latency-critical path on which an allocation (and the synchronisation it may
 * imply) is not acceptable.
 *
 * Arguments and results are those of kda_layer_core.  The scratch it needs is
 * taken from a fixed array of KDA_NOALLOC_SCRATCH_BYTES bytes in the library's
 * own device memory, which every GPU that loads the library holds until the
 * process exits.  The call allocates nothing and frees nothing.
 *   - Sizes whose scratch, kda_layer_core_workspace_size(), exceeds
 *     KDA_NOALLOC_SCRATCH_BYTES are rejected with KDA_ERR_UNSUPPORTED before any
 *     launch (with fp32 intermediates that is about 26,000 (token, head) rows).
 *   - All calls share the one array, and it keeps the last call's contents.
 *     Nothing in it has to start at zero: every stage writes its part in full
 *     before the next stage reads it.  Calls that overlap on the GPU (two
 *     streams, or two host threads, at once) race on the array and corrupt each
 *     other's results, so serialise them.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is kept for the life of the
 *     process: after cudaDeviceReset (or any other teardown of the device's
 *     primary context) it no longer names live memory, so a process that
 *     resets a device must not call this entry point on it again.
 */
#define KDA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
kda_status kda_layer_core_noalloc(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                                  const void *qp, const void *kp, const void *vp,
                                  const float *conv_w, const void *z, const float *A,
                                  const float *b, const void *beta_logit, const void *g,
                                  const int32_t *cu_seqlens, const float *S0, float scale,
                                  float l2_eps, float rms_eps, kda_dtype out_dtype, void *o_gated,
                                  float *S_final, void *stream);

/*
 * kda_layer_core_fused - the same layer core as kda_layer_core in ONE
 * tensor-core kernel: only the layer's inputs and outputs cross HBM ("Kimi K3 ·
 * KDA layer", KDA equation list: short convolution, SiLU, L2 norm, the decay and
 * write-strength gates, the delta-rule recurrence, the sigmoid-gated RMSNorm).
 *
 * Inside the kernel every intermediate (q^, k^, v, log_alpha, beta, o~) is fp32
 * and enters each tensor-core product as a bf16 hi + lo pair, so the result
 * matches kda_layer_core's within the 2e-3 (row-conditioned) bound; it is not
 * bit-identical to it.  No workspace; nothing is allocated.
 *
 *   Arguments as kda_layer_core (without workspace).  qp, kp, vp, z, g and
 *   o_gated must be 16-byte aligned (qp, kp, vp are read with TMA);
 *   beta_logit needs 2-byte alignment; log_alpha's floor of -5 holds by
 *   construction (-5 sigmoid(.)).
 * Errors: KDA_ERR_INVALID_ARGUMENT (null/misaligned pointers, bad sizes or dtype,
 * S0/S_final partially overlapping), KDA_ERR_UNSUPPORTED (more than 65535 heads
 * or sequences), KDA_ERR_CUDA (launch failure); a kernel that gives up waiting
 * on the tensor core reports KDA_ERR_DEVICE_TIMEOUT through
 * kda_get_device_status.
 */
kda_status kda_layer_core_fused(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                                const void *qp, const void *kp, const void *vp,
                                const float *conv_w, const void *z, const float *A,
                                const float *b, const void *beta_logit, const void *g,
                                const int32_t *cu_seqlens, const float *S0, float scale,
                                float l2_eps, float rms_eps, kda_dtype out_dtype, void *o_gated,
                                float *S_final, void *stream);

/*
 * kda_layer_core_fused_unbounded_decay - kda_layer_core_fused with Kimi Linear's decay
 * gate log alpha = -e^{A_h} softplus(z + b), which has no floor ("Kimi K3's
 * Architecture: Kimi Delta Attention, Attention Residuals, and 896 Experts", section
 * "Channel-wise decay, and the floor K3 puts under it": K3 bounds the decay so that the
 * chunk's reciprocal decays stay in range; Kimi Linear did not).  Arguments, results and
 * errors are those of kda_layer_core_fused.
 * Each 32-token chunk takes the tensor-core form when every one of its decay factors lies
 * within the range that the -5 floor would guarantee (about e^{+-80} around the chunk's
 * middle), and otherwise runs token by token on the state inside the same kernel, exactly
 * for any decay (log alpha = -inf included).  On inputs like the 16-sequence layer workload
 * (A ~ N(0, 0.5), z ~ N(0, 1)) about one chunk in 10^5 takes the token-by-token form.
 */
kda_status kda_layer_core_fused_unbounded_decay(
    int32_t num_seqs, int32_t total_tokens, int32_t num_heads, const void *qp, const void *kp,
    const void *vp, const float *conv_w, const void *z, const float *A, const float *b,
    const void *beta_logit, const void *g, const int32_t *cu_seqlens, const float *S0, float scale,
    float l2_eps, float rms_eps, kda_dtype out_dtype, void *o_gated, float *S_final, void *stream);

/*
 * kda_layer_core_fused_with_checkpoints - kda_layer_core_fused that also leaves
 * the recurrent state's snapshots every ckpt_every tokens of each sequence, as
 * kda_prefill_with_checkpoints does (same ckpt_every, ckpt_base, ckpt_states
 * meaning, layout and errors).  A snapshot holds only the recurrent state; the
 * short convolution's state at that token is the three pre-convolution inputs
 * before it, which the caller already holds in qp, kp, vp.
 */
kda_status kda_layer_core_fused_with_checkpoints(
    int32_t num_seqs, int32_t total_tokens, int32_t num_heads, const void *qp, const void *kp,
    const void *vp, const float *conv_w, const void *z, const float *A, const float *b,
    const void *beta_logit, const void *g, const int32_t *cu_seqlens, const float *S0, float scale,
    float l2_eps, float rms_eps, kda_dtype out_dtype, void *o_gated, float *S_final,
    int32_t ckpt_every, const int32_t *ckpt_base, float *ckpt_states, void *stream);

/*
 * kda_decode_layer - one decode step of the whole layer core for a batch of
 * requests whose recurrent state and short-convolution state live in pools
 * ("Kimi K3 · KDA layer", KDA equation list; a decoding request carries its own
 * KDA state and short-convolution state: "Inside Kimi K3: How KDA, AttnRes, and
 * 896 Experts Work", section "KDA writes corrections into a recurrent matrix";
 * fixed per-request state blocks in a pool, mutated only in the request's own
 * working slot: "Kimi K3: Architecture and SGLang Day-0 Support", sections
 * "RadixAttention: prefix caching for KDA state" and "Memory management for two
 * state types").
 *
 * For request b and head h, with n = slot[b]:
 *   x^c = SiLU(w0 x^p + w1 x_{t-1} + w2 x_{t-2} + w3 x_{t-3}) for x in q, k, v, the three
 *         previous inputs taken from conv_pool row n (which then shifts by one token);
 *   q^, k^ = L2-normalised q^c, k^c; log_alpha = -5 sigmoid(e^A (z + b)); beta = sigmoid(beta_logit);
 *   the recurrence step of kda_decode_step on S_pool row n (updated in place);
 *   o = sigmoid(g) o~ / sqrt(mean(o~^2) + rms_eps).
 * A request at the start of its sequence has a zeroed conv_pool row (zero history,
 * as in the prefill) and the S0 it starts from in its S_pool row.
 *
 *   batch, num_heads, pool_size >= 1; P = pool_size rows in each pool
 *   qp, kp, vp  [B][H][128] bf16: this token's pre-convolution projections
 *   conv_w      [3][H*128][4] fp32 (taps: w0 multiplies the current token)
 *   z, g        [B][H][128] bf16;  A [H] fp32;  b [H][128] fp32 or NULL (zero)
 *   beta_logit  [B][H] bf16
 *   slot        [B] int32, device: the pool row of each request; rows must be
 *               distinct within a call (repeated rows race).  A row outside
 *               [0, P) leaves that request untouched and records
 *               KDA_ERR_DEVICE_CHECK (detail = b) in the device status word.
 *   S_pool      [P][H][128][128] fp32, row j = key channel, updated in place
 *   conv_pool   [P][3][3][H][128] bf16: stream (q, k, v), tap (t-1, t-2, t-3);
 *               updated in place
 *   o           [B][H][128] out_dtype
 * All pointers are caller-owned device memory; qp, kp, vp, z, g, conv_w, S_pool,
 * conv_pool and o 16-byte aligned; the pools must not overlap.  Nothing is
 * allocated.
 * Errors: KDA_ERR_INVALID_ARGUMENT (null/misaligned pointers, bad sizes or dtype,
 * overlapping pools), KDA_ERR_UNSUPPORTED (batch * heads above 2^31 - 1),
 * KDA_ERR_CUDA (launch failure).
 */
kda_status kda_decode_layer(int32_t batch, int32_t num_heads, int32_t pool_size,
                            const void *qp, const void *kp, const void *vp, const float *conv_w,
                            const void *z, const float *A, const float *b, const void *beta_logit,
                            const void *g, const int32_t *slot, float *S_pool, void *conv_pool,
                            float scale, float l2_eps, float rms_eps, kda_dtype out_dtype,
                            void *o, void *stream);

/*
 * kda_decode_tokens - a few tokens per request from a state held in a pool:
 * the verify and replay steps of speculative decoding.
 *
 * For each request b, its tokens t in [cu_tokens[b], cu_tokens[b+1]) run the
 * recurrence in order, starting from S_pool[slot[b]][h], exactly as kda_prefill
 * over that sequence with S0 = that row.  o~ is written for every token.  The
 * state after the request's last token goes back to the pool row when
 * write_back = 1, and to S_final[b] when S_final is not NULL.
 *   Verify (write_back = 0): the draft tokens are scored against the row
 *   without changing it, so rows may be shared by several requests (branches
 *   from one cached state).  Replay (write_back = 1): the accepted tokens are
 *   run again and the row advances ("Inside Kimi K3: How KDA, AttnRes, and 896
 *   Experts Work", section "What could go wrong": a rejected draft cannot be
 *   rolled back in a recurrent state, so the accepted inputs are replayed;
 *   "Kimi K3: Architecture and SGLang Day-0 Support", section "RadixAttention:
 *   prefix caching for KDA state": a request mutates only its own slot).
 * Each (request, head) reads its state once and writes it at most twice, with
 * all of the request's tokens applied in registers in between: meant for a few
 * tokens (a speculative draft); longer inputs belong to kda_prefill.
 *
 *   in_dtype, out_dtype  as kda_decode_step
 *   batch        B >= 1 requests; num_heads H >= 1; pool_size P >= 1 rows
 *   total_tokens T >= 0 rows of q, k, v, log_alpha, beta, o
 *   cu_tokens    [B+1] int32 (device): 0 <= cu[b] <= cu[b+1] <= T (request b
 *                may have zero tokens: its state is then copied unchanged)
 *   slot         [B] int32 (device) pool rows in [0, P); with write_back = 1
 *                no two requests may name the same row
 *   q, k         [T][H][128] in_dtype, expected unit-norm per head
 *   v            [T][H][128] in_dtype
 *   log_alpha    [T][H][128] fp32 (-inf allowed: alpha = 0)
 *   beta         [T][H] fp32
 *   S_pool       [P][H][128][128] fp32
 *   write_back   0 or 1
 *   S_final      [B][H][128][128] fp32 or NULL; must not overlap S_pool
 *   o            [T][H][128] out_dtype
 * Pointers are caller-owned device memory, 16-byte aligned (beta, cu_tokens and
 * slot 4-byte); q, k, v, log_alpha, beta and o may be NULL when T = 0.
 * Errors: KDA_ERR_INVALID_ARGUMENT (null/misaligned pointers, bad sizes, dtype
 * or write_back, S_final overlapping the pool), KDA_ERR_UNSUPPORTED (B * H above
 * 2^31 - 2^16 or T * H above 2^31 - 1), KDA_ERR_CUDA (launch failure).  A request whose slot
 * lies outside [0, P) or whose token range lies outside [0, T) is refused by
 * the kernel: nothing is read or written for it and kda_get_device_status
 * reports KDA_ERR_DEVICE_CHECK with detail = b.
 */
kda_status kda_decode_tokens(kda_dtype in_dtype, kda_dtype out_dtype, int32_t batch,
                             int32_t num_heads, int32_t pool_size, int32_t total_tokens,
                             const int32_t *cu_tokens, const int32_t *slot, const void *q,
                             const void *k, const void *v, const float *log_alpha,
                             const float *beta, float *S_pool, int32_t write_back, float *S_final,
                             float scale, void *o, void *stream);

/* Most tokens one request may bring to kda_decode_layer_tokens in one call. */
#define KDA_DECODE_LAYER_MAX_TOKENS 16

/*
 * kda_decode_layer_tokens - the whole layer core (short convolution, L2 norms,
 * gates, recurrence, output gate) for a few tokens per request whose recurrent
 * and short-convolution states live in pools: the layer-level verify and replay
 * steps of speculative decoding ("Kimi K3 · KDA layer", KDA equation list;
 * "Inside Kimi K3: How KDA, AttnRes, and 896 Experts Work", sections "KDA writes
 * corrections into a recurrent matrix" and "What could go wrong").
 *
 * Request b's tokens are rows [cu_tokens[b], cu_tokens[b+1]) (at most
 * KDA_DECODE_LAYER_MAX_TOKENS).  Its convolution window is the row's
 * convolution state (the three earlier pre-convolution inputs) followed by its
 * tokens' q^p, k^p, v^p; the recurrence runs from S_pool[slot[b]] over the
 * tokens; o_gated is written for every token.  Exactly as kda_decode_layer
 * applied to the tokens one after another, except that with write_back = 0
 * (verify) neither pool changes (rows may then be shared by several requests),
 * and with write_back = 1 (replay; distinct rows) both rows advance past the
 * last token.  A request with no tokens changes nothing.
 *
 *   Pools, weights and per-token inputs as kda_decode_layer, with the per-token
 *   inputs packed over all requests' tokens: qp, kp, vp, z, g [T][H][128] bf16,
 *   beta_logit [T][H] bf16, o_gated [T][H][128] out_dtype; cu_tokens [B+1] and
 *   slot [B] int32 (device).  Per-token pointers may be NULL when T = 0.
 * Errors: KDA_ERR_INVALID_ARGUMENT (null/misaligned pointers, bad sizes, dtype or
 * write_back, overlapping pools), KDA_ERR_UNSUPPORTED (B * H or T * H above
 * 2^31 - 1), KDA_ERR_CUDA (launch failure).  A request whose slot lies outside
 * [0, P), whose token range lies outside [0, T) or holds more than
 * KDA_DECODE_LAYER_MAX_TOKENS tokens is refused by the kernel (nothing read or
 * written for it; KDA_ERR_DEVICE_CHECK with detail = b).
 */
kda_status kda_decode_layer_tokens(int32_t batch, int32_t num_heads, int32_t pool_size,
                                   int32_t total_tokens, const int32_t *cu_tokens,
                                   const int32_t *slot, const void *qp, const void *kp,
                                   const void *vp, const float *conv_w, const void *z,
                                   const float *A, const float *b, const void *beta_logit,
                                   const void *g, float *S_pool, void *conv_pool,
                                   int32_t write_back, float scale, float l2_eps, float rms_eps,
                                   kda_dtype out_dtype, void *o, void *stream);

/*
 * kda_check_prefill_inputs - the contents checks the host cannot make before a
 * prefill: cu_seqlens starts at 0, never decreases and ends at total_tokens;
 * every log alpha lies in [-5, 0] and is not NaN (the floor g_min = -5 bounds the
 * chunk's reciprocal decays: "Kimi K3's Architecture: Kimi Delta Attention,
 * Attention Residuals, and 896 Experts", section "Channel-wise decay, and the
 * floor K3 puts under it").  One read of log_alpha on `stream`; a failure is
 * reported by kda_get_device_status as KDA_ERR_DEVICE_CHECK with detail =
 * (kind << 28) | index, kind 1 = cu_seqlens (index = n), kind 2 = log alpha
 * (index = the token of a failing value).  A library built with KDA_DEBUG
 * defined runs these checks inside every kda_prefill* call.
 *
 *   log_alpha    [T][H][128] fp32 (16-byte aligned), or [T][H] (4-byte aligned)
 *                with head_decay = 1, or NULL to check cu_seqlens only
 *   head_decay   0 or 1
 *   cu_seqlens   [N+1] int32 (device)
 * Errors: KDA_ERR_INVALID_ARGUMENT (sizes, flags, null or misaligned pointers),
 * KDA_ERR_CUDA (launch failure).
 */
kda_status kda_check_prefill_inputs(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                                    const float *log_alpha, int32_t head_decay,
                                    const int32_t *cu_seqlens, void *stream);

/*
 * kda_get_device_status - synchronises `stream`, then returns and clears the
 * device status word: KDA_OK, KDA_ERR_DEVICE_TIMEOUT or KDA_ERR_DEVICE_CHECK
 * (KDA_ERR_CUDA if the synchronisation itself fails).  If detail is not
 * NULL it receives the kernel-specific code recorded with the status (0 if
 * none).
 */
kda_status kda_get_device_status(void *stream, uint32_t *detail);

/*
 * kda_debug_inject_handoff_timeout - test-only fault injection that lets a test
 * check, on a GPU, that a device-side wait which runs out is reported through
 * the status word and leaves the context usable.  The pages have no counterpart:
 * this is failure-detection plumbing.
 *
 * In a library built with KDA_DEBUG defined it arms the NEXT launch of the
 * tensor-core prefill (kda_prefill, kda_prefill_with_checkpoints and
 * kda_prefill_head_decay with bf16 inputs).  In that launch the warps that build
 * each chunk's operands skip their first "chunk ready" hand-off (nothing has been
 * issued into that chunk's slot by then), and every wait of the launch gives up
 * after 1 ms instead of 2 s.  The warps that consume the chunk give up waiting
 * for it, the launch leaves without writing its results, and
 * kda_get_device_status reports KDA_ERR_DEVICE_TIMEOUT with detail 20 (the wait
 * for a ready chunk).  A sequence of two chunks (33 to 64 tokens) keeps that the
 * only wait that runs out.  Later launches are unaffected.
 * The normal library arms nothing and returns KDA_ERR_UNSUPPORTED.  The armed
 * state is shared by the process: do not call it while other threads launch
 * prefills.
 */
kda_status kda_debug_inject_handoff_timeout(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
