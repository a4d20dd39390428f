// C ABI of libkda: argument validation on the host, then kernel launches.
// Nothing here allocates device memory.
#include <atomic>
#include <cstring>

#include "kda_common.cuh"

namespace kda {
namespace {

// Device status word ([0] = kda_status, [1] = detail); see kda_get_device_status.
__device__ uint32_t g_status_word[2];

constexpr int kMaxDevices = 64;
std::atomic<uint32_t *> g_status_ptr[kMaxDevices];

DeviceStatus device_status() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return {nullptr};
    uint32_t *p = g_status_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return {nullptr};
        p = static_cast<uint32_t *>(addr);
        g_status_ptr[dev].store(p, std::memory_order_release);
    }
    return {p};
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok_ptr(const void *p) { return p != nullptr && aligned16(p); }
bool ok_opt_ptr(const void *p) { return p == nullptr || aligned16(p); }
// Per-row scalars (beta, cu_seqlens, beta_logit) need only their element alignment.
bool ok_ptr_elem(const void *p, size_t align) {
    return p != nullptr && (reinterpret_cast<uintptr_t>(p) & (align - 1)) == 0;
}
bool ok_dtype(kda_dtype d) { return d == KDA_BF16 || d == KDA_FP32; }

bool overlap(const void *a, const void *b, size_t bytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bytes && y < x + bytes;
}

kda_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

// Checkpoint arguments: none (every == 0), or every a positive multiple of the prefill's
// 32-token chunk with the offsets and the states both given.
bool ok_checkpoints(int32_t every, const int32_t *base, const float *states) {
    if (every == 0) return true;
    return every > 0 && every % 32 == 0 && ok_ptr_elem(base, 4) && ok_ptr(states);
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" {

const char *kda_status_string(kda_status status) {
    switch (status) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARGUMENT: return "KDA_ERR_INVALID_ARGUMENT";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_DEVICE_TIMEOUT: return "KDA_ERR_DEVICE_TIMEOUT";
        case KDA_ERR_DEVICE_CHECK: return "KDA_ERR_DEVICE_CHECK";
    }
    return "KDA_UNKNOWN_STATUS";
}

int32_t kda_version(void) { return 200; }  // 0.2.0: snapshots, multi-token decode, decay variants, checks

size_t kda_prefill_workspace_size(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                                  kda_dtype in_dtype) {
    (void)num_seqs; (void)total_tokens; (void)num_heads; (void)in_dtype;
    return 0;
}

kda_status kda_prefill(kda_dtype in_dtype, kda_dtype out_dtype, int32_t num_seqs,
                       int32_t total_tokens, int32_t num_heads, const void *q, const void *k,
                       const void *v, const float *log_alpha, const float *beta,
                       const float *S0, const int32_t *cu_seqlens, float scale, void *o,
                       float *S_final, void *workspace, size_t workspace_bytes, void *stream) {
    return kda_prefill_with_checkpoints(in_dtype, out_dtype, num_seqs, total_tokens, num_heads, q,
                                        k, v, log_alpha, beta, S0, cu_seqlens, scale, o, S_final,
                                        workspace, workspace_bytes, 0, nullptr, nullptr, stream);
}

}  // extern "C"

namespace {
// kda_prefill in full: per-channel decay ([T][H][128]) or one decay per (token, head) ([T][H]).
kda_status prefill_impl(kda_dtype in_dtype, kda_dtype out_dtype, int32_t num_seqs,
                        int32_t total_tokens, int32_t num_heads, const void *q, const void *k,
                        const void *v, const float *log_alpha, bool head_decay, bool unbounded,
                        const float *beta,
                        const float *S0, const int32_t *cu_seqlens, float scale, void *o,
                        float *S_final, void *workspace, size_t workspace_bytes,
                        int32_t ckpt_every, const int32_t *ckpt_base, float *ckpt_states,
                        void *stream) {
    if (!ok_dtype(in_dtype) || !ok_dtype(out_dtype)) return KDA_ERR_INVALID_ARGUMENT;
    if (!ok_checkpoints(ckpt_every, ckpt_base, ckpt_states)) return KDA_ERR_INVALID_ARGUMENT;
    if (num_seqs < 1 || total_tokens < 0 || num_heads < 1) return KDA_ERR_INVALID_ARGUMENT;
    if (!ok_ptr_elem(cu_seqlens, 4)) return KDA_ERR_INVALID_ARGUMENT;
    if (total_tokens > 0) {
        const bool la_ok = head_decay ? ok_ptr_elem(log_alpha, 4) : ok_ptr(log_alpha);
        if (!ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !la_ok || !ok_ptr_elem(beta, 4) || !ok_ptr(o))
            return KDA_ERR_INVALID_ARGUMENT;
    }
    if (!ok_opt_ptr(S0) || !ok_opt_ptr(S_final)) return KDA_ERR_INVALID_ARGUMENT;
    const size_t state_bytes = (size_t)num_seqs * num_heads * kD * kD * sizeof(float);
    if (S0 && S_final && S0 != S_final && overlap(S0, S_final, state_bytes))
        return KDA_ERR_INVALID_ARGUMENT;
    if (num_heads > 65535 || num_seqs > 65535) return KDA_ERR_UNSUPPORTED;
    const size_t need = kda_prefill_workspace_size(num_seqs, total_tokens, num_heads, in_dtype);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
        return KDA_ERR_WORKSPACE;

#ifdef KDA_DEBUG
    // debug builds: the contents checks run before every prefill with the decay floor
    if (!unbounded) {
        CheckArgs c{num_seqs, total_tokens, num_heads, head_decay ? 1 : 0,
                    total_tokens > 0 ? log_alpha : nullptr, cu_seqlens, device_status()};
        if (launch_check_prefill(c, static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return KDA_ERR_CUDA;
    }
#endif
    PrefillArgs a;
    a.in_dtype = in_dtype; a.out_dtype = out_dtype;
    a.num_seqs = num_seqs; a.total_tokens = total_tokens; a.num_heads = num_heads;
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.S0 = S0;
    a.cu_seqlens = cu_seqlens; a.scale = scale; a.o = o; a.S_final = S_final;
    a.workspace = workspace; a.workspace_bytes = workspace_bytes;
    a.ckpt = Checkpoints{ckpt_every, ckpt_base, ckpt_states};
    a.head_decay = head_decay ? 1 : 0;
    a.unbounded = unbounded ? 1 : 0;
    a.status = device_status();
    // bf16 inputs: chunked tensor-core kernel (without the floor, chunks out of its range run
    // token by token inside it); fp32 inputs: the token-by-token kernel, exact for any decay.
    if (in_dtype == KDA_BF16)
        return from_cuda(launch_prefill_tc(a, static_cast<cudaStream_t>(stream)));
    return from_cuda(launch_prefill_recurrent(a, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

kda_status kda_prefill_with_checkpoints(kda_dtype in_dtype, kda_dtype out_dtype, int32_t num_seqs,
                                        int32_t total_tokens, int32_t num_heads, const void *q,
                                        const void *k, const void *v, const float *log_alpha,
                                        const float *beta, const float *S0,
                                        const int32_t *cu_seqlens, float scale, void *o,
                                        float *S_final, void *workspace, size_t workspace_bytes,
                                        int32_t ckpt_every, const int32_t *ckpt_base,
                                        float *ckpt_states, void *stream) {
    return prefill_impl(in_dtype, out_dtype, num_seqs, total_tokens, num_heads, q, k, v, log_alpha,
                        false, false, beta, S0, cu_seqlens, scale, o, S_final, workspace,
                        workspace_bytes, ckpt_every, ckpt_base, ckpt_states, stream);
}

kda_status kda_prefill_head_decay(kda_dtype in_dtype, kda_dtype out_dtype, int32_t num_seqs,
                                  int32_t total_tokens, int32_t num_heads, const void *q,
                                  const void *k, const void *v, const float *log_alpha,
                                  const float *beta, const float *S0, const int32_t *cu_seqlens,
                                  float scale, void *o, float *S_final, void *workspace,
                                  size_t workspace_bytes, int32_t ckpt_every,
                                  const int32_t *ckpt_base, float *ckpt_states, void *stream) {
    return prefill_impl(in_dtype, out_dtype, num_seqs, total_tokens, num_heads, q, k, v, log_alpha,
                        true, false, beta, S0, cu_seqlens, scale, o, S_final, workspace,
                        workspace_bytes, ckpt_every, ckpt_base, ckpt_states, stream);
}

kda_status kda_prefill_unbounded_decay(kda_dtype in_dtype, kda_dtype out_dtype, int32_t num_seqs,
                                       int32_t total_tokens, int32_t num_heads, const void *q,
                                       const void *k, const void *v, const float *log_alpha,
                                       const float *beta, const float *S0,
                                       const int32_t *cu_seqlens, float scale, void *o,
                                       float *S_final, void *workspace, size_t workspace_bytes,
                                       void *stream) {
    return prefill_impl(in_dtype, out_dtype, num_seqs, total_tokens, num_heads, q, k, v, log_alpha,
                        false, true, beta, S0, cu_seqlens, scale, o, S_final, workspace,
                        workspace_bytes, 0, nullptr, nullptr, stream);
}

}  // extern "C"

namespace {
kda_status decode_impl(kda_dtype in_dtype, kda_dtype out_dtype, int32_t batch, int32_t num_heads,
                       const void *q, const void *k, const void *v, const float *log_alpha,
                       bool head_decay, const float *beta, float *S_inout, float scale, void *o,
                       void *stream) {
    if (!ok_dtype(in_dtype) || !ok_dtype(out_dtype)) return KDA_ERR_INVALID_ARGUMENT;
    if (batch < 1 || num_heads < 1) return KDA_ERR_INVALID_ARGUMENT;
    const bool la_ok = head_decay ? ok_ptr_elem(log_alpha, 4) : ok_ptr(log_alpha);
    if (!ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !la_ok || !ok_ptr_elem(beta, 4) ||
        !ok_ptr(S_inout) || !ok_ptr(o))
        return KDA_ERR_INVALID_ARGUMENT;
    if ((int64_t)batch * num_heads > 0x7fffffffLL) return KDA_ERR_UNSUPPORTED;
    DecodeArgs a;
    a.in_dtype = in_dtype; a.out_dtype = out_dtype;
    a.batch = batch; a.num_heads = num_heads;
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta;
    a.head_decay = head_decay ? 1 : 0;
    a.S = S_inout; a.scale = scale; a.o = o;
    a.status = device_status();
    return from_cuda(launch_decode(a, static_cast<cudaStream_t>(stream)));
}
}  // namespace

extern "C" {

kda_status kda_decode_step(kda_dtype in_dtype, kda_dtype out_dtype, int32_t batch,
                           int32_t num_heads, const void *q, const void *k, const void *v,
                           const float *log_alpha, const float *beta, float *S_inout,
                           float scale, void *o, void *stream) {
    return decode_impl(in_dtype, out_dtype, batch, num_heads, q, k, v, log_alpha, false, beta,
                       S_inout, scale, o, stream);
}

kda_status kda_decode_step_head_decay(kda_dtype in_dtype, kda_dtype out_dtype, int32_t batch,
                                      int32_t num_heads, const void *q, const void *k,
                                      const void *v, const float *log_alpha, const float *beta,
                                      float *S_inout, float scale, void *o, void *stream) {
    return decode_impl(in_dtype, out_dtype, batch, num_heads, q, k, v, log_alpha, true, beta,
                       S_inout, scale, o, stream);
}

}  // extern "C"

namespace {
kda_status frontend_impl(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                         const void *qp, const void *kp, const void *vp, const float *conv_w,
                         const void *z, const float *A, const float *b, const void *beta_logit,
                         const int32_t *cu_seqlens, float l2_eps, kda_dtype out_dtype,
                         void *q_hat, void *k_hat, void *v_out, float *log_alpha, float *beta,
                         bool unbounded_decay, void *stream) {
    if (!ok_dtype(out_dtype)) return KDA_ERR_INVALID_ARGUMENT;
    if (num_seqs < 1 || total_tokens < 0 || num_heads < 1) return KDA_ERR_INVALID_ARGUMENT;
    if (!ok_ptr_elem(cu_seqlens, 4) || !ok_ptr(conv_w) || !ok_ptr_elem(A, 4) || !ok_opt_ptr(b))
        return KDA_ERR_INVALID_ARGUMENT;
    if (total_tokens > 0) {
        if (!ok_ptr(qp) || !ok_ptr(kp) || !ok_ptr(vp) || !ok_ptr(z) || !ok_ptr_elem(beta_logit, 2) ||
            !ok_ptr(q_hat) || !ok_ptr(k_hat) || !ok_ptr(v_out) || !ok_ptr(log_alpha) ||
            !ok_ptr_elem(beta, 4))
            return KDA_ERR_INVALID_ARGUMENT;
    }
    if ((int64_t)total_tokens * num_heads / 8 >= 0x7fffffffLL) return KDA_ERR_UNSUPPORTED;
    FrontendArgs a;
    a.num_seqs = num_seqs; a.total_tokens = total_tokens; a.num_heads = num_heads;
    a.qp = static_cast<const __nv_bfloat16 *>(qp);
    a.kp = static_cast<const __nv_bfloat16 *>(kp);
    a.vp = static_cast<const __nv_bfloat16 *>(vp);
    a.z = static_cast<const __nv_bfloat16 *>(z);
    a.beta_logit = static_cast<const __nv_bfloat16 *>(beta_logit);
    a.conv_w = conv_w; a.A = A; a.b = b; a.cu_seqlens = cu_seqlens; a.l2_eps = l2_eps;
    a.out_dtype = out_dtype; a.q_hat = q_hat; a.k_hat = k_hat; a.v_out = v_out;
    a.log_alpha = log_alpha; a.beta = beta;
    a.unbounded_decay = unbounded_decay ? 1 : 0;
    return from_cuda(launch_frontend(a, static_cast<cudaStream_t>(stream)));
}
}  // namespace

extern "C" {

kda_status kda_frontend(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                        const void *qp, const void *kp, const void *vp, const float *conv_w,
                        const void *z, const float *A, const float *b, const void *beta_logit,
                        const int32_t *cu_seqlens, float l2_eps, kda_dtype out_dtype,
                        void *q_hat, void *k_hat, void *v_out, float *log_alpha, float *beta,
                        void *stream) {
    return frontend_impl(num_seqs, total_tokens, num_heads, qp, kp, vp, conv_w, z, A, b,
                         beta_logit, cu_seqlens, l2_eps, out_dtype, q_hat, k_hat, v_out,
                         log_alpha, beta, false, stream);
}

kda_status kda_frontend_unbounded_decay(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                                        const void *qp, const void *kp, const void *vp,
                                        const float *conv_w, const void *z, const float *A,
                                        const float *b, const void *beta_logit,
                                        const int32_t *cu_seqlens, float l2_eps,
                                        kda_dtype out_dtype, void *q_hat, void *k_hat,
                                        void *v_out, float *log_alpha, float *beta,
                                        void *stream) {
    return frontend_impl(num_seqs, total_tokens, num_heads, qp, kp, vp, conv_w, z, A, b,
                         beta_logit, cu_seqlens, l2_eps, out_dtype, q_hat, k_hat, v_out,
                         log_alpha, beta, true, stream);
}

kda_status kda_output_gate(int64_t num_rows, kda_dtype in_dtype, const void *o_tilde,
                           const void *g, float eps, kda_dtype out_dtype, void *out,
                           void *stream) {
    if (!ok_dtype(in_dtype) || !ok_dtype(out_dtype) || num_rows < 0)
        return KDA_ERR_INVALID_ARGUMENT;
    if (num_rows > 0 && (!ok_ptr(o_tilde) || !ok_ptr(g) || !ok_ptr(out)))
        return KDA_ERR_INVALID_ARGUMENT;
    if (num_rows / 8 >= 0x7fffffffLL) return KDA_ERR_UNSUPPORTED;
    GateArgs a;
    a.num_rows = num_rows; a.in_dtype = in_dtype; a.out_dtype = out_dtype;
    a.o_tilde = o_tilde; a.g = static_cast<const __nv_bfloat16 *>(g); a.eps = eps; a.out = out;
    return from_cuda(launch_output_gate(a, static_cast<cudaStream_t>(stream)));
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t kda_layer_core_workspace_size(int32_t num_seqs, int32_t total_tokens, int32_t num_heads) {
    (void)num_seqs;
    if (total_tokens < 0 || num_heads < 1) return 0;
    const size_t rows = (size_t)total_tokens * num_heads;
    return 3 * align256(rows * kD * 4)    /* q^, k^, v fp32 */
           + align256(rows * kD * 4)      /* log_alpha fp32 */
           + align256(rows * 4)           /* beta fp32 */
           + align256(rows * kD * 4)      /* o~ fp32 */
           + kda_prefill_workspace_size(num_seqs, total_tokens, num_heads, KDA_FP32);
}

}  // extern "C"

namespace {
kda_status layer_core_impl(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                           const void *qp, const void *kp, const void *vp, const float *conv_w,
                           const void *z, const float *A, const float *b, const void *beta_logit,
                           const void *g, const int32_t *cu_seqlens, const float *S0, float scale,
                           float l2_eps, float rms_eps, kda_dtype out_dtype, void *o_gated,
                           float *S_final, void *workspace, size_t workspace_bytes,
                           bool unbounded_decay, void *stream) {
    if (!ok_dtype(out_dtype)) return KDA_ERR_INVALID_ARGUMENT;
    if (num_seqs < 1 || total_tokens < 0 || num_heads < 1) return KDA_ERR_INVALID_ARGUMENT;
    if (total_tokens > 0 && (!ok_ptr(g) || !ok_ptr(o_gated))) return KDA_ERR_INVALID_ARGUMENT;
    const size_t need = kda_layer_core_workspace_size(num_seqs, total_tokens, num_heads);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
        return KDA_ERR_WORKSPACE;
    const size_t rows = (size_t)total_tokens * num_heads;
    unsigned char *w = static_cast<unsigned char *>(workspace);
    void *q_hat = w;
    void *k_hat = w + align256(rows * kD * 4);
    void *v_out = w + 2 * align256(rows * kD * 4);
    float *log_alpha = reinterpret_cast<float *>(w + 3 * align256(rows * kD * 4));
    float *beta = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(log_alpha) +
                                            align256(rows * kD * 4));
    float *o_tilde = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(beta) +
                                               align256(rows * 4));
    void *pre_ws = reinterpret_cast<unsigned char *>(o_tilde) + align256(rows * kD * 4);
    const size_t pre_ws_bytes = kda_prefill_workspace_size(num_seqs, total_tokens, num_heads,
                                                           KDA_FP32);
    kda_status st = frontend_impl(num_seqs, total_tokens, num_heads, qp, kp, vp, conv_w, z, A, b,
                                  beta_logit, cu_seqlens, l2_eps, KDA_FP32, q_hat, k_hat, v_out,
                                  log_alpha, beta, unbounded_decay, stream);
    if (st != KDA_OK) return st;
    // (the unbounded gate has no decay floor: its prefill skips the debug contents checks)
    st = (unbounded_decay ? kda_prefill_unbounded_decay : kda_prefill)(
        KDA_FP32, KDA_FP32, num_seqs, total_tokens, num_heads, q_hat, k_hat, v_out, log_alpha,
        beta, S0, cu_seqlens, scale, o_tilde, S_final, pre_ws, pre_ws_bytes, stream);
    if (st != KDA_OK) return st;
    return kda_output_gate((int64_t)rows, KDA_FP32, o_tilde, g, rms_eps, out_dtype, o_gated,
                           stream);
}
}  // namespace

extern "C" {

kda_status kda_layer_core(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                          const void *qp, const void *kp, const void *vp, const float *conv_w,
                          const void *z, const float *A, const float *b, const void *beta_logit,
                          const void *g, const int32_t *cu_seqlens, const float *S0, float scale,
                          float l2_eps, float rms_eps, kda_dtype out_dtype, void *o_gated,
                          float *S_final, void *workspace, size_t workspace_bytes, void *stream) {
    return layer_core_impl(num_seqs, total_tokens, num_heads, qp, kp, vp, conv_w, z, A, b,
                           beta_logit, g, cu_seqlens, S0, scale, l2_eps, rms_eps, out_dtype,
                           o_gated, S_final, workspace, workspace_bytes, false, stream);
}

kda_status kda_layer_core_unbounded_decay(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                                          const void *qp, const void *kp, const void *vp,
                                          const float *conv_w, const void *z, const float *A,
                                          const float *b, const void *beta_logit, const void *g,
                                          const int32_t *cu_seqlens, const float *S0, float scale,
                                          float l2_eps, float rms_eps, kda_dtype out_dtype,
                                          void *o_gated, float *S_final, void *workspace,
                                          size_t workspace_bytes, void *stream) {
    return layer_core_impl(num_seqs, total_tokens, num_heads, qp, kp, vp, conv_w, z, A, b,
                           beta_logit, g, cu_seqlens, S0, scale, l2_eps, rms_eps, out_dtype,
                           o_gated, S_final, workspace, workspace_bytes, true, stream);
}

kda_status kda_layer_core_fused(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                                const void *qp, const void *kp, const void *vp,
                                const float *conv_w, const void *z, const float *A,
                                const float *b, const void *beta_logit, const void *g,
                                const int32_t *cu_seqlens, const float *S0, float scale,
                                float l2_eps, float rms_eps, kda_dtype out_dtype, void *o_gated,
                                float *S_final, void *stream) {
    return kda_layer_core_fused_with_checkpoints(num_seqs, total_tokens, num_heads, qp, kp, vp,
                                                 conv_w, z, A, b, beta_logit, g, cu_seqlens, S0,
                                                 scale, l2_eps, rms_eps, out_dtype, o_gated, S_final,
                                                 0, nullptr, nullptr, stream);
}

static kda_status layer_core_fused_impl(
    int32_t num_seqs, int32_t total_tokens, int32_t num_heads, const void *qp, const void *kp,
    const void *vp, const float *conv_w, const void *z, const float *A, const float *b,
    const void *beta_logit, const void *g, const int32_t *cu_seqlens, const float *S0, float scale,
    float l2_eps, float rms_eps, kda_dtype out_dtype, void *o_gated, float *S_final,
    int32_t ckpt_every, const int32_t *ckpt_base, float *ckpt_states, bool unbounded,
    void *stream) {
    if (!ok_dtype(out_dtype)) return KDA_ERR_INVALID_ARGUMENT;
    if (!ok_checkpoints(ckpt_every, ckpt_base, ckpt_states)) return KDA_ERR_INVALID_ARGUMENT;
    if (num_seqs < 1 || total_tokens < 0 || num_heads < 1) return KDA_ERR_INVALID_ARGUMENT;
    if (!ok_ptr_elem(cu_seqlens, 4) || !ok_ptr(conv_w) || !ok_ptr_elem(A, 4) || !ok_opt_ptr(b))
        return KDA_ERR_INVALID_ARGUMENT;
    if (total_tokens > 0) {
        if (!ok_ptr(qp) || !ok_ptr(kp) || !ok_ptr(vp) || !ok_ptr(z) || !ok_ptr_elem(beta_logit, 2) ||
            !ok_ptr(g) || !ok_ptr(o_gated))
            return KDA_ERR_INVALID_ARGUMENT;
    }
    if (!ok_opt_ptr(S0) || !ok_opt_ptr(S_final)) return KDA_ERR_INVALID_ARGUMENT;
    const size_t state_bytes = (size_t)num_seqs * num_heads * kD * kD * sizeof(float);
    if (S0 && S_final && S0 != S_final && overlap(S0, S_final, state_bytes))
        return KDA_ERR_INVALID_ARGUMENT;
    if (num_heads > 65535 || num_seqs > 65535) return KDA_ERR_UNSUPPORTED;
    LayerArgs a;
    a.num_seqs = num_seqs; a.total_tokens = total_tokens; a.num_heads = num_heads;
    a.qp = static_cast<const __nv_bfloat16 *>(qp);
    a.kp = static_cast<const __nv_bfloat16 *>(kp);
    a.vp = static_cast<const __nv_bfloat16 *>(vp);
    a.z = static_cast<const __nv_bfloat16 *>(z);
    a.beta_logit = static_cast<const __nv_bfloat16 *>(beta_logit);
    a.g = static_cast<const __nv_bfloat16 *>(g);
    a.conv_w = conv_w; a.A = A; a.b = b; a.S0 = S0; a.cu_seqlens = cu_seqlens;
    a.scale = scale; a.l2_eps = l2_eps; a.rms_eps = rms_eps;
    a.out_dtype = out_dtype; a.o = o_gated; a.S_final = S_final;
    a.ckpt = Checkpoints{ckpt_every, ckpt_base, ckpt_states};
    a.unbounded_decay = unbounded ? 1 : 0;
    a.status = device_status();
    return from_cuda(launch_layer_tc(a, static_cast<cudaStream_t>(stream)));
}

kda_status kda_layer_core_fused_with_checkpoints(
    int32_t num_seqs, int32_t total_tokens, int32_t num_heads, const void *qp, const void *kp,
    const void *vp, const float *conv_w, const void *z, const float *A, const float *b,
    const void *beta_logit, const void *g, const int32_t *cu_seqlens, const float *S0, float scale,
    float l2_eps, float rms_eps, kda_dtype out_dtype, void *o_gated, float *S_final,
    int32_t ckpt_every, const int32_t *ckpt_base, float *ckpt_states, void *stream) {
    return layer_core_fused_impl(num_seqs, total_tokens, num_heads, qp, kp, vp, conv_w, z, A, b,
                                 beta_logit, g, cu_seqlens, S0, scale, l2_eps, rms_eps, out_dtype,
                                 o_gated, S_final, ckpt_every, ckpt_base, ckpt_states, false,
                                 stream);
}

kda_status kda_layer_core_fused_unbounded_decay(
    int32_t num_seqs, int32_t total_tokens, int32_t num_heads, const void *qp, const void *kp,
    const void *vp, const float *conv_w, const void *z, const float *A, const float *b,
    const void *beta_logit, const void *g, const int32_t *cu_seqlens, const float *S0, float scale,
    float l2_eps, float rms_eps, kda_dtype out_dtype, void *o_gated, float *S_final, void *stream) {
    return layer_core_fused_impl(num_seqs, total_tokens, num_heads, qp, kp, vp, conv_w, z, A, b,
                                 beta_logit, g, cu_seqlens, S0, scale, l2_eps, rms_eps, out_dtype,
                                 o_gated, S_final, 0, nullptr, nullptr, true, stream);
}

kda_status kda_decode_layer(int32_t batch, int32_t num_heads, int32_t pool_size,
                            const void *qp, const void *kp, const void *vp, const float *conv_w,
                            const void *z, const float *A, const float *b, const void *beta_logit,
                            const void *g, const int32_t *slot, float *S_pool, void *conv_pool,
                            float scale, float l2_eps, float rms_eps, kda_dtype out_dtype,
                            void *o, void *stream) {
    if (!ok_dtype(out_dtype)) return KDA_ERR_INVALID_ARGUMENT;
    if (batch < 1 || num_heads < 1 || pool_size < 1) return KDA_ERR_INVALID_ARGUMENT;
    if (!ok_ptr(qp) || !ok_ptr(kp) || !ok_ptr(vp) || !ok_ptr(z) || !ok_ptr(g) || !ok_ptr(conv_w) ||
        !ok_ptr_elem(A, 4) || !ok_opt_ptr(b) || !ok_ptr_elem(beta_logit, 2) || !ok_ptr_elem(slot, 4) ||
        !ok_ptr(S_pool) || !ok_ptr(conv_pool) || !ok_ptr(o))
        return KDA_ERR_INVALID_ARGUMENT;
    const size_t state_bytes = (size_t)pool_size * num_heads * kD * kD * sizeof(float);
    const size_t conv_bytes = (size_t)pool_size * 9 * num_heads * kD * sizeof(__nv_bfloat16);
    const uintptr_t sp = reinterpret_cast<uintptr_t>(S_pool), cp = reinterpret_cast<uintptr_t>(conv_pool);
    if (sp < cp + conv_bytes && cp < sp + state_bytes) return KDA_ERR_INVALID_ARGUMENT;  // pools overlap
    if ((int64_t)batch * num_heads > 0x7fffffffLL) return KDA_ERR_UNSUPPORTED;
    DecodeLayerArgs a;
    a.batch = batch; a.num_heads = num_heads; a.pool_size = pool_size;
    a.qp = static_cast<const __nv_bfloat16 *>(qp);
    a.kp = static_cast<const __nv_bfloat16 *>(kp);
    a.vp = static_cast<const __nv_bfloat16 *>(vp);
    a.z = static_cast<const __nv_bfloat16 *>(z);
    a.beta_logit = static_cast<const __nv_bfloat16 *>(beta_logit);
    a.g = static_cast<const __nv_bfloat16 *>(g);
    a.conv_w = conv_w; a.A = A; a.b = b; a.slot = slot;
    a.S_pool = S_pool;
    a.conv_pool = static_cast<__nv_bfloat16 *>(conv_pool);
    a.scale = scale; a.l2_eps = l2_eps; a.rms_eps = rms_eps;
    a.out_dtype = out_dtype; a.o = o;
    a.status = device_status();
    return from_cuda(launch_decode_layer(a, static_cast<cudaStream_t>(stream)));
}

kda_status kda_decode_tokens(kda_dtype in_dtype, kda_dtype out_dtype, int32_t batch,
                             int32_t num_heads, int32_t pool_size, int32_t total_tokens,
                             const int32_t *cu_tokens, const int32_t *slot, const void *q,
                             const void *k, const void *v, const float *log_alpha,
                             const float *beta, float *S_pool, int32_t write_back, float *S_final,
                             float scale, void *o, void *stream) {
    if (!ok_dtype(in_dtype) || !ok_dtype(out_dtype)) return KDA_ERR_INVALID_ARGUMENT;
    if (batch < 1 || num_heads < 1 || pool_size < 1 || total_tokens < 0)
        return KDA_ERR_INVALID_ARGUMENT;
    if (write_back != 0 && write_back != 1) return KDA_ERR_INVALID_ARGUMENT;
    if (!ok_ptr_elem(cu_tokens, 4) || !ok_ptr_elem(slot, 4) || !ok_ptr(S_pool) ||
        !ok_opt_ptr(S_final))
        return KDA_ERR_INVALID_ARGUMENT;
    if (total_tokens > 0 && (!ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !ok_ptr(log_alpha) ||
                             !ok_ptr_elem(beta, 4) || !ok_ptr(o)))
        return KDA_ERR_INVALID_ARGUMENT;
    const size_t unit_bytes = (size_t)num_heads * kD * kD * sizeof(float);
    if (S_final != nullptr) {
        const uintptr_t sp = reinterpret_cast<uintptr_t>(S_pool), fp = reinterpret_cast<uintptr_t>(S_final);
        if (sp < fp + batch * unit_bytes && fp < sp + pool_size * unit_bytes)
            return KDA_ERR_INVALID_ARGUMENT;  // S_final overlaps the pool
    }
    // (the persistent kernel steps unit indices by its grid: they stay below 2^31)
    if ((int64_t)batch * num_heads > 0x7fff0000LL || (int64_t)total_tokens * num_heads > 0x7fffffffLL)
        return KDA_ERR_UNSUPPORTED;
    DecodeTokensArgs a;
    a.in_dtype = in_dtype; a.out_dtype = out_dtype;
    a.batch = batch; a.num_heads = num_heads; a.pool_size = pool_size; a.total_tokens = total_tokens;
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta;
    a.cu_tokens = cu_tokens; a.slot = slot;
    a.S_pool = S_pool; a.write_back = write_back; a.S_final = S_final;
    a.scale = scale; a.o = o;
    a.status = device_status();
    return from_cuda(launch_decode_tokens(a, static_cast<cudaStream_t>(stream)));
}

kda_status kda_decode_layer_tokens(int32_t batch, int32_t num_heads, int32_t pool_size,
                                   int32_t total_tokens, const int32_t *cu_tokens,
                                   const int32_t *slot, const void *qp, const void *kp,
                                   const void *vp, const float *conv_w, const void *z,
                                   const float *A, const float *b, const void *beta_logit,
                                   const void *g, float *S_pool, void *conv_pool,
                                   int32_t write_back, float scale, float l2_eps, float rms_eps,
                                   kda_dtype out_dtype, void *o, void *stream) {
    if (!ok_dtype(out_dtype)) return KDA_ERR_INVALID_ARGUMENT;
    if (batch < 1 || num_heads < 1 || pool_size < 1 || total_tokens < 0)
        return KDA_ERR_INVALID_ARGUMENT;
    if (write_back != 0 && write_back != 1) return KDA_ERR_INVALID_ARGUMENT;
    if (!ok_ptr_elem(cu_tokens, 4) || !ok_ptr_elem(slot, 4) || !ok_ptr(S_pool) ||
        !ok_ptr(conv_pool) || !ok_ptr(conv_w) || !ok_ptr_elem(A, 4) || !ok_opt_ptr(b))
        return KDA_ERR_INVALID_ARGUMENT;
    if (total_tokens > 0 && (!ok_ptr(qp) || !ok_ptr(kp) || !ok_ptr(vp) || !ok_ptr(z) || !ok_ptr(g) ||
                             !ok_ptr_elem(beta_logit, 2) || !ok_ptr(o)))
        return KDA_ERR_INVALID_ARGUMENT;
    const size_t state_bytes = (size_t)pool_size * num_heads * kD * kD * sizeof(float);
    const size_t conv_bytes = (size_t)pool_size * 9 * num_heads * kD * sizeof(__nv_bfloat16);
    const uintptr_t sp = reinterpret_cast<uintptr_t>(S_pool), cp = reinterpret_cast<uintptr_t>(conv_pool);
    if (sp < cp + conv_bytes && cp < sp + state_bytes) return KDA_ERR_INVALID_ARGUMENT;  // pools overlap
    if ((int64_t)batch * num_heads > 0x7fffffffLL || (int64_t)total_tokens * num_heads > 0x7fffffffLL)
        return KDA_ERR_UNSUPPORTED;
    DecodeLayerTokensArgs a;
    a.batch = batch; a.num_heads = num_heads; a.pool_size = pool_size; a.total_tokens = total_tokens;
    a.qp = static_cast<const __nv_bfloat16 *>(qp);
    a.kp = static_cast<const __nv_bfloat16 *>(kp);
    a.vp = static_cast<const __nv_bfloat16 *>(vp);
    a.z = static_cast<const __nv_bfloat16 *>(z);
    a.beta_logit = static_cast<const __nv_bfloat16 *>(beta_logit);
    a.g = static_cast<const __nv_bfloat16 *>(g);
    a.conv_w = conv_w; a.A = A; a.b = b;
    a.cu_tokens = cu_tokens; a.slot = slot;
    a.S_pool = S_pool;
    a.conv_pool = static_cast<__nv_bfloat16 *>(conv_pool);
    a.write_back = write_back;
    a.scale = scale; a.l2_eps = l2_eps; a.rms_eps = rms_eps;
    a.out_dtype = out_dtype; a.o = o;
    a.status = device_status();
    return from_cuda(launch_decode_layer_tokens(a, static_cast<cudaStream_t>(stream)));
}

kda_status kda_check_prefill_inputs(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                                    const float *log_alpha, int32_t head_decay,
                                    const int32_t *cu_seqlens, void *stream) {
    if (num_seqs < 1 || total_tokens < 0 || num_heads < 1) return KDA_ERR_INVALID_ARGUMENT;
    if (head_decay != 0 && head_decay != 1) return KDA_ERR_INVALID_ARGUMENT;
    if (!ok_ptr_elem(cu_seqlens, 4)) return KDA_ERR_INVALID_ARGUMENT;
    if (log_alpha != nullptr && !(head_decay ? ok_ptr_elem(log_alpha, 4) : ok_ptr(log_alpha)))
        return KDA_ERR_INVALID_ARGUMENT;
    CheckArgs a{num_seqs, total_tokens, num_heads, head_decay, log_alpha, cu_seqlens,
                device_status()};
    return from_cuda(launch_check_prefill(a, static_cast<cudaStream_t>(stream)));
}

kda_status kda_get_device_status(void *stream, uint32_t *detail) {
    if (detail) *detail = 0;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KDA_ERR_CUDA;
    DeviceStatus st = device_status();
    if (st.word == nullptr) return KDA_ERR_CUDA;
    uint32_t host[2] = {0, 0};
    if (cudaMemcpy(host, st.word, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (host[0] != 0) {
        const uint32_t zero[2] = {0, 0};
        if (cudaMemcpy(st.word, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return KDA_ERR_CUDA;
    }
    if (detail) *detail = host[1];
    return static_cast<kda_status>(host[0]);
}

}  // extern "C"
