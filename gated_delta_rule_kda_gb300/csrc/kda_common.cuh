// Shared device helpers and launcher declarations of libkda (sm_103a).
#pragma once

#include <atomic>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

constexpr int kD = KDA_HEAD_DIM;  // d_k = d_v = 128

// Device status word: [0] = kda_status code, [1] = kernel-specific detail.
// The first writer wins (atomicCAS on [0]).
struct DeviceStatus {
    uint32_t *word;
};

__device__ __forceinline__ void record_status(DeviceStatus st, uint32_t code, uint32_t detail) {
    if (st.word == nullptr) return;
    if (atomicCAS(st.word, 0u, code) == 0u) atomicExch(st.word + 1, detail);
}

// Ask L2 to fetch [p, p + bytes) ahead of its use (bytes a multiple of 16; p must lie in an
// allocation the caller owns).  The one-CTA-per-unit decode kernels use it for the state of
// the unit one resident wave ahead, so that HBM keeps streaming while resident CTAs compute.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Streaming multiprocessors of the current device (cached per device; a racing first call
// stores the same value).
inline int device_sm_count() {
    constexpr int kMaxDevices = 64;
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    const int slot = dev >= 0 && dev < kMaxDevices ? dev : 0;
    int sms = cache[slot].load(std::memory_order_relaxed);
    if (sms == 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
            sms = 1;
        cache[slot].store(sms, std::memory_order_relaxed);
    }
    return sms;
}

template <typename T>
struct Elem;
template <>
struct Elem<float> {
    static __device__ __forceinline__ float load(const float *p) { return *p; }
    static __device__ __forceinline__ void store(float *p, float x) { *p = x; }
};
template <>
struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16 *p) {
        return __bfloat162float(*p);
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, float x) {
        *p = __float2bfloat16_rn(x);
    }
};

// Load 4 consecutive elements (16-byte aligned for fp32, 8-byte for bf16).
__device__ __forceinline__ float4 load4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
    uint2 raw = *reinterpret_cast<const uint2 *>(p);
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162 *>(&raw.x);
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162 *>(&raw.y);
    float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
    return make_float4(fa.x, fa.y, fb.x, fb.y);
}
__device__ __forceinline__ void store4(float *p, float4 x) {
    *reinterpret_cast<float4 *>(p) = x;
}
__device__ __forceinline__ void store4(__nv_bfloat16 *p, float4 x) {
    __nv_bfloat162 a = __floats2bfloat162_rn(x.x, x.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(x.z, x.w);
    uint2 raw;
    raw.x = *reinterpret_cast<uint32_t *>(&a);
    raw.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = raw;
}

// ---------------------------------------------------------------------------
// Launcher argument blocks (host side).  Pointers are device pointers that the
// ABI layer has already validated.
// ---------------------------------------------------------------------------
struct DecodeArgs {
    kda_dtype in_dtype, out_dtype;
    int32_t batch, num_heads;
    const void *q, *k, *v;
    const float *log_alpha, *beta;
    int32_t head_decay;  // 1: log_alpha is [B][H], one decay per (request, head)
    int32_t prefetch_ahead;  // units between a CTA and the one whose state it prefetches (0: none)
    float *S;
    float scale;
    void *o;
    DeviceStatus status;
};

// The whole layer core for a few tokens per request from pooled recurrent and
// short-convolution states (speculative verify / replay at the layer level).
constexpr int kDecodeLayerMaxTokens = KDA_DECODE_LAYER_MAX_TOKENS;
struct DecodeLayerTokensArgs {
    int32_t batch, num_heads, pool_size, total_tokens;
    const __nv_bfloat16 *qp, *kp, *vp, *z, *beta_logit, *g;  // [T][H][128] ([T][H] for beta_logit)
    const float *conv_w, *A, *b;                            // [3][H*128][4], [H], [H][128] or null
    const int32_t *cu_tokens, *slot;                        // [B+1], [B]
    float *S_pool;                                          // [P][H][128][128]
    __nv_bfloat16 *conv_pool;                               // [P][3][3][H][128]
    int32_t write_back;
    float scale, l2_eps, rms_eps;
    kda_dtype out_dtype;
    void *o;                                                // [T][H][128]
    int32_t prefetch_ahead;  // units between a CTA and the one whose state it prefetches (0: none)
    DeviceStatus status;
};

// Several tokens per request from a pooled state: request b's tokens are rows
// [cu_tokens[b], cu_tokens[b+1]) of q, k, v, log_alpha, beta; its state is S_pool[slot[b]].
struct DecodeTokensArgs {
    kda_dtype in_dtype, out_dtype;
    int32_t batch, num_heads, pool_size, total_tokens;
    const void *q, *k, *v;                 // [T][H][128]
    const float *log_alpha, *beta;         // [T][H][128], [T][H]
    const int32_t *cu_tokens, *slot;       // [B+1], [B]
    float *S_pool;                         // [P][H][128][128]
    int32_t write_back;                    // 1: the final state goes back to the pool row
    float *S_final;                        // [B][H][128][128] or null
    float scale;
    void *o;                               // [T][H][128]
    int32_t prefetch_ahead;  // units between a CTA and the one whose state it prefetches (0: none)
    DeviceStatus status;
};

// State snapshots during a prefill: for sequence n, snapshot k (k = 0, 1, ...) is the state
// after its first (k + 1) * every tokens, written to states[(base[n] + k)][h][j][c] while
// k < base[n + 1] - base[n].  every == 0: none.
struct Checkpoints {
    int32_t every;
    const int32_t *base;
    float *states;
};

// One decode step of the whole layer core for a batch of requests whose recurrent state
// and short-convolution state live in pools indexed by slot.
struct DecodeLayerArgs {
    int32_t batch, num_heads, pool_size;
    const __nv_bfloat16 *qp, *kp, *vp, *z, *beta_logit, *g;  // [B][H][128] ([B][H] for beta_logit)
    const float *conv_w, *A, *b;                            // [3][H*128][4], [H], [H][128] or null
    const int32_t *slot;                                    // [B]
    float *S_pool;                                          // [P][H][128][128]
    __nv_bfloat16 *conv_pool;                               // [P][3][3][H][128]
    float scale, l2_eps, rms_eps;
    kda_dtype out_dtype;
    void *o;                                                // [B][H][128]
    int32_t prefetch_ahead;  // units between a CTA and the one whose state it prefetches (0: none)
    DeviceStatus status;
};

struct PrefillArgs {
    kda_dtype in_dtype, out_dtype;
    int32_t num_seqs, total_tokens, num_heads;
    const void *q, *k, *v;
    const float *log_alpha, *beta, *S0;
    const int32_t *cu_seqlens;
    float scale;
    void *o;
    float *S_final;
    void *workspace;
    size_t workspace_bytes;
    Checkpoints ckpt;
    int32_t head_decay;  // 1: log_alpha is [T][H], one decay per (token, head)
    int32_t unbounded;   // 1: any decay <= 0 (no -5 floor): chunks out of the tensor-core range
                         //    run token by token; fp32 inputs run the token-by-token kernel
    DeviceStatus status;
};

struct FrontendArgs {
    int32_t num_seqs, total_tokens, num_heads;
    const __nv_bfloat16 *qp, *kp, *vp, *z, *beta_logit;
    const float *conv_w, *A, *b;
    const int32_t *cu_seqlens;
    float l2_eps;
    kda_dtype out_dtype;
    void *q_hat, *k_hat, *v_out;
    float *log_alpha, *beta;
    int32_t unbounded_decay;  // 1: log_alpha = -e^A softplus(z + b) instead of -5 sigmoid(e^A (z + b))
};

struct GateArgs {
    int64_t num_rows;
    kda_dtype in_dtype, out_dtype;
    const void *o_tilde;
    const __nv_bfloat16 *g;
    float eps;
    void *out;
};

// One KDA layer core in a single tensor-core kernel (front end and gate fused).
struct LayerArgs {
    int32_t num_seqs, total_tokens, num_heads;
    const __nv_bfloat16 *qp, *kp, *vp, *z, *beta_logit, *g;
    const float *conv_w, *A, *b, *S0;
    const int32_t *cu_seqlens;
    float scale, l2_eps, rms_eps;
    kda_dtype out_dtype;
    void *o;
    float *S_final;
    Checkpoints ckpt;
    int32_t unbounded_decay;  // 1: log_alpha = -e^A softplus(z + b) (no floor), chunk fallback
    DeviceStatus status;
};

// Contents checks of prefill inputs (offsets monotonic, log alpha in [-5, 0]).
struct CheckArgs {
    int32_t num_seqs, total_tokens, num_heads, head_decay;
    const float *log_alpha;  // [T][H][128] ([T][H] with head_decay) or null
    const int32_t *cu_seqlens;
    DeviceStatus status;
};

cudaError_t launch_check_prefill(const CheckArgs &a, cudaStream_t stream);
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream);
cudaError_t launch_decode_layer(const DecodeLayerArgs &a, cudaStream_t stream);
cudaError_t launch_decode_tokens(const DecodeTokensArgs &a, cudaStream_t stream);
cudaError_t launch_decode_layer_tokens(const DecodeLayerTokensArgs &a, cudaStream_t stream);
cudaError_t launch_prefill_recurrent(const PrefillArgs &a, cudaStream_t stream);
cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t stream);
cudaError_t launch_layer_tc(const LayerArgs &a, cudaStream_t stream);
cudaError_t launch_frontend(const FrontendArgs &a, cudaStream_t stream);
cudaError_t launch_output_gate(const GateArgs &a, cudaStream_t stream);

}  // namespace kda
