// KDA front end and output gate (elementwise, HBM-bound).
//
// Front end ("Kimi K3 · KDA layer", KDA equation list; "Inside Kimi K3: How
// KDA, AttnRes, and 896 Experts Work", section "Short convolutions give KDA
// local order before recurrence"), per token t, head h, channel i:
//   x^c = SiLU( sum_{j=0..3} w[x][h*128+i][j] * x^p_{t-j} )   (zero before the sequence start)
//   q^, k^ = x^c / sqrt(sum_i x^c^2 + l2_eps)                  (v is not normalised)
//   log_alpha = -5 sigmoid(e^{A_h} (z + b));   beta = sigmoid(beta_logit)
// or, with the unbounded gate of Kimi Linear ("Kimi K3's Architecture: Kimi Delta
// Attention, Attention Residuals, and 896 Experts", section "Channel-wise decay, and the
// floor K3 puts under it"), log_alpha = -e^{A_h} softplus(z + b), in (-inf, 0).
// Output gate (same equation list): o^g = sigmoid(g) * o~ / sqrt(mean(o~^2) + eps).
//
// Both kernels give one warp to one (token, head) row of 128 channels: lane l
// owns channels [4l, 4l+4), so every row access is one coalesced 256-byte
// (bf16) or 512-byte (fp32) transaction and the per-head reductions are warp
// shuffles.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kWarpsPerBlock = kThreads / 32;

__device__ __forceinline__ float sigmoidf_(float x) { return 1.f / (1.f + expf(-x)); }
__device__ __forceinline__ float siluf_(float x) { return x * sigmoidf_(x); }
// softplus(x) = log(1 + e^x); above 20 it equals x to fp32 precision.
__device__ __forceinline__ float softplusf_(float x) { return x > 20.f ? x : log1pf(expf(x)); }
__device__ __forceinline__ float log_decay(float eA, float zb, bool unbounded) {
    return unbounded ? -eA * softplusf_(zb) : -5.f * sigmoidf_(eA * zb);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// Start of the sequence that owns token t (largest n with cu[n] <= t).
__device__ __forceinline__ int seq_start(const int32_t *cu, int num_seqs, int t) {
    int lo = 0, hi = num_seqs;  // invariant: cu[lo] <= t < cu[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu[mid] <= t) lo = mid;
        else hi = mid;
    }
    return cu[lo];
}

template <typename Tout>
__global__ void __launch_bounds__(kThreads)
frontend_kernel(FrontendArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    const int H = a.num_heads;
    if (row >= (int64_t)a.total_tokens * H) return;
    const int t = (int)(row / H), h = (int)(row % H);
    const int start = seq_start(a.cu_seqlens, a.num_seqs, t);
    const int c0 = 4 * lane;
    const __nv_bfloat16 *src[3] = {a.qp, a.kp, a.vp};
    void *dst[3] = {a.q_hat, a.k_hat, a.v_out};

#pragma unroll
    for (int s = 0; s < 3; ++s) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const float *w = a.conv_w + ((size_t)s * H * kD + (size_t)h * kD + c0) * 4;
        float4 wt[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) wt[c] = *reinterpret_cast<const float4 *>(w + 4 * c);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            // taps before the sequence start read as zero (predicated, so all four loads of a
            // stream are in flight at once)
            const float4 x = t - j >= start ? load4(src[s] + ((size_t)(t - j) * H + h) * kD + c0)
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
            const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float wj = j == 0 ? wt[c].x : j == 1 ? wt[c].y : j == 2 ? wt[c].z : wt[c].w;
                acc[c] = fmaf(wj, xs[c], acc[c]);
            }
        }
        float4 y = make_float4(siluf_(acc[0]), siluf_(acc[1]), siluf_(acc[2]), siluf_(acc[3]));
        if (s < 2) {
            const float ss = warp_sum(y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w);
            const float inv = rsqrtf(ss + a.l2_eps);
            y.x *= inv; y.y *= inv; y.z *= inv; y.w *= inv;
        }
        store4(static_cast<Tout *>(dst[s]) + (size_t)row * kD + c0, y);
    }

    const float eA = expf(a.A[h]);
    const float4 z = load4(a.z + (size_t)row * kD + c0);
    float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
    if (a.b != nullptr) b = *reinterpret_cast<const float4 *>(a.b + (size_t)h * kD + c0);
    const bool ub = a.unbounded_decay != 0;
    float4 la;
    la.x = log_decay(eA, z.x + b.x, ub);
    la.y = log_decay(eA, z.y + b.y, ub);
    la.z = log_decay(eA, z.z + b.z, ub);
    la.w = log_decay(eA, z.w + b.w, ub);
    *reinterpret_cast<float4 *>(a.log_alpha + (size_t)row * kD + c0) = la;
    if (lane == 0) a.beta[row] = sigmoidf_(__bfloat162float(a.beta_logit[row]));
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kThreads)
gate_kernel(int64_t rows, const Tin *__restrict__ ot, const __nv_bfloat16 *__restrict__ g,
            float eps, Tout *__restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (row >= rows) return;
    const size_t off = (size_t)row * kD + 4 * lane;
    const float4 x = load4(ot + off);
    const float4 gg = load4(g + off);
    const float ms = warp_sum(x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w) * (1.f / kD);
    const float inv = rsqrtf(ms + eps);
    float4 y;
    y.x = sigmoidf_(gg.x) * x.x * inv;
    y.y = sigmoidf_(gg.y) * x.y * inv;
    y.z = sigmoidf_(gg.z) * x.z * inv;
    y.w = sigmoidf_(gg.w) * x.w * inv;
    store4(out + off, y);
}

}  // namespace

cudaError_t launch_frontend(const FrontendArgs &a, cudaStream_t stream) {
    const int64_t rows = (int64_t)a.total_tokens * a.num_heads;
    if (rows == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((rows + kWarpsPerBlock - 1) / kWarpsPerBlock);
    if (a.out_dtype == KDA_BF16) frontend_kernel<__nv_bfloat16><<<blocks, kThreads, 0, stream>>>(a);
    else frontend_kernel<float><<<blocks, kThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_output_gate(const GateArgs &a, cudaStream_t stream) {
    if (a.num_rows == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((a.num_rows + kWarpsPerBlock - 1) / kWarpsPerBlock);
    const bool in_bf = a.in_dtype == KDA_BF16, out_bf = a.out_dtype == KDA_BF16;
    if (in_bf && out_bf)
        gate_kernel<__nv_bfloat16, __nv_bfloat16><<<blocks, kThreads, 0, stream>>>(
            a.num_rows, static_cast<const __nv_bfloat16 *>(a.o_tilde), a.g, a.eps,
            static_cast<__nv_bfloat16 *>(a.out));
    else if (in_bf)
        gate_kernel<__nv_bfloat16, float><<<blocks, kThreads, 0, stream>>>(
            a.num_rows, static_cast<const __nv_bfloat16 *>(a.o_tilde), a.g, a.eps,
            static_cast<float *>(a.out));
    else if (out_bf)
        gate_kernel<float, __nv_bfloat16><<<blocks, kThreads, 0, stream>>>(
            a.num_rows, static_cast<const float *>(a.o_tilde), a.g, a.eps,
            static_cast<__nv_bfloat16 *>(a.out));
    else
        gate_kernel<float, float><<<blocks, kThreads, 0, stream>>>(
            a.num_rows, static_cast<const float *>(a.o_tilde), a.g, a.eps,
            static_cast<float *>(a.out));
    return cudaGetLastError();
}

}  // namespace kda
