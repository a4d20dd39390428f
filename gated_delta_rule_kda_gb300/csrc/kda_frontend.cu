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
// Lane l owns channels [4l, 4l+4) of a (token, head) row, so every row access is one
// coalesced 256-byte (bf16) or 512-byte (fp32) transaction and the per-head reductions are
// warp shuffles.  The gate gives one warp one row; the front end gives one warp two
// consecutive tokens of one head.
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

// One warp takes tokens t0 = 2 tp and t0 + 1 of head h: the head's taps are loaded once for
// both, and the five input rows t0 - 3 .. t0 + 1 once per stream (the two tokens' windows
// overlap in three of them).  The rows are requested before the search for the sequence start,
// so the two overlap; rows before a token's sequence start are zeroed afterwards (token t0 + 1
// may open the next sequence).
// Five blocks per SM (48 registers a thread, a few spilled): 4.9 % faster than four
// (64 registers, none spilled); more warps in flight matter more here than the spills.
template <typename Tout>
__global__ void __launch_bounds__(kThreads, 5)
frontend_kernel(FrontendArgs a) {
    const int lane = threadIdx.x & 31;
    const int H = a.num_heads, T = a.total_tokens;
    const int64_t wi = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (wi >= (int64_t)((T + 1) / 2) * H) return;
    const int tp = (int)(wi / H), h = (int)(wi - (int64_t)tp * H);
    const int t0 = 2 * tp;
    const bool two = t0 + 1 < T;
    const int c0 = 4 * lane;
    const __nv_bfloat16 *src[3] = {a.qp, a.kp, a.vp};
    void *dst[3] = {a.q_hat, a.k_hat, a.v_out};
    auto row_ptr = [&](const __nv_bfloat16 *base, int t) {
        return base + ((size_t)t * H + h) * kD + c0;
    };
    // stream 0's rows first: in flight while the sequence start is looked up
    float4 xr[5];  // rows t0 - 3 .. t0 + 1
#pragma unroll
    for (int k = 0; k < 5; ++k) {
        const int t = t0 - 3 + k;
        xr[k] = t >= 0 && t < T ? load4(row_ptr(src[0], t)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // starts of t0's sequence and of t0 + 1's (t0 + 1 opens the next one when it is a cu entry)
    int lo = 0, hi = a.num_seqs;  // invariant: cu[lo] <= t0 < cu[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (a.cu_seqlens[mid] <= t0) lo = mid;
        else hi = mid;
    }
    const int start0 = a.cu_seqlens[lo];
    const int start1 = a.cu_seqlens[lo + 1] == t0 + 1 ? t0 + 1 : start0;

#pragma unroll
    for (int s = 0; s < 3; ++s) {
        if (s > 0) {
#pragma unroll
            for (int k = 0; k < 5; ++k) {
                const int t = t0 - 3 + k;
                xr[k] = t >= 0 && t < T ? load4(row_ptr(src[s], t)) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        const float *w = a.conv_w + ((size_t)s * H * kD + (size_t)h * kD + c0) * 4;
        float4 wt[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) wt[c] = *reinterpret_cast<const float4 *>(w + 4 * c);
#pragma unroll
        for (int u = 0; u < 2; ++u) {  // token t0 + u: taps j = 0..3 read row t0 + u - j
            if (u == 1 && !two) break;
            const int st = u == 0 ? start0 : start1;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int k = 3 + u - j;  // index of row t0 + u - j in xr
                const bool in = t0 + u - j >= st;
                const float xs[4] = {xr[k].x, xr[k].y, xr[k].z, xr[k].w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float wj = j == 0 ? wt[c].x : j == 1 ? wt[c].y : j == 2 ? wt[c].z : wt[c].w;
                    acc[c] = fmaf(wj, in ? xs[c] : 0.f, acc[c]);
                }
            }
            float4 y = make_float4(siluf_(acc[0]), siluf_(acc[1]), siluf_(acc[2]), siluf_(acc[3]));
            if (s < 2) {
                const float ss = warp_sum(y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w);
                const float inv = rsqrtf(ss + a.l2_eps);
                y.x *= inv; y.y *= inv; y.z *= inv; y.w *= inv;
            }
            store4(static_cast<Tout *>(dst[s]) + ((size_t)(t0 + u) * H + h) * kD + c0, y);
        }
    }

    const float eA = expf(a.A[h]);
    float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
    if (a.b != nullptr) b = *reinterpret_cast<const float4 *>(a.b + (size_t)h * kD + c0);
    const bool ub = a.unbounded_decay != 0;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        if (u == 1 && !two) break;
        const size_t row = (size_t)(t0 + u) * H + h;
        const float4 z = load4(a.z + row * kD + c0);
        float4 la;
        la.x = log_decay(eA, z.x + b.x, ub);
        la.y = log_decay(eA, z.y + b.y, ub);
        la.z = log_decay(eA, z.z + b.z, ub);
        la.w = log_decay(eA, z.w + b.w, ub);
        *reinterpret_cast<float4 *>(a.log_alpha + row * kD + c0) = la;
        if (lane == 0) a.beta[row] = sigmoidf_(__bfloat162float(a.beta_logit[row]));
    }
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
    const int64_t warps = (int64_t)((a.total_tokens + 1) / 2) * a.num_heads;  // token pairs x heads
    if (warps == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((warps + kWarpsPerBlock - 1) / kWarpsPerBlock);
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
