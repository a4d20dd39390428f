// Contents checks of prefill inputs that the argument checks on the host cannot make: the
// sequence offsets and the decay range the chunked kernels rely on.
//
// cu_seqlens must start at 0, never decrease and end at T (packed variable-length
// sequences).  Every log alpha must lie in [-5, 0]: the floor g_min = -5 is what bounds the
// chunk's reciprocal decays ("Kimi K3's Architecture: Kimi Delta Attention, Attention
// Residuals, and 896 Experts", section "Channel-wise decay, and the floor K3 puts under
// it"); NaN fails too.  A failure is recorded in the device status word as
// KDA_ERR_DEVICE_CHECK with detail = (kind << 28) | index: kind 1 = cu_seqlens (index n),
// kind 2 = log alpha (index = token).  One read of log alpha: HBM-bound.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr uint32_t kIndexMask = (1u << 28) - 1;

__device__ __forceinline__ bool decay_ok(float x) { return x >= -5.f && x <= 0.f; }

__global__ void __launch_bounds__(kThreads) check_prefill_kernel(const CheckArgs a) {
    const int tid = threadIdx.x;
    if (blockIdx.x == 0) {
        for (int n = tid; n <= a.num_seqs; n += kThreads) {
            const int c = a.cu_seqlens[n];
            const bool bad = (n == 0 && c != 0) || (n == a.num_seqs && c != a.total_tokens) ||
                             (n > 0 && c < a.cu_seqlens[n - 1]);
            if (bad) record_status(a.status, KDA_ERR_DEVICE_CHECK, (1u << 28) | ((uint32_t)n & kIndexMask));
        }
    }
    if (a.log_alpha == nullptr) return;
    const size_t per_token = (size_t)a.num_heads * (a.head_decay ? 1 : kD);
    const size_t total = (size_t)a.total_tokens * per_token;
    const size_t stride = (size_t)gridDim.x * kThreads;
    if (!a.head_decay) {  // [T][H][128]: four values per load, four loads in flight
        const float4 *p = reinterpret_cast<const float4 *>(a.log_alpha);
        const size_t n4 = total / 4;
        for (size_t i0 = (size_t)blockIdx.x * kThreads + tid; i0 < n4; i0 += 4 * stride) {
            float4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const size_t i = i0 + u * stride;
                x[u] = i < n4 ? __ldcs(p + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const size_t i = i0 + u * stride;
                if (!(decay_ok(x[u].x) && decay_ok(x[u].y) && decay_ok(x[u].z) && decay_ok(x[u].w)))
                    record_status(a.status, KDA_ERR_DEVICE_CHECK,
                                  (2u << 28) | ((uint32_t)(4 * i / per_token) & kIndexMask));
            }
        }
    } else {  // [T][H]
        for (size_t i = (size_t)blockIdx.x * kThreads + tid; i < total; i += stride)
            if (!decay_ok(__ldcs(a.log_alpha + i)))
                record_status(a.status, KDA_ERR_DEVICE_CHECK,
                              (2u << 28) | ((uint32_t)(i / per_token) & kIndexMask));
    }
}

}  // namespace

cudaError_t launch_check_prefill(const CheckArgs &a, cudaStream_t stream) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms = 1;
    check_prefill_kernel<<<4 * sms, kThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
