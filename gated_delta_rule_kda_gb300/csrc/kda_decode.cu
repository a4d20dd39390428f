// KDA decode step: one token per (request, head), fp32 state updated in place.
//
// Per unit (request b, head h), with S the 128x128 fp32 state (row j = key
// channel), the recurrence step ("Kimi K3 · KDA layer", KDA equation list) is
//   S' = Diag(alpha) S,  r = S'^T k,  u = beta (v - r),  S <- S' + k u^T,
//   o~ = scale S^T q = scale (S'^T q + (k.q) u)
// The last form needs S only once: both reductions r = S'^T k and p = S'^T q
// come from the same pass over the decayed state, then the rank-1 write is
// applied while the state is still in registers.  The state therefore crosses
// HBM exactly twice (64 KiB read + 64 KiB written), which is the whole cost of
// the step: the kernel is HBM-bound by construction.
//
// Layout: one 256-thread CTA per unit.  Warp w owns rows [16w, 16w+16); lane l
// owns columns [4l, 4l+4), so every row is one coalesced 512-byte warp access
// and each thread keeps 64 state values in registers.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = kD / kWarps;  // 16

__device__ __forceinline__ float4 ld_stream(const float *p) {
    return __ldcs(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ void st_stream(float *p, float4 x) {
    __stcs(reinterpret_cast<float4 *>(p), x);
}

template <typename Tin, typename Tout, bool kHeadDecay>
__global__ void __launch_bounds__(kThreads, 2)
decode_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
              const float *__restrict__ log_alpha, const float *__restrict__ beta,
              float *__restrict__ S, float scale, Tout *__restrict__ o, int prefetch_ahead) {
    __shared__ float s_q[kD], s_k[kD], s_a[kD], s_v[kD], s_u[kD];
    __shared__ float s_red_r[kWarps][kD], s_red_p[kWarps][kD];
    __shared__ float s_kq;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t unit = blockIdx.x;
    float *Su = S + unit * (size_t)(kD * kD);
    // L2 prefetch of the state one resident wave ahead (HBM keeps streaming while resident
    // CTAs compute)
    if (tid == 0 && prefetch_ahead > 0 && unit + prefetch_ahead < gridDim.x)
        prefetch_l2(S + (unit + prefetch_ahead) * (size_t)(kD * kD), kD * kD * sizeof(float));

    // 1. Issue the whole state load first: 16 x 16 B per thread in flight.
    float4 s[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i)
        s[i] = ld_stream(Su + (size_t)(warp * kRowsPerWarp + i) * kD + 4 * lane);

    // 2. The per-token vectors (q, k, v, alpha = exp(log_alpha)).
    if (tid < kD) {
        s_q[tid] = Elem<Tin>::load(q + unit * kD + tid);
        s_k[tid] = Elem<Tin>::load(k + unit * kD + tid);
    } else {
        const int c = tid - kD;
        s_v[c] = Elem<Tin>::load(v + unit * kD + c);
        // kHeadDecay: one decay per (request, head), log_alpha [B][H]
        s_a[c] = expf(kHeadDecay ? log_alpha[unit] : log_alpha[unit * kD + c]);
    }
    __syncthreads();

    // 3. Decay the rows, and reduce r = S'^T k, p = S'^T q over this warp's rows.
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f), p = r;
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const int j = warp * kRowsPerWarp + i;
        const float a = s_a[j], kj = s_k[j], qj = s_q[j];
        s[i].x *= a; s[i].y *= a; s[i].z *= a; s[i].w *= a;
        r.x = fmaf(s[i].x, kj, r.x); r.y = fmaf(s[i].y, kj, r.y);
        r.z = fmaf(s[i].z, kj, r.z); r.w = fmaf(s[i].w, kj, r.w);
        p.x = fmaf(s[i].x, qj, p.x); p.y = fmaf(s[i].y, qj, p.y);
        p.z = fmaf(s[i].z, qj, p.z); p.w = fmaf(s[i].w, qj, p.w);
    }
    *reinterpret_cast<float4 *>(&s_red_r[warp][4 * lane]) = r;
    *reinterpret_cast<float4 *>(&s_red_p[warp][4 * lane]) = p;
    if (warp == 0) {  // k . q
        float kq = 0.f;
#pragma unroll
        for (int m = 0; m < kD / 32; ++m) kq = fmaf(s_k[lane + 32 * m], s_q[lane + 32 * m], kq);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
        if (lane == 0) s_kq = kq;
    }
    __syncthreads();

    // 4. u = beta (v - r) and the readout o = scale (p + (k.q) u), one column per thread.
    if (tid < kD) {
        float rr = 0.f, pp = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            rr += s_red_r[w][tid];
            pp += s_red_p[w][tid];
        }
        const float u = beta[unit] * (s_v[tid] - rr);
        s_u[tid] = u;
        Elem<Tout>::store(o + unit * kD + tid, scale * fmaf(s_kq, u, pp));
    }
    __syncthreads();

    // 5. Rank-1 write S = S' + k u^T and stream the state back.
    const float4 u4 = *reinterpret_cast<const float4 *>(&s_u[4 * lane]);
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const int j = warp * kRowsPerWarp + i;
        const float kj = s_k[j];
        s[i].x = fmaf(kj, u4.x, s[i].x); s[i].y = fmaf(kj, u4.y, s[i].y);
        s[i].z = fmaf(kj, u4.z, s[i].z); s[i].w = fmaf(kj, u4.w, s[i].w);
        st_stream(Su + (size_t)j * kD + 4 * lane, s[i]);
    }
}

template <typename Tin, typename Tout>
cudaError_t launch_typed(const DecodeArgs &a, cudaStream_t stream) {
    const size_t units = (size_t)a.batch * a.num_heads;
    auto kernel = a.head_decay ? decode_kernel<Tin, Tout, true> : decode_kernel<Tin, Tout, false>;
    kernel<<<(unsigned)units, kThreads, 0, stream>>>(
        static_cast<const Tin *>(a.q), static_cast<const Tin *>(a.k),
        static_cast<const Tin *>(a.v), a.log_alpha, a.beta, a.S, a.scale,
        static_cast<Tout *>(a.o), 2 * device_sm_count());
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream) {
    const bool in_bf = a.in_dtype == KDA_BF16, out_bf = a.out_dtype == KDA_BF16;
    if (in_bf && out_bf) return launch_typed<__nv_bfloat16, __nv_bfloat16>(a, stream);
    if (in_bf) return launch_typed<__nv_bfloat16, float>(a, stream);
    if (out_bf) return launch_typed<float, __nv_bfloat16>(a, stream);
    return launch_typed<float, float>(a, stream);
}

}  // namespace kda
