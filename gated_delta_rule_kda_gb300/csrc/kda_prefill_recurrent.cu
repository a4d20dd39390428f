// KDA prefill, token-by-token form on the fp32 CUDA cores.
//
// This is the full-precision path (fp32 inputs) and the reference-order GPU
// path: it runs the recurrence exactly as defined ("Kimi K3 · KDA layer", KDA
// equation list), one token after another:
//   S <- Diag(alpha_t) S;  r = S^T k_t;  S <- S + beta_t k_t (v_t - r)^T;  o~_t = scale S^T q_t
//
// Parallel decomposition.  Value columns of the state evolve independently
// (column c only needs k, alpha, beta and v[c]), so a (sequence, head) unit is
// split into 4 CTAs of 32 columns.  Inside a CTA, 8 adjacent lanes share a pair
// of columns and each holds 16 of their 128 rows in registers (so every alpha,
// k and q value read from shared memory serves two columns); the two reductions
// over rows per token are 3-step xor shuffles.  No state ever leaves registers
// until the sequence ends.
//
// Token inputs are staged through shared memory 16 tokens at a time; the next
// batch is fetched into registers while the current one is processed.  Vectors
// indexed by row are stored with 4 floats of padding after every 16 rows so that
// the 8 row groups of a warp read 8 different bank groups.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kThreads = 128;
constexpr int kCols = 32;        // value columns per CTA
constexpr int kSplit = kD / kCols;
constexpr int kRows = 16;        // rows per thread (and two columns)
constexpr int kTB = 16;          // tokens per staged batch
constexpr int kPadRow = kD + 32; // padded vector: 4 floats after every 16 rows

__device__ __forceinline__ int prow(int row) { return row + 4 * (row >> 4); }

template <typename Tin, typename Tout, bool kCkpt, bool kHeadDecay>
__global__ void __launch_bounds__(kThreads)
prefill_recurrent_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                         const Tin *__restrict__ v, const float *__restrict__ log_alpha,
                         const float *__restrict__ beta, const float *__restrict__ S0,
                         const int32_t *__restrict__ cu_seqlens, int H, float scale,
                         Tout *__restrict__ o, float *__restrict__ S_final, const Checkpoints ckpt) {
    __shared__ __align__(16) float s_q[kTB][kPadRow];
    __shared__ __align__(16) float s_k[kTB][kPadRow];
    __shared__ __align__(16) float s_a[kTB][kPadRow];
    __shared__ __align__(16) float s_v[kTB][kCols];
    __shared__ float s_b[kTB];
    __shared__ __align__(16) float s_o[kTB][kCols];

    const int tid = threadIdx.x;
    const int cp = tid >> 3, rq = tid & 7;  // column pair (columns 2 cp, 2 cp + 1), row group
    const int col0 = blockIdx.x * kCols;
    const int h = blockIdx.y, n = blockIdx.z;
    const int t_begin = cu_seqlens[n], t_end = cu_seqlens[n + 1];
    const size_t state_off = ((size_t)n * H + h) * (size_t)(kD * kD);

    float2 s[kRows];  // rows kRows rq + i, columns col0 + 2 cp + {0, 1}
    if (S0 != nullptr) {
#pragma unroll
        for (int i = 0; i < kRows; ++i)
            s[i] = *reinterpret_cast<const float2 *>(S0 + state_off + (size_t)(kRows * rq + i) * kD + col0 + 2 * cp);
    } else {
#pragma unroll
        for (int i = 0; i < kRows; ++i) s[i] = make_float2(0.f, 0.f);
    }

    // Register prefetch buffers for one batch: 16 tokens x 3 vectors x 32 quads
    // = 1536 quads -> 12 per thread; v: 16 x 8 quads -> 1 per thread; beta: 16.
    constexpr int kQuadsPerThread = (3 * kTB * (kD / 4)) / kThreads;  // 12
    float4 pre[kQuadsPerThread];
    float4 pre_v;
    float pre_b = 0.f;

    auto fetch = [&](int t0) {
#pragma unroll
        for (int m = 0; m < kQuadsPerThread; ++m) {
            const int idx = tid + kThreads * m;
            const int arr = idx / (kTB * 32), rem = idx % (kTB * 32);
            const int tok = rem / 32, quad = rem % 32;
            const int t = t0 + tok;
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < t_end) {
                const size_t off = ((size_t)t * H + h) * kD + 4 * quad;
                if (arr == 0) x = load4(q + off);
                else if (arr == 1) x = load4(k + off);
                else if constexpr (kHeadDecay) {  // one decay per (token, head): [T][H]
                    const float y = log_alpha[(size_t)t * H + h];
                    x = make_float4(y, y, y, y);
                } else x = load4(log_alpha + off);
            }
            pre[m] = x;
        }
        {
            const int tok = tid / 8, quad = tid % 8;
            const int t = t0 + tok;
            pre_v = t < t_end ? load4(v + ((size_t)t * H + h) * kD + col0 + 4 * quad)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (tid < kTB) pre_b = (t0 + tid < t_end) ? beta[(size_t)(t0 + tid) * H + h] : 0.f;
    };
    auto stash = [&]() {
#pragma unroll
        for (int m = 0; m < kQuadsPerThread; ++m) {
            const int idx = tid + kThreads * m;
            const int arr = idx / (kTB * 32), rem = idx % (kTB * 32);
            const int tok = rem / 32, quad = rem % 32;
            float4 x = pre[m];
            if (arr == 2) x = make_float4(expf(x.x), expf(x.y), expf(x.z), expf(x.w));
            float *dst = arr == 0 ? &s_q[tok][prow(4 * quad)]
                       : arr == 1 ? &s_k[tok][prow(4 * quad)]
                                  : &s_a[tok][prow(4 * quad)];
            *reinterpret_cast<float4 *>(dst) = x;
        }
        *reinterpret_cast<float4 *>(&s_v[tid / 8][4 * (tid % 8)]) = pre_v;
        if (tid < kTB) s_b[tid] = pre_b;
    };

    if (t_begin < t_end) fetch(t_begin);
    for (int t0 = t_begin; t0 < t_end; t0 += kTB) {
        __syncthreads();  // previous batch fully consumed
        stash();
        __syncthreads();
        if (t0 + kTB < t_end) fetch(t0 + kTB);
        const int nb = min(kTB, t_end - t0);
        for (int tt = 0; tt < nb; ++tt) {
            const float *a_row = &s_a[tt][prow(kRows * rq)];
            const float *k_row = &s_k[tt][prow(kRows * rq)];
            const float *q_row = &s_q[tt][prow(kRows * rq)];
            // decay, then the prediction r = S^T k (this thread's 16 rows, both columns)
            float2 r = make_float2(0.f, 0.f);
            float4 kr[kRows / 4];  // this thread's k rows, used again by the delta write
#pragma unroll
            for (int i = 0; i < kRows; i += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(a_row + i);
                const float4 k4 = *reinterpret_cast<const float4 *>(k_row + i);
                kr[i / 4] = k4;
                const float av[4] = {a4.x, a4.y, a4.z, a4.w}, kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    s[i + e].x *= av[e]; s[i + e].y *= av[e];
                    r.x = fmaf(s[i + e].x, kv[e], r.x); r.y = fmaf(s[i + e].y, kv[e], r.y);
                }
            }
#pragma unroll
            for (int m = 1; m < 8; m <<= 1) {
                r.x += __shfl_xor_sync(0xffffffffu, r.x, m);
                r.y += __shfl_xor_sync(0xffffffffu, r.y, m);
            }
            const float2 v2 = *reinterpret_cast<const float2 *>(&s_v[tt][2 * cp]);
            const float bt = s_b[tt];
            const float u0 = bt * (v2.x - r.x), u1 = bt * (v2.y - r.y);
            // delta write, then the readout of the updated state
            float2 p = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < kRows; i += 4) {
                const float4 k4 = kr[i / 4];
                const float4 q4 = *reinterpret_cast<const float4 *>(q_row + i);
                const float kv[4] = {k4.x, k4.y, k4.z, k4.w}, qv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    s[i + e].x = fmaf(kv[e], u0, s[i + e].x); s[i + e].y = fmaf(kv[e], u1, s[i + e].y);
                    p.x = fmaf(s[i + e].x, qv[e], p.x); p.y = fmaf(s[i + e].y, qv[e], p.y);
                }
            }
#pragma unroll
            for (int m = 1; m < 8; m <<= 1) {
                p.x += __shfl_xor_sync(0xffffffffu, p.x, m);
                p.y += __shfl_xor_sync(0xffffffffu, p.y, m);
            }
            if (rq == 0) *reinterpret_cast<float2 *>(&s_o[tt][2 * cp]) = make_float2(scale * p.x, scale * p.y);
            if (kCkpt) {  // snapshot after every `every` tokens of the sequence
                const int done = t0 + tt + 1 - t_begin;
                if (done % ckpt.every == 0) {
                    const int kk = done / ckpt.every - 1;
                    const int base = ckpt.base[n];
                    if (kk < ckpt.base[n + 1] - base) {
                        float *dst = ckpt.states + ((size_t)(base + kk) * H + h) * (size_t)(kD * kD);
#pragma unroll
                        for (int i = 0; i < kRows; ++i)
                            *reinterpret_cast<float2 *>(dst + (size_t)(kRows * rq + i) * kD + col0 + 2 * cp) = s[i];
                    }
                }
            }
        }
        __syncthreads();
        // write the batch's outputs: nb tokens x 32 columns
        for (int idx = tid; idx < nb * kCols; idx += kThreads) {
            const int tok = idx / kCols, c = idx % kCols;
            Elem<Tout>::store(o + ((size_t)(t0 + tok) * H + h) * kD + col0 + c, s_o[tok][c]);
        }
    }

    if (S_final != nullptr) {
#pragma unroll
        for (int i = 0; i < kRows; ++i)
            *reinterpret_cast<float2 *>(S_final + state_off + (size_t)(kRows * rq + i) * kD + col0 + 2 * cp) = s[i];
    }
}

template <typename Tin, typename Tout>
cudaError_t launch_typed(const PrefillArgs &a, cudaStream_t stream) {
    dim3 grid(kSplit, a.num_heads, a.num_seqs);
    // snapshots and the per-head decay are separate instantiations, so the loop without
    // them is untouched
    auto kernel = a.head_decay
                      ? (a.ckpt.every > 0 ? prefill_recurrent_kernel<Tin, Tout, true, true>
                                          : prefill_recurrent_kernel<Tin, Tout, false, true>)
                      : (a.ckpt.every > 0 ? prefill_recurrent_kernel<Tin, Tout, true, false>
                                          : prefill_recurrent_kernel<Tin, Tout, false, false>);
    kernel<<<grid, kThreads, 0, stream>>>(
        static_cast<const Tin *>(a.q), static_cast<const Tin *>(a.k),
        static_cast<const Tin *>(a.v), a.log_alpha, a.beta, a.S0, a.cu_seqlens, a.num_heads,
        a.scale, static_cast<Tout *>(a.o), a.S_final, a.ckpt);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_recurrent(const PrefillArgs &a, cudaStream_t stream) {
    const bool in_bf = a.in_dtype == KDA_BF16, out_bf = a.out_dtype == KDA_BF16;
    if (in_bf && out_bf) return launch_typed<__nv_bfloat16, __nv_bfloat16>(a, stream);
    if (in_bf) return launch_typed<__nv_bfloat16, float>(a, stream);
    if (out_bf) return launch_typed<float, __nv_bfloat16>(a, stream);
    return launch_typed<float, float>(a, stream);
}

}  // namespace kda
