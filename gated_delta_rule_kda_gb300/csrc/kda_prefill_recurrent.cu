// KDA prefill, token-by-token form on the fp32 CUDA cores.
//
// This is the full-precision path (fp32 inputs) and the reference-order GPU
// path: it runs the recurrence exactly as defined ("Kimi K3 · KDA layer", KDA
// equation list), one token after another:
//   S <- Diag(alpha_t) S;  r = S^T k_t;  S <- S + beta_t k_t (v_t - r)^T;  o~_t = scale S^T q_t
//
// Parallel decomposition.  Value columns of the state evolve independently
// (column c only needs k, alpha, beta and v[c]), so a (sequence, head) unit is
// split into 4 CTAs of 32 columns.  Inside a CTA, 4 adjacent lanes share one
// column and each holds 32 of its 128 rows in registers; the two reductions
// over rows per token are 2-step xor shuffles.  No state ever leaves registers
// until the sequence ends.
//
// Token inputs are staged through shared memory 16 tokens at a time; the next
// batch is fetched into registers while the current one is processed.  Vectors
// indexed by row are stored with 4 floats of padding after every 32 rows so that
// the 4 row-quarters of a warp read 4 different bank groups.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kThreads = 128;
constexpr int kCols = 32;        // value columns per CTA
constexpr int kSplit = kD / kCols;
constexpr int kRows = 32;        // rows per thread
constexpr int kTB = 16;          // tokens per staged batch
constexpr int kPadRow = kD + 16; // padded vector: 4 floats after every 32 rows

__device__ __forceinline__ int prow(int row) { return row + 4 * (row >> 5); }

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
    const int cl = tid >> 2, rq = tid & 3;
    const int col0 = blockIdx.x * kCols;
    const int h = blockIdx.y, n = blockIdx.z;
    const int t_begin = cu_seqlens[n], t_end = cu_seqlens[n + 1];
    const size_t state_off = ((size_t)n * H + h) * (size_t)(kD * kD);

    float s[kRows];
    if (S0 != nullptr) {
#pragma unroll
        for (int i = 0; i < kRows; ++i)
            s[i] = S0[state_off + (size_t)(kRows * rq + i) * kD + col0 + cl];
    } else {
#pragma unroll
        for (int i = 0; i < kRows; ++i) s[i] = 0.f;
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
            // decay, then the prediction r = S^T k (this thread's 32 rows)
            float r0 = 0.f, r1 = 0.f;
#pragma unroll
            for (int i = 0; i < kRows; i += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(a_row + i);
                const float4 k4 = *reinterpret_cast<const float4 *>(k_row + i);
                s[i] *= a4.x; s[i + 1] *= a4.y; s[i + 2] *= a4.z; s[i + 3] *= a4.w;
                r0 = fmaf(s[i], k4.x, r0); r1 = fmaf(s[i + 1], k4.y, r1);
                r0 = fmaf(s[i + 2], k4.z, r0); r1 = fmaf(s[i + 3], k4.w, r1);
            }
            float r = r0 + r1;
            r += __shfl_xor_sync(0xffffffffu, r, 1);
            r += __shfl_xor_sync(0xffffffffu, r, 2);
            const float u = s_b[tt] * (s_v[tt][cl] - r);
            // delta write, then the readout of the updated state
            float p0 = 0.f, p1 = 0.f;
#pragma unroll
            for (int i = 0; i < kRows; i += 4) {
                const float4 k4 = *reinterpret_cast<const float4 *>(k_row + i);
                const float4 q4 = *reinterpret_cast<const float4 *>(q_row + i);
                s[i] = fmaf(k4.x, u, s[i]); s[i + 1] = fmaf(k4.y, u, s[i + 1]);
                s[i + 2] = fmaf(k4.z, u, s[i + 2]); s[i + 3] = fmaf(k4.w, u, s[i + 3]);
                p0 = fmaf(s[i], q4.x, p0); p1 = fmaf(s[i + 1], q4.y, p1);
                p0 = fmaf(s[i + 2], q4.z, p0); p1 = fmaf(s[i + 3], q4.w, p1);
            }
            float p = p0 + p1;
            p += __shfl_xor_sync(0xffffffffu, p, 1);
            p += __shfl_xor_sync(0xffffffffu, p, 2);
            if (rq == 0) s_o[tt][cl] = scale * p;
            if (kCkpt) {  // snapshot after every `every` tokens of the sequence
                const int done = t0 + tt + 1 - t_begin;
                if (done % ckpt.every == 0) {
                    const int kk = done / ckpt.every - 1;
                    const int base = ckpt.base[n];
                    if (kk < ckpt.base[n + 1] - base) {
                        float *dst = ckpt.states + ((size_t)(base + kk) * H + h) * (size_t)(kD * kD);
#pragma unroll
                        for (int i = 0; i < kRows; ++i) dst[(size_t)(kRows * rq + i) * kD + col0 + cl] = s[i];
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
            S_final[state_off + (size_t)(kRows * rq + i) * kD + col0 + cl] = s[i];
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
