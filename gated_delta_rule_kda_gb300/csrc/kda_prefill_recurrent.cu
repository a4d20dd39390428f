// KDA prefill, token-by-token form on the fp32 CUDA cores.
//
// This is the full-precision path (fp32 inputs) and the reference-order GPU
// path: it runs the recurrence exactly as defined ("Kimi K3 · KDA layer", KDA
// equation list), one token after another:
//   S <- Diag(alpha_t) S;  r = S^T k_t;  S <- S + beta_t k_t (v_t - r)^T;  o~_t = scale S^T q_t
//
// Parallel decomposition.  Value columns of the state evolve independently
// (column c only needs k, alpha, beta and v[c]), so a (sequence, head) unit is
// split into 2 CTAs of 64 columns.  Inside a CTA, 8 adjacent lanes share a quad
// of columns and each holds 16 of their 128 rows in registers, so every alpha,
// k and q value read from shared memory serves four columns.  The two reductions
// over rows per token are transposed butterflies: at each of three xor steps a
// lane sends half of the partial sums it holds and keeps the other half, so that
// it ends with the full sum of one column (four shuffles for four columns); u is
// gathered back to all eight lanes in three more shuffles.  Each lane keeps its four
// columns in a lane-dependent register order (column quad_col(rq) ^ m in component m),
// which lets every butterfly step run without lane-dependent selects; the order is
// applied when the state is loaded and undone when it is stored.  No state ever leaves
// registers until the sequence ends.
//
// Each token costs one pass over the state: the delta write and readout of
// token t, then the decay and prediction of token t + 1.  Token inputs are
// staged through shared memory 8 tokens at a time in two buffers (the last
// token of a batch reads the next batch's first decay and key); the batch after
// that is fetched into registers while the current one is processed.  Vectors
// indexed by row are stored with 4 floats of padding after every 16 rows so that
// the 8 row groups of a warp read 8 different bank groups.
#include "kda_column_quads.cuh"
#include "kda_common.cuh"
#include "tc_primitives.cuh"

namespace kda {
namespace {

constexpr int kThreads = 128;
constexpr int kCols = 64;        // value columns per CTA
constexpr int kSplit = kD / kCols;
constexpr int kRows = 16;        // rows per thread (and four columns)
constexpr int kTB = 8;           // tokens per staged batch
constexpr int kCtasPerSm = 3;
using quads::kPadRow;
using quads::prow;
using quads::quad_col;
using quads::quad_gather;
using quads::quad_reduce;
using quads::lane_order;

template <typename Tin, typename Tout, bool kCkpt, bool kHeadDecay>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
prefill_recurrent_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                         const Tin *__restrict__ v, const float *__restrict__ log_alpha,
                         const float *__restrict__ beta, const float *__restrict__ S0,
                         const int32_t *__restrict__ cu_seqlens, int H, float scale,
                         Tout *__restrict__ o, float *__restrict__ S_final, const Checkpoints ckpt) {
    // Staged token inputs, double-buffered: the last token of a batch already reads the
    // decay and key of the next batch's first token.
    struct Batch {
        float q[kTB][kPadRow], k[kTB][kPadRow], a[kTB][kPadRow], v[kTB][kCols], b[kTB];
    };
    __shared__ __align__(16) Batch sb[2];
    __shared__ __align__(16) float s_o[kTB][kCols];

    const int tid = threadIdx.x;
    const int cq = tid >> 3, rq = tid & 7;  // column quad (columns 4 cq .. 4 cq + 3), row group
    const int jc = quad_col(rq);            // the column whose reductions this lane finishes
    const int col0 = blockIdx.x * kCols;
    const int h = blockIdx.y, n = blockIdx.z;
    const int t_begin = cu_seqlens[n], t_end = cu_seqlens[n + 1];
    const size_t state_off = ((size_t)n * H + h) * (size_t)(kD * kD);
    // this thread's part of a [128][128] state: rows kRows rq + i, columns col0 + 4 cq ..
    const size_t my_off = (size_t)(kRows * rq) * kD + col0 + 4 * cq;

    float4 s[kRows];
    if (S0 != nullptr) {
#pragma unroll
        for (int i = 0; i < kRows; ++i)
            s[i] = lane_order(*reinterpret_cast<const float4 *>(S0 + state_off + my_off + (size_t)i * kD),
                              jc);
    } else {
#pragma unroll
        for (int i = 0; i < kRows; ++i) s[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // Register prefetch buffers for one batch: 8 tokens x 3 vectors x 32 quads = 768
    // quads -> 6 per thread; v: 8 tokens x 16 quads -> 1 per thread; beta: 8.
    constexpr int kQuadsPerThread = (3 * kTB * (kD / 4)) / kThreads;  // 6
    constexpr int kVQuads = kCols / 4;                                // 16 per token
    static_assert(kTB * kVQuads == kThreads, "one v quad per thread");
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
            const int tok = tid / kVQuads, quad = tid % kVQuads;
            const int t = t0 + tok;
            pre_v = t < t_end ? load4(v + ((size_t)t * H + h) * kD + col0 + 4 * quad)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (tid < kTB) pre_b = (t0 + tid < t_end) ? beta[(size_t)(t0 + tid) * H + h] : 0.f;
    };
    auto stash = [&](Batch &B) {
#pragma unroll
        for (int m = 0; m < kQuadsPerThread; ++m) {
            const int idx = tid + kThreads * m;
            const int arr = idx / (kTB * 32), rem = idx % (kTB * 32);
            const int tok = rem / 32, quad = rem % 32;
            float4 x = pre[m];
            if (arr == 2) x = make_float4(expf(x.x), expf(x.y), expf(x.z), expf(x.w));
            float *dst = arr == 0 ? &B.q[tok][prow(4 * quad)]
                       : arr == 1 ? &B.k[tok][prow(4 * quad)]
                                  : &B.a[tok][prow(4 * quad)];
            *reinterpret_cast<float4 *>(dst) = x;
        }
        *reinterpret_cast<float4 *>(&B.v[tid / kVQuads][4 * (tid % kVQuads)]) = pre_v;
        if (tid < kTB) B.b[tid] = pre_b;
    };

    // Tokens are processed in one pass over the state each: the delta write and readout of
    // token t, then the decay and prediction of token t + 1, so the two reductions of a step
    // run side by side.  Rows past the sequence end are staged as zeros (alpha = 1, k = 0,
    // beta = 0), which leaves the state as it is after the last token.
    float4 kr[kRows / 4];  // this thread's rows of the current token's k
    float4 u = make_float4(0.f, 0.f, 0.f, 0.f);  // the current token's u, all four columns
    // u of column jc from its prediction r (held for column jc) and token (B, tn)
    auto u_of = [&](const Batch &B, int tn, float rj) {
        return quad_gather(B.b[tn] * (B.v[tn][4 * cq + jc] - rj));
    };
    if (t_begin < t_end) {
        fetch(t_begin);
        stash(sb[0]);
        fetch(t_begin + kTB);
        __syncthreads();
        {  // the first token: decay and prediction
            const float *a_row = &sb[0].a[0][prow(kRows * rq)];
            const float *k_row = &sb[0].k[0][prow(kRows * rq)];
            float2 r01 = make_float2(0.f, 0.f), r23 = r01;
#pragma unroll
            for (int i = 0; i < kRows; i += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(a_row + i);
                const float4 k4 = *reinterpret_cast<const float4 *>(k_row + i);
                kr[i / 4] = k4;
                const float av[4] = {a4.x, a4.y, a4.z, a4.w}, kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float4 &x = s[i + e];
                    const float2 a2 = make_float2(av[e], av[e]), k2 = make_float2(kv[e], kv[e]);
                    const float2 x01 = tc::mul2(make_float2(x.x, x.y), a2);
                    const float2 x23 = tc::mul2(make_float2(x.z, x.w), a2);
                    x = make_float4(x01.x, x01.y, x23.x, x23.y);
                    r01 = tc::fma2(x01, k2, r01);
                    r23 = tc::fma2(x23, k2, r23);
                }
            }
            u = u_of(sb[0], 0, quad_reduce(make_float4(r01.x, r01.y, r23.x, r23.y)));
        }
    }
    int cur = 0;
    for (int t0 = t_begin; t0 < t_end; t0 += kTB, cur ^= 1) {
        __syncthreads();  // the other buffer (the previous batch) and s_o are no longer read
        stash(sb[cur ^ 1]);
        __syncthreads();
        fetch(t0 + 2 * kTB);
        const int nb = min(kTB, t_end - t0);
        // Two tokens per loop trip (their buffer choices and offsets become constants): 4.8 %
        // faster on the fp32 prefill.  The snapshot instantiations keep one, which spills less.
        constexpr int kTokUnroll = kCkpt ? 1 : 2;
#pragma unroll kTokUnroll
        for (int tt = 0; tt < nb; ++tt) {
            const Batch &B = sb[cur];
            const Batch &N = tt + 1 < kTB ? sb[cur] : sb[cur ^ 1];  // the next token's batch
            const int tn = tt + 1 < kTB ? tt + 1 : 0;
            const float *q_row = &B.q[tt][prow(kRows * rq)];
            const float *a_row = &N.a[tn][prow(kRows * rq)];
            const float *k_row = &N.k[tn][prow(kRows * rq)];
            float *snap = nullptr;  // snapshot after every `every` tokens of the sequence
            if constexpr (kCkpt) {
                const int done = t0 + tt + 1 - t_begin;
                if (done % ckpt.every == 0) {
                    const int kk = done / ckpt.every - 1;
                    const int base = ckpt.base[n];
                    if (kk < ckpt.base[n + 1] - base)
                        snap = ckpt.states + ((size_t)(base + kk) * H + h) * (size_t)(kD * kD) + my_off;
                }
            }
            float2 p01 = make_float2(0.f, 0.f), p23 = p01, r01 = p01, r23 = p01;
            const float2 u01 = make_float2(u.x, u.y), u23 = make_float2(u.z, u.w);
#pragma unroll
            for (int i = 0; i < kRows; i += 4) {
                const float4 k4 = kr[i / 4];
                const float4 q4 = *reinterpret_cast<const float4 *>(q_row + i);
                const float4 a4 = *reinterpret_cast<const float4 *>(a_row + i);
                const float4 n4 = *reinterpret_cast<const float4 *>(k_row + i);
                kr[i / 4] = n4;
                const float kv[4] = {k4.x, k4.y, k4.z, k4.w}, qv[4] = {q4.x, q4.y, q4.z, q4.w};
                const float av[4] = {a4.x, a4.y, a4.z, a4.w}, nv[4] = {n4.x, n4.y, n4.z, n4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {  // delta write and readout of token t
                    float4 &x = s[i + e];
                    const float2 k2 = make_float2(kv[e], kv[e]), q2 = make_float2(qv[e], qv[e]);
                    const float2 x01 = tc::fma2(k2, u01, make_float2(x.x, x.y));
                    const float2 x23 = tc::fma2(k2, u23, make_float2(x.z, x.w));
                    x = make_float4(x01.x, x01.y, x23.x, x23.y);
                    p01 = tc::fma2(x01, q2, p01);
                    p23 = tc::fma2(x23, q2, p23);
                }
                if (kCkpt && snap != nullptr) {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        *reinterpret_cast<float4 *>(snap + (size_t)(i + e) * kD) = lane_order(s[i + e], jc);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {  // decay and prediction of token t + 1
                    float4 &x = s[i + e];
                    const float2 a2 = make_float2(av[e], av[e]), n2 = make_float2(nv[e], nv[e]);
                    const float2 x01 = tc::mul2(make_float2(x.x, x.y), a2);
                    const float2 x23 = tc::mul2(make_float2(x.z, x.w), a2);
                    x = make_float4(x01.x, x01.y, x23.x, x23.y);
                    r01 = tc::fma2(x01, n2, r01);
                    r23 = tc::fma2(x23, n2, r23);
                }
            }
            const float pj = quad_reduce(make_float4(p01.x, p01.y, p23.x, p23.y));
            const float rj = quad_reduce(make_float4(r01.x, r01.y, r23.x, r23.y));
            if ((rq & 1) == 0) s_o[tt][4 * cq + jc] = scale * pj;
            u = u_of(N, tn, rj);
        }
        __syncthreads();
        // write the batch's outputs: nb tokens x 64 columns
        for (int idx = tid; idx < nb * kCols; idx += kThreads) {
            const int tok = idx / kCols, c = idx % kCols;
            Elem<Tout>::store(o + ((size_t)(t0 + tok) * H + h) * kD + col0 + c, s_o[tok][c]);
        }
    }

    if (S_final != nullptr) {
#pragma unroll
        for (int i = 0; i < kRows; ++i)
            *reinterpret_cast<float4 *>(S_final + state_off + my_off + (size_t)i * kD) = lane_order(s[i], jc);
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
