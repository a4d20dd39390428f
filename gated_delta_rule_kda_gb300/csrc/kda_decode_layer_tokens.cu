// KDA layer core for a few tokens per request from pooled states: the layer-level verify
// and replay steps of speculative decoding.
//
// Per unit (request b, head h), with the request's pool row n = slot[b] and its tokens
// t in [cu_tokens[b], cu_tokens[b+1]) (at most kMaxTok), following the KDA equation list
// ("Kimi K3 · KDA layer"):
//   window     the three inputs before the first token (the row's short-convolution
//              state, taps t-1, t-2, t-3), then the tokens' own q^p, k^p, v^p
//   front end  x^c = SiLU(w0 x^p_t + w1 x^p_{t-1} + w2 x^p_{t-2} + w3 x^p_{t-3}) over the
//              window; q^, k^ L2-normalised per head; log alpha = -5 sigmoid(e^A (z + b));
//              beta = sigmoid(beta_logit)
//   recurrence from S = S_pool[n][h], token by token (as the decode step)
//   gate       o = sigmoid(g) o~ / sqrt(mean(o~^2) + eps)
// Verify (write_back = 0) changes neither pool; replay (write_back = 1) stores the state
// after the last token and the last three inputs as the row's new convolution state
// ("Inside Kimi K3: How KDA, AttnRes, and 896 Experts Work", sections "KDA writes
// corrections into a recurrent matrix" and "What could go wrong").
//
// Layout: one 256-thread CTA per unit, two per SM.  All of the unit's inputs are copied
// (with the head's convolution taps) into shared memory by cp.async at once while the
// state streams into registers (warp w owns rows [16w, 16w+16), lane l columns
// [4l, 4l+4)).  Front end: two tasks per token, (q, k) and (v, decay), over the warps,
// lane l channels [4l, 4l+4), so each token's L2 sums are warp reductions.
// Recurrence: per token the decay and both column reductions (packed fp32x2), a CTA
// barrier, warp w finishing columns [16w, 16w+16) once (u and o~), a barrier, the rank-1
// write with each lane's four columns of u.  Gate:
// warp w again takes tokens w and w + 8.
#include "kda_common.cuh"
#include "tc_primitives.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = kD / kWarps;  // 16
constexpr int kMaxTok = kDecodeLayerMaxTokens;
constexpr int kHist = 3;                   // taps before the first token

__device__ __forceinline__ float4 ld_stream(const float *p) {
    return __ldcs(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ void st_stream(float *p, float4 x) {
    __stcs(reinterpret_cast<float4 *>(p), x);
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ float sigmoidf_(float x) { return 1.f / (1.f + expf(-x)); }
__device__ __forceinline__ float2 lo2(float4 x) { return make_float2(x.x, x.y); }
__device__ __forceinline__ float2 hi2(float4 x) { return make_float2(x.z, x.w); }
__device__ __forceinline__ float4 cat4(float2 a, float2 b) { return make_float4(a.x, a.y, b.x, b.y); }
__device__ __forceinline__ float2 dup2(float x) { return make_float2(x, x); }
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// Width-4 causal convolution + SiLU of channels 4 l .. 4 l + 3 at window row r (x points at
// row r, channel 4 l; rows r-1 .. r-3 lie kD elements apart before it).
__device__ __forceinline__ float4 conv_silu4(const float4 (&cw)[4][32], const __nv_bfloat16 *x,
                                             int lane) {
    const float4 w0 = cw[0][lane], w1 = cw[1][lane], w2 = cw[2][lane], w3 = cw[3][lane];
    const float4 x0 = load4(x), x1 = load4(x - kD), x2 = load4(x - 2 * kD), x3 = load4(x - 3 * kD);
    float c[4];
    c[0] = fmaf(w0.w, x3.x, fmaf(w0.z, x2.x, fmaf(w0.y, x1.x, w0.x * x0.x)));
    c[1] = fmaf(w1.w, x3.y, fmaf(w1.z, x2.y, fmaf(w1.y, x1.y, w1.x * x0.y)));
    c[2] = fmaf(w2.w, x3.z, fmaf(w2.z, x2.z, fmaf(w2.y, x1.z, w2.x * x0.z)));
    c[3] = fmaf(w3.w, x3.w, fmaf(w3.z, x2.w, fmaf(w3.y, x1.w, w3.x * x0.w)));
    return make_float4(c[0] * sigmoidf_(c[0]), c[1] * sigmoidf_(c[1]), c[2] * sigmoidf_(c[2]),
                       c[3] * sigmoidf_(c[3]));
}

struct Smem {
    float q[kMaxTok][kD], k[kMaxTok][kD], v[kMaxTok][kD], a[kMaxTok][kD];  // front-end outputs
    float ot[kMaxTok][kD];                                                   // o~ before the gate
    __nv_bfloat16 x[3][kHist + kMaxTok][kD];  // q^p, k^p, v^p windows (rows 0-2: t-3, t-2, t-1)
    __nv_bfloat16 z[kMaxTok][kD], g[kMaxTok][kD];
    float4 cw[3][4][32];  // this head's taps (w0 .. w3) of channel 4 l + e at [stream][e][l]
    float b[kMaxTok];
    float red_r[2][kWarps][kD], red_p[2][kWarps][kD];
    float u[2][kD];  // u of every column, double-buffered by token parity
    float kq[2];
};

template <typename Tout>
__global__ void __launch_bounds__(kThreads, 2) decode_layer_tokens_kernel(const DecodeLayerTokensArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.num_heads;
    const int b = blockIdx.x / H, h = blockIdx.x % H;
    const int n = a.slot[b];
    const int t_begin = a.cu_tokens[b], t_end = a.cu_tokens[b + 1];
    const int ntok = t_end - t_begin;
    // Refused units read and write nothing (the whole CTA leaves before any access).
    if (n < 0 || n >= a.pool_size || t_begin < 0 || t_end < t_begin || t_end > a.total_tokens ||
        ntok > kMaxTok) {
        if (tid == 0) record_status(a.status, KDA_ERR_DEVICE_CHECK, (uint32_t)b);
        return;
    }
    const size_t HD = (size_t)H * kD;
    float *Su = a.S_pool + ((size_t)n * H + h) * (size_t)(kD * kD);
    if (tid == 0 && a.prefetch_ahead > 0) {  // L2 prefetch: the state one resident wave ahead
        const size_t u2 = blockIdx.x + (size_t)a.prefetch_ahead;
        if (u2 < gridDim.x) {
            const int n2 = a.slot[u2 / H];
            if (n2 >= 0 && n2 < a.pool_size)
                prefetch_l2(a.S_pool + ((size_t)n2 * H + u2 % H) * (size_t)(kD * kD), kD * kD * sizeof(float));
        }
    }
    __nv_bfloat16 *cpool = a.conv_pool + (size_t)n * 9 * HD;  // [stream][tap][H][128]
    const int row0 = warp * kRowsPerWarp;

    // 1. All of the unit's inputs into shared memory (8-byte quads), then the state into
    //    registers: the copies and the state stream are in flight together.
    {
        const int rows_x = kHist + ntok, tasks = (3 * rows_x + 2 * ntok) * 32;
        for (int task = tid; task < tasks; task += kThreads) {
            const int row = task >> 5, qd = task & 31;
            const void *src;
            __nv_bfloat16 *dst;
            if (row < 3 * rows_x) {
                // stream s and window row r of `row` (compares: no division by a runtime value)
                int s = 0, r = row;
                if (r >= rows_x) {
                    r -= rows_x;
                    s = 1;
                    if (r >= rows_x) {
                        r -= rows_x;
                        s = 2;
                    }
                }
                dst = &sm.x[s][r][4 * qd];
                src = r < kHist ? cpool + ((size_t)(3 * s + (kHist - 1 - r)) * HD + (size_t)h * kD + 4 * qd)
                                : (s == 0 ? a.qp : s == 1 ? a.kp : a.vp) +
                                      (((size_t)(t_begin + r - kHist) * H + h) * kD + 4 * qd);
            } else {
                const int rr = row - 3 * rows_x, which = rr >= ntok ? 1 : 0, r = rr - which * ntok;
                dst = which == 0 ? &sm.z[r][4 * qd] : &sm.g[r][4 * qd];
                src = (which == 0 ? a.z : a.g) + (((size_t)(t_begin + r) * H + h) * kD + 4 * qd);
            }
            cp_async8(smem_u32(dst), src);
        }
        for (int task = tid; task < 3 * kD; task += kThreads) {  // the head's convolution taps
            const int st = task / kD, c = task % kD;
            cp_async16(smem_u32(&sm.cw[st][c & 3][c >> 2]),
                       a.conv_w + ((size_t)st * HD + (size_t)h * kD + c) * 4, 16);
        }
        cp_async_commit();
    }
    float4 s[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i)
        s[i] = ld_stream(Su + (size_t)(row0 + i) * kD + 4 * lane);
    float bl = 0.f;
    if (tid < ntok) bl = __bfloat162float(a.beta_logit[(size_t)(t_begin + tid) * H + h]);
    cp_async_wait_all();
    __syncthreads();

    // 2. Front end: two tasks per token, (q, k) and (v, decay), spread over the warps;
    //    lane l takes channels 4l .. 4l + 3, so each token's L2 sums are warp reductions.
    if (tid < ntok) sm.b[tid] = sigmoidf_(bl);
    const size_t ch = (size_t)h * kD + 4 * lane;
    const float ea = expf(a.A[h]);
#pragma unroll 1
    for (int task = warp; task < 2 * ntok; task += kWarps) {
        const int tk = task >> 1, r = kHist + tk;  // the token and its row of the windows
        if ((task & 1) == 0) {
            // q and k: convolution + SiLU, then the L2 norms over the token's 128 channels
            float4 y[2];
            float ss[2];
#pragma unroll
            for (int st = 0; st < 2; ++st) {
                const float4 y4 = conv_silu4(sm.cw[st], &sm.x[st][r][4 * lane], lane);
                y[st] = y4;
                ss[st] = y4.x * y4.x + y4.y * y4.y + y4.z * y4.z + y4.w * y4.w;
            }
            const float nq = rsqrtf(warp_sum(ss[0]) + a.l2_eps), nk = rsqrtf(warp_sum(ss[1]) + a.l2_eps);
            *reinterpret_cast<float4 *>(&sm.q[tk][4 * lane]) =
                make_float4(y[0].x * nq, y[0].y * nq, y[0].z * nq, y[0].w * nq);
            *reinterpret_cast<float4 *>(&sm.k[tk][4 * lane]) =
                make_float4(y[1].x * nk, y[1].y * nk, y[1].z * nk, y[1].w * nk);
        } else {
            // v: convolution + SiLU; the decay alpha = exp(-5 sigmoid(e^A (z + b)))
            *reinterpret_cast<float4 *>(&sm.v[tk][4 * lane]) = conv_silu4(sm.cw[2], &sm.x[2][r][4 * lane], lane);
            const float4 z4 = load4(&sm.z[tk][4 * lane]);
            const float4 b4 = a.b != nullptr ? *reinterpret_cast<const float4 *>(a.b + ch)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4 *>(&sm.a[tk][4 * lane]) =
                make_float4(expf(-5.f * sigmoidf_(ea * (z4.x + b4.x))), expf(-5.f * sigmoidf_(ea * (z4.y + b4.y))),
                            expf(-5.f * sigmoidf_(ea * (z4.z + b4.z))), expf(-5.f * sigmoidf_(ea * (z4.w + b4.w))));
        }
    }
    // Replay: the row's new convolution state is the last three inputs of the window.
    if (a.write_back && ntok > 0 && warp < kHist) {
        const int tap = warp, r = kHist + ntok - 1 - tap;
#pragma unroll
        for (int st = 0; st < 3; ++st)
            *reinterpret_cast<uint2 *>(cpool + (size_t)(3 * st + tap) * HD + ch) =
                *reinterpret_cast<const uint2 *>(&sm.x[st][r][4 * lane]);
    }
    __syncthreads();

    // 3. Recurrence, token by token; o~ to shared memory for the gate.
    int par = 0;
#pragma unroll 1
    for (int tt = 0; tt < ntok; ++tt, par ^= 1) {
        float2 r01 = make_float2(0.f, 0.f), r23 = r01, p01 = r01, p23 = r01;
#pragma unroll
        for (int i4 = 0; i4 < kRowsPerWarp; i4 += 4) {
            const float4 al4 = *reinterpret_cast<const float4 *>(&sm.a[tt][row0 + i4]);
            const float4 k4 = *reinterpret_cast<const float4 *>(&sm.k[tt][row0 + i4]);
            const float4 q4 = *reinterpret_cast<const float4 *>(&sm.q[tt][row0 + i4]);
            const float alv[4] = {al4.x, al4.y, al4.z, al4.w};
            const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
            const float qv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float4 &x = s[i4 + e];
                const float2 x01 = mul2(lo2(x), dup2(alv[e]));
                const float2 x23 = mul2(hi2(x), dup2(alv[e]));
                x = cat4(x01, x23);
                r01 = fma2(x01, dup2(kv[e]), r01); r23 = fma2(x23, dup2(kv[e]), r23);
                p01 = fma2(x01, dup2(qv[e]), p01); p23 = fma2(x23, dup2(qv[e]), p23);
            }
        }
        *reinterpret_cast<float4 *>(&sm.red_r[par][warp][4 * lane]) = cat4(r01, r23);
        *reinterpret_cast<float4 *>(&sm.red_p[par][warp][4 * lane]) = cat4(p01, p23);
        if (warp == 0) {  // k . q
            float kq = 0.f;
#pragma unroll
            for (int m = 0; m < kD / 32; ++m)
                kq = fmaf(sm.k[tt][lane + 32 * m], sm.q[tt][lane + 32 * m], kq);
            kq = warp_sum(kq);
            if (lane == 0) sm.kq[par] = kq;
        }
        __syncthreads();
        // Warp w finishes columns 16 w .. 16 w + 15 once: lanes 0-15 sum r over the warps'
        // partials and form u = beta (v - r), lanes 16-31 sum p and form o~ with u from their
        // partner lane; after a second barrier each lane reads its four columns of u.
        {
            const int c = 16 * warp + (lane & 15);
            const float(*part)[kD] = lane < 16 ? sm.red_r[par] : sm.red_p[par];
            float x = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) x += part[w][c];
            const float uc = sm.b[tt] * (sm.v[tt][c] - x);  // lanes 0-15
            const float uo = __shfl_sync(0xffffffffu, uc, lane & 15);
            if (lane < 16)
                sm.u[par][c] = uc;
            else
                sm.ot[tt][c] = a.scale * fmaf(sm.kq[par], uo, x);
        }
        __syncthreads();
        const float4 u4 = *reinterpret_cast<const float4 *>(&sm.u[par][4 * lane]);
        const float2 u01 = lo2(u4), u23 = hi2(u4);
#pragma unroll
        for (int i4 = 0; i4 < kRowsPerWarp; i4 += 4) {
            const float4 k4 = *reinterpret_cast<const float4 *>(&sm.k[tt][row0 + i4]);
            const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float4 &x = s[i4 + e];
                x = cat4(fma2(dup2(kv[e]), u01, lo2(x)), fma2(dup2(kv[e]), u23, hi2(x)));
            }
        }
    }
    if (a.write_back && ntok > 0) {  // the state goes back before the gate
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i)
            st_stream(Su + (size_t)(row0 + i) * kD + 4 * lane, s[i]);
    }
    __syncthreads();

    // 4. Output gate per token: warp w, tokens w and w + 8.
    Tout *o = static_cast<Tout *>(a.o);
#pragma unroll 1
    for (int tk = warp; tk < ntok; tk += kWarps) {
        const float4 x = *reinterpret_cast<const float4 *>(&sm.ot[tk][4 * lane]);
        const float ms = warp_sum(x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w) * (1.f / kD);
        const float rs = rsqrtf(ms + a.rms_eps);
        const float4 gg = load4(&sm.g[tk][4 * lane]);
        store4(o + ((size_t)(t_begin + tk) * H + h) * kD + 4 * lane,
               make_float4(sigmoidf_(gg.x) * x.x * rs, sigmoidf_(gg.y) * x.y * rs,
                           sigmoidf_(gg.z) * x.z * rs, sigmoidf_(gg.w) * x.w * rs));
    }
}

}  // namespace

cudaError_t launch_decode_layer_tokens(const DecodeLayerTokensArgs &args, cudaStream_t stream) {
    DecodeLayerTokensArgs a = args;
    a.prefetch_ahead = 2 * device_sm_count();  // two CTAs per SM: one resident wave
    const size_t units = (size_t)a.batch * a.num_heads;
    const int bytes = (int)sizeof(Smem);
    if (a.out_dtype == KDA_BF16) {
        cudaError_t e = cudaFuncSetAttribute(decode_layer_tokens_kernel<__nv_bfloat16>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        decode_layer_tokens_kernel<__nv_bfloat16><<<(unsigned)units, kThreads, bytes, stream>>>(a);
    } else {
        cudaError_t e = cudaFuncSetAttribute(decode_layer_tokens_kernel<float>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        decode_layer_tokens_kernel<float><<<(unsigned)units, kThreads, bytes, stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace kda
