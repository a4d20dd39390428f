// KDA decode step of the whole layer core, for requests whose state lives in a pool.
//
// Per unit (request b, head h), with the request's pool row n = slot[b]
// ("Kimi K3 · KDA layer", KDA equation list; the short-convolution state that each
// request carries beside its recurrent state is the pages' own description of a
// decoding request, "Kimi Linear", section on serving state):
//   x^c   = SiLU(w0 x^p_t + w1 x^p_{t-1} + w2 x^p_{t-2} + w3 x^p_{t-3})  for x in q, k, v,
//           the three previous inputs read from the convolution state of row n;
//   q^ = q^c / |q^c|,  k^ = k^c / |k^c|,  v = v^c
//   log alpha = -5 sigmoid(e^A (z + b)),  beta = sigmoid(beta_logit)
//   S' = Diag(alpha) S,  u = beta (v - S'^T k^),  S <- S' + k^ u^T
//   o~ = scale S^T q^ = scale (S'^T q^ + (k^.q^) u)
//   o  = sigmoid(g) o~ / sqrt(mean(o~^2) + eps)
// and the convolution state of row n shifts by one token (x^p_t becomes the newest).
// As in the plain decode step the state is read and written once, in registers, so
// the kernel is HBM-bound; the front end and the gate add ~3 KB to its 128 KB.
//
// Layout: one 256-thread CTA per unit.  Warp w owns state rows [16w, 16w+16); lane l
// owns columns [4l, 4l+4).  Front end: threads 0-127 take channel tid of q and k,
// threads 128-255 channel tid-128 of v and of the decay.  The convolution state of a
// pool row is [3 streams (q, k, v)][3 taps (t-1, t-2, t-3)][H][128] bf16: every
// (stream, tap) of a head is one contiguous 256-byte row.
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
__device__ __forceinline__ float bf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ float sigmoidf_(float x) { return 1.f / (1.f + expf(-x)); }

// Width-4 causal convolution of one channel followed by SiLU; shifts the channel's
// convolution state (taps t-1, t-2, t-3 at hist[0], hist[HD], hist[2 HD]).
__device__ __forceinline__ float conv_silu(const __nv_bfloat16 *xp_t, __nv_bfloat16 *hist,
                                           size_t HD, const float4 w) {
    const __nv_bfloat16 x0 = *xp_t, h1 = hist[0], h2 = hist[HD], h3 = hist[2 * HD];
    float a = w.x * __bfloat162float(x0);
    a = fmaf(w.y, __bfloat162float(h1), a);
    a = fmaf(w.z, __bfloat162float(h2), a);
    a = fmaf(w.w, __bfloat162float(h3), a);
    hist[0] = x0;  // the newest input becomes tap t-1 of the next step
    hist[HD] = h1;
    hist[2 * HD] = h2;
    return a * sigmoidf_(a);
}

// Sum over the 128 threads 0-127 (warps 0-3) of two values; every one of them gets both sums.
__device__ __forceinline__ float2 sum128(float x, float y, float2 (*part)[4]) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        x += __shfl_xor_sync(0xffffffffu, x, off);
        y += __shfl_xor_sync(0xffffffffu, y, off);
    }
    if (lane == 0) (*part)[warp] = make_float2(x, y);
    asm volatile("bar.sync 1, 128;" ::: "memory");  // threads 0-127 only
    const float2 a = (*part)[0], b = (*part)[1], c = (*part)[2], d = (*part)[3];
    return make_float2((a.x + b.x) + (c.x + d.x), (a.y + b.y) + (c.y + d.y));
}

template <typename Tout>
__global__ void __launch_bounds__(kThreads, 2) decode_layer_kernel(const DecodeLayerArgs a) {
    __shared__ float s_q[kD], s_k[kD], s_a[kD], s_v[kD], s_u[kD];
    __shared__ float s_red_r[kWarps][kD], s_red_p[kWarps][kD];
    __shared__ float2 s_part[4], s_part2[4];
    __shared__ float s_kq;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.num_heads;
    const int b = blockIdx.x / H, h = blockIdx.x % H;
    const int n = a.slot[b];
    if (n < 0 || n >= a.pool_size) {  // the whole CTA leaves: nothing is read or written
        if (tid == 0) record_status(a.status, KDA_ERR_DEVICE_CHECK, (uint32_t)b);
        return;
    }
    const size_t unit = (size_t)b * H + h;
    float *Su = a.S_pool + ((size_t)n * H + h) * (size_t)(kD * kD);

    // 1. Issue the whole state load first: 16 x 16 B per thread in flight.
    float4 s[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i)
        s[i] = ld_stream(Su + (size_t)(warp * kRowsPerWarp + i) * kD + 4 * lane);

    // 2. Front end while the state streams in.
    const size_t HD = (size_t)H * kD;
    __nv_bfloat16 *cpool = a.conv_pool + (size_t)n * 9 * HD;  // [stream][tap][H][128]
    if (tid < kD) {
        const int c = tid;
        const size_t ch = (size_t)h * kD + c;
        const float4 wq = *reinterpret_cast<const float4 *>(a.conv_w + (0 * HD + ch) * 4);
        const float4 wk = *reinterpret_cast<const float4 *>(a.conv_w + (1 * HD + ch) * 4);
        const float yq = conv_silu(a.qp + unit * kD + c, cpool + 0 * 3 * HD + ch, HD, wq);
        const float yk = conv_silu(a.kp + unit * kD + c, cpool + 1 * 3 * HD + ch, HD, wk);
        const float2 ss = sum128(yq * yq, yk * yk, &s_part);
        s_q[c] = yq * rsqrtf(ss.x + a.l2_eps);
        s_k[c] = yk * rsqrtf(ss.y + a.l2_eps);
    } else {
        const int c = tid - kD;
        const size_t ch = (size_t)h * kD + c;
        const float4 wv = *reinterpret_cast<const float4 *>(a.conv_w + (2 * HD + ch) * 4);
        s_v[c] = conv_silu(a.vp + unit * kD + c, cpool + 2 * 3 * HD + ch, HD, wv);
        const float bias = a.b != nullptr ? a.b[ch] : 0.f;
        const float la = -5.f * sigmoidf_(expf(a.A[h]) * (bf(a.z + unit * kD + c) + bias));
        s_a[c] = expf(la);
    }
    __syncthreads();

    // 3. Decay the rows, and reduce r = S'^T k, p = S'^T q over this warp's rows.
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f), p = r;
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const int j = warp * kRowsPerWarp + i;
        const float al = s_a[j], kj = s_k[j], qj = s_q[j];
        s[i].x *= al; s[i].y *= al; s[i].z *= al; s[i].w *= al;
        r.x = fmaf(s[i].x, kj, r.x); r.y = fmaf(s[i].y, kj, r.y);
        r.z = fmaf(s[i].z, kj, r.z); r.w = fmaf(s[i].w, kj, r.w);
        p.x = fmaf(s[i].x, qj, p.x); p.y = fmaf(s[i].y, qj, p.y);
        p.z = fmaf(s[i].z, qj, p.z); p.w = fmaf(s[i].w, qj, p.w);
    }
    *reinterpret_cast<float4 *>(&s_red_r[warp][4 * lane]) = r;
    *reinterpret_cast<float4 *>(&s_red_p[warp][4 * lane]) = p;
    if (warp == 0) {  // k^ . q^
        float kq = 0.f;
#pragma unroll
        for (int m = 0; m < kD / 32; ++m) kq = fmaf(s_k[lane + 32 * m], s_q[lane + 32 * m], kq);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
        if (lane == 0) s_kq = kq;
    }
    __syncthreads();

    // 4. u = beta (v - r), o~ = scale (p + (k.q) u), then the gate (one channel per thread).
    if (tid < kD) {
        float rr = 0.f, pp = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            rr += s_red_r[w][tid];
            pp += s_red_p[w][tid];
        }
        const float beta = sigmoidf_(bf(a.beta_logit + unit));
        const float u = beta * (s_v[tid] - rr);
        s_u[tid] = u;
        const float ot = a.scale * fmaf(s_kq, u, pp);
        const float ms = sum128(ot * ot, 0.f, &s_part2).x * (1.f / kD);
        const float og = sigmoidf_(bf(a.g + unit * kD + tid)) * ot * rsqrtf(ms + a.rms_eps);
        Elem<Tout>::store(static_cast<Tout *>(a.o) + unit * kD + tid, og);
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

}  // namespace

cudaError_t launch_decode_layer(const DecodeLayerArgs &a, cudaStream_t stream) {
    const size_t units = (size_t)a.batch * a.num_heads;
    if (a.out_dtype == KDA_BF16)
        decode_layer_kernel<__nv_bfloat16><<<(unsigned)units, kThreads, 0, stream>>>(a);
    else
        decode_layer_kernel<float><<<(unsigned)units, kThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
