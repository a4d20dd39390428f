// KDA decode step of the whole layer core, for requests whose state lives in a pool.
//
// Per unit (request b, head h), with the request's pool row n = slot[b]
// ("Kimi K3 · KDA layer", KDA equation list; each decoding request carries a
// short-convolution state beside its recurrent state: "Inside Kimi K3: How KDA,
// AttnRes, and 896 Experts Work", section "KDA writes corrections into a recurrent
// matrix"):
//   x^c   = SiLU(w0 x^p_t + w1 x^p_{t-1} + w2 x^p_{t-2} + w3 x^p_{t-3})  for x in q, k, v,
//           the three previous inputs read from the convolution state of row n;
//   q^ = q^c / |q^c|,  k^ = k^c / |k^c|,  v = v^c   (|x| = sqrt(sum x^2 + l2_eps))
//   log alpha = -5 sigmoid(e^A (z + b)),  beta = sigmoid(beta_logit)
//   S' = Diag(alpha) S,  u = beta (v - S'^T k^),  S <- S' + k^ u^T
//   o~ = scale S^T q^ = scale (S'^T q^ + (k^.q^) u)
//   o  = sigmoid(g) o~ / sqrt(mean(o~^2) + eps)
// and the convolution state of row n shifts by one token (x^p_t becomes the newest).
// As in the plain decode step the state is read and written once, in registers, so
// the kernel is HBM-bound; the front end and the gate add ~6 KB to its 128 KB.  The
// front end's inputs are fetched before the state stream, and the state goes back
// before the gate's reduction, so that neither lengthens a CTA's life.
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

// One channel of one stream: the current input, its three previous inputs (taps t-1, t-2,
// t-3 at hist[0], hist[HD], hist[2 HD] of the convolution state) and the four weights.
struct ConvIn {
    __nv_bfloat16 x0, h1, h2, h3;
    float4 w;
};
__device__ __forceinline__ ConvIn conv_load(const __nv_bfloat16 *xp_t, const __nv_bfloat16 *hist,
                                            size_t HD, const float *w) {
    ConvIn c;
    c.x0 = *xp_t;
    c.h1 = hist[0];
    c.h2 = hist[HD];
    c.h3 = hist[2 * HD];
    c.w = *reinterpret_cast<const float4 *>(w);
    return c;
}
// Width-4 causal convolution followed by SiLU; shifts the convolution state by one token.
__device__ __forceinline__ float conv_silu(const ConvIn &c, __nv_bfloat16 *hist, size_t HD) {
    float a = c.w.x * __bfloat162float(c.x0);
    a = fmaf(c.w.y, __bfloat162float(c.h1), a);
    a = fmaf(c.w.z, __bfloat162float(c.h2), a);
    a = fmaf(c.w.w, __bfloat162float(c.h3), a);
    hist[0] = c.x0;  // the newest input becomes tap t-1 of the next step
    hist[HD] = c.h1;
    hist[2 * HD] = c.h2;
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
    if (tid == 0 && a.prefetch_ahead > 0) {  // L2 prefetch: the state one resident wave ahead
        const size_t u2 = blockIdx.x + (size_t)a.prefetch_ahead;
        if (u2 < gridDim.x) {
            const int n2 = a.slot[u2 / H];
            if (n2 >= 0 && n2 < a.pool_size)
                prefetch_l2(a.S_pool + ((size_t)n2 * H + u2 % H) * (size_t)(kD * kD), kD * kD * sizeof(float));
        }
    }

    // 1. The front end's few inputs first (they decide when the state work can start),
    //    then the whole state load: 16 x 16 B per thread in flight.
    const size_t HD = (size_t)H * kD;
    __nv_bfloat16 *cpool = a.conv_pool + (size_t)n * 9 * HD;  // [stream][tap][H][128]
    const int c = tid & (kD - 1);
    const size_t ch = (size_t)h * kD + c;
    ConvIn in0, in1;  // q, k (threads 0-127) or v (threads 128-255, in0 only)
    float zb = 0.f, gl = 0.f, bl = 0.f;
    if (tid < kD) {
        in0 = conv_load(a.qp + unit * kD + c, cpool + 0 * 3 * HD + ch, HD, a.conv_w + (0 * HD + ch) * 4);
        in1 = conv_load(a.kp + unit * kD + c, cpool + 1 * 3 * HD + ch, HD, a.conv_w + (1 * HD + ch) * 4);
        gl = bf(a.g + unit * kD + c);
        bl = bf(a.beta_logit + unit);
    } else {
        in0 = conv_load(a.vp + unit * kD + c, cpool + 2 * 3 * HD + ch, HD, a.conv_w + (2 * HD + ch) * 4);
        zb = bf(a.z + unit * kD + c) + (a.b != nullptr ? a.b[ch] : 0.f);
    }
    float4 s[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i)
        s[i] = ld_stream(Su + (size_t)(warp * kRowsPerWarp + i) * kD + 4 * lane);

    // 2. Front end while the state streams in.
    if (tid < kD) {
        const float yq = conv_silu(in0, cpool + 0 * 3 * HD + ch, HD);
        const float yk = conv_silu(in1, cpool + 1 * 3 * HD + ch, HD);
        const float2 ss = sum128(yq * yq, yk * yk, &s_part);
        s_q[c] = yq * rsqrtf(ss.x + a.l2_eps);
        s_k[c] = yk * rsqrtf(ss.y + a.l2_eps);
    } else {
        s_v[c] = conv_silu(in0, cpool + 2 * 3 * HD + ch, HD);
        const float la = -5.f * sigmoidf_(expf(a.A[h]) * zb);
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

    // 4. u = beta (v - r) and o~ = scale (p + (k.q) u), one channel per thread.
    float ot = 0.f;
    if (tid < kD) {
        float rr = 0.f, pp = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            rr += s_red_r[w][tid];
            pp += s_red_p[w][tid];
        }
        const float u = sigmoidf_(bl) * (s_v[tid] - rr);
        s_u[tid] = u;
        ot = a.scale * fmaf(s_kq, u, pp);
    }
    __syncthreads();

    // 5. Rank-1 write S = S' + k u^T and stream the state back (before the gate's reduction).
    const float4 u4 = *reinterpret_cast<const float4 *>(&s_u[4 * lane]);
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const int j = warp * kRowsPerWarp + i;
        const float kj = s_k[j];
        s[i].x = fmaf(kj, u4.x, s[i].x); s[i].y = fmaf(kj, u4.y, s[i].y);
        s[i].z = fmaf(kj, u4.z, s[i].z); s[i].w = fmaf(kj, u4.w, s[i].w);
        st_stream(Su + (size_t)j * kD + 4 * lane, s[i]);
    }

    // 6. Output gate: sigmoid(g) o~ / sqrt(mean(o~^2) + eps) over the head's 128 channels.
    if (tid < kD) {
        const float ms = sum128(ot * ot, 0.f, &s_part2).x * (1.f / kD);
        const float og = sigmoidf_(gl) * ot * rsqrtf(ms + a.rms_eps);
        Elem<Tout>::store(static_cast<Tout *>(a.o) + unit * kD + tid, og);
    }
}

}  // namespace

cudaError_t launch_decode_layer(const DecodeLayerArgs &args, cudaStream_t stream) {
    DecodeLayerArgs a = args;
    a.prefetch_ahead = 2 * device_sm_count();  // two CTAs per SM: one resident wave
    const size_t units = (size_t)a.batch * a.num_heads;
    if (a.out_dtype == KDA_BF16)
        decode_layer_kernel<__nv_bfloat16><<<(unsigned)units, kThreads, 0, stream>>>(a);
    else
        decode_layer_kernel<float><<<(unsigned)units, kThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
