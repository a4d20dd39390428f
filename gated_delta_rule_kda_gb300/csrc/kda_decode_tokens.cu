// KDA decode of a few tokens per request from a pooled state: speculative verify and replay.
//
// Per unit (request b, head h), with the request's pool row n = slot[b] and its tokens
// t in [cu_tokens[b], cu_tokens[b+1]), the recurrence ("Kimi K3 · KDA layer", KDA
// equation list) is stepped token by token from S = S_pool[n][h]:
//   S' = Diag(alpha_t) S,  r = S'^T k_t,  u = beta_t (v_t - r),  S <- S' + k_t u^T,
//   o~_t = scale S^T q_t = scale (S'^T q_t + (k_t.q_t) u)
// A draft of several tokens is checked against the state without changing it (verify:
// the row is only read), and the accepted tokens are then run again from the same row
// with the result written back (replay), so no state per draft step is ever stored
// ("Inside Kimi K3: How KDA, AttnRes, and 896 Experts Work", section "What could go
// wrong": speculative rejection replays the accepted inputs).  The final state can also
// go to a separate buffer.
//
// Each state is read once and (with write-back) written once; between the two it stays
// in registers for all of the unit's tokens.  Work per unit grows with its tokens while
// its bytes do not, and only two units fit an SM (the state takes 64 registers a thread),
// so the kernel is persistent: each CTA walks a list of units, and while it computes one
// from registers the next unit's state streams into shared memory by one bulk async copy
// (and its first tokens by cp.async), keeping HBM busy through the compute.
//
// Layout: 256 threads per CTA, two CTAs per SM.  Warp w owns state rows [16w, 16w+16);
// lane l owns columns [4l, 4l+4).  Tokens are copied kTB at a time and widened to fp32
// once per batch.  Per token: decay and the two column reductions (packed fp32x2), a
// barrier, then warp w finishes columns [16w, 16w+16) once (lanes 0-15 u = beta (v - r),
// lanes 16-31 o~), a barrier, and every warp reads u for its own columns and applies the
// rank-1 write.
#include "kda_common.cuh"
#include "tc_primitives.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = kD / kWarps;  // 16
constexpr int kTB = 4;                     // tokens staged per batch
constexpr int kCtasPerSm = 2;
constexpr uint32_t kStateBytes = kD * kD * sizeof(float);
constexpr uint64_t kWaitNs = 2000000000ull;  // bound on the wait for a state copy

__device__ __forceinline__ void st_stream(float *p, float4 x) {
    __stcs(reinterpret_cast<float4 *>(p), x);
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
// One quad (four consecutive elements) of a token vector into shared memory, as given.
__device__ __forceinline__ void copy_quad(float *dst, const float *src) {
    cp_async16(smem_u32(dst), src, 16);
}
__device__ __forceinline__ void copy_quad(__nv_bfloat16 *dst, const __nv_bfloat16 *src) {
    cp_async8(smem_u32(dst), src);
}
// Bulk async copy global -> shared, completing `bar`'s transaction count.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ float2 lo2(float4 x) { return make_float2(x.x, x.y); }
__device__ __forceinline__ float2 hi2(float4 x) { return make_float2(x.z, x.w); }
__device__ __forceinline__ float4 cat4(float2 a, float2 b) { return make_float4(a.x, a.y, b.x, b.y); }
__device__ __forceinline__ float2 dup2(float x) { return make_float2(x, x); }

// Shared memory (dynamic): the next unit's state, the batch as fp32 (q, k, v, alpha) and as
// copied (q, k, v in the input type, log alpha), beta, and the per-warp column partials of r
// and p, double-buffered by token parity so that one barrier per token suffices.
template <typename Tin>
struct Smem {
    float state[kD][kD];
    float q[kTB][kD], k[kTB][kD], v[kTB][kD], a[kTB][kD];
    Tin rq[kTB][kD], rk[kTB][kD], rv[kTB][kD];
    float rla[kTB][kD];
    float rb[kTB], b[kTB];
    float red_r[2][kWarps][kD], red_p[2][kWarps][kD];
    float u[2][kD];  // u of every column, double-buffered by token parity
    float kq[2];
    uint64_t bar;
};

// A unit (request, head) and the bounds checks that decide whether it may be touched.
struct Unit {
    int b, h, n, t_begin, t_end;
    bool ok;
};
__device__ __forceinline__ Unit unit_at(const DecodeTokensArgs &a, int u) {
    Unit x;
    x.b = u / a.num_heads;
    x.h = u % a.num_heads;
    x.n = a.slot[x.b];
    x.t_begin = a.cu_tokens[x.b];
    x.t_end = a.cu_tokens[x.b + 1];
    x.ok = x.n >= 0 && x.n < a.pool_size && x.t_begin >= 0 && x.t_end >= x.t_begin &&
           x.t_end <= a.total_tokens;
    return x;
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) decode_tokens_kernel(const DecodeTokensArgs a) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem<Tin> &sm = *reinterpret_cast<Smem<Tin> *>(smem_raw);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.num_heads;
    const int units = a.batch * H;  // the host keeps units + gridDim.x below 2^31
    const Tin *q = static_cast<const Tin *>(a.q), *k = static_cast<const Tin *>(a.k),
              *v = static_cast<const Tin *>(a.v);
    Tout *o = static_cast<Tout *>(a.o);
    const int row0 = warp * kRowsPerWarp;

    // Thread tid copies quad fq of token ft of two vectors of a batch: (q, k) for
    // pair 0, (v, log alpha) for pair 1; later it widens exactly the quads it copied, so
    // the copy buffer needs no barrier of its own.
    const int ft = tid >> 6, pair = (tid >> 5) & 1, fq = tid & 31;
    auto fetch = [&](const Unit &x, int t0) {
        if (t0 + ft < x.t_end) {
            const size_t off = ((size_t)(t0 + ft) * H + x.h) * kD + 4 * fq;
            if (pair == 0) {
                copy_quad(&sm.rq[ft][4 * fq], q + off);
                copy_quad(&sm.rk[ft][4 * fq], k + off);
            } else {
                copy_quad(&sm.rv[ft][4 * fq], v + off);
                copy_quad(&sm.rla[ft][4 * fq], a.log_alpha + off);
            }
        }
        if (tid < kTB && t0 + tid < x.t_end)
            cp_async4(smem_u32(&sm.rb[tid]), a.beta + (size_t)(t0 + tid) * H + x.h, 4);
        cp_async_commit();
    };
    // Request unit x's state into shared memory (one thread).
    auto request_state = [&](const Unit &x) {
        if (tid == 0) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&sm.bar, kStateBytes);
            bulk_load(&sm.state[0][0], a.S_pool + ((size_t)x.n * H + x.h) * (size_t)(kD * kD),
                      kStateBytes, &sm.bar);
        }
    };

    if (tid == 0) {
        mbar_init(&sm.bar, 1);
        fence_mbar_init();
    }
    __syncthreads();

    int u = blockIdx.x;
    Unit cur = u < units ? unit_at(a, u) : Unit{0, 0, 0, 0, 0, false};
    bool copy_pending = u < units && cur.ok;
    if (copy_pending) {
        request_state(cur);
        fetch(cur, cur.t_begin);
    }
    uint32_t ph = 0;
    int par = 0;  // token parity: which partial buffers this token uses
    for (; u < units; u += gridDim.x) {
        const int un = u + gridDim.x;
        const Unit nxt = un < units ? unit_at(a, un) : Unit{0, 0, 0, 0, 0, false};
        const bool nxt_ok = un < units && nxt.ok;
        if (!cur.ok) {  // refused: nothing of this unit is read or written
            if (tid == 0) record_status(a.status, KDA_ERR_DEVICE_CHECK, (uint32_t)cur.b);
            if (nxt_ok) {  // the state buffer is idle: start the next unit's copies
                request_state(nxt);
                fetch(nxt, nxt.t_begin);
                copy_pending = true;
            }
            cur = nxt;
            continue;
        }

        // The state has landed in shared memory: into registers, then free the buffer.  (The
        // CTA gives up as one if any thread's bounded wait ran out.)
        if (!__syncthreads_and(mbar_wait_bounded(&sm.bar, ph, kWaitNs))) {
            if (tid == 0) record_status(a.status, KDA_ERR_DEVICE_TIMEOUT, 1u);
            break;
        }
        ph ^= 1;
        copy_pending = false;
        float4 s[kRowsPerWarp];
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i)
            s[i] = *reinterpret_cast<const float4 *>(&sm.state[row0 + i][4 * lane]);
        __syncthreads();  // every thread has its rows: the buffer may take the next state
        if (nxt_ok) {
            request_state(nxt);
            copy_pending = true;
        }

        for (int t0 = cur.t_begin; t0 < cur.t_end; t0 += kTB) {
            cp_async_wait_all();  // this thread's copies of the batch have landed
            __syncthreads();      // the previous batch's fp32 vectors are no longer read
            if (t0 + ft < cur.t_end) {  // widen the quads this thread copied
                if (pair == 0) {
                    store4(&sm.q[ft][4 * fq], load4(&sm.rq[ft][4 * fq]));
                    store4(&sm.k[ft][4 * fq], load4(&sm.rk[ft][4 * fq]));
                } else {
                    store4(&sm.v[ft][4 * fq], load4(&sm.rv[ft][4 * fq]));
                    const float4 la = load4(&sm.rla[ft][4 * fq]);
                    store4(&sm.a[ft][4 * fq],
                           make_float4(expf(la.x), expf(la.y), expf(la.z), expf(la.w)));
                }
            }
            if (tid < kTB) sm.b[tid] = sm.rb[tid];
            // The copy buffer is free: the next batch, or the next unit's first batch.
            if (t0 + kTB < cur.t_end)
                fetch(cur, t0 + kTB);
            else if (nxt_ok)
                fetch(nxt, nxt.t_begin);
            __syncthreads();  // the batch's fp32 vectors are visible
            const int nb = min(kTB, cur.t_end - t0);
#pragma unroll 1
            for (int tt = 0; tt < nb; ++tt, par ^= 1) {
                // Decay this warp's rows and reduce r = S'^T k, p = S'^T q over them (four
                // rows of alpha, k and q per broadcast load, two columns per instruction).
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
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
                    if (lane == 0) sm.kq[par] = kq;
                }
                __syncthreads();
                // Warp w finishes columns 16 w .. 16 w + 15 once: lanes 0-15 sum r over the
                // warps' partials and form u = beta (v - r), lanes 16-31 sum p and write
                // o~ = scale (p + (k.q) u) with u from their partner lane.  u goes to shared
                // memory, and after a second barrier each lane reads its four columns of it.
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
                        Elem<Tout>::store(o + ((size_t)(t0 + tt) * H + cur.h) * kD + c,
                                          a.scale * fmaf(sm.kq[par], uo, x));
                }
                __syncthreads();
                const float4 u4 = *reinterpret_cast<const float4 *>(&sm.u[par][4 * lane]);
                // Rank-1 write S = S' + k u^T.
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
        }
        if (cur.t_end == cur.t_begin && nxt_ok) fetch(nxt, nxt.t_begin);  // no batch ran

        // The state after the last token: back to the pool row and/or to S_final[b].
        float *Su = a.S_pool + ((size_t)cur.n * H + cur.h) * (size_t)(kD * kD);
        float *Sf = a.S_final != nullptr
                        ? a.S_final + ((size_t)cur.b * H + cur.h) * (size_t)(kD * kD)
                        : nullptr;
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            const size_t off = (size_t)(row0 + i) * kD + 4 * lane;
            if (a.write_back) st_stream(Su + off, s[i]);
            if (Sf != nullptr) st_stream(Sf + off, s[i]);
        }
        cur = nxt;
    }
    // Nothing may still be landing in this CTA's shared memory when it exits.
    cp_async_wait_all();
    if (copy_pending && tid == 0) mbar_wait_bounded(&sm.bar, ph, kWaitNs);
    __syncthreads();
}

// CTAs resident at once on the current device.
int resident_ctas() { return kCtasPerSm * device_sm_count(); }

template <typename Tin, typename Tout>
cudaError_t launch_typed(const DecodeTokensArgs &a, cudaStream_t stream) {
    const int64_t units = (int64_t)a.batch * a.num_heads;
    const int bytes = (int)sizeof(Smem<Tin>);
    cudaError_t e = cudaFuncSetAttribute(decode_tokens_kernel<Tin, Tout>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    const int grid = units < resident_ctas() ? (int)units : resident_ctas();
    decode_tokens_kernel<Tin, Tout><<<grid, kThreads, bytes, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_tokens(const DecodeTokensArgs &a, cudaStream_t stream) {
    const bool in_bf = a.in_dtype == KDA_BF16, out_bf = a.out_dtype == KDA_BF16;
    if (in_bf && out_bf) return launch_typed<__nv_bfloat16, __nv_bfloat16>(a, stream);
    if (in_bf) return launch_typed<__nv_bfloat16, float>(a, stream);
    if (out_bf) return launch_typed<float, __nv_bfloat16>(a, stream);
    return launch_typed<float, float>(a, stream);
}

}  // namespace kda
