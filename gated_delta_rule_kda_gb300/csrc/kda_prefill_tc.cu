// KDA prefill on the 5th-generation tensor cores (tcgen05 + TMEM), bf16 inputs.
//
// One CTA owns one (sequence, head) unit and walks its chunks of C = 32 tokens
// in order, keeping the 128x128 fp32 state in TMEM for the whole sequence.
// Chunk-wise form ("Kimi K3's Architecture: Kimi Delta Attention, Attention
// Residuals, and 896 Experts", section "Channel-wise decay, and the floor K3
// puts under it": parallel inside a chunk, recurrent across chunks, keys
// rescaled by reciprocal cumulative decay).  Per chunk, with S0 the entering
// state, gamma the in-chunk inclusive cumulative log-decay per channel and
// Gamma = e^gamma:
//
//   A[r,i] = beta_r sum_c k_r[c] k_i[c] e^{gamma_r[c]-gamma_i[c]}   (i < r)
//   P[r,i] =        sum_c q_r[c] k_i[c] e^{gamma_r[c]-gamma_i[c]}   (i <= r)
//   T      = (I + A)^-1,  Tb = T diag(beta)
//   W      = Tb (k (.) Gamma),   U~ = Tb V
//   U      = U~ - W S0
//   O      = scale ((q (.) Gamma) S0 + P U)
//   S_C    = Diag(Gamma_C) S0 + (k (.) e^{gamma_C - gamma})^T U
//
// Decay factors.  Each pair (r, i) inside the chunk is written with one
// reference per channel, m = gamma_15 (the middle of the chunk):
// e^{gamma_r - gamma_i} = e^{D_r} e^{-D_i} with D = gamma - m.  With the decay
// floor log alpha >= -5 (the pages' g_min), |D| <= 5 * 16 = 80 for every row,
// so both factors stay inside the bf16/fp32 range (e^80 < 3.4e38) and the whole
// causal 32 x 32 Gram block is ONE dense tensor-core product; the pairs i > r
// that the range does not cover are masked out afterwards.
//
// The state is held TRANSPOSED (TMEM lane = value channel c, column = key
// channel j), so every product is an M = 128 tcgen05.mma:
//   M1  G = [k E ; q E] . (k E^-1)^T                  (lanes 0-31 -> A, 32-63 -> P)
//   M2  U~^T = V^T . Tb^T                            (V read MN-major from its staged tile)
//   M2b W = Tb . (k Gamma)       (rows r in lanes 0-31; B read MN-major)
//   M3  [ (W S0)^T | (Q~ S0)^T ] = S0^T . [W ; Q~]^T   (A = S0^T from TMEM)
//   M4  (Q~ S0 + P U)^T += U^T . P^T
//   M5  S^T += U^T . K^        (S^T scaled by Gamma_C along j first; B read MN-major)
//
// Precision: an fp32 quantity x enters an MMA as x = hi + lo (two bf16,
// round-to-nearest), and a product X.Y is formed as hi.hi + hi.lo + lo.hi
// (fp32 accumulation); V is exact in bf16 and enters once.
//
// Inputs of chunk c+1 are staged with cp.async while chunk c is processed.
#include "kda_common.cuh"
#include "tc_primitives.cuh"

namespace kda {
namespace {
using namespace tc;

constexpr int kC = 32;
constexpr int kThreads = 256;
constexpr uint64_t kWaitNs = 2000000000ull;  // bound on every wait for the tensor core

// ---- shared memory map (bytes from a 1024-aligned base) --------------------
// Two input buffers, each: q, k, v tiles (bf16 [32][128] in the swizzled tile
// layout below), log_alpha (fp32 [32][128] natural), beta [32].
constexpr uint32_t IB_Q = 0, IB_K = 8192, IB_V = 16384, IB_LA = 24576, IB_BETA = 40960;
constexpr uint32_t IB_SIZE = 43008;
constexpr uint32_t W_E = 2 * IB_SIZE;     // fp32 [32][128]  e^{D}
constexpr uint32_t W_EI = W_E + 16384;    // fp32 [32][128]  e^{-D}
constexpr uint32_t W_R = W_EI + 16384;    // R hi|lo (M1 B); then Tb hi|lo, P hi|lo (4 KB each)
constexpr uint32_t W_KT = W_R + 16384;    // (k Gamma) hi|lo, MN-major A of M2
constexpr uint32_t W_KH = W_KT + 16384;   // K^ hi|lo, MN-major B of M5
constexpr uint32_t W_WQ = W_KH + 16384;   // [W ; Q~] hi (16 KB) | lo (16 KB), B of M3
constexpr uint32_t W_A = W_WQ + 32768;    // fp32 [32][33]
constexpr uint32_t W_T = W_A + 4224;      // fp32 [32][33]
constexpr uint32_t W_VEC = W_T + 4224;    // per-channel vectors (below)
constexpr uint32_t W_BAR = W_VEC + 5 * 512;
constexpr uint32_t W_TSLOT = W_BAR + 8;
constexpr uint32_t SM_DYN = W_TSLOT + 8 + 1024;  // + alignment slack
constexpr int V_M = 0, V_EM = 128, V_D31 = 256, V_E31 = 384, V_GC = 512;  // float offsets
constexpr int kLd = 33;  // padded row stride of A and T

// ---- TMEM column map (512 columns) -----------------------------------------
constexpr uint32_t TM_ST = 0;    // S^T fp32 [c][j]
constexpr uint32_t TM_D1 = 128;  // [(W S0)^T | (Q~ S0 + P U)^T] (32 + 32); Gram result during M1
constexpr uint32_t TM_DW = 192;  // [unused | U~^T] (32 + 32)
constexpr uint32_t TM_OPG = 256; // M1's A operand: hi (64) | lo (64); then W (lanes 0-31, 128 cols)
constexpr uint32_t TM_OPS = 384; // M3's A operand S^T hi (64) | lo (64); then U^T hi (16) | lo (16)

// Swizzled [32 rows][128 bf16] tile: two 64-column blocks of 32 x 128 bytes,
// 16-byte chunk j of row i at chunk position j ^ (i % 8).  Read as a K-major
// operand it has 32 rows and K = 128; read MN-major it has K = 32 rows and
// MN = 128 (64-element blocks 4096 bytes apart).
__device__ __forceinline__ uint32_t tile_chunk(int i, int cc) {
    return (uint32_t)((cc >> 3) * 4096 + i * 128 + (((cc & 7) ^ (i & 7)) << 4));
}
// fp32 [32][128] with 16-byte chunks swizzled by row.
__device__ __forceinline__ uint32_t e_chunk(int r, int q) {  // q = 4-float chunk 0..31
    return (uint32_t)(r * 512 + (((q ^ r) & 31) << 4));
}

struct Params {
    const __nv_bfloat16 *q, *k, *v;
    const float *log_alpha, *beta, *S0;
    const int32_t *cu_seqlens;
    int H;
    float scale;
    void *o;
    float *S_final;
    DeviceStatus status;
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &u, float (&x)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// Store 8 fp32 values as a hi 16-byte chunk and a lo 16-byte chunk.
__device__ __forceinline__ void store_split_chunk(unsigned char *hi, unsigned char *lo,
                                                  const float (&x)[8]) {
    uint4 h, l;
    split2(x[0], x[1], h.x, l.x);
    split2(x[2], x[3], h.y, l.y);
    split2(x[4], x[5], h.z, l.z);
    split2(x[6], x[7], h.w, l.w);
    *reinterpret_cast<uint4 *>(hi) = h;
    *reinterpret_cast<uint4 *>(lo) = l;
}

// One thread waits for the tensor core (bounded); the CTA barrier then orders
// every other thread after the completed MMAs.
__device__ __forceinline__ bool wait_mma(uint64_t *bar, uint32_t &phase, DeviceStatus st,
                                         uint32_t where) {
    bool ok = true;
    if (threadIdx.x == 0) {
        ok = mbar_wait_bounded(bar, phase & 1u, kWaitNs);
        if (!ok) record_status(st, KDA_ERR_DEVICE_TIMEOUT, where);
    }
    ++phase;
    ok = __syncthreads_and(ok) != 0;
    fence_after_sync();
    return ok;
}

// Operand writes (generic-proxy smem stores and tcgen05.st) -> visible to the MMA.
__device__ __forceinline__ void publish_operands() {
    tmem_wait_st();
    fence_proxy_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
}

// Stage chunk [t0, t0 + nrow) of this head into input buffer `buf` (zero rows past nrow).
__device__ __forceinline__ void issue_loads(const Params &p, unsigned char *buf, int t0, int nrow,
                                            int h, int tid) {
    const int H = p.H;
    const __nv_bfloat16 *src[3] = {p.q, p.k, p.v};
    const uint32_t dst[3] = {IB_Q, IB_K, IB_V};
#pragma unroll
    for (int m = 0; m < 6; ++m) {
        const int e = tid + kThreads * m;  // 1536 chunks of 16 bytes
        const int a = e >> 9, rem = e & 511;
        const int i = rem >> 4, cc = rem & 15;
        const bool ok = i < nrow;
        const __nv_bfloat16 *s = ok ? src[a] + ((size_t)(t0 + i) * H + h) * kD + 8 * cc : src[a];
        cp_async16(smem_u32(buf + dst[a] + tile_chunk(i, cc)), s, ok ? 16u : 0u);
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const int e = tid + kThreads * m;  // 1024 chunks of 4 floats
        const int i = e >> 5, qq = e & 31;
        const bool ok = i < nrow;
        const float *s = ok ? p.log_alpha + ((size_t)(t0 + i) * H + h) * kD + 4 * qq : p.log_alpha;
        cp_async16(smem_u32(buf + IB_LA + i * 512 + qq * 16), s, ok ? 16u : 0u);
    }
    if (tid < kC) {
        const bool ok = tid < nrow;
        const float *s = ok ? p.beta + (size_t)(t0 + tid) * H + h : p.beta;
        cp_async4(smem_u32(buf + IB_BETA + 4 * tid), s, ok ? 4u : 0u);
    }
    cp_async_commit();
}

template <typename Tout>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(Params p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float *vec = reinterpret_cast<float *>(sm + W_VEC);
    float *sA = reinterpret_cast<float *>(sm + W_A);
    float *sT = reinterpret_cast<float *>(sm + W_T);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + W_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + W_TSLOT);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int trow = 32 * quarter + lane;  // this thread's TMEM lane
    const int H = p.H;
    const int h = blockIdx.x % H, n = blockIdx.x / H;
    const int t_begin = p.cu_seqlens[n], t_end = p.cu_seqlens[n + 1];
    const size_t state_off = ((size_t)n * H + h) * (size_t)(kD * kD);

    if (warp == 0) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    if (t_begin < t_end) issue_loads(p, sm, t_begin, min(kC, t_end - t_begin), h, tid);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tb = *tslot;
    const uint32_t tl = tb + ((uint32_t)(32 * quarter) << 16);  // this warp's lane quarter
    uint32_t phase = 0;

    // ---- entering state -> TMEM, transposed (lane c, column j) ----
    {
        const int c = trow;
        uint32_t w[32];
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            const int j0 = 64 * half + 32 * part;
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
                w[jj] = p.S0 ? __float_as_uint(p.S0[state_off + (size_t)(j0 + jj) * kD + c]) : 0u;
            tmem_st32(tl + TM_ST + j0, w);
        }
        tmem_wait_st();
    }

    bool alive = true;
    int chunk = 0;
    for (int t0 = t_begin; t0 < t_end && alive; t0 += kC, ++chunk) {
        const int nrow = min(kC, t_end - t0);
        unsigned char *buf = sm + (chunk & 1) * IB_SIZE;
        const float *beta_s = reinterpret_cast<const float *>(buf + IB_BETA);

        // ---- F1: this chunk's inputs have landed; stage the next chunk ----
        cp_async_wait_all();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        if (t0 + kC < t_end)
            issue_loads(p, sm + ((chunk + 1) & 1) * IB_SIZE, t0 + kC, min(kC, t_end - t0 - kC), h,
                        tid);

        // ---- F2: decay factors in log2 units: D = (gamma - gamma_15) log2(e),
        //      E = 2^D, E^-1 = 2^-D ----
        {
            const int c = tid & 127;
            const float *la = reinterpret_cast<const float *>(buf + IB_LA);
            const float kL2E = 1.4426950408889634f;
            const uint32_t cq = (uint32_t)(c >> 2), cb = (uint32_t)((c & 3) << 2);
            float acc = 0.f;
            if (half == 0) {  // rows 15..0: D_r = -(sum of log alpha over rows r+1..15)
#pragma unroll
                for (int r = 15; r >= 0; --r) {
                    const uint32_t off = (uint32_t)(r * 512) + ((cq ^ (uint32_t)r) << 4) + cb;
                    *reinterpret_cast<float *>(sm + W_E + off) = ex2_approx(-acc);
                    *reinterpret_cast<float *>(sm + W_EI + off) = ex2_approx(acc);
                    acc = fmaf(la[r * kD + c], kL2E, acc);
                }
                vec[V_M + c] = acc;  // gamma_15 log2(e)
                vec[V_EM + c] = ex2_approx(acc);
            } else {  // rows 16..31: D_r = sum of log alpha over rows 16..r
#pragma unroll
                for (int r = 16; r < 32; ++r) {
                    acc = fmaf(la[r * kD + c], kL2E, acc);
                    const uint32_t off = (uint32_t)(r * 512) + ((cq ^ (uint32_t)r) << 4) + cb;
                    *reinterpret_cast<float *>(sm + W_E + off) = ex2_approx(acc);
                    *reinterpret_cast<float *>(sm + W_EI + off) = ex2_approx(-acc);
                }
                vec[V_D31 + c] = acc;
                vec[V_E31 + c] = ex2_approx(acc);
            }
        }
        __syncthreads();

        // ---- F3: operands that do not depend on the state ----
        if (tid < kD) vec[V_GC + tid] = ex2_approx(vec[V_M + tid] + vec[V_D31 + tid]);  // Gamma_C
        if (trow < 64) {  // M1's A operand into TMEM: rows 0..31 k E, rows 32..63 q E
            const int r = trow & 31;
            const unsigned char *src = buf + (trow < 32 ? IB_K : IB_Q);
            uint32_t hw[32], lw[32];
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8) {
                const int cc = 8 * half + q8;
                float x[8];
                bf16x8_to_f32(*reinterpret_cast<const uint4 *>(src + tile_chunk(r, cc)), x);
                const float4 e0 = *reinterpret_cast<const float4 *>(sm + W_E + e_chunk(r, 2 * cc));
                const float4 e1 =
                    *reinterpret_cast<const float4 *>(sm + W_E + e_chunk(r, 2 * cc + 1));
                split2(x[0] * e0.x, x[1] * e0.y, hw[4 * q8 + 0], lw[4 * q8 + 0]);
                split2(x[2] * e0.z, x[3] * e0.w, hw[4 * q8 + 1], lw[4 * q8 + 1]);
                split2(x[4] * e1.x, x[5] * e1.y, hw[4 * q8 + 2], lw[4 * q8 + 2]);
                split2(x[6] * e1.z, x[7] * e1.w, hw[4 * q8 + 3], lw[4 * q8 + 3]);
            }
            tmem_st32(tl + TM_OPG + 32 * half, hw);
            tmem_st32(tl + TM_OPG + 64 + 32 * half, lw);
        }
        // 16-byte-chunk jobs: R = k E^-1 (M1 B), k Gamma (M2b B), K^ (M5 B), Q~ (M3 B rows 32..63)
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int job = m >> 1;
            const int rem = tid + kThreads * (m & 1);
            const int i = rem >> 4, cc = rem & 15;
            float x[8];
            bf16x8_to_f32(*reinterpret_cast<const uint4 *>(buf + (job == 3 ? IB_Q : IB_K) +
                                                           tile_chunk(i, cc)),
                          x);
            const uint32_t fsrc = (job == 0 || job == 2) ? W_EI : W_E;
            float4 f0 = *reinterpret_cast<const float4 *>(sm + fsrc + e_chunk(i, 2 * cc));
            float4 f1 = *reinterpret_cast<const float4 *>(sm + fsrc + e_chunk(i, 2 * cc + 1));
            if (job != 0) {  // channel factor: e^m (k Gamma, Q~) or E_31 (K^)
                const float *cf = vec + (job == 2 ? V_E31 : V_EM) + 8 * cc;
                const float4 c0 = *reinterpret_cast<const float4 *>(cf);
                const float4 c1 = *reinterpret_cast<const float4 *>(cf + 4);
                f0.x *= c0.x; f0.y *= c0.y; f0.z *= c0.z; f0.w *= c0.w;
                f1.x *= c1.x; f1.y *= c1.y; f1.z *= c1.z; f1.w *= c1.w;
            }
            const float2 p0 = mul2(make_float2(x[0], x[1]), make_float2(f0.x, f0.y));
            const float2 p1 = mul2(make_float2(x[2], x[3]), make_float2(f0.z, f0.w));
            const float2 p2 = mul2(make_float2(x[4], x[5]), make_float2(f1.x, f1.y));
            const float2 p3 = mul2(make_float2(x[6], x[7]), make_float2(f1.z, f1.w));
            const float y[8] = {p0.x, p0.y, p1.x, p1.y, p2.x, p2.y, p3.x, p3.y};
            unsigned char *hi;
            uint32_t lo_off;
            if (job == 0) {
                hi = sm + W_R + tile_chunk(i, cc);
                lo_off = 8192;
            } else if (job == 1) {
                hi = sm + W_KT + tile_chunk(i, cc);
                lo_off = 8192;
            } else if (job == 2) {
                hi = sm + W_KH + tile_chunk(i, cc);
                lo_off = 8192;
            } else {
                hi = sm + W_WQ + sw128_chunk_offset(64, 32 + i, cc);
                lo_off = 16384;
            }
            store_split_chunk(hi, hi + lo_off, y);
        }
        publish_operands();
        if (tid == 0) {  // M1: Gram
            const uint32_t id = idesc_bf16_f32(128, 32);
            const uint32_t rh = smem_u32(sm + W_R), rl = rh + 8192;
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16_tmem_a(tb + TM_D1, tb + TM_OPG + 8 * s, sw128_desc_k(rh, 32, s), id, s > 0);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16_tmem_a(tb + TM_D1, tb + TM_OPG + 8 * s, sw128_desc_k(rl, 32, s), id, 1);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16_tmem_a(tb + TM_D1, tb + TM_OPG + 64 + 8 * s, sw128_desc_k(rh, 32, s), id,
                                1);
            mma_commit(bar);
        }

        // ---- F4 (while M1 runs): S0^T -> M3's A operand; S^T *= Gamma_C along j ----
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            const int j0 = 64 * half + 32 * part;
            float sv[32];
            tmem_ld32(tl + TM_ST + j0, sv);
            uint32_t hw[16], lw[16], sc[32];
#pragma unroll
            for (int pp = 0; pp < 16; ++pp) split2(sv[2 * pp], sv[2 * pp + 1], hw[pp], lw[pp]);
#pragma unroll
            for (int jj = 0; jj < 32; jj += 4) {
                const float4 g4 = *reinterpret_cast<const float4 *>(vec + V_GC + j0 + jj);
                const float2 a = mul2(make_float2(sv[jj], sv[jj + 1]), make_float2(g4.x, g4.y));
                const float2 b = mul2(make_float2(sv[jj + 2], sv[jj + 3]), make_float2(g4.z, g4.w));
                sc[jj] = __float_as_uint(a.x);
                sc[jj + 1] = __float_as_uint(a.y);
                sc[jj + 2] = __float_as_uint(b.x);
                sc[jj + 3] = __float_as_uint(b.y);
            }
            tmem_st16u(tl + TM_OPS + (j0 >> 1), hw);
            tmem_st16u(tl + TM_OPS + 64 + (j0 >> 1), lw);
            tmem_st32(tl + TM_ST + j0, sc);
        }
        alive = wait_mma(bar, phase, p.status, 1);
        if (!alive) break;

        // ---- F5: A (k rows, scaled by beta, strictly lower) and P (q rows, lower) ----
        if (trow < 64) {
            float g[16];
            tmem_ld16(tl + TM_D1 + 16 * half, g);
            if (trow < 32) {
                const int r = trow;
                const float br = beta_s[r];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int i = 16 * half + e;
                    sA[r * kLd + i] = i < r ? br * g[e] : 0.f;
                }
            } else {
                const int r = trow - 32;
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int i = 16 * half + 8 * c2 + e;
                        x[e] = i <= r ? g[8 * c2 + e] : 0.f;
                    }
                    const int ch = 2 * half + c2;
                    store_split_chunk(sm + W_R + 8192 + sw128_chunk_offset(32, r, ch),
                                      sm + W_R + 12288 + sw128_chunk_offset(32, r, ch), x);
                }
            }
        }
        __syncthreads();

        // ---- F6: T = (I + A)^-1 on 2 x 2 tiles of 16, then Tb = T diag(beta) ----
        if (tid < 32) {  // diagonal tiles, one column per thread
            const int blk = tid >> 4, jj = tid & 15;
            float x[16];
#pragma unroll
            for (int m = 0; m < 16; ++m) x[m] = m == jj ? 1.f : 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i)
#pragma unroll
                for (int m = i + 1; m < 16; ++m)
                    x[m] = fmaf(-sA[(16 * blk + m) * kLd + 16 * blk + i], x[i], x[m]);
#pragma unroll
            for (int m = 0; m < 16; ++m) sT[(16 * blk + m) * kLd + 16 * blk + jj] = x[m];
        }
        __syncthreads();
        {  // T_10 = -T_11 (A_10 T_00)
            const int r = tid >> 4, i = tid & 15;
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) acc = fmaf(sA[(16 + r) * kLd + m], sT[m * kLd + i], acc);
            sT[(16 + r) * kLd + i] = acc;  // X = A_10 T_00 in the T_10 slot
            __syncthreads();
            float y = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m)
                y = fmaf(sT[(16 + r) * kLd + 16 + m], sT[(16 + m) * kLd + i], y);
            __syncthreads();
            sT[(16 + r) * kLd + i] = -y;
        }
        __syncthreads();
        if (tid < 128) {  // Tb -> M2's B operand and M2b's A operand (32 rows x 32 K)
            const int r = tid >> 2, cc = tid & 3;
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int i = 8 * cc + e;
                x[e] = i <= r ? sT[r * kLd + i] * beta_s[i] : 0.f;
            }
            store_split_chunk(sm + W_R + sw128_chunk_offset(32, r, cc),
                              sm + W_R + 4096 + sw128_chunk_offset(32, r, cc), x);
        }
        publish_operands();
        if (tid == 0) {
            const uint32_t th = smem_u32(sm + W_R), tlo = th + 4096;
            // M2: U~^T = V^T Tb^T  (V exact in bf16, read MN-major from the staged tile)
            const uint32_t idv = idesc_bf16_f32(128, 32) | kIdescAMN;
            const uint32_t va = smem_u32(buf + IB_V);
#pragma unroll
            for (int s = 0; s < 2; ++s)
                mma_bf16(tb + TM_DW + 32, sw128_desc_mn(va + 2048 * s, 4096),
                         sw128_desc_k(th, 32, s), idv, s > 0);
#pragma unroll
            for (int s = 0; s < 2; ++s)
                mma_bf16(tb + TM_DW + 32, sw128_desc_mn(va + 2048 * s, 4096),
                         sw128_desc_k(tlo, 32, s), idv, 1);
            // M2b: W = Tb (k Gamma): A = Tb (rows r; lanes >= 32 unused), B = (k Gamma) MN-major
            const uint32_t idw = idesc_bf16_f32(128, 128) | kIdescBMN;
            const uint32_t kh = smem_u32(sm + W_KT), kl = kh + 8192;
#pragma unroll
            for (int s = 0; s < 2; ++s)
                mma_bf16(tb + TM_OPG, sw128_desc_k(th, 128, s), sw128_desc_mn(kh + 2048 * s, 4096),
                         idw, s > 0);
#pragma unroll
            for (int s = 0; s < 2; ++s)
                mma_bf16(tb + TM_OPG, sw128_desc_k(th, 128, s), sw128_desc_mn(kl + 2048 * s, 4096),
                         idw, 1);
#pragma unroll
            for (int s = 0; s < 2; ++s)
                mma_bf16(tb + TM_OPG, sw128_desc_k(tlo, 128, s), sw128_desc_mn(kh + 2048 * s, 4096),
                         idw, 1);
            mma_commit(bar);
        }
        alive = wait_mma(bar, phase, p.status, 2);
        if (!alive) break;

        // ---- F7: W rows (TMEM lanes 0..31) -> rows 0..31 of M3's B operand ----
        if (quarter == 0) {
            const int r = lane;
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                const int j0 = 64 * half + 32 * part;
                float w[32];
                tmem_ld32(tl + TM_OPG + j0, w);
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8) {
                    const float x[8] = {w[8 * q8], w[8 * q8 + 1], w[8 * q8 + 2], w[8 * q8 + 3],
                                        w[8 * q8 + 4], w[8 * q8 + 5], w[8 * q8 + 6], w[8 * q8 + 7]};
                    const int cc = (j0 >> 3) + q8;
                    unsigned char *hi = sm + W_WQ + sw128_chunk_offset(64, r, cc);
                    store_split_chunk(hi, hi + 16384, x);
                }
            }
        }
        publish_operands();
        if (tid == 0) {  // M3: [(W S0)^T | (Q~ S0)^T] = S0^T [W ; Q~]^T
            const uint32_t id = idesc_bf16_f32(128, 64);
            const uint32_t bh = smem_u32(sm + W_WQ), bl = bh + 16384;
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16_tmem_a(tb + TM_D1, tb + TM_OPS + 8 * s, sw128_desc_k(bh, 64, s), id, s > 0);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16_tmem_a(tb + TM_D1, tb + TM_OPS + 8 * s, sw128_desc_k(bl, 64, s), id, 1);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16_tmem_a(tb + TM_D1, tb + TM_OPS + 64 + 8 * s, sw128_desc_k(bh, 64, s), id,
                                1);
            mma_commit(bar);
        }
        alive = wait_mma(bar, phase, p.status, 3);
        if (!alive) break;

        // ---- F8: U^T = U~^T - (W S0)^T -> A operand of M4 / M5 ----
        {
            float ut[16], ws[16];
            tmem_ld16(tl + TM_DW + 32 + 16 * half, ut);
            tmem_ld16(tl + TM_D1 + 16 * half, ws);
            uint32_t hw[8], lw[8];
#pragma unroll
            for (int pp = 0; pp < 8; ++pp)
                split2(ut[2 * pp] - ws[2 * pp], ut[2 * pp + 1] - ws[2 * pp + 1], hw[pp], lw[pp]);
            tmem_st8u(tl + TM_OPS + 8 * half, hw);
            tmem_st8u(tl + TM_OPS + 16 + 8 * half, lw);
        }
        publish_operands();
        if (tid == 0) {
            const uint32_t id32 = idesc_bf16_f32(128, 32);
            const uint32_t id128 = idesc_bf16_f32(128, 128) | kIdescBMN;
            const uint32_t ph = smem_u32(sm + W_R + 8192), pl = ph + 4096;
            const uint32_t kh = smem_u32(sm + W_KH), kl = kh + 8192;
            // M4: (Q~ S0 + P U)^T += U^T P^T
#pragma unroll
            for (int s = 0; s < 2; ++s)
                mma_bf16_tmem_a(tb + TM_D1 + 32, tb + TM_OPS + 8 * s, sw128_desc_k(ph, 32, s), id32,
                                1);
#pragma unroll
            for (int s = 0; s < 2; ++s)
                mma_bf16_tmem_a(tb + TM_D1 + 32, tb + TM_OPS + 8 * s, sw128_desc_k(pl, 32, s), id32,
                                1);
#pragma unroll
            for (int s = 0; s < 2; ++s)
                mma_bf16_tmem_a(tb + TM_D1 + 32, tb + TM_OPS + 16 + 8 * s, sw128_desc_k(ph, 32, s),
                                id32, 1);
            // M5: S^T += U^T K^
#pragma unroll
            for (int s = 0; s < 2; ++s)
                mma_bf16_tmem_a(tb + TM_ST, tb + TM_OPS + 8 * s, sw128_desc_mn(kh + 2048 * s, 4096),
                                id128, 1);
#pragma unroll
            for (int s = 0; s < 2; ++s)
                mma_bf16_tmem_a(tb + TM_ST, tb + TM_OPS + 8 * s, sw128_desc_mn(kl + 2048 * s, 4096),
                                id128, 1);
#pragma unroll
            for (int s = 0; s < 2; ++s)
                mma_bf16_tmem_a(tb + TM_ST, tb + TM_OPS + 16 + 8 * s,
                                sw128_desc_mn(kh + 2048 * s, 4096), id128, 1);
            mma_commit(bar);
        }
        alive = wait_mma(bar, phase, p.status, 4);
        if (!alive) break;

        // ---- F9: readout o[r][c] = scale (Q~ S0 + P U)^T[c][r] ----
        {
            const int c = trow;
            float ov[16];
            tmem_ld16(tl + TM_D1 + 32 + 16 * half, ov);
            Tout *o = static_cast<Tout *>(p.o);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int r = 16 * half + e;
                if (r < nrow)
                    Elem<Tout>::store(o + ((size_t)(t0 + r) * H + h) * kD + c, p.scale * ov[e]);
            }
        }
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
    }

    cp_async_wait_all();  // nothing may still be in flight into shared memory on exit
    // ---- final state (lane c, column j) -> S_final[j][c] ----
    if (alive && p.S_final != nullptr) {
        const int c = trow;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            const int j0 = 64 * half + 32 * part;
            float sv[32];
            tmem_ld32(tl + TM_ST + j0, sv);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
                p.S_final[state_off + (size_t)(j0 + jj) * kD + c] = sv[jj];
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

template <typename Tout>
cudaError_t launch_typed(const PrefillArgs &a, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<Tout>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SM_DYN);
    if (e != cudaSuccess) return e;
    Params p;
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.k = static_cast<const __nv_bfloat16 *>(a.k);
    p.v = static_cast<const __nv_bfloat16 *>(a.v);
    p.log_alpha = a.log_alpha;
    p.beta = a.beta;
    p.S0 = a.S0;
    p.cu_seqlens = a.cu_seqlens;
    p.H = a.num_heads;
    p.scale = a.scale;
    p.o = a.o;
    p.S_final = a.S_final;
    p.status = a.status;
    const unsigned grid = (unsigned)a.num_seqs * (unsigned)a.num_heads;
    prefill_tc_kernel<Tout><<<grid, kThreads, SM_DYN, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t stream) {
    if (a.out_dtype == KDA_BF16) return launch_typed<__nv_bfloat16>(a, stream);
    return launch_typed<float>(a, stream);
}

}  // namespace kda
