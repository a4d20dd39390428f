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
//   M2b W' = Tb . (k E)          (Tb repeated in all four lane quarters; B read MN-major)
//   M3  [ (W S0)^T | (Q~ S0)^T ] = S0^T . [W ; Q~]^T   (A = S0^T from TMEM)
//   M4  (Q~ S0 + P U)^T += U^T . P^T
//   M5  X^T += U^T . (k E^-1)    (the state kept as X = S / e31; B read MN-major)
//
// Precision: an fp32 quantity x enters an MMA as x = hi + lo (two bf16,
// round-to-nearest), and a product X.Y is formed as hi.hi + hi.lo + lo.hi
// (fp32 accumulation); V is exact in bf16 and enters once.
//
// Inputs of chunk c+1 are staged with TMA (q, k, v, log_alpha) and cp.async (beta)
// while chunk c is processed.
#include <cuda.h>
#include <cstring>
#include <cudaTypedefs.h>

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
// layout below, written by TMA with 128-byte swizzle), log_alpha (fp32, four
// [32 rows][32 channels] boxes of 4096 bytes), beta [32].
constexpr uint32_t IB_Q = 0, IB_K = 8192, IB_V = 16384, IB_LA = 24576, IB_BETA = 40960;
constexpr uint32_t IB_SIZE = 43008;
constexpr uint32_t W_E = 2 * IB_SIZE;    // fp32 [32][128] 2^D, then (solve) Tb x4 hi (16 KB)
constexpr uint32_t W_EI = W_E + 16384;   // fp32 [32][128] 2^-D, then Tb x4 lo (16 KB)
constexpr uint32_t W_X = W_EI + 16384;   // [k E ; q E] hi (16 KB) | lo (16 KB), 64 rows x 128 K
constexpr uint32_t W_R = W_X + 32768;    // R = k E^-1 hi (8 KB) | lo (8 KB), 32 rows x 128 K
constexpr uint32_t W_WQ = W_R + 16384;   // [W ; Q~] hi (16 KB) | lo (16 KB), 64 rows x 128 K
constexpr uint32_t W_P = W_WQ + 32768;   // P hi (4 KB) | lo (4 KB), 32 rows x 32 K
constexpr uint32_t W_A = W_P + 8192;     // fp32 [32][33]
constexpr uint32_t W_T = W_A + 4224;     // fp32 [32][33]
constexpr uint32_t W_VEC = W_T + 4224;   // em[2][128], e31[2][128] (by chunk parity)
constexpr uint32_t W_BAR = W_VEC + 4 * 512;   // two MMA mbarriers, then two TMA mbarriers
constexpr uint32_t W_TSLOT = W_BAR + 32;
constexpr uint32_t kTmaBytes = 10 * 4096;        // 6 bf16 boxes (q, k, v) + 4 fp32 boxes
constexpr uint32_t SM_DYN = W_TSLOT + 8 + 1024;  // + alignment slack
constexpr int kLd = 33;  // padded row stride of A and T

// ---- TMEM column map (512 columns) -----------------------------------------
constexpr uint32_t TM_ST = 0;    // state, stored as S^T / e31 (lane c, column j), fp32
constexpr uint32_t TM_D1 = 128;  // [(W S0)^T | (Q~ S0 + P U)^T] (32 + 32)
constexpr uint32_t TM_DG = 192;  // Gram result, K steps 0-3 (lanes 0-31 k rows, 32-63 q rows)
constexpr uint32_t TM_DU = 224;  // Gram result, K steps 4-7; then U~^T (32 columns)
constexpr uint32_t TM_WT = 256;  // W' = Tb (k E) (rows r repeated in every lane quarter), 128
                                 // columns; then the K steps 4-7 half of M3 (64 columns)
constexpr uint32_t TM_OPS = 384; // M3's A operand S0^T hi (64) | lo (64); then U^T hi (16) | lo (16)

// Swizzled [rows][128 bf16] operand tile with `rows` rows: two 64-column blocks
// of rows x 128 bytes, 16-byte chunk j of row i at chunk position j ^ (i % 8).
// Read K-major it has `rows` rows and K = 128; read MN-major (K = the rows) its
// 64-element MN blocks are rows * 128 bytes apart.
__device__ __forceinline__ uint32_t tile_chunk(int rows, int i, int cc) {
    return (uint32_t)((cc >> 3) * rows * 128 + i * 128 + (((cc & 7) ^ (i & 7)) << 4));
}
// fp32 [32][128] with 16-byte chunks swizzled by row.
__device__ __forceinline__ uint32_t e_chunk(int r, int q) {  // q = 4-float chunk 0..31
    return (uint32_t)(r * 512 + (((q ^ r) & 31) << 4));
}

struct Params {
    CUtensorMap tm_q, tm_k, tm_v, tm_la;  // [T][H*128] with boxes of 32 tokens
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

__device__ __forceinline__ void mul8(float (&x)[8], const float4 &a, const float4 &b) {
    const float2 p0 = mul2(make_float2(x[0], x[1]), make_float2(a.x, a.y));
    const float2 p1 = mul2(make_float2(x[2], x[3]), make_float2(a.z, a.w));
    const float2 p2 = mul2(make_float2(x[4], x[5]), make_float2(b.x, b.y));
    const float2 p3 = mul2(make_float2(x[6], x[7]), make_float2(b.z, b.w));
    x[0] = p0.x; x[1] = p0.y; x[2] = p1.x; x[3] = p1.y;
    x[4] = p2.x; x[5] = p2.y; x[6] = p3.x; x[7] = p3.y;
}

// MMAs are issued by two threads (lane 0 of warps 0 and 1), each tracking its
// own work on its own mbarrier.  Those two threads wait (bounded) for their
// barrier; the CTA barrier then orders every other thread after both.
constexpr int kIssuerA = 0, kIssuerB = 32;
__device__ __forceinline__ bool wait_mma(uint64_t *bar, uint32_t &phase, DeviceStatus st,
                                         uint32_t where) {
    bool ok = true;
    if (threadIdx.x == kIssuerA || threadIdx.x == kIssuerB) {
        ok = mbar_wait_bounded(bar + (threadIdx.x == kIssuerB), phase & 1u, kWaitNs);
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

// Stage chunk [t0, t0 + 32) of this head into input buffer `buf`: one thread
// issues the TMA boxes, threads 0..31 fetch beta (zero past nrow).  Rows past the
// sequence end are not masked here: log_alpha and beta are masked where they are
// used, which keeps those rows out of every product (see the kernel).
constexpr int kTmaThread = 64;
__device__ __forceinline__ void issue_loads(const Params &p, unsigned char *buf, uint64_t *tbar,
                                            int t0, int nrow, int h, int tid) {
    if (tid == kTmaThread) {
        fence_proxy_async_smem();  // earlier generic accesses to this buffer come first
        mbar_arrive_expect_tx(tbar, kTmaBytes);
        const CUtensorMap *maps[3] = {&p.tm_q, &p.tm_k, &p.tm_v};
        const uint32_t dst[3] = {IB_Q, IB_K, IB_V};
#pragma unroll
        for (int a = 0; a < 3; ++a)
#pragma unroll
            for (int b = 0; b < 2; ++b)
                tma_load_2d(smem_u32(buf + dst[a] + 4096 * b), maps[a], h * kD + 64 * b, t0, tbar);
#pragma unroll
        for (int b = 0; b < 4; ++b)
            tma_load_2d(smem_u32(buf + IB_LA + 4096 * b), &p.tm_la, h * kD + 32 * b, t0, tbar);
    }
    if (tid < kC) {
        const bool ok = tid < nrow;
        const float *s = ok ? p.beta + (size_t)(t0 + tid) * p.H + h : p.beta;
        cp_async4(smem_u32(buf + IB_BETA + 4 * tid), s, ok ? 4u : 0u);
        cp_async_commit();
    }
}

// Algebra per chunk (log2 units, D_r = (gamma_r - gamma_15) log2 e, E = 2^D,
// em = e^{gamma_15}, e31 = 2^{D_31}, so Gamma_r = em E_r and Gamma_C = em e31):
//   Gram:  G = [k E ; q E] (k E^-1)^T  ->  A = beta_r G_k (i < r), P = G_q (i <= r)
//   W = Tb (k Gamma) = (Tb (k E)) diag(em),   Q~ = (q E) diag(em),   U~ = Tb V
//   K^ = (k E^-1) diag(e31)  =>  S_C = Diag(e31) [ Diag(em) S0 + (k E^-1)^T U ]
// The state is kept in TMEM as X = S / e31 (per key channel), so the update is
// X <- Diag(em) S0 + (k E^-1)^T U with the Gram's own R = k E^-1 tile as M5's
// B operand, and S0 = Diag(e31_prev) X is formed once per chunk in the pass that
// also builds M3's A operand.
template <typename Tout>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ Params p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float *vec = reinterpret_cast<float *>(sm + W_VEC);  // em[2][128] | e31[2][128]
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
    uint64_t *tbar = bar + 2;  // TMA barriers, one per input buffer
    if (tid == kTmaThread) {
        mbar_init(bar, 1);
        mbar_init(bar + 1, 1);
        mbar_init(tbar, 1);
        mbar_init(tbar + 1, 1);
        fence_mbar_init();
    }
    if (tid < kD) vec[2 * kD + kD + tid] = 1.f;  // e31 of "chunk -1": the entering state is exact
    __syncthreads();
    if (t_begin < t_end) issue_loads(p, sm, tbar, t_begin, min(kC, t_end - t_begin), h, tid);
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

    // Readout of a finished chunk: o[t0 + r][c] = scale (Q~ S0 + P U)^T[c][r], the two K
    // halves of M3 summed.  Done by warps 4..7 (one per lane quarter): the tile is staged
    // row-major in the (dead) E^-1 table, then written out as 16-byte row chunks.
    Tout *o = static_cast<Tout *>(p.o);
    auto readout = [&](int t0r, int nrowr) {
        Tout *ot = reinterpret_cast<Tout *>(sm + W_EI);  // [32][128]
        const int c = trow;
#pragma unroll
        for (int r0 = 0; r0 < 32; r0 += 16) {
            float ov[16], ov2[16];
            tmem_ld16(tl + TM_D1 + 32 + r0, ov);
            tmem_ld16(tl + TM_WT + 32 + r0, ov2);
#pragma unroll
            for (int e = 0; e < 16; ++e)
                Elem<Tout>::store(ot + (r0 + e) * kD + c, p.scale * (ov[e] + ov2[e]));
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");  // warps 4..7 only
        constexpr int kPerRow = kD * (int)sizeof(Tout) / 16;  // 16-byte chunks per row
        const int lt = tid - 128;
        for (int e = lt; e < kC * kPerRow; e += 128) {
            const int r = e / kPerRow, ch = e % kPerRow;
            if (r < nrowr)
                *reinterpret_cast<uint4 *>(reinterpret_cast<unsigned char *>(
                    o + ((size_t)(t0r + r) * H + h) * kD) + 16 * ch) =
                    *reinterpret_cast<const uint4 *>(reinterpret_cast<const unsigned char *>(ot) +
                                                     r * kD * sizeof(Tout) + 16 * ch);
        }
    };

    bool alive = true;
    int chunk = 0, t0_prev = 0, nrow_prev = 0;
    for (int t0 = t_begin; t0 < t_end && alive; t0 += kC, ++chunk) {
        const int nrow = min(kC, t_end - t0);
        const int par = chunk & 1;
        unsigned char *buf = sm + par * IB_SIZE;
        const float *beta_s = reinterpret_cast<const float *>(buf + IB_BETA);
        float *em = vec + par * kD;
        float *e31 = vec + 2 * kD + par * kD;
        const float *e31_prev = vec + 2 * kD + (par ^ 1) * kD;

        // ---- F1: this chunk's inputs have landed; stage the next chunk ----
        {
            bool ok = true;
            if (tid == kTmaThread) {
                ok = mbar_wait_bounded(tbar + par, (uint32_t)(chunk >> 1) & 1u, kWaitNs);
                if (!ok) record_status(p.status, KDA_ERR_DEVICE_TIMEOUT, 0);
            }
            if (tid < kC) cp_async_wait_all();
            if (!__syncthreads_and(ok)) {
                alive = false;
                break;
            }
            fence_after_sync();
        }
        if (t0 + kC < t_end)
            issue_loads(p, sm + (par ^ 1) * IB_SIZE, tbar + (par ^ 1), t0 + kC,
                        min(kC, t_end - t0 - kC), h, tid);

        // ---- F2: decay factors; threads c and c + 128 share key channel c ----
        {
            const int c = tid & 127;
            const float *la = reinterpret_cast<const float *>(buf + IB_LA);
            const float kL2E = 1.4426950408889634f;
            const uint32_t cq = (uint32_t)(c >> 2), cb = (uint32_t)((c & 3) << 2);
            float pre[16];
            float acc = 0.f;
            const int r0 = 16 * half;
#pragma unroll
            const float *lac = la + (c >> 5) * 1024 + (c & 31);  // box c/32, row stride 32
            for (int r = 0; r < 16; ++r) {
                const float x = (r0 + r) < nrow ? lac[(r0 + r) * 32] : 0.f;  // rows past the end
                acc = fmaf(x, kL2E, acc);
                pre[r] = acc;
            }
            // rows 0..15: D = prefix - prefix_15;  rows 16..31: D = sum of rows 16..r
            const float sub = half == 0 ? pre[15] : 0.f;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const float d = pre[r] - sub;
                const uint32_t off =
                    (uint32_t)((r0 + r) * 512) + ((cq ^ (uint32_t)(r0 + r)) << 4) + cb;
                *reinterpret_cast<float *>(sm + W_E + off) = ex2_approx(d);
                *reinterpret_cast<float *>(sm + W_EI + off) = ex2_approx(-d);
            }
            if (half == 0) em[c] = ex2_approx(pre[15]);
            else e31[c] = ex2_approx(pre[15]);
        }
        __syncthreads();

        // ---- F3: [k E ; q E], R = k E^-1, Q~ = q E em (one 16-byte chunk per job) ----
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int e = tid + kThreads * m;  // 512 jobs: row i, chunk cc
            const int i = e >> 4, cc = e & 15;
            float xk[8], xq[8];
            bf16x8_to_f32(*reinterpret_cast<const uint4 *>(buf + IB_K + tile_chunk(32, i, cc)), xk);
            bf16x8_to_f32(*reinterpret_cast<const uint4 *>(buf + IB_Q + tile_chunk(32, i, cc)), xq);
            const float4 e0 = *reinterpret_cast<const float4 *>(sm + W_E + e_chunk(i, 2 * cc));
            const float4 e1 = *reinterpret_cast<const float4 *>(sm + W_E + e_chunk(i, 2 * cc + 1));
            const float4 f0 = *reinterpret_cast<const float4 *>(sm + W_EI + e_chunk(i, 2 * cc));
            const float4 f1 = *reinterpret_cast<const float4 *>(sm + W_EI + e_chunk(i, 2 * cc + 1));
            const float4 m0 = *reinterpret_cast<const float4 *>(em + 8 * cc);
            const float4 m1 = *reinterpret_cast<const float4 *>(em + 8 * cc + 4);
            float r8[8] = {xk[0], xk[1], xk[2], xk[3], xk[4], xk[5], xk[6], xk[7]};
            mul8(r8, f0, f1);   // k E^-1
            mul8(xk, e0, e1);   // k E
            mul8(xq, e0, e1);   // q E
            unsigned char *xh = sm + W_X + tile_chunk(64, i, cc);
            store_split_chunk(xh, xh + 16384, xk);
            xh = sm + W_X + tile_chunk(64, 32 + i, cc);
            store_split_chunk(xh, xh + 16384, xq);
            unsigned char *rh = sm + W_R + tile_chunk(32, i, cc);
            store_split_chunk(rh, rh + 8192, r8);
            mul8(xq, m0, m1);   // Q~ = q E em
            unsigned char *qh = sm + W_WQ + tile_chunk(64, 32 + i, cc);
            store_split_chunk(qh, qh + 16384, xq);
        }
        publish_operands();
        if (tid == kIssuerA || tid == kIssuerB) {  // M1: Gram, K steps split over two issuers
            // A = [k E ; q E] (rows 64..127 of the view are ignored), B = R
            const uint32_t id = idesc_bf16_f32(128, 32);
            const int s0 = tid == kIssuerA ? 0 : 4;
            const uint32_t d = tb + (tid == kIssuerA ? TM_DG : TM_DU);
            const uint32_t xh = smem_u32(sm + W_X), xl = xh + 16384;
            const uint32_t rh = smem_u32(sm + W_R), rl = rh + 8192;
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(d, sw128_desc_k(xh, 64, s0 + s), sw128_desc_k(rh, 32, s0 + s), id, s > 0);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(d, sw128_desc_k(xh, 64, s0 + s), sw128_desc_k(rl, 32, s0 + s), id, 1);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(d, sw128_desc_k(xl, 64, s0 + s), sw128_desc_k(rh, 32, s0 + s), id, 1);
            mma_commit(bar + (tid == kIssuerB));
        }

        // ---- F4 (while M1 runs): S0 = e31_prev X -> M3's A operand; X <- em S0 ----
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            const int j0 = 64 * half + 32 * part;
            float sv[32];
            tmem_ld32(tl + TM_ST + j0, sv);
            uint32_t hw[16], lw[16], sc[32];
#pragma unroll
            for (int jj = 0; jj < 32; jj += 4) {
                const float4 g = *reinterpret_cast<const float4 *>(e31_prev + j0 + jj);
                const float2 a = mul2(make_float2(sv[jj], sv[jj + 1]), make_float2(g.x, g.y));
                const float2 b = mul2(make_float2(sv[jj + 2], sv[jj + 3]), make_float2(g.z, g.w));
                sv[jj] = a.x; sv[jj + 1] = a.y; sv[jj + 2] = b.x; sv[jj + 3] = b.y;
            }
#pragma unroll
            for (int pp = 0; pp < 16; ++pp) split2(sv[2 * pp], sv[2 * pp + 1], hw[pp], lw[pp]);
#pragma unroll
            for (int jj = 0; jj < 32; jj += 4) {
                const float4 g = *reinterpret_cast<const float4 *>(em + j0 + jj);
                const float2 a = mul2(make_float2(sv[jj], sv[jj + 1]), make_float2(g.x, g.y));
                const float2 b = mul2(make_float2(sv[jj + 2], sv[jj + 3]), make_float2(g.z, g.w));
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
            float g[16], g2[16];
            tmem_ld16(tl + TM_DG + 16 * half, g);
            tmem_ld16(tl + TM_DU + 16 * half, g2);
#pragma unroll
            for (int e = 0; e < 16; ++e) g[e] += g2[e];
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
                    unsigned char *ph = sm + W_P + sw128_chunk_offset(32, r, 2 * half + c2);
                    store_split_chunk(ph, ph + 4096, x);
                }
            }
        }
        __syncthreads();

        // ---- F6: T = (I + A)^-1 on 2 x 2 tiles of 16, then Tb = T diag(beta); while warp 0
        //      solves the diagonal tiles, warps 4..7 read out the previous chunk ----
        if (half == 1 && chunk > 0) readout(t0_prev, nrow_prev);
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
        {  // Tb (32 rows x 32 K) written 4 times: rows 32 q + r, so W' lands in every lane quarter
            const int r = tid >> 3, cc = tid & 3, copy2 = (tid >> 2) & 1;
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int i = 8 * cc + e;
                x[e] = i <= r ? sT[r * kLd + i] * beta_s[i] : 0.f;
            }
#pragma unroll
            for (int cp = 0; cp < 2; ++cp) {
                const int row = 32 * (2 * cp + copy2) + r;
                unsigned char *th = sm + W_E + sw128_chunk_offset(128, row, cc);
                store_split_chunk(th, th + 16384, x);
            }
        }
        publish_operands();
        if (tid == kIssuerA) {  // M2: U~^T = V^T Tb^T  (V exact in bf16, read MN-major)
            const uint32_t th = smem_u32(sm + W_E), tlo = th + 16384;
            const uint32_t idv = idesc_bf16_f32(128, 32) | kIdescAMN;
            const uint32_t va = smem_u32(buf + IB_V);
#pragma unroll
            for (int s = 0; s < 2; ++s)
                mma_bf16(tb + TM_DU, sw128_desc_mn(va + 2048 * s, 4096), sw128_desc_k(th, 128, s),
                         idv, s > 0);
#pragma unroll
            for (int s = 0; s < 2; ++s)
                mma_bf16(tb + TM_DU, sw128_desc_mn(va + 2048 * s, 4096), sw128_desc_k(tlo, 128, s),
                         idv, 1);
            mma_commit(bar);
        } else if (tid == kIssuerB) {
            // M2b: W' = Tb (k E): A = Tb x4 (128 rows), B = rows 0..31 of [k E ; q E] MN-major
            const uint32_t th = smem_u32(sm + W_E), tlo = th + 16384;
            const uint32_t idw = idesc_bf16_f32(128, 128) | kIdescBMN;
            const uint32_t xh = smem_u32(sm + W_X), xl = xh + 16384;
#pragma unroll
            for (int s = 0; s < 2; ++s)
                mma_bf16(tb + TM_WT, sw128_desc_k(th, 128, s), sw128_desc_mn(xh + 2048 * s, 8192),
                         idw, s > 0);
#pragma unroll
            for (int s = 0; s < 2; ++s)
                mma_bf16(tb + TM_WT, sw128_desc_k(th, 128, s), sw128_desc_mn(xl + 2048 * s, 8192),
                         idw, 1);
#pragma unroll
            for (int s = 0; s < 2; ++s)
                mma_bf16(tb + TM_WT, sw128_desc_k(tlo, 128, s), sw128_desc_mn(xh + 2048 * s, 8192),
                         idw, 1);
            mma_commit(bar + 1);
        }
        alive = wait_mma(bar, phase, p.status, 2);
        if (!alive) break;

        // ---- F7: W = W' diag(em) -> rows 0..31 of M3's B operand (all 8 warps) ----
        {
            const int r = lane;
            const int c0 = 16 * (2 * quarter + half);
            float w[16];
            tmem_ld16(tl + TM_WT + c0, w);
#pragma unroll
            for (int h8 = 0; h8 < 2; ++h8) {
                float x[8] = {w[8 * h8], w[8 * h8 + 1], w[8 * h8 + 2], w[8 * h8 + 3],
                              w[8 * h8 + 4], w[8 * h8 + 5], w[8 * h8 + 6], w[8 * h8 + 7]};
                const float4 m0 = *reinterpret_cast<const float4 *>(em + c0 + 8 * h8);
                const float4 m1 = *reinterpret_cast<const float4 *>(em + c0 + 8 * h8 + 4);
                mul8(x, m0, m1);
                unsigned char *wh = sm + W_WQ + tile_chunk(64, r, (c0 >> 3) + h8);
                store_split_chunk(wh, wh + 16384, x);
            }
        }
        publish_operands();
        if (tid == kIssuerA || tid == kIssuerB) {
            // M3: [(W S0)^T | (Q~ S0)^T] = S0^T [W ; Q~]^T, K steps 0-3 -> D1, 4-7 -> WT
            const uint32_t id = idesc_bf16_f32(128, 64);
            const int s0 = tid == kIssuerA ? 0 : 4;
            const uint32_t d = tb + (tid == kIssuerA ? TM_D1 : TM_WT);
            const uint32_t bh = smem_u32(sm + W_WQ), bl = bh + 16384;
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16_tmem_a(d, tb + TM_OPS + 8 * (s0 + s), sw128_desc_k(bh, 64, s0 + s), id,
                                s > 0);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16_tmem_a(d, tb + TM_OPS + 8 * (s0 + s), sw128_desc_k(bl, 64, s0 + s), id, 1);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16_tmem_a(d, tb + TM_OPS + 64 + 8 * (s0 + s), sw128_desc_k(bh, 64, s0 + s), id,
                                1);
            mma_commit(bar + (tid == kIssuerB));
        }
        alive = wait_mma(bar, phase, p.status, 3);
        if (!alive) break;

        // ---- F8: U^T = U~^T - (W S0)^T -> A operand of M4 / M5 ----
        {
            float ut[16], ws[16], ws2[16];
            tmem_ld16(tl + TM_DU + 16 * half, ut);
            tmem_ld16(tl + TM_D1 + 16 * half, ws);
            tmem_ld16(tl + TM_WT + 16 * half, ws2);
#pragma unroll
            for (int e = 0; e < 16; ++e) ws[e] += ws2[e];
            uint32_t hw[8], lw[8];
#pragma unroll
            for (int pp = 0; pp < 8; ++pp)
                split2(ut[2 * pp] - ws[2 * pp], ut[2 * pp + 1] - ws[2 * pp + 1], hw[pp], lw[pp]);
            tmem_st8u(tl + TM_OPS + 8 * half, hw);
            tmem_st8u(tl + TM_OPS + 16 + 8 * half, lw);
        }
        publish_operands();
        if (tid == kIssuerA) {  // M4: (Q~ S0 + P U)^T += U^T P^T
            const uint32_t id32 = idesc_bf16_f32(128, 32);
            const uint32_t ph = smem_u32(sm + W_P), pl = ph + 4096;
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
            mma_commit(bar);
        } else if (tid == kIssuerB) {  // M5: X += U^T (k E^-1)  (the Gram's R tile, read MN-major)
            const uint32_t id128 = idesc_bf16_f32(128, 128) | kIdescBMN;
            const uint32_t rh = smem_u32(sm + W_R), rl = rh + 8192;
#pragma unroll
            for (int s = 0; s < 2; ++s)
                mma_bf16_tmem_a(tb + TM_ST, tb + TM_OPS + 8 * s, sw128_desc_mn(rh + 2048 * s, 4096),
                                id128, 1);
#pragma unroll
            for (int s = 0; s < 2; ++s)
                mma_bf16_tmem_a(tb + TM_ST, tb + TM_OPS + 8 * s, sw128_desc_mn(rl + 2048 * s, 4096),
                                id128, 1);
#pragma unroll
            for (int s = 0; s < 2; ++s)
                mma_bf16_tmem_a(tb + TM_ST, tb + TM_OPS + 16 + 8 * s,
                                sw128_desc_mn(rh + 2048 * s, 4096), id128, 1);
            mma_commit(bar + 1);
        }
        alive = wait_mma(bar, phase, p.status, 4);
        if (!alive) break;

        t0_prev = t0;
        nrow_prev = nrow;  // read out during the next chunk's solve (or after the loop)
    }

    if (alive && chunk > 0 && half == 1) readout(t0_prev, nrow_prev);  // the last chunk
    cp_async_wait_all();  // nothing may still be in flight into shared memory on exit
    if (tid == kTmaThread && !alive) {  // let an outstanding TMA load land before leaving
        // loads were issued for chunks 0 .. n_issued-1; chunks 0 .. chunk-1 were consumed
        const int n_issued = (t_end - t_begin + kC - 1) / kC < chunk + 2
                                 ? (t_end - t_begin + kC - 1) / kC
                                 : chunk + 2;
        for (int c = chunk; c < n_issued; ++c)
            mbar_wait_bounded(tbar + (c & 1), (uint32_t)(c >> 1) & 1u, kWaitNs);
    }
    // ---- final state S = Diag(e31_last) X (lane c, column j) -> S_final[j][c] ----
    if (alive && p.S_final != nullptr) {
        const int c = trow;
        const float *e31_last = vec + 2 * kD + ((chunk - 1) & 1) * kD;  // chunk 0 -> slot 1 = 1
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            const int j0 = 64 * half + 32 * part;
            float sv[32];
            tmem_ld32(tl + TM_ST + j0, sv);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
                p.S_final[state_off + (size_t)(j0 + jj) * kD + c] = sv[jj] * e31_last[j0 + jj];
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// [T][H*128] tensor, boxes of 32 tokens x box_cols elements.
bool encode_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int elem_bytes, int T,
                int H, int box_cols, CUtensorMapSwizzle swz) {
    auto fn = tensor_map_encoder();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)H * kD, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)H * kD * elem_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)kC};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename Tout>
cudaError_t launch_typed(const PrefillArgs &a, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<Tout>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SM_DYN);
    if (e != cudaSuccess) return e;
    Params p;
    memset(&p, 0, sizeof(p));
    if (a.total_tokens > 0) {
        const int T = a.total_tokens, H = a.num_heads;
        if (!encode_map(&p.tm_q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, H, 64,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_map(&p.tm_k, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, H, 64,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_map(&p.tm_v, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, H, 64,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_map(&p.tm_la, a.log_alpha, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, T, H, 32,
                        CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
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
