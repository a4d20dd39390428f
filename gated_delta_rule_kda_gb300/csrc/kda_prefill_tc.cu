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
// In log2 units, D_r = (gamma_r - gamma_15) log2 e, E = 2^D, em = e^{gamma_15},
// e31 = 2^{D_31}, so Gamma_r = em E_r and Gamma_C = em e31.  The state is kept
// in TMEM as X = S / e31 of the chunk that produced it (per key channel):
//   W  = (Tb (k E)) Diag(em),  Q~ = (q E) Diag(em)   (both bounded by |k|, |q|)
//   S0 = Diag(e31_prev) X,     X_new = Diag(em) S0 + (k E^-1)^T U
// em multiplies the q / W side of every product, never the state operand: em
// can be as small as e^-80, and a state operand scaled by it would lose its low
// bf16 half to the subnormal range.
//
// The state is held TRANSPOSED (TMEM lane = value channel c, column = key
// channel j), so every product is an M = 128 tcgen05.mma:
//   M1  G = [k E ; q E] . (k E^-1)^T                  (lanes 0-31 -> A, 32-63 -> P)
//   M2  U~^T = V^T . Tb^T                            (V read MN-major from its staged tile)
//   M2b W'^T = (k E)^T . Tb^T                        ((k E)^T K-major; lane = key channel)
//   M3  [ (W S0)^T | (Q~ S0)^T ] = S0^T . [W ; Q~]^T   (A = S0^T from TMEM, B read MN-major)
//   M4  (Q~ S0 + P U)^T += U^T . P^T
//   M5  X^T = (Diag(em) S0)^T + U^T . (k E^-1)        (the Gram's B tile, read MN-major)
//
// Precision: an fp32 quantity x enters an MMA as x = hi + lo (two bf16,
// round-to-nearest), and a product X.Y is formed as hi.hi + hi.lo + lo.hi
// (fp32 accumulation); V is exact in bf16 and enters once.
//
// Warp roles.  Only M3 .. M5 depend on the state; everything before them
// depends on the chunk's inputs alone.  Warps 4-11 (the prep group) therefore
// build chunk c+1's operands (decay, [k E ; q E], k E^-1 and Q~, the Gram, the
// triangular solve, Tb) while warps 0-3 (the chain group) run chunk c: the U~
// and W' products, W, and the state-dependent products.  The operands of a
// chunk live in one of two slots (shared-memory tiles); the groups hand slots
// over with mbarriers ("full" prep -> chain, "empty" chain -> prep, "v free"
// chain -> prep once M2 has read the slot's v tile), and every wait is bounded
// in time.
//
// Layer mode (kLayer): the same kernel also runs one whole KDA layer core
// ("Kimi K3 · KDA layer", KDA equation list) with nothing but the layer's inputs
// and outputs crossing HBM.  The prep group computes the front end from the raw
// pre-convolution q^p, k^p, v^p tiles: the width-4 causal short convolution
// (the three previous tokens come from an 8-row TMA box; zero before the
// sequence start), SiLU, the per-head L2 normalisation of q and k, log alpha =
// -5 sigmoid(e^A (z + b)) and beta = sigmoid(beta_logit).  v is then fp32, so it
// enters M2 as hi + lo like every other operand.  The chain group's readout
// applies the output gate sigmoid(g) * RMSNorm(o~) per (token, head) row.
#include <atomic>
#include <cuda.h>
#include <cstring>
#include <cudaTypedefs.h>

#include "kda_common.cuh"
#include "tc_primitives.cuh"

namespace kda {
namespace {
using namespace tc;

constexpr int kC = 32;
constexpr int kThreads = 384;  // chain group: warps 0-3, prep group: warps 4-11
constexpr uint64_t kWaitNs = 2000000000ull;  // bound on every wait
constexpr int kMaxOrderedSeqs = 64;  // longest-first CTA order for up to this many sequences

// ---- shared memory map (bytes from a 1024-aligned base) --------------------
// q, k, v tiles (bf16 [32][128], two 64-column blocks with 128-byte swizzle, as
// written by TMA) for two chunks.  log_alpha travels through registers.
constexpr uint32_t S_QKV = 0, QKV_SIZE = 24576, QO = 0, KO = 8192, VO = 16384;
// Tb by slot (32 rows, K = 32: hi in K steps 0-1, lo in K steps 2-3 of one swizzled
// tile), built by the prep group and read by the chain group's M2 / M2b; A (fp32
// [32][32], column-major) for the prep group's solve; T by slot (fp32 [32][33]).
constexpr uint32_t S_DT = 2 * QKV_SIZE;
constexpr uint32_t S_TB = S_DT, TB_SIZE = 4096;
constexpr uint32_t S_A = S_DT + 2 * TB_SIZE;
constexpr uint32_t S_TS = S_A + 4096;
constexpr int kLdT = 33;
constexpr uint32_t T_SIZE = 32 * kLdT * 4;
// [k E ; q E] hi | lo (64 rows), private to the prep group.
constexpr uint32_t S_WX = (S_TS + 2 * T_SIZE + 1023) & ~1023u;
// Per slot: [W ; Q~]^T hi | lo, key-channel major (128 rows j of 64 elements: W[., j] in
// elements 0-31, Q~[., j] in 32-63; elements 0-31 hold (k E)^T until W replaces them), so
// that M3 reads it MN-major and M2b reads (k E)^T K-major,
// R = k E^-1 hi | lo (32 rows), P (32 rows, K = 32: hi in K steps 0-1, lo in 2-3).
constexpr uint32_t S_WQ = S_WX + 32768, WQ_SIZE = 32768;
constexpr uint32_t S_R = S_WQ + 2 * WQ_SIZE, R_SIZE = 16384;
constexpr uint32_t S_P = S_R + 2 * R_SIZE, P_SIZE = 4096;
constexpr uint32_t S_STG = S_P + 2 * P_SIZE;  // bf16 output staging [32][128]; layer mode: g tile
constexpr uint32_t S_VEC = S_STG + 8192;      // em[2][128], e31p[2][128], e31[2][128]
constexpr uint32_t S_BETA = S_VEC + 3072;     // beta [2][32]
// Layer mode: conv history (q^p, k^p, v^p rows t0-8 .. t0-1: three [8][128] bf16
// swizzled tiles) and the gate's row reductions.
constexpr uint32_t S_HIST = (S_BETA + 256 + 1023) & ~1023u;
constexpr uint32_t S_GATE = S_HIST + 3 * 2048;  // [4 warps][32 rows] partials, then [32] 1/rms
constexpr uint32_t S_BAR = S_GATE + 640;
constexpr uint32_t S_TSLOT = S_BAR + 128;
constexpr uint32_t SM_DYN = S_TSLOT + 16 + 1024;  // + alignment slack
static_assert(SM_DYN <= 232448, "shared memory map exceeds 227 KB");
// M1 reads 128 rows of the 64-row [k E ; q E] tile (rows 64-127 are ignored):
// what follows the tile must still be inside the map.
static_assert(S_WX + 32768 + 8192 <= S_STG, "M1's A view leaves the map");

// mbarriers (8 bytes each, from S_BAR)
constexpr int B_TQKV = 0;   // [2] TMA q/k/v by slot
constexpr int B_CA = 2, B_CB = 3, B_PA = 4, B_PB = 5;  // MMA completion, one per issuer
constexpr int B_FULL = 6;   // [2] prep -> chain: slot holds a chunk's operands
constexpr int B_EMPTY = 8;  // [2] chain -> prep: slot consumed
constexpr int B_VFREE = 10; // [2] chain -> prep: M2 has read the slot's v tile
constexpr int B_TG = 12;    // layer mode: TMA of the chunk's g tile (chain group)
constexpr int kNumBars = 13;

// ---- TMEM column map (512 columns) -----------------------------------------
constexpr uint32_t TM_ST = 0;    // state X^T (lane c, column j), fp32
constexpr uint32_t TM_OPS = 128; // M3's A operand S0^T hi (64) | lo (64); then U^T hi (16) | lo (16)
constexpr uint32_t TM_D3A = 256; // M3 [(W S0)^T | (Q~ S0)^T (+ M4)]: K steps 0-3 (prefill),
                                 // the hi.hi and lo.hi products (layer mode)
constexpr uint32_t TM_D3B = 320; // M3: K steps 4-7 (prefill), the hi.lo products (layer mode)
constexpr uint32_t TM_DG = 384;  // Gram, K steps 0-3
constexpr uint32_t TM_DU = 416;  // Gram, K steps 4-7
constexpr uint32_t TM_UT = 448;  // U~^T (32 columns)
constexpr uint32_t TM_WT = 480;  // W'^T (lane = key channel j, column = row r)

// Threads with a fixed job.
constexpr int kCA = 0, kCB = 32;            // chain-group MMA issuers
constexpr int kPA = 128, kPB = 160;         // prep-group MMA issuers
constexpr int kTmaThread = 192;             // prep-group TMA issuer
constexpr int kChainBar = 1, kPrepBar = 2;  // named barriers
constexpr int kChainThreads = 128, kPrepThreads = 256;

// Swizzled [rows][128 bf16] operand tile with `rows` rows: two 64-column blocks
// of rows x 128 bytes, 16-byte chunk j of row i at chunk position j ^ (i % 8).
__device__ __forceinline__ uint32_t tile_chunk(int rows, int i, int cc) {
    return (uint32_t)((cc >> 3) * rows * 128 + i * 128 + (((cc & 7) ^ (i & 7)) << 4));
}
struct Params {
    CUtensorMap tm_q, tm_k, tm_v;     // [T][H*128] bf16 with boxes of 32 tokens x 64 channels
    CUtensorMap tm_qh, tm_kh, tm_vh;  // layer mode: the same tensors, boxes of 8 tokens
    CUtensorMap tm_g;                 // layer mode: g [T][H*128] bf16, boxes of 32 tokens x 128
    const float *log_alpha, *beta, *S0;
    const int32_t *cu_seqlens;
    int H;
    float scale;
    void *o;
    float *S_final;
    DeviceStatus status;
    // layer mode (front end and output gate fused)
    const __nv_bfloat16 *z, *beta_logit, *g;
    const float *conv_w, *A, *b;
    float l2_eps, rms_eps;
    Checkpoints ckpt;  // read only by the instantiation that takes snapshots
    // Test-only fault injection, read only by the debug library (KDA_DEBUG): the prep group
    // skips its first "slot full" hand-off, and every wait gives up after wait_ns.
    int32_t skip_first_full;
    uint64_t wait_ns;
};

// 1 / (1 + 2^(-x log2 e)) on the SFU: ex2.approx and rcp.approx, each within about
// 2^-22 relative; tends to 0 (not NaN) for x -> -inf.
__device__ __forceinline__ float sigmoid_(float x) {
    const float e = ex2_approx(-1.4426950408889634f * x);
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + e));
    return r;
}
// log(1 + e^x) on the SFU (ex2.approx, lg2.approx: about 2^-22 relative); above 20 it equals x to
// fp32 precision, and where e^x is below half an ulp of 1 it returns 0 (alpha = 1 to within
// 6e-8).  Kimi Linear's decay gate.
__device__ __forceinline__ float softplus_(float x) {
    if (x > 20.f) return x;
    float l;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l) : "f"(1.f + ex2_approx(1.4426950408889634f * x)));
    return 0.6931471805599453f * l;
}
__device__ __forceinline__ void bf16x4_to_f32(uint2 u, float (&x)[4]) {
    x[0] = __uint_as_float(u.x << 16);
    x[1] = __uint_as_float(u.x & 0xFFFF0000u);
    x[2] = __uint_as_float(u.y << 16);
    x[3] = __uint_as_float(u.y & 0xFFFF0000u);
}

// Store 8 fp32 values as a hi 16-byte chunk and a lo 16-byte chunk; with lo_first the lo
// chunk is stored by the first of the two instructions.
__device__ __forceinline__ void store_split_chunk(unsigned char *hi, unsigned char *lo,
                                                  const float (&x)[8], bool lo_first = false) {
    uint4 h, l;
    split2(x[0], x[1], h.x, l.x);
    split2(x[2], x[3], h.y, l.y);
    split2(x[4], x[5], h.z, l.z);
    split2(x[6], x[7], h.w, l.w);
    *reinterpret_cast<uint4 *>(lo_first ? lo : hi) = lo_first ? l : h;
    *reinterpret_cast<uint4 *>(lo_first ? hi : lo) = lo_first ? h : l;
}

// Elements e0 .. e0 + 3 (e0 % 4 == 0) of row j of a key-channel-major [128][64] bf16 tile
// (128-byte swizzle), as hi and lo halves.
__device__ __forceinline__ void store_t4(unsigned char *tile, int j, int e0, const float (&v)[4]) {
    uint2 h, l;
    split2(v[0], v[1], h.x, l.x);
    split2(v[2], v[3], h.y, l.y);
    const uint32_t o = (uint32_t)(j * 128 + ((((e0 >> 3) ^ (j & 7))) << 4) + (e0 & 4) * 2);
    *reinterpret_cast<uint2 *>(tile + o) = h;
    *reinterpret_cast<uint2 *>(tile + 16384 + o) = l;
}

// ---- group synchronisation (128-thread named barriers) ----------------------
__device__ __forceinline__ int group_size(int id) {
    return id == kChainBar ? kChainThreads : kPrepThreads;
}
__device__ __forceinline__ void group_sync(int id) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(group_size(id)) : "memory");
}
// Barrier over the group that also ANDs a predicate across it.
__device__ __forceinline__ bool group_and(int id, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(group_size(id))
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Bounded wait by one thread; a timeout is recorded with `where`.
__device__ __forceinline__ bool wait_one(uint64_t *bar, uint32_t parity, const Params &p,
                                         uint32_t where) {
#ifdef KDA_DEBUG
    const uint64_t limit = p.wait_ns;
#else
    const uint64_t limit = kWaitNs;
#endif
    const bool ok = mbar_wait_bounded(bar, parity, limit);
    if (!ok) record_status(p.status, KDA_ERR_DEVICE_TIMEOUT, where);
    return ok;
}
// Operand writes (generic-proxy smem stores and tcgen05.st) -> visible to an MMA
// issued by a thread of the same group after this barrier.
__device__ __forceinline__ void publish(int id) {
    tmem_wait_st();
    fence_proxy_async_smem();
    fence_before_sync();
    group_sync(id);
    fence_after_sync();
}

// Stage chunk [t0, t0 + 32) of head h: q/k/v into slot `slot` (TMA, one
// thread), beta by threads pt < 32 (cp.async, zero past nrow).  Rows past the
// sequence end are not masked here: log_alpha is zero and beta is zero there,
// which keeps those rows out of every product (see the kernel).
template <bool kLayer>
__device__ __forceinline__ void issue_loads(const Params &p, unsigned char *sm, uint64_t *bar,
                                            int slot, int t0, int nrow, int h, int tid,
                                            bool history) {
    if (tid == kTmaThread) {
        fence_proxy_async_smem();  // earlier generic accesses to these buffers come first
        unsigned char *qkv = sm + S_QKV + slot * QKV_SIZE;
        const bool hist = kLayer && history;
        mbar_arrive_expect_tx(bar + B_TQKV + slot, 6 * 4096 + (hist ? 6 * 1024 : 0));
        if (hist) {  // tokens t0-8 .. t0-1 (t0 - 8 >= 0: history is loaded only inside a sequence)
            const CUtensorMap *hm[3] = {&p.tm_qh, &p.tm_kh, &p.tm_vh};
#pragma unroll
            for (int a = 0; a < 3; ++a)
#pragma unroll
                for (int b = 0; b < 2; ++b)
                    tma_load_2d(smem_u32(sm + S_HIST + 2048 * a + 1024 * b), hm[a], h * kD + 64 * b,
                                t0 - 8, bar + B_TQKV + slot);
        }
        const CUtensorMap *maps[3] = {&p.tm_q, &p.tm_k, &p.tm_v};
        const uint32_t dst[3] = {QO, KO, VO};
#pragma unroll
        for (int a = 0; a < 3; ++a)
#pragma unroll
            for (int b = 0; b < 2; ++b)
                tma_load_2d(smem_u32(qkv + dst[a] + 4096 * b), maps[a], h * kD + 64 * b, t0,
                            bar + B_TQKV + slot);
    }
    const int pt = tid - 128;
    if (!kLayer && pt >= 0 && pt < kC) {
        const bool ok = pt < nrow;
        const float *s = ok ? p.beta + (size_t)(t0 + pt) * p.H + h : p.beta;
        cp_async4(smem_u32(sm + S_BETA + 128 * slot + 4 * pt), s, ok ? 4u : 0u);
        cp_async_commit();
    }
}

// log_alpha of chunk [t0, t0 + 32): rows 4 rg .. 4 rg + 3, channels 4 q4 .. 4 q4 + 3
// (rows past nrow zero).  kHeadDecay: log_alpha is [T][H], one decay per (token, head)
// shared by all channels (the Gated DeltaNet case), broadcast here.
template <bool kHeadDecay>
__device__ __forceinline__ void load_log_alpha(const Params &p, int t0, int nrow, int h, int q4,
                                               int rg, float4 (&la)[4]) {
    if constexpr (kHeadDecay) {
        const float *src = p.log_alpha + (size_t)t0 * p.H + h;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int r = 4 * rg + k;
            const float x = r < nrow ? __ldg(src + (size_t)r * p.H) : 0.f;
            la[k] = make_float4(x, x, x, x);
        }
    } else {
        const float *src = p.log_alpha + ((size_t)t0 * p.H + h) * kD + 4 * q4;
        const size_t stride = (size_t)p.H * kD;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int r = 4 * rg + k;
            la[k] = r < nrow ? __ldg(reinterpret_cast<const float4 *>(src + r * stride))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
}

// Layer mode: z of rows 4 rg .. 4 rg + 3, channels 4 q4 .. 4 q4 + 3 (zero past nrow), and
// beta_logit of row pt for pt < 32.
__device__ __forceinline__ void load_gate_inputs(const Params &p, int t0, int nrow, int h, int q4,
                                                 int rg, int pt, uint2 (&z)[4], uint32_t &bl) {
    const __nv_bfloat16 *src = p.z + ((size_t)t0 * p.H + h) * kD + 4 * q4;
    const size_t stride = (size_t)p.H * kD;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int r = 4 * rg + k;
        z[k] = r < nrow ? __ldg(reinterpret_cast<const uint2 *>(src + r * stride)) : make_uint2(0, 0);
    }
    bl = 0;
    if (pt < kC && pt < nrow)
        bl = __bfloat16_as_ushort(p.beta_logit[(size_t)(t0 + pt) * p.H + h]);
}

// ============================================================================
// Prep group (warps 4-11, 256 threads): operands of every chunk, in order.
// ============================================================================
template <bool kLayer, bool kHeadDecay, bool kUnb>
__device__ __forceinline__ void prep_group(const Params &p, unsigned char *sm, uint32_t tb,
                                           int h, int t_begin, int t_end, int nchunks) {
    const int tid = threadIdx.x, pt = tid - 128, lane = tid & 31;
    const int quarter = (pt >> 5) & 3, half = pt >> 7;  // TMEM lane quarter; second warp of it
    const uint32_t tl = tb + ((uint32_t)(32 * quarter) << 16);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + S_BAR);
    float *vec = reinterpret_cast<float *>(sm + S_VEC);
    float *sAt = reinterpret_cast<float *>(sm + S_A);  // A^T: sAt[i * 32 + r] = A[r][i]
    float *sT_base = reinterpret_cast<float *>(sm + S_TS);
    unsigned char *wx = sm + S_WX;
    // Decay pass layout: channels 4 q4 .. 4 q4 + 3, rows 4 rg .. 4 rg + 3; the
    // eight row groups of a channel quad sit in lanes (lane & 3) + 4 rg of a warp.
    const int q4 = 4 * (pt >> 5) + (lane & 3), rg = lane >> 2;
    float4 e31_prev = make_float4(1.f, 1.f, 1.f, 1.f);  // 1: the entering state is exact
    uint32_t ph = 0;   // MMA barrier phase (PA and PB)
    int consumed = 0;  // chunks whose q/k/v were waited for
    int issued = 0;    // chunks whose q/k/v loads were issued
    bool alive = true;
    float4 la[4];      // log_alpha of the next chunk (this thread's 4 rows x 4 channels)
    uint2 zr[4];       // layer mode: z of the next chunk (same rows and channels)
    uint32_t bl = 0;   // layer mode: beta_logit of row pt of the next chunk (bf16 bits)
    float eA = 0.f;    // layer mode: e^{A_h}
    float4 bb = make_float4(0.f, 0.f, 0.f, 0.f);  // layer mode: b[h][4 q4 ..]
    if constexpr (kLayer) {
        eA = expf(p.A[h]);
        if (p.b != nullptr) bb = *reinterpret_cast<const float4 *>(p.b + (size_t)h * kD + 4 * q4);
    }

    if (nchunks > 0) {
        const int n0 = min(kC, t_end - t_begin);
        issue_loads<kLayer>(p, sm, bar, 0, t_begin, n0, h, tid, false);
        issued = 1;
        if constexpr (kLayer) load_gate_inputs(p, t_begin, n0, h, q4, rg, pt, zr, bl);
        else load_log_alpha<kHeadDecay>(p, t_begin, n0, h, q4, rg, la);
    }

    for (int c = 0; c < nchunks; ++c) {
        const int s = c & 1;
        const int t0 = t_begin + kC * c;
        const int nrow = min(kC, t_end - t0);
        const unsigned char *qkv = sm + S_QKV + s * QKV_SIZE;
        const float *beta_s = reinterpret_cast<const float *>(sm + S_BETA + 128 * s);
        unsigned char *wq = sm + S_WQ + s * WQ_SIZE;
        unsigned char *rr = sm + S_R + s * R_SIZE;
        unsigned char *pp = sm + S_P + s * P_SIZE;
        float *em_s = vec + s * kD, *e31p_s = vec + 2 * kD + s * kD, *e31_s = vec + 4 * kD + s * kD;
        float *sT = sT_base + s * (32 * kLdT);
        // kUnb: the chunk takes the tensor-core form (every decay factor in range) or is handed
        // to the chain group to run token by token
        bool fast = true, in_range = true;

        // ---- slot s free again (chunk c-2 finished); chunk c's inputs landed ----
        {
            bool ok = true;
            if (tid == kPA && c >= 2)
                ok = wait_one(bar + B_EMPTY + s, ((c >> 1) - 1) & 1, p, 10);
            if (tid == kTmaThread) ok = wait_one(bar + B_TQKV + s, (c >> 1) & 1, p, 11);
            if (pt < kC) cp_async_wait_all();
            if constexpr (kLayer) {  // beta = sigmoid(beta_logit); rows past the end write nothing
                if (pt < kC)
                    const_cast<float *>(beta_s)[pt] =
                        pt < nrow ? sigmoid_(__uint_as_float(bl << 16)) : 0.f;
            }
            alive = group_and(kPrepBar, ok);
            fence_after_sync();
            if (!alive) break;
            consumed = c + 1;
        }

        // ---- F2/F3: decay and operands, thread = 4 rows x 4 channels (4 q4 .. 4 q4 + 3).
        //      D (log2 units): rows 0..15 prefix - prefix_15, rows 16..31 the sum of rows
        //      16..r (two scan segments of 4 row groups).  Then [k E ; q E] -> wx and
        //      R = k E^-1 -> rr (the Gram's operands) ----
        {
            const int cc = q4 >> 1, hb = (q4 & 1) * 8;
            float qh[4][4], kh[4][4];  // layer mode: q^, k^ of rows 4 rg + k
            if constexpr (kLayer) {
                // ---- front end: short conv + SiLU for q^p, k^p, v^p ----
                float y[3][4][4];
#pragma unroll
                for (int X = 0; X < 3; ++X) {
                    const unsigned char *tile = qkv + (X == 0 ? QO : X == 1 ? KO : VO);
                    const unsigned char *hist = sm + S_HIST + 2048 * X;
                    const float *wsrc = p.conv_w + (((size_t)X * p.H + h) * kD + 4 * q4) * 4;
                    float4 w4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) w4[e] = __ldg(reinterpret_cast<const float4 *>(wsrc) + e);
                    float raw[7][4];  // rows 4 rg - 3 .. 4 rg + 3
#pragma unroll
                    for (int lr = 0; lr < 7; ++lr) {
                        const int row = 4 * rg - 3 + lr;
                        uint2 u = make_uint2(0, 0);
                        if (row >= 0)
                            u = *reinterpret_cast<const uint2 *>(tile + tile_chunk(32, row, cc) + hb);
                        else if (c > 0)  // previous tokens of this sequence; zero before its start
                            u = *reinterpret_cast<const uint2 *>(hist + tile_chunk(8, 8 + row, cc) + hb);
                        bf16x4_to_f32(u, raw[lr]);
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            // tap j multiplies token t - j (tap 0: the current token)
                            float a = w4[e].x * raw[k + 3][e];
                            a = fmaf(w4[e].y, raw[k + 2][e], a);
                            a = fmaf(w4[e].z, raw[k + 1][e], a);
                            a = fmaf(w4[e].w, raw[k][e], a);
                            y[X][k][e] = a * sigmoid_(a);
                        }
                }
                // ---- L2 norms of q and k per (token, head) row: 4 lanes, then 8 warps ----
                // [2][32 rows][8 warps]; A is not in use here.  Warp w's partial of row r sits in
                // word w ^ rg of the row, so that the eight row groups storing at once hit eight
                // banks; a row's reader sums all eight words, in either half order.
                float* part = sAt;
                float ss[2][4];
#pragma unroll
                for (int X = 0; X < 2; ++X)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        float v = y[X][k][0] * y[X][k][0];
                        v = fmaf(y[X][k][1], y[X][k][1], v);
                        v = fmaf(y[X][k][2], y[X][k][2], v);
                        v = fmaf(y[X][k][3], y[X][k][3], v);
                        v += __shfl_xor_sync(0xffffffffu, v, 1);
                        v += __shfl_xor_sync(0xffffffffu, v, 2);
                        ss[X][k] = v;
                    }
                if ((lane & 3) == 0) {
#pragma unroll
                    for (int X = 0; X < 2; ++X)
#pragma unroll
                        for (int k = 0; k < 4; ++k) part[(X * 32 + 4 * rg + k) * 8 + ((pt >> 5) ^ rg)] = ss[X][k];
                }
                group_sync(kPrepBar);  // partials complete; every raw tile read is done
#pragma unroll
                for (int X = 0; X < 2; ++X)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        // odd row groups read the upper half first (rows 4 apart share banks)
                        const float *row = part + (X * 32 + 4 * rg + k) * 8;
                        const float4 a = *reinterpret_cast<const float4 *>(row + 4 * (rg & 1));
                        const float4 b = *reinterpret_cast<const float4 *>(row + 4 * ((rg & 1) ^ 1));
                        const float inv = rsqrtf(((a.x + a.y) + (a.z + a.w)) + ((b.x + b.y) + (b.z + b.w)) + p.l2_eps);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            if (X == 0) qh[k][e] = y[0][k][e] * inv;
                            else kh[k][e] = y[1][k][e] * inv;
                        }
                    }
                // ---- v (fp32) -> V hi over the v^p tile, V lo over the q^p tile ----
#pragma unroll
                for (int k = 0; k < 4; ++k) {  // rows in the order of F2/F3 (bank groups)
                    const bool sw = (rg & 2) != 0;
                    const int r = 4 * rg + (k ^ (rg & 2));
                    float vv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) vv[e] = sw ? y[2][k ^ 2][e] : y[2][k][e];
                    uint2 h2, l2;
                    split2(vv[0], vv[1], h2.x, l2.x);
                    split2(vv[2], vv[3], h2.y, l2.y);
                    unsigned char *qkvw = const_cast<unsigned char *>(qkv);
                    *reinterpret_cast<uint2 *>(qkvw + VO + tile_chunk(32, r, cc) + hb) = h2;
                    *reinterpret_cast<uint2 *>(qkvw + QO + tile_chunk(32, r, cc) + hb) = l2;
                }
                // ---- log alpha = -5 sigmoid(e^A (z + b)), or with kUnb Kimi Linear's
                //      -e^A softplus(z + b) (rows past the end: 0) ----
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float zf[4];
                    bf16x4_to_f32(zr[k], zf);
                    const bool in = 4 * rg + k < nrow;
                    if constexpr (kUnb) {
                        la[k].x = in ? -eA * softplus_(zf[0] + bb.x) : 0.f;
                        la[k].y = in ? -eA * softplus_(zf[1] + bb.y) : 0.f;
                        la[k].z = in ? -eA * softplus_(zf[2] + bb.z) : 0.f;
                        la[k].w = in ? -eA * softplus_(zf[3] + bb.w) : 0.f;
                    } else {
                        la[k].x = in ? -5.f * sigmoid_(eA * (zf[0] + bb.x)) : 0.f;
                        la[k].y = in ? -5.f * sigmoid_(eA * (zf[1] + bb.y)) : 0.f;
                        la[k].z = in ? -5.f * sigmoid_(eA * (zf[2] + bb.z)) : 0.f;
                        la[k].w = in ? -5.f * sigmoid_(eA * (zf[3] + bb.w)) : 0.f;
                    }
                }
            }
            const float kL2E = 1.4426950408889634f;
            float4 pre[4];
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                acc.x = fmaf(la[k].x, kL2E, acc.x);
                acc.y = fmaf(la[k].y, kL2E, acc.y);
                acc.z = fmaf(la[k].z, kL2E, acc.z);
                acc.w = fmaf(la[k].w, kL2E, acc.w);
                pre[k] = acc;
            }
            float4 incl = acc;  // inclusive scan over the row groups of the segment
#pragma unroll
            for (int d = 1; d <= 2; d <<= 1) {
                float4 y;
                y.x = __shfl_up_sync(0xffffffffu, incl.x, 4 * d);
                y.y = __shfl_up_sync(0xffffffffu, incl.y, 4 * d);
                y.z = __shfl_up_sync(0xffffffffu, incl.z, 4 * d);
                y.w = __shfl_up_sync(0xffffffffu, incl.w, 4 * d);
                if ((rg & 3) >= d) {
                    incl.x += y.x; incl.y += y.y; incl.z += y.z; incl.w += y.w;
                }
            }
            float4 mid, last;  // prefix_15 and the sum of rows 16..31
            mid.x = __shfl_sync(0xffffffffu, incl.x, 12 + (lane & 3));
            mid.y = __shfl_sync(0xffffffffu, incl.y, 12 + (lane & 3));
            mid.z = __shfl_sync(0xffffffffu, incl.z, 12 + (lane & 3));
            mid.w = __shfl_sync(0xffffffffu, incl.w, 12 + (lane & 3));
            last.x = __shfl_sync(0xffffffffu, incl.x, 28 + (lane & 3));
            last.y = __shfl_sync(0xffffffffu, incl.y, 28 + (lane & 3));
            last.z = __shfl_sync(0xffffffffu, incl.z, 28 + (lane & 3));
            last.w = __shfl_sync(0xffffffffu, incl.w, 28 + (lane & 3));
            // base = exclusive prefix of this row group, minus prefix_15 in the first segment
            float4 base;
            base.x = incl.x - acc.x - (rg < 4 ? mid.x : 0.f);
            base.y = incl.y - acc.y - (rg < 4 ? mid.y : 0.f);
            base.z = incl.z - acc.z - (rg < 4 ? mid.z : 0.f);
            base.w = incl.w - acc.w - (rg < 4 ? mid.w : 0.f);
            const float em4[4] = {ex2_approx(mid.x), ex2_approx(mid.y), ex2_approx(mid.z),
                                  ex2_approx(mid.w)};
            if constexpr (kUnb) {
                // Without the decay floor the chunk takes the tensor-core form only when every
                // factor 2^{+-D} stays inside 2^115 (about e^80, the range the floor guarantees);
                // otherwise (a decay of -inf included) the chain group runs it token by token.
                // Layer mode votes here, while the thread still holds q^, k^; with bf16 inputs
                // the vote rides on the operand pass's closing barrier instead.
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    in_range = in_range && fabsf(base.x + pre[k].x) <= 115.f &&
                               fabsf(base.y + pre[k].y) <= 115.f && fabsf(base.z + pre[k].z) <= 115.f &&
                               fabsf(base.w + pre[k].w) <= 115.f;
                if constexpr (kLayer) fast = group_and(kPrepBar, in_range);
            }
            if (rg == 0) {
                // a chunk run token by token leaves the state unscaled: e31 = 1
                const float4 e31 = fast ? make_float4(ex2_approx(last.x), ex2_approx(last.y),
                                                      ex2_approx(last.z), ex2_approx(last.w))
                                        : make_float4(1.f, 1.f, 1.f, 1.f);
                *reinterpret_cast<float4 *>(em_s + 4 * q4) =
                    make_float4(em4[0], em4[1], em4[2], em4[3]);
                *reinterpret_cast<float4 *>(e31p_s + 4 * q4) = e31_prev;
                *reinterpret_cast<float4 *>(e31_s + 4 * q4) = e31;
                e31_prev = e31;
            }
            // Row order: threads with bit 1 of rg set take their rows in the order 2, 3, 0, 1,
            // so that the four rows a half-warp stores at once (8-byte accesses are served a
            // half-warp at a time) fall in four distinct 32-byte bank groups of the swizzled tile.
            if (kUnb && kLayer && !fast) {
                // Out of range (layer mode): raw q^, k^ (fp32) into slot s's [W ; Q~] tile and
                // alpha (fp32; row 0 times the entering state's scale e31) into its R tile,
                // [32][128] each, for the chain group's token-by-token pass.  Nothing else of the
                // chunk is built.  (bf16 inputs write the same after the pass's closing vote.)
                float *kf = reinterpret_cast<float *>(wq), *qf = kf + kC * kD;
                float *af = reinterpret_cast<float *>(rr);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r = 4 * rg + k;
                    float kv[4], qv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        kv[e] = kh[k][e];
                        qv[e] = qh[k][e];
                    }
                    float4 al4 = make_float4(ex2_approx(la[k].x * kL2E), ex2_approx(la[k].y * kL2E),
                                             ex2_approx(la[k].z * kL2E), ex2_approx(la[k].w * kL2E));
                    if (r == 0) {  // the entering state's scale, stored above by this thread
                        const float4 ep = *reinterpret_cast<const float4 *>(e31p_s + 4 * q4);
                        al4.x *= ep.x; al4.y *= ep.y; al4.z *= ep.z; al4.w *= ep.w;
                    }
                    *reinterpret_cast<float4 *>(kf + r * kD + 4 * q4) = make_float4(kv[0], kv[1], kv[2], kv[3]);
                    *reinterpret_cast<float4 *>(qf + r * kD + 4 * q4) = make_float4(qv[0], qv[1], qv[2], qv[3]);
                    *reinterpret_cast<float4 *>(af + r * kD + 4 * q4) = al4;
                }
            } else {
            float kT[4][4];  // bf16 inputs: k E by channel t and loop step k
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const bool sw = (rg & 2) != 0;
                const int kk = k ^ (rg & 2);
                const int r = 4 * rg + kk;
                const float4 pk = sw ? pre[k ^ 2] : pre[k];
                const float dv[4] = {base.x + pk.x, base.y + pk.y, base.z + pk.z, base.w + pk.w};
                float kv[4], qv[4];
                if constexpr (kLayer) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        kv[e] = sw ? kh[k ^ 2][e] : kh[k][e];
                        qv[e] = sw ? qh[k ^ 2][e] : qh[k][e];
                    }
                } else {
                    bf16x4_to_f32(*reinterpret_cast<const uint2 *>(qkv + KO + tile_chunk(32, r, cc) + hb), kv);
                    bf16x4_to_f32(*reinterpret_cast<const uint2 *>(qkv + QO + tile_chunk(32, r, cc) + hb), qv);
                }
                float xk[4], xq[4], xr[4];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float E = ex2_approx(dv[t]), EI = ex2_approx(-dv[t]);
                    xk[t] = kv[t] * E;    // k E
                    xq[t] = qv[t] * E;    // q E
                    xr[t] = kv[t] * EI;   // k E^-1
                    if constexpr (!kLayer && !kUnb) kT[t][k] = xk[t];
                }
                uint2 h2, l2;
                split2(xk[0], xk[1], h2.x, l2.x);
                split2(xk[2], xk[3], h2.y, l2.y);
                unsigned char *dst = wx + tile_chunk(64, r, cc) + hb;
                *reinterpret_cast<uint2 *>(dst) = h2;
                *reinterpret_cast<uint2 *>(dst + 16384) = l2;
                split2(xq[0], xq[1], h2.x, l2.x);
                split2(xq[2], xq[3], h2.y, l2.y);
                dst = wx + tile_chunk(64, 32 + r, cc) + hb;
                *reinterpret_cast<uint2 *>(dst) = h2;
                *reinterpret_cast<uint2 *>(dst + 16384) = l2;
                split2(xr[0], xr[1], h2.x, l2.x);
                split2(xr[2], xr[3], h2.y, l2.y);
                dst = rr + tile_chunk(32, r, cc) + hb;
                *reinterpret_cast<uint2 *>(dst) = h2;
                *reinterpret_cast<uint2 *>(dst + 8192) = l2;
            }
            if constexpr (!kLayer && !kUnb) {
                // (k E)^T -> wq elements 4 rg .. 4 rg + 3 of rows j = 4 q4 + t (M2b's A operand;
                // layer mode and the unbounded variant write it during the Gram instead, where it
                // costs no registers here)
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const bool sw = (rg & 2) != 0;
                    const float v[4] = {sw ? kT[t][2] : kT[t][0], sw ? kT[t][3] : kT[t][1],
                                        sw ? kT[t][0] : kT[t][2], sw ? kT[t][1] : kT[t][3]};
                    store_t4(wq, 4 * q4 + t, 4 * rg, v);
                }
            }
            }
        }
        if (c + 1 < nchunks) {
            if constexpr (kLayer) load_gate_inputs(p, t0 + kC, min(kC, t_end - t0 - kC), h, q4, rg, pt, zr, bl);
            else load_log_alpha<kHeadDecay>(p, t0 + kC, min(kC, t_end - t0 - kC), h, q4, rg, la);
        }
        if constexpr (kUnb && !kLayer) {
            // the range vote on the closing barrier; an out-of-range chunk then replaces what the
            // pass wrote for the tensor-core form by raw k, q and alpha (log alpha read again)
            tmem_wait_st();
            fence_proxy_async_smem();
            fence_before_sync();
            fast = group_and(kPrepBar, in_range);
            fence_after_sync();
            if (!fast) {
                const int cc = q4 >> 1, hb = (q4 & 1) * 8;
                float4 lac[4];
                load_log_alpha<false>(p, t0, nrow, h, q4, rg, lac);
                float *kf = reinterpret_cast<float *>(wq), *qf = kf + kC * kD;
                float *af = reinterpret_cast<float *>(rr);
                const float4 ep = *reinterpret_cast<const float4 *>(e31p_s + 4 * q4);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r = 4 * rg + k;
                    float kv[4], qv[4];
                    bf16x4_to_f32(*reinterpret_cast<const uint2 *>(qkv + KO + tile_chunk(32, r, cc) + hb), kv);
                    bf16x4_to_f32(*reinterpret_cast<const uint2 *>(qkv + QO + tile_chunk(32, r, cc) + hb), qv);
                    const float kL2E = 1.4426950408889634f;
                    float4 al4 = make_float4(ex2_approx(lac[k].x * kL2E), ex2_approx(lac[k].y * kL2E),
                                             ex2_approx(lac[k].z * kL2E), ex2_approx(lac[k].w * kL2E));
                    if (r == 0) { al4.x *= ep.x; al4.y *= ep.y; al4.z *= ep.z; al4.w *= ep.w; }
                    *reinterpret_cast<float4 *>(kf + r * kD + 4 * q4) = make_float4(kv[0], kv[1], kv[2], kv[3]);
                    *reinterpret_cast<float4 *>(qf + r * kD + 4 * q4) = make_float4(qv[0], qv[1], qv[2], qv[3]);
                    *reinterpret_cast<float4 *>(af + r * kD + 4 * q4) = al4;
                }
                if (rg == 0) {  // the chunk leaves the state unscaled
                    *reinterpret_cast<float4 *>(e31_s + 4 * q4) = make_float4(1.f, 1.f, 1.f, 1.f);
                    e31_prev = make_float4(1.f, 1.f, 1.f, 1.f);
                }
            }
        } else {
            publish(kPrepBar);
        }
        if (c + 1 < nchunks) {  // stage chunk c+1 into slot s^1 once chunk c-1 no longer needs it
            bool ok = true;
            if (tid == kTmaThread && c >= 1)
                ok = wait_one(bar + B_VFREE + (s ^ 1), ((c - 1) >> 1) & 1, p, 12);
            alive = group_and(kPrepBar, ok);
            if (!alive) break;
            issue_loads<kLayer>(p, sm, bar, s ^ 1, t0 + kC, min(kC, t_end - t0 - kC), h, tid, true);
            issued = c + 2;
        }
        // Gram, solve and Tb: the tensor-core form only (a chunk run token by token needs none)
        if (!kUnb || fast) {
            if (tid == kPA || tid == kPB) {  // M1: Gram, K steps split over the two issuers
                // M = 64 ([k E ; q E] has 64 rows): D row m lands in TMEM lane 32 (m / 16) + m % 16
                const uint32_t id = idesc_bf16_f32(64, 32);
                const int s0 = tid == kPA ? 0 : 4;
                const uint32_t d = tb + (tid == kPA ? TM_DG : TM_DU);
                const uint32_t xh = smem_u32(wx), xl = xh + 16384;
                const uint32_t rh = smem_u32(rr), rl = rh + 8192;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16(d, sw128_desc_k(xh, 64, s0 + k), sw128_desc_k(rh, 32, s0 + k), id, k > 0);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16(d, sw128_desc_k(xh, 64, s0 + k), sw128_desc_k(rl, 32, s0 + k), id, 1);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16(d, sw128_desc_k(xl, 64, s0 + k), sw128_desc_k(rh, 32, s0 + k), id, 1);
                mma_commit(bar + (tid == kPA ? B_PA : B_PB));
            }
            // ---- while M1 runs: Q~ = (q E) em, rebuilt from its hi + lo in wx (the Gram only reads
            //      wx) -> wq elements 32 + r of rows j; layer mode also (k E)^T -> elements r of rows
            //      j (M2b's A operand), the hi and lo words of wx's k rows transposed 4 x 4 ----
            {
                const int cc = q4 >> 1, hb = (q4 & 1) * 8;
                const float4 em4 = *reinterpret_cast<const float4 *>(em_s + 4 * q4);
                float qT[4][4];  // Q~ by channel t and loop step k (row 4 rg + (k ^ (rg & 2)))
                uint2 kw[2][4];  // k E hi / lo words by loop step k
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r = 4 * rg + (k ^ (rg & 2));  // the row order of F2/F3
                    const uint32_t oq = tile_chunk(64, 32 + r, cc) + hb;
                    const uint32_t ok2 = tile_chunk(64, r, cc) + hb;
                    if constexpr (kLayer || kUnb) {
                        kw[0][k] = *reinterpret_cast<const uint2 *>(wx + ok2);
                        kw[1][k] = *reinterpret_cast<const uint2 *>(wx + 16384 + ok2);
                    }
                    float qh4[4], ql4[4];
                    bf16x4_to_f32(*reinterpret_cast<const uint2 *>(wx + oq), qh4);
                    bf16x4_to_f32(*reinterpret_cast<const uint2 *>(wx + 16384 + oq), ql4);
                    qT[0][k] = (qh4[0] + ql4[0]) * em4.x;
                    qT[1][k] = (qh4[1] + ql4[1]) * em4.y;
                    qT[2][k] = (qh4[2] + ql4[2]) * em4.z;
                    qT[3][k] = (qh4[3] + ql4[3]) * em4.w;
                }
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const bool sw = (rg & 2) != 0;
                    const float v[4] = {sw ? qT[t][2] : qT[t][0], sw ? qT[t][3] : qT[t][1],
                                        sw ? qT[t][0] : qT[t][2], sw ? qT[t][1] : qT[t][3]};
                    store_t4(wq, 4 * q4 + t, 32 + 4 * rg, v);
                }
                const bool sw = (rg & 2) != 0;
#pragma unroll
                for (int hl = 0; hl < ((kLayer || kUnb) ? 2 : 0); ++hl) {
                    // rows 4 rg .. 4 rg + 3 in order
                    const uint2 a = sw ? kw[hl][2] : kw[hl][0], b = sw ? kw[hl][3] : kw[hl][1];
                    const uint2 c2 = sw ? kw[hl][0] : kw[hl][2], d = sw ? kw[hl][1] : kw[hl][3];
                    const int e0 = 4 * rg;
#pragma unroll
                    for (int t = 0; t < 4; ++t) {  // channel 4 q4 + t: 16-bit half t & 1 of word t >> 1
                        const uint32_t sel = (t & 1) ? 0x7632u : 0x5410u;
                        const uint32_t wa = (t >> 1) ? a.y : a.x, wb = (t >> 1) ? b.y : b.x;
                        const uint32_t wc = (t >> 1) ? c2.y : c2.x, wd = (t >> 1) ? d.y : d.x;
                        const int j = 4 * q4 + t;
                        const uint32_t o = (uint32_t)(j * 128 + ((((e0 >> 3) ^ (j & 7))) << 4) + (e0 & 4) * 2);
                        *reinterpret_cast<uint2 *>(wq + 16384 * hl + o) =
                            make_uint2(__byte_perm(wa, wb, sel), __byte_perm(wc, wd, sel));
                    }
                }
            }
            {
                bool ok = true;
                if (tid == kPA || tid == kPB)
                    ok = wait_one(bar + (tid == kPA ? B_PA : B_PB), ph & 1, p, 13);
                ++ph;
                alive = group_and(kPrepBar, ok);
                fence_after_sync();
                if (!alive) break;
            }

            // ---- F5: A (k rows, scaled by beta, strictly lower; stored column-major) and
            //      P (q rows, lower).  The M = 64 Gram holds its rows in lanes 0-15 of each lane
            //      quarter: quarters 0-1 the k rows 0-15 / 16-31, quarters 2-3 the q rows; each of
            //      the two warps of a quarter takes 16 columns ----
            {
                float g[16], g2[16];
                tmem_ld16(tl + TM_DG + 16 * half, g);
                tmem_ld16(tl + TM_DU + 16 * half, g2);
                const int r = 16 * (quarter & 1) + lane;
                if (lane >= 16) {
                    // lanes 16-31 of each quarter hold no Gram rows
                } else if (quarter < 2) {
                    const float br = beta_s[r];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int i = 16 * half + e;
                        sAt[i * 32 + r] = i < r ? br * (g[e] + g2[e]) : 0.f;
                    }
                } else {
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {
                        float x[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int i = 16 * half + 8 * c2 + e;
                            x[e] = i <= r ? g[8 * c2 + e] + g2[8 * c2 + e] : 0.f;
                        }
                        store_split_chunk(pp + sw128_chunk_offset(32, r, 2 * half + c2),
                                          pp + sw128_chunk_offset(32, r, 4 + 2 * half + c2), x);
                    }
                }
            }
            group_sync(kPrepBar);

            // ---- F6: T = (I + A)^-1.  One warp inverts both 16 x 16 diagonal blocks by
            //      forward substitution (lane = column: lanes 0-15 the upper block, 16-31 the
            //      lower), then T_10 = -T_11 (A_10 T_00) with one entry per thread, then
            //      T goes to slot s for the chain group ----
            if (pt < 32) {
                const int o = 16 * (lane >> 4), j = lane & 15;
                float x[16];
#pragma unroll
                for (int m = 0; m < 16; ++m) x[m] = m == j ? 1.f : 0.f;
#pragma unroll
                for (int i = 0; i < 15; ++i) {
                    float a[16];  // column o + i of A, rows o .. o + 15
#pragma unroll
                    for (int q = (i + 1) >> 2; q < 4; ++q) {
                        const float4 v = *reinterpret_cast<const float4 *>(sAt + (o + i) * 32 + o + 4 * q);
                        a[4 * q] = v.x; a[4 * q + 1] = v.y; a[4 * q + 2] = v.z; a[4 * q + 3] = v.w;
                    }
#pragma unroll
                    for (int m = i + 1; m < 16; ++m) x[m] = fmaf(-a[m], x[i], x[m]);
                }
#pragma unroll
                for (int m = 0; m < 16; ++m) sT[(o + m) * kLdT + o + j] = x[m];
            }
            group_sync(kPrepBar);
            if constexpr (kLayer) {
                // Layer mode: this group sets the pace there, so the chain group forms T_10 and
                // Tb itself; A_10 goes to T's upper-right block (which T never uses) for it.
                const int r = pt >> 4, m = pt & 15;
                sT[r * kLdT + 16 + m] = sAt[m * 32 + 16 + r];
            } else {
                {  // 32 x 32: T_10 = -T_11 (A_10 T_00), one entry per thread (row 16 + r, column i)
                    const int r = pt >> 4, i = pt & 15;
                    float x0 = 0.f, x1 = 0.f;
#pragma unroll
                    for (int m = 0; m < 16; m += 2) {
                        x0 = fmaf(sAt[m * 32 + 16 + r], sT[m * kLdT + i], x0);
                        x1 = fmaf(sAt[(m + 1) * 32 + 16 + r], sT[(m + 1) * kLdT + i], x1);
                    }
                    // X = A_10 T_00 (row r, column i) goes to T's upper-right block, which T never uses
                    sT[r * kLdT + 16 + i] = x0 + x1;
                    group_sync(kPrepBar);
                    float y0 = 0.f, y1 = 0.f;
#pragma unroll
                    for (int m = 0; m < 16; m += 2) {
                        y0 = fmaf(sT[(16 + r) * kLdT + 16 + m], sT[m * kLdT + 16 + i], y0);
                        y1 = fmaf(sT[(16 + r) * kLdT + 17 + m], sT[(m + 1) * kLdT + 16 + i], y1);
                    }
                    sT[(16 + r) * kLdT + i] = -(y0 + y1);
                }
                group_sync(kPrepBar);
                // ---- Tb = T diag(beta) (32 rows x K 32) -> slot s: one 16-byte chunk per thread ----
                if (pt < 128) {
                    const int r = pt >> 2, cc = pt & 3;
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int i = 8 * cc + e;
                        x[e] = i <= r ? sT[r * kLdT + i] * beta_s[i] : 0.f;
                    }
                    // a quarter-warp holds rows r and r + 1: odd rows store their lo chunk first, so
                    // that each instruction's 8 chunks fall in 8 distinct 16-byte bank groups
                    unsigned char *tbs = sm + S_TB + s * TB_SIZE;
                    store_split_chunk(tbs + sw128_chunk_offset(32, r, cc), tbs + sw128_chunk_offset(32, r, 4 + cc),
                                      x, (r & 1) != 0);
                }
            }
        }
        if constexpr (kUnb) {
            if (tid == kPA) reinterpret_cast<int *>(sm + S_TSLOT + 8)[s] = fast ? 0 : 1;
        }
        fence_proxy_async_smem();  // wq, P and Tb are MMA operands of the chain group
        group_sync(kPrepBar);
#ifdef KDA_DEBUG
        if (tid == kPA && !(p.skip_first_full && c == 0)) mbar_arrive(bar + B_FULL + s);
#else
        if (tid == kPA) mbar_arrive(bar + B_FULL + s);
#endif
    }

    if (pt < kC) cp_async_wait_all();  // nothing may still be in flight into shared memory
    if (!alive && tid == kTmaThread) {  // let outstanding TMA loads land before leaving
        for (int c = consumed; c < issued; ++c)
            mbar_wait_bounded(bar + B_TQKV + (c & 1), (c >> 1) & 1, kWaitNs);
    }
}

// ============================================================================
// Chain group (warps 0-3): the state-dependent products, chunk by chunk.
// ============================================================================
template <bool B>
struct BoolTag {
    static constexpr bool value = B;
};

// Snapshot slot for the state after `done` tokens of a sequence whose slots are
// [base, base + count) (head h), or null when `done` is not a positive multiple of the
// interval or the sequence has no slot for it.
__device__ __forceinline__ float *snapshot_dst(const Params &p, int base, int count, int h,
                                               int done) {
    if (done <= 0 || done % p.ckpt.every != 0) return nullptr;
    const int k = done / p.ckpt.every - 1;
    if (k >= count) return nullptr;
    return p.ckpt.states + ((size_t)(base + k) * p.H + h) * (size_t)(kD * kD);
}

// A chunk out of the tensor-core range (kUnb), run token by token on column c_lane of the
// state (TMEM lane c_lane): S <- Diag(alpha_t) S, r = S^T k_t, u = beta_t (v_t - r),
// S <- S + k_t u, then S^T q_t (unscaled) into the readout accumulator's TMEM column t.  Out of
// line, so that the tensor-core loop keeps its code size.
template <bool kLayer>
__device__ __noinline__ void token_by_token_chunk(unsigned char *sm, uint32_t tl, int s, int nrow,
                                                   int c_lane) {
    const unsigned char *wq = sm + S_WQ + s * WQ_SIZE, *rr = sm + S_R + s * R_SIZE;
    const unsigned char *qkv = sm + S_QKV + s * QKV_SIZE;
    const float *kf = reinterpret_cast<const float *>(wq), *qf = kf + kC * kD;
    const float *af = reinterpret_cast<const float *>(rr);
    const float *beta_c = reinterpret_cast<const float *>(sm + S_BETA + 128 * s);
    for (int t = 0; t < nrow; ++t) {
        const float *at = af + t * kD, *kt = kf + t * kD, *qt = qf + t * kD;
        // v_t[c] (bf16 tile; layer mode: hi in the v^p tile, lo in the q^p tile's place)
        const uint32_t vo = tile_chunk(32, t, c_lane >> 3) + (c_lane & 7) * 2;
        float vc = __uint_as_float((uint32_t)*reinterpret_cast<const unsigned short *>(qkv + VO + vo) << 16);
        if constexpr (kLayer)
            vc += __uint_as_float((uint32_t)*reinterpret_cast<const unsigned short *>(qkv + QO + vo) << 16);
        float r4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int part = 0; part < 4; ++part) {  // decay and prediction
            float sv[32];
            uint32_t st[32];
            tmem_ld32(tl + TM_ST + 32 * part, sv);
#pragma unroll
            for (int jj = 0; jj < 32; jj += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(at + 32 * part + jj);
                const float4 k4 = *reinterpret_cast<const float4 *>(kt + 32 * part + jj);
                const float av[4] = {a4.x, a4.y, a4.z, a4.w}, kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float x = sv[jj + e] * av[e];
                    r4[e] = fmaf(x, kv[e], r4[e]);
                    st[jj + e] = __float_as_uint(x);
                }
            }
            tmem_st32(tl + TM_ST + 32 * part, st);
        }
        tmem_wait_st();
        const float u = beta_c[t] * (vc - ((r4[0] + r4[1]) + (r4[2] + r4[3])));
        float o4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int part = 0; part < 4; ++part) {  // delta write and readout
            float sv[32];
            uint32_t st[32];
            tmem_ld32(tl + TM_ST + 32 * part, sv);
#pragma unroll
            for (int jj = 0; jj < 32; jj += 4) {
                const float4 k4 = *reinterpret_cast<const float4 *>(kt + 32 * part + jj);
                const float4 q4 = *reinterpret_cast<const float4 *>(qt + 32 * part + jj);
                const float kv[4] = {k4.x, k4.y, k4.z, k4.w}, qv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float x = fmaf(kv[e], u, sv[jj + e]);
                    o4[e] = fmaf(x, qv[e], o4[e]);
                    st[jj + e] = __float_as_uint(x);
                }
            }
            tmem_st32(tl + TM_ST + 32 * part, st);
        }
        tmem_st1u(tl + TM_D3A + 32 + t,
                  __float_as_uint((o4[0] + o4[1]) + (o4[2] + o4[3])));
        tmem_wait_st();
    }
}

template <typename Tout, bool kLayer, bool kCkpt, bool kUnb>
__device__ __forceinline__ void chain_group(const Params &p, unsigned char *sm, uint32_t tb,
                                            int h, int n, int t_begin, int t_end, int nchunks) {
    const int tid = threadIdx.x, warp = tid >> 5;
    const int c_lane = tid;  // TMEM lane = value channel
    const uint32_t tl = tb + ((uint32_t)(32 * warp) << 16);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + S_BAR);
    const float *vec = reinterpret_cast<const float *>(sm + S_VEC);
    const int H = p.H;
    const size_t state_off = ((size_t)n * H + h) * (size_t)(kD * kD);
    Tout *o = static_cast<Tout *>(p.o);
    uint32_t ph = 0;  // MMA barrier phase (CA and CB)
    bool alive = true;
    int snap_base = 0, snap_count = 0;  // this sequence's snapshot slots
    if constexpr (kCkpt) {
        snap_base = p.ckpt.base[n];
        snap_count = p.ckpt.base[n + 1] - snap_base;
    }

    // ---- entering state -> TMEM, transposed (lane c, column j) ----
#pragma unroll
    for (int part = 0; part < 4; ++part) {
        uint32_t w[32];
        const int j0 = 32 * part;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj)
            w[jj] = p.S0 ? __float_as_uint(p.S0[state_off + (size_t)(j0 + jj) * kD + c_lane]) : 0u;
        tmem_st32(tl + TM_ST + j0, w);
    }
    tmem_wait_st();

    // Layer mode: the chunk's g tile arrives by TMA in the staging buffer's place
    // (the gated output is stored directly); chunk c+1's tile is requested once
    // chunk c's readout has read its own.
    int g_issued = 0;
    auto issue_g = [&](int t0g) {
        if (tid == 0) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar + B_TG, kC * kD * 2);
            tma_load_2d(smem_u32(sm + S_STG), &p.tm_g, h * kD, t0g, bar + B_TG);
        }
    };
    if constexpr (kLayer) {
        if (nchunks > 0) {
            issue_g(t_begin);
            g_issued = 1;
        }
    }

    // bf16 output: a finished chunk is staged row-major in shared memory and
    // copied out with 16-byte stores while the next chunk's M3 runs.
    __nv_bfloat16 *stg = reinterpret_cast<__nv_bfloat16 *>(sm + S_STG);
    int pend_t0 = 0, pend_rows = 0;
    auto copy_out = [&]() {  // warps 2-3 (warps 0-1 issue M3 meanwhile)
        if (tid < 64) return;
        for (int e = tid - 64; e < kC * 16; e += 64) {
            const int r = e >> 4, chn = e & 15;
            if (r < pend_rows)
                *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(o) +
                                           ((size_t)(pend_t0 + r) * H + h) * kD + 8 * chn) =
                    *reinterpret_cast<const uint4 *>(stg + r * kD + 8 * chn);
        }
        pend_rows = 0;
    };

    for (int c = 0; c < nchunks; ++c) {
        const int s = c & 1;
        const int t0 = t_begin + kC * c;
        const int nrow = min(kC, t_end - t0);
        unsigned char *wq = sm + S_WQ + s * WQ_SIZE;
        const unsigned char *rr = sm + S_R + s * R_SIZE;
        const unsigned char *pp = sm + S_P + s * P_SIZE;
        const unsigned char *qkv = sm + S_QKV + s * QKV_SIZE;
        const float *em = vec + s * kD;

        // ---- the prep group has filled slot s ----
        {
            bool ok = true;
            if (tid == 0) ok = wait_one(bar + B_FULL + s, (c >> 1) & 1, p, 20);
            alive = group_and(kChainBar, ok);
            fence_after_sync();
            if (!alive) break;
        }

        // kUnb: a chunk out of the tensor-core range runs token by token on the state in TMEM
        const bool fb = kUnb && reinterpret_cast<const int *>(sm + S_TSLOT + 8)[s] != 0;
        if (fb) {
            // The recurrence itself, token by token, on column c_lane of the state (TMEM lane
            // c_lane): S <- Diag(alpha_t) S, r = S^T k_t, u = beta_t (v_t - r), S <- S + k_t u,
            // o~ = scale S^T q_t.  The prep group left raw k, q and alpha (fp32, [32][128]) in the
            // slot's [W ; Q~] and R tiles, alpha of row 0 times the entering state's scale, so the
            // state comes out unscaled (the prep group set this chunk's e31 to 1).  Exact for any
            // decay, alpha = 0 included.  Each token's S^T q_t goes to the readout accumulator's
            // TMEM column (its partner columns zero), so the readout below serves both forms.
            if constexpr (sizeof(Tout) == 2 && !kLayer) copy_out();  // the previous chunk's rows
            {
                uint32_t zero[32];
#pragma unroll
                for (int r = 0; r < 32; ++r) zero[r] = 0u;
                tmem_st32(tl + TM_D3A + 32, zero);
                tmem_st32(tl + TM_D3B + 32, zero);
            }
            token_by_token_chunk<kLayer>(sm, tl, s, nrow, c_lane);
            // every thread is done with slot s: its v tile and its operand tiles go back
            fence_before_sync();
            group_sync(kChainBar);
            fence_after_sync();
            if (tid == 0) {
                mbar_arrive(bar + B_VFREE + s);
                mbar_arrive(bar + B_EMPTY + s);
            }
        } else {
        if constexpr (kLayer) {
            // ---- layer mode: T_10 = -T_11 (A_10 T_00) and Tb = T diag(beta) for slot s, here
            //      (the prep group, the slower one in layer mode, left T_00, T_11 and A_10 in the
            //      slot's T: A_10 in the upper-right block, which T never uses) ----
            float *sTs = reinterpret_cast<float *>(sm + S_TS) + s * (32 * kLdT);
            const float *beta_s = reinterpret_cast<const float *>(sm + S_BETA + 128 * s);
            const int r = tid >> 4, i = tid & 15;  // entries (r, i) and (r + 8, i)
            float x[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {  // X = A_10 T_00
                const int rr = r + 8 * hh;
                float x0 = 0.f, x1 = 0.f;
#pragma unroll
                for (int m = 0; m < 16; m += 2) {
                    x0 = fmaf(sTs[rr * kLdT + 16 + m], sTs[m * kLdT + i], x0);
                    x1 = fmaf(sTs[rr * kLdT + 17 + m], sTs[(m + 1) * kLdT + i], x1);
                }
                x[hh] = x0 + x1;
            }
            group_sync(kChainBar);  // every read of A_10 is done: X goes in its place
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) sTs[(r + 8 * hh) * kLdT + 16 + i] = x[hh];
            group_sync(kChainBar);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {  // T_10 = -T_11 X
                const int rr = r + 8 * hh;
                float y0 = 0.f, y1 = 0.f;
#pragma unroll
                for (int m = 0; m < 16; m += 2) {
                    y0 = fmaf(sTs[(16 + rr) * kLdT + 16 + m], sTs[m * kLdT + 16 + i], y0);
                    y1 = fmaf(sTs[(16 + rr) * kLdT + 17 + m], sTs[(m + 1) * kLdT + 16 + i], y1);
                }
                sTs[(16 + rr) * kLdT + i] = -(y0 + y1);
            }
            group_sync(kChainBar);
            {  // Tb (32 rows x K 32) -> slot s: one 16-byte chunk per thread
                const int r2 = tid >> 2, cc = tid & 3;
                float xb[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int i2 = 8 * cc + e;
                    xb[e] = i2 <= r2 ? sTs[r2 * kLdT + i2] * beta_s[i2] : 0.f;
                }
                unsigned char *tbs = sm + S_TB + s * TB_SIZE;
                store_split_chunk(tbs + sw128_chunk_offset(32, r2, cc),
                                  tbs + sw128_chunk_offset(32, r2, 4 + cc), xb, (r2 & 1) != 0);
            }
            fence_proxy_async_smem();  // Tb is M2's and M2b's operand
            group_sync(kChainBar);
        }
        // (Tb, W's k E and Q~ came with the slot: the prep group published them)
        if (tid == kCA) {  // M2: U~^T = V^T Tb^T  (V read MN-major: exact bf16, or hi + lo)
            const uint32_t th = smem_u32(sm + S_TB + s * TB_SIZE);
            const uint32_t idv = idesc_bf16_f32(128, 32) | kIdescAMN;
            const uint32_t va = smem_u32(qkv + VO);
#pragma unroll
            for (int k = 0; k < 2; ++k)
                mma_bf16(tb + TM_UT, sw128_desc_mn(va + 2048 * k, 4096), sw128_desc_k(th, 32, k), idv,
                         k > 0);
#pragma unroll
            for (int k = 0; k < 2; ++k)
                mma_bf16(tb + TM_UT, sw128_desc_mn(va + 2048 * k, 4096), sw128_desc_k(th, 32, 2 + k), idv,
                         1);
            if constexpr (kLayer) {  // V lo (in the q^p tile's place)
                const uint32_t vl = smem_u32(qkv + QO);
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    mma_bf16(tb + TM_UT, sw128_desc_mn(vl + 2048 * k, 4096), sw128_desc_k(th, 32, k), idv,
                             1);
            }
            mma_commit(bar + B_CA);
        } else if (tid == kCB) {  // M2b: W'^T = (k E)^T Tb^T, (k E)^T (wq elements 0-31) K-major
            const uint32_t th = smem_u32(sm + S_TB + s * TB_SIZE);
            const uint32_t idw = idesc_bf16_f32(128, 32);
            const uint32_t xh = smem_u32(wq), xl = xh + 16384;
#pragma unroll
            for (int k = 0; k < 2; ++k)
                mma_bf16(tb + TM_WT, sw128_desc_k(xh, 128, k), sw128_desc_k(th, 32, k), idw, k > 0);
#pragma unroll
            for (int k = 0; k < 2; ++k)
                mma_bf16(tb + TM_WT, sw128_desc_k(xh, 128, k), sw128_desc_k(th, 32, 2 + k), idw, 1);
#pragma unroll
            for (int k = 0; k < 2; ++k)
                mma_bf16(tb + TM_WT, sw128_desc_k(xl, 128, k), sw128_desc_k(th, 32, k), idw, 1);
            mma_commit(bar + B_CB);
        }

        // ---- F4 (while M2 and M2b run): S0 = Diag(e31_prev) X -> M3's A operand (hi | lo);
        //      X <- Diag(em) S0.  After the first quarter each issuer waits for its own
        //      products, and M2's issuer releases slot s's v tile, so that the prep group can
        //      stage the chunk after next early ----
        bool m2_ok = true;
        {
            const float *e31p = vec + 2 * kD + s * kD;
            auto f4 = [&](auto with_snapshot, float *snap) {
                constexpr bool kSnap = decltype(with_snapshot)::value;
                // the state's columns 32 part .. 32 part + 31; the next part's load is in flight
                // while this part is split and stored
                uint32_t sr[2][32];
                tmem_ld32_async(tl + TM_ST, sr[0]);
                tmem_ld_wait32(sr[0]);
#pragma unroll
                for (int part = 0; part < 4; ++part) {
                    if (part < 3) tmem_ld32_async(tl + TM_ST + 32 * (part + 1), sr[(part + 1) & 1]);
                    if (part == 1 && (tid == kCA || tid == kCB)) {
                        m2_ok = wait_one(bar + (tid == kCA ? B_CA : B_CB), ph & 1, p, 24);
                        if (m2_ok && tid == kCA) mbar_arrive(bar + B_VFREE + s);
                    }
                    const int j0 = 32 * part;
                    float sv[32];
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) sv[jj] = __uint_as_float(sr[part & 1][jj]);
                    uint32_t hw[16], lw[16], yv[32];
#pragma unroll
                    for (int jj = 0; jj < 32; jj += 4) {
                        const float4 ep = *reinterpret_cast<const float4 *>(e31p + j0 + jj);
                        const float4 mm = *reinterpret_cast<const float4 *>(em + j0 + jj);
                        const float2 a = mul2(make_float2(sv[jj], sv[jj + 1]), make_float2(ep.x, ep.y));
                        const float2 b =
                            mul2(make_float2(sv[jj + 2], sv[jj + 3]), make_float2(ep.z, ep.w));
                        split2(a.x, a.y, hw[jj >> 1], lw[jj >> 1]);
                        split2(b.x, b.y, hw[(jj >> 1) + 1], lw[(jj >> 1) + 1]);
                        if constexpr (kSnap) {
                            float *d = snap + (size_t)(j0 + jj) * kD + c_lane;
                            d[0] = a.x; d[kD] = a.y; d[2 * kD] = b.x; d[3 * kD] = b.y;
                        }
                        const float2 ya = mul2(a, make_float2(mm.x, mm.y));
                        const float2 yb = mul2(b, make_float2(mm.z, mm.w));
                        yv[jj] = __float_as_uint(ya.x);
                        yv[jj + 1] = __float_as_uint(ya.y);
                        yv[jj + 2] = __float_as_uint(yb.x);
                        yv[jj + 3] = __float_as_uint(yb.y);
                    }
                    tmem_st16u(tl + TM_OPS + (j0 >> 1), hw);
                    tmem_st16u(tl + TM_OPS + 64 + (j0 >> 1), lw);
                    tmem_st32(tl + TM_ST + j0, yv);
                    if (part < 3) tmem_ld_wait32(sr[(part + 1) & 1]);
                }
            };
            // Layer mode keeps this loop rolled: its larger code (the front end) makes
            // instruction fetch the tighter limit there (measured: 45.2 ms against 46.0 ms per
            // step on the layer workload); the prefill unrolls it and keeps the next part's TMEM
            // load in flight (1.14 ms against 1.22 ms).
            auto f4_rolled = [&](auto with_snapshot, float *snap) {
                constexpr bool kSnap = decltype(with_snapshot)::value;
#pragma unroll 1
                for (int part = 0; part < 4; ++part) {
                    if (part == 1 && (tid == kCA || tid == kCB)) {
                        m2_ok = wait_one(bar + (tid == kCA ? B_CA : B_CB), ph & 1, p, 24);
                        if (m2_ok && tid == kCA) mbar_arrive(bar + B_VFREE + s);
                    }
                    const int j0 = 32 * part;
                    float sv[32];
                    tmem_ld32(tl + TM_ST + j0, sv);
                    uint32_t hw[16], lw[16], yv[32];
#pragma unroll
                    for (int jj = 0; jj < 32; jj += 4) {
                        const float4 ep = *reinterpret_cast<const float4 *>(e31p + j0 + jj);
                        const float4 mm = *reinterpret_cast<const float4 *>(em + j0 + jj);
                        const float2 a = mul2(make_float2(sv[jj], sv[jj + 1]), make_float2(ep.x, ep.y));
                        const float2 b =
                            mul2(make_float2(sv[jj + 2], sv[jj + 3]), make_float2(ep.z, ep.w));
                        split2(a.x, a.y, hw[jj >> 1], lw[jj >> 1]);
                        split2(b.x, b.y, hw[(jj >> 1) + 1], lw[(jj >> 1) + 1]);
                        if constexpr (kSnap) {
                            float *d = snap + (size_t)(j0 + jj) * kD + c_lane;
                            d[0] = a.x; d[kD] = a.y; d[2 * kD] = b.x; d[3 * kD] = b.y;
                        }
                        const float2 ya = mul2(a, make_float2(mm.x, mm.y));
                        const float2 yb = mul2(b, make_float2(mm.z, mm.w));
                        yv[jj] = __float_as_uint(ya.x);
                        yv[jj + 1] = __float_as_uint(ya.y);
                        yv[jj + 2] = __float_as_uint(yb.x);
                        yv[jj + 3] = __float_as_uint(yb.y);
                    }
                    tmem_st16u(tl + TM_OPS + (j0 >> 1), hw);
                    tmem_st16u(tl + TM_OPS + 64 + (j0 >> 1), lw);
                    tmem_st32(tl + TM_ST + j0, yv);
                }
            };
            // The entering state S0 is the state after kC c tokens: a snapshot when that is a
            // multiple of the interval (F4 computes S0 in fp32 anyway).  Chunks without one
            // run the loop without the stores.
            float *snap = nullptr;
            if constexpr (kCkpt) snap = snapshot_dst(p, snap_base, snap_count, h, kC * c);
            if constexpr (kLayer) {
                if (kCkpt && snap != nullptr)
                    f4_rolled(BoolTag<true>{}, snap);
                else
                    f4_rolled(BoolTag<false>{}, nullptr);
            } else {
                if (kCkpt && snap != nullptr)
                    f4(BoolTag<true>{}, snap);
                else
                    f4(BoolTag<false>{}, nullptr);
            }
        }
        // ---- M2 and M2b done (W'^T is read next) ----
        {
            ++ph;
            alive = group_and(kChainBar, m2_ok);
            fence_after_sync();
            if (!alive) break;
        }
        // ---- F7: W = W' Diag(em) -> wq elements 0-31 of row j ((k E)^T is dead); thread = key
        //      channel j, four 16-byte chunks per half ----
        {
            const int j = tid;
            float w[32];
            tmem_ld32(tl + TM_WT, w);
            const float emj = em[j];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = w[8 * q + e] * emj;
                const uint32_t o = (uint32_t)(j * 128 + ((q ^ (j & 7)) << 4));
                store_split_chunk(wq + o, wq + 16384 + o, x);
            }
        }
        publish(kChainBar);
        // M3: [(W S0)^T | (Q~ S0)^T] = S0^T [W ; Q~]^T ([W ; Q~] read MN-major: K step k = rows
        // 16 k .. 16 k + 15 of the key-channel-major tile).  The tensor pipe shares its slots
        // among the threads issuing at once, and M3 runs while the prep group issues its Gram
        // from two threads.  The prefill, where this group sets the pace, issues M3 from two
        // threads too (K steps 0-3 -> D3A, 4-7 -> D3B, three products of N = 64 each).  Layer
        // mode, where the prep group sets it, issues M3 from one thread as 16 MMAs: S0 hi .
        // [B hi | B lo] (N = 128 through the descriptor's second 64-element block, 16 KB on) into
        // D3A (hi.hi) and D3B (hi.lo), then S0 lo . B hi (N = 64) onto D3A; fewer, wider MMAs
        // and a larger share of the pipe for the Gram.  Either way the U split and the readout
        // read D3A + D3B.
        if constexpr (kLayer) {
            if (tid == kCA) {
                const uint32_t id128 = idesc_bf16_f32(128, 128) | kIdescBMN;
                const uint32_t id64 = idesc_bf16_f32(128, 64) | kIdescBMN;
                const uint32_t bh = smem_u32(wq);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint64_t bd = sw128_desc_mn(bh + 2048 * k, 16384);
                    mma_bf16_tmem_a(tb + TM_D3A, tb + TM_OPS + 8 * k, bd, id128, k > 0);
                    mma_bf16_tmem_a(tb + TM_D3A, tb + TM_OPS + 64 + 8 * k, bd, id64, 1);
                }
                mma_commit(bar + B_CA);
            } else if (tid == kCB) {
                mma_commit(bar + B_CB);  // (no products: keeps B_CB at one phase per product group)
            }
        } else if (tid == kCA || tid == kCB) {
            const uint32_t id = idesc_bf16_f32(128, 64) | kIdescBMN;
            const int s0 = tid == kCA ? 0 : 4;
            const uint32_t d = tb + (tid == kCA ? TM_D3A : TM_D3B);
            const uint32_t bh = smem_u32(wq), bl = bh + 16384;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16_tmem_a(d, tb + TM_OPS + 8 * (s0 + k), sw128_desc_mn(bh + 2048 * (s0 + k), 16384),
                                id, k > 0);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16_tmem_a(d, tb + TM_OPS + 8 * (s0 + k), sw128_desc_mn(bl + 2048 * (s0 + k), 16384),
                                id, 1);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16_tmem_a(d, tb + TM_OPS + 64 + 8 * (s0 + k),
                                sw128_desc_mn(bh + 2048 * (s0 + k), 16384), id, 1);
            mma_commit(bar + (tid == kCA ? B_CA : B_CB));
        }
        if constexpr (sizeof(Tout) == 2 && !kLayer) copy_out();  // previous chunk, while M3 runs
        {
            bool ok = true;
            if (tid == kCA || tid == kCB)
                ok = wait_one(bar + (tid == kCA ? B_CA : B_CB), ph & 1, p, 21);
            ++ph;
            alive = group_and(kChainBar, ok);
            fence_after_sync();
            if (!alive) break;
        }

        // ---- F8: U^T = U~^T - (W S0)^T -> A operand of M4 / M5 ----
        {
            float ut[32], a[32], b[32];
            tmem_ld32(tl + TM_UT, ut);
            tmem_ld32(tl + TM_D3A, a);
            tmem_ld32(tl + TM_D3B, b);
            uint32_t hw[16], lw[16];
#pragma unroll
            for (int q = 0; q < 16; ++q)
                split2(ut[2 * q] - (a[2 * q] + b[2 * q]), ut[2 * q + 1] - (a[2 * q + 1] + b[2 * q + 1]),
                       hw[q], lw[q]);
            tmem_st16u(tl + TM_OPS, hw);
            tmem_st16u(tl + TM_OPS + 16, lw);
        }
        publish(kChainBar);
        if (tid == kCA) {  // M4: (Q~ S0 + P U)^T += U^T P^T
            const uint32_t id32 = idesc_bf16_f32(128, 32);
            const uint32_t ph2 = smem_u32(pp);
#pragma unroll
            for (int k = 0; k < 2; ++k)
                mma_bf16_tmem_a(tb + TM_D3A + 32, tb + TM_OPS + 8 * k, sw128_desc_k(ph2, 32, k), id32, 1);
#pragma unroll
            for (int k = 0; k < 2; ++k)
                mma_bf16_tmem_a(tb + TM_D3A + 32, tb + TM_OPS + 8 * k, sw128_desc_k(ph2, 32, 2 + k), id32,
                                1);
#pragma unroll
            for (int k = 0; k < 2; ++k)
                mma_bf16_tmem_a(tb + TM_D3A + 32, tb + TM_OPS + 16 + 8 * k, sw128_desc_k(ph2, 32, k),
                                id32, 1);
            mma_commit(bar + B_CA);
        } else if (tid == kCB) {  // M5: X += U^T (k E^-1)  (R read MN-major)
            const uint32_t id128 = idesc_bf16_f32(128, 128) | kIdescBMN;
            const uint32_t rh = smem_u32(rr), rl = rh + 8192;
#pragma unroll
            for (int k = 0; k < 2; ++k)
                mma_bf16_tmem_a(tb + TM_ST, tb + TM_OPS + 8 * k, sw128_desc_mn(rh + 2048 * k, 4096),
                                id128, 1);
#pragma unroll
            for (int k = 0; k < 2; ++k)
                mma_bf16_tmem_a(tb + TM_ST, tb + TM_OPS + 8 * k, sw128_desc_mn(rl + 2048 * k, 4096),
                                id128, 1);
#pragma unroll
            for (int k = 0; k < 2; ++k)
                mma_bf16_tmem_a(tb + TM_ST, tb + TM_OPS + 16 + 8 * k,
                                sw128_desc_mn(rh + 2048 * k, 4096), id128, 1);
            mma_commit(bar + B_CB);
        }
        // ---- M4 and M5 done: hand slot s back, then read out o = scale (D3A + D3B)[:, 32:64] ----
        {
            bool ok = true;
            if (tid == kCA || tid == kCB)
                ok = wait_one(bar + (tid == kCA ? B_CA : B_CB), ph & 1, p, 22);
            ++ph;
            fence_before_sync();
            alive = group_and(kChainBar, ok);
            fence_after_sync();
            if (!alive) break;
            if (tid == 0) mbar_arrive(bar + B_EMPTY + s);
        }
        }  // the tensor-core form
        {
            float a[32], b[32];
            tmem_ld32(tl + TM_D3A + 32, a);
            tmem_ld32(tl + TM_D3B + 32, b);
#pragma unroll
            for (int r = 0; r < 32; ++r) a[r] = p.scale * (a[r] + b[r]);  // o~[t0 + r][c]
            if constexpr (kLayer) {
                // Output gate: o^g = sigmoid(g) o~ / sqrt(mean_c o~^2 + eps) per (token, head)
                // row.  Sum of squares over this warp's 32 channels for all 32 rows at once:
                // five halving steps leave lane l with row l's sum.
#pragma unroll
                for (int r = 0; r < 32; ++r) b[r] = a[r] * a[r];
#pragma unroll
                for (int o2 = 16; o2 >= 1; o2 >>= 1) {
                    const bool up = (c_lane & o2) != 0;
#pragma unroll
                    for (int i = 0; i < o2; ++i) {
                        const float keep = up ? b[i + o2] : b[i];
                        const float send = up ? b[i] : b[i + o2];
                        b[i] = keep + __shfl_xor_sync(0xffffffffu, send, o2);
                    }
                }
                float *gate = reinterpret_cast<float *>(sm + S_GATE);
                gate[warp * 32 + (c_lane & 31)] = b[0];
                bool ok = true;
                if (tid == 0) ok = wait_one(bar + B_TG, c & 1, p, 25);  // chunk c's g tile
                ok = group_and(kChainBar, ok);
                if (!ok) {
                    alive = false;
                    break;
                }
                if (tid < 32)
                    gate[128 + tid] = rsqrtf((gate[tid] + gate[32 + tid] + gate[64 + tid] + gate[96 + tid]) *
                                                 (1.f / kD) + p.rms_eps);
                group_sync(kChainBar);
                const unsigned short *gs = reinterpret_cast<const unsigned short *>(sm + S_STG);
#pragma unroll
                for (int r = 0; r < 32; ++r)
                    a[r] *= sigmoid_(__uint_as_float((uint32_t)gs[r * kD + c_lane] << 16)) * gate[128 + r];
                group_sync(kChainBar);  // every read of the g tile is done
                if constexpr (sizeof(Tout) == 2) {
                    // stage the gated rows in the g tile's place, then 16-byte stores
#pragma unroll
                    for (int r = 0; r < 32; ++r) stg[r * kD + c_lane] = __float2bfloat16_rn(a[r]);
                    group_sync(kChainBar);
                    for (int e = tid; e < kC * 16; e += 128) {
                        const int r = e >> 4, chn = e & 15;
                        if (r < nrow)
                            *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(o) +
                                                       ((size_t)(t0 + r) * H + h) * kD + 8 * chn) =
                                *reinterpret_cast<const uint4 *>(stg + r * kD + 8 * chn);
                    }
                    group_sync(kChainBar);  // the staged rows are out
                } else {
#pragma unroll
                    for (int r = 0; r < 32; ++r)
                        if (r < nrow) o[((size_t)(t0 + r) * H + h) * kD + c_lane] = a[r];
                }
                if (c + 1 < nchunks) {
                    issue_g(t0 + kC);
                    g_issued = c + 2;
                }
            } else if constexpr (sizeof(Tout) == 2) {
#pragma unroll
                for (int r = 0; r < 32; ++r) stg[r * kD + c_lane] = __float2bfloat16_rn(a[r]);
                pend_t0 = t0;
                pend_rows = nrow;
            } else {
#pragma unroll
                for (int r = 0; r < 32; ++r)
                    if (r < nrow) o[((size_t)(t0 + r) * H + h) * kD + c_lane] = a[r];
            }
        }
    }
    if constexpr (sizeof(Tout) == 2 && !kLayer) {
        if (alive) copy_out();
    }
    if constexpr (kLayer) {  // a g tile still in flight (only after an early exit) must land first
        if (tid == 0 && !alive && g_issued > 0)  // at most the last one is outstanding
            mbar_wait_bounded(bar + B_TG, (g_issued - 1) & 1, kWaitNs);
    }

    // ---- final state S = Diag(e31_last) X (lane c, column j) -> S_final[j][c], and the
    //      last snapshot when the sequence ends on one ----
    float *snap = nullptr;
    if constexpr (kCkpt) {
        if (nchunks > 0) snap = snapshot_dst(p, snap_base, snap_count, h, t_end - t_begin);
    }
    if (alive && (p.S_final != nullptr || snap != nullptr)) {
        const float *e31_last = vec + 4 * kD + ((nchunks - 1) & 1) * kD;
#pragma unroll
        for (int part = 0; part < 4; ++part) {
            const int j0 = 32 * part;
            float sv[32];
            tmem_ld32(tl + TM_ST + j0, sv);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const float x = nchunks > 0 ? sv[jj] * e31_last[j0 + jj] : sv[jj];
                if (p.S_final != nullptr) p.S_final[state_off + (size_t)(j0 + jj) * kD + c_lane] = x;
                if (kCkpt && snap != nullptr) snap[(size_t)(j0 + jj) * kD + c_lane] = x;
            }
        }
    }
}

template <typename Tout, bool kLayer, bool kCkpt, bool kHeadDecay, bool kUnb>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ Params p) {
    extern __shared__ unsigned char smem_raw[];
    // The map starts at the first 1024-byte boundary of the dynamic window (the swizzled
    // tiles need it).  The offset is added to the array itself, not through an integer
    // round trip, so that the compiler keeps every access in the shared address space
    // (32-bit shared loads and stores instead of generic ones).
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + S_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + S_TSLOT);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int H = p.H;
    const int h = blockIdx.x % H, r = blockIdx.x / H;
    // CTA r x H + h takes the r-th longest sequence (ties in index order): blocks start
    // roughly in index order, so the longest (sequence, head) units start in the first
    // wave and shorter ones fill in behind them.  Thread j < N ranks sequence j.
    const int nseq = gridDim.x / H;
    const bool ordered = nseq > 1 && nseq <= kMaxOrderedSeqs;
    int *nslot = reinterpret_cast<int *>(sm + S_TSLOT + 4);
    if (ordered && tid < nseq) {
        const int len = p.cu_seqlens[tid + 1] - p.cu_seqlens[tid];
        int rank = 0;
        for (int j = 0; j < nseq; ++j) {
            const int lj = p.cu_seqlens[j + 1] - p.cu_seqlens[j];
            rank += (lj > len || (lj == len && j < tid)) ? 1 : 0;
        }
        if (rank == r) *nslot = tid;  // ranks are a permutation: exactly one writer
    }

    if (warp == 0) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    if (tid == kTmaThread) {
        for (int i = 0; i < kNumBars; ++i) mbar_init(bar + i, 1);
        fence_mbar_init();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tb = *tslot;
    const int n = ordered ? *nslot : r;
    const int t_begin = p.cu_seqlens[n], t_end = p.cu_seqlens[n + 1];
    const int nchunks = t_end > t_begin ? (t_end - t_begin + kC - 1) / kC : 0;

    if (warp >= 4)
        prep_group<kLayer, kHeadDecay, kUnb>(p, sm, tb, h, t_begin, t_end, nchunks);
    else
        chain_group<Tout, kLayer, kCkpt, kUnb>(p, sm, tb, h, n, t_begin, t_end, nchunks);

    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

// The driver's tensor-map encoder, looked up once (a function-local static: thread-safe).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        return nullptr;
    }();
    return fn;
}

// [T][H*128] tensor, boxes of box_rows tokens x box_cols elements.
bool encode_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int elem_bytes, int T,
                int H, int box_cols, int box_rows, CUtensorMapSwizzle swz) {
    auto fn = tensor_map_encoder();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)H * kD, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)H * kD * elem_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_bf16_tiles(CUtensorMap *m, const void *base, int T, int H, int box_rows) {
    return encode_map(m, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, H, 64, box_rows,
                      CU_TENSOR_MAP_SWIZZLE_128B);
}

template <typename Tout, bool kLayer, bool kCkpt, bool kHeadDecay, bool kUnb = false>
cudaError_t launch_kernel(const Params &p, int num_seqs, int num_heads, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<Tout, kLayer, kCkpt, kHeadDecay, kUnb>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SM_DYN);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)num_seqs * (unsigned)num_heads;
    prefill_tc_kernel<Tout, kLayer, kCkpt, kHeadDecay, kUnb><<<grid, kThreads, SM_DYN, stream>>>(p);
    return cudaGetLastError();
}

// Snapshots and the per-head decay are separate instantiations: the kernel without them is
// compiled as if their code did not exist.
template <typename Tout, bool kLayer, bool kHeadDecay>
cudaError_t launch_params(const Params &p, int num_seqs, int num_heads, cudaStream_t stream) {
    if (p.ckpt.every > 0)
        return launch_kernel<Tout, kLayer, true, kHeadDecay>(p, num_seqs, num_heads, stream);
    return launch_kernel<Tout, kLayer, false, kHeadDecay>(p, num_seqs, num_heads, stream);
}

#ifdef KDA_DEBUG
// Armed by kda_debug_inject_handoff_timeout, consumed by the next prefill launch.
std::atomic<int> g_inject_handoff_timeout{0};
#endif

template <typename Tout>
cudaError_t launch_typed(const PrefillArgs &a, cudaStream_t stream) {
    Params p;
    memset(&p, 0, sizeof(p));
    p.wait_ns = kWaitNs;
#ifdef KDA_DEBUG
    if (g_inject_handoff_timeout.exchange(0) != 0) {
        p.skip_first_full = 1;
        p.wait_ns = 1000000ull;  // 1 ms
    }
#endif
    if (a.total_tokens > 0) {
        const int T = a.total_tokens, H = a.num_heads;
        if (!encode_bf16_tiles(&p.tm_q, a.q, T, H, kC) || !encode_bf16_tiles(&p.tm_k, a.k, T, H, kC) ||
            !encode_bf16_tiles(&p.tm_v, a.v, T, H, kC))
            return cudaErrorInvalidValue;
    }
    p.log_alpha = a.log_alpha;
    p.beta = a.beta;
    p.S0 = a.S0;
    p.cu_seqlens = a.cu_seqlens;
    p.H = a.num_heads;
    p.scale = a.scale;
    p.o = a.o;
    p.S_final = a.S_final;
    p.ckpt = a.ckpt;
    p.status = a.status;
    if (a.unbounded)  // no decay floor: chunks out of the tensor-core range run token by token
        return launch_kernel<Tout, false, false, false, true>(p, a.num_seqs, a.num_heads, stream);
    if (a.head_decay) return launch_params<Tout, false, true>(p, a.num_seqs, a.num_heads, stream);
    return launch_params<Tout, false, false>(p, a.num_seqs, a.num_heads, stream);
}

template <typename Tout>
cudaError_t launch_layer_typed(const LayerArgs &a, cudaStream_t stream) {
    Params p;
    memset(&p, 0, sizeof(p));
    p.wait_ns = kWaitNs;
    if (a.total_tokens > 0) {
        const int T = a.total_tokens, H = a.num_heads;
        if (!encode_bf16_tiles(&p.tm_q, a.qp, T, H, kC) || !encode_bf16_tiles(&p.tm_k, a.kp, T, H, kC) ||
            !encode_bf16_tiles(&p.tm_v, a.vp, T, H, kC) || !encode_bf16_tiles(&p.tm_qh, a.qp, T, H, 8) ||
            !encode_bf16_tiles(&p.tm_kh, a.kp, T, H, 8) || !encode_bf16_tiles(&p.tm_vh, a.vp, T, H, 8) ||
            !encode_map(&p.tm_g, a.g, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, H, kD, kC,
                        CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    p.S0 = a.S0;
    p.cu_seqlens = a.cu_seqlens;
    p.H = a.num_heads;
    p.scale = a.scale;
    p.o = a.o;
    p.S_final = a.S_final;
    p.ckpt = a.ckpt;
    p.status = a.status;
    p.z = a.z;
    p.beta_logit = a.beta_logit;
    p.g = a.g;
    p.conv_w = a.conv_w;
    p.A = a.A;
    p.b = a.b;
    p.l2_eps = a.l2_eps;
    p.rms_eps = a.rms_eps;
    if (a.unbounded_decay)
        return launch_kernel<Tout, true, false, false, true>(p, a.num_seqs, a.num_heads, stream);
    return launch_params<Tout, true, false>(p, a.num_seqs, a.num_heads, stream);
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t stream) {
    if (a.out_dtype == KDA_BF16) return launch_typed<__nv_bfloat16>(a, stream);
    return launch_typed<float>(a, stream);
}

cudaError_t launch_layer_tc(const LayerArgs &a, cudaStream_t stream) {
    if (a.out_dtype == KDA_BF16) return launch_layer_typed<__nv_bfloat16>(a, stream);
    return launch_layer_typed<float>(a, stream);
}

}  // namespace kda

extern "C" kda_status kda_debug_inject_handoff_timeout(void) {
#ifdef KDA_DEBUG
    kda::g_inject_handoff_timeout.store(1);
    return KDA_OK;
#else
    return KDA_ERR_UNSUPPORTED;
#endif
}
