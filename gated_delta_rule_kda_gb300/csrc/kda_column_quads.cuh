// Column-quad layout of a 128 x 128 fp32 state held in registers, shared by the
// token-by-token kernels (prefill and multi-token decode).
//
// Value columns of the KDA state evolve independently: column c needs only k,
// alpha, beta and v[c] of each token.  Eight adjacent lanes (row groups
// rq = lane & 7) share a quad of four columns, and each holds 16 of the 128 rows
// of all four, so every alpha, k and q value read from shared memory serves
// four columns.  The two reductions over rows per token (r = S^T k, p = S^T q)
// are transposed butterflies over the eight lanes: at each of three xor steps a
// lane sends half of the partial sums it holds and keeps the other half, so it
// ends with the full sum of one column (four shuffles for four columns); a
// value per column goes back to all eight lanes in three more shuffles.
#pragma once

#include "kda_common.cuh"

namespace kda {
namespace quads {

constexpr unsigned kFull = 0xffffffffu;

// Row-indexed vectors in shared memory carry 4 floats of padding after every 16
// rows, so that the 8 row groups of a warp read 8 different bank groups.
constexpr int kPadRow = kD + 32;
__device__ __forceinline__ int prow(int row) { return row + 4 * (row >> 4); }

// Column of its quad whose full sum a lane holds after quad_reduce (row group rq = lane & 7).
__device__ __forceinline__ int quad_col(int rq) { return 2 * ((rq >> 2) & 1) + ((rq >> 1) & 1); }

// Sum of x (one partial sum per column of the quad) over the 8 lanes of a row-group set
// (lanes that differ in bits 0-2): the lane returns the sum for column quad_col(rq).
__device__ __forceinline__ float quad_reduce(float4 x, int rq) {
    const bool hi = (rq & 4) != 0;  // keeps columns 2, 3; its partner keeps 0, 1
    float a = hi ? x.z : x.x, b = hi ? x.w : x.y;
    const float sa = hi ? x.x : x.z, sb = hi ? x.y : x.w;
    a += __shfl_xor_sync(kFull, sa, 4);
    b += __shfl_xor_sync(kFull, sb, 4);
    const bool mid = (rq & 2) != 0;  // keeps the odd column of the pair
    float c = mid ? b : a;
    const float sc = mid ? a : b;
    c += __shfl_xor_sync(kFull, sc, 2);
    c += __shfl_xor_sync(kFull, c, 1);
    return c;
}

// The four columns' values to every lane of the row-group set, from x held for column
// quad_col(rq) (lanes rq and rq ^ 1 hold the same column).
__device__ __forceinline__ float4 quad_gather(float x, int rq) {
    const float xo = __shfl_xor_sync(kFull, x, 2);  // the other column of the pair
    const bool mid = (rq & 2) != 0;
    const float p0 = mid ? xo : x, p1 = mid ? x : xo;  // columns 2 hi, 2 hi + 1
    const float o0 = __shfl_xor_sync(kFull, p0, 4), o1 = __shfl_xor_sync(kFull, p1, 4);
    return (rq & 4) ? make_float4(o0, o1, p0, p1) : make_float4(p0, p1, o0, o1);
}

}  // namespace quads
}  // namespace kda
