// Column-quad layout of a 128 x 128 fp32 state held in registers, used by the
// token-by-token prefill kernel.
//
// Value columns of the KDA state evolve independently: column c needs only k,
// alpha, beta and v[c] of each token.  Eight adjacent lanes (row groups
// rq = lane & 7) share a quad of four columns, and each holds 16 of the 128 rows
// of all four, so every alpha, k and q value read from shared memory serves
// four columns.  The two reductions over rows per token (r = S^T k, p = S^T q)
// are transposed butterflies over the eight lanes: at each of three xor steps a
// lane sends half of the partial sums it holds and keeps the other half, so it
// ends with the full sum of one column (four shuffles for four columns); a
// value per column goes back to all eight lanes in three more shuffles.  Each
// lane keeps its four columns in a lane-dependent order (lane_order) that makes
// both free of selects.
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

// Register order of a lane's four columns.  Component m of the lane's float4s holds column
// quad_col(rq) ^ m of its quad: first the column whose full sum the lane ends with, then that
// column's pair partner, then the other pair in the same order.  With this order every step
// of the butterflies below keeps components 0-1 and sends 2-3 (or keeps 0 and sends 1) on
// every lane, so they need no lane-dependent selects.  The map is its own inverse.
__device__ __forceinline__ float4 lane_order(float4 x, int jc) {
    const bool b2 = (jc & 2) != 0, b1 = (jc & 1) != 0;
    const float p0 = b2 ? x.z : x.x, p1 = b2 ? x.w : x.y;
    const float p2 = b2 ? x.x : x.z, p3 = b2 ? x.y : x.w;
    return b1 ? make_float4(p1, p0, p3, p2) : make_float4(p0, p1, p2, p3);
}

// Sum of y (one partial sum per column of the quad, in lane order) over the 8 lanes of a
// row-group set (lanes that differ in bits 0-2): the lane returns the sum for column
// quad_col(rq).  The xor-4 partner holds this lane's two columns in its components 2-3, the
// xor-2 partner this lane's column in its component 1, the xor-1 partner the same column.
__device__ __forceinline__ float quad_reduce(float4 y) {
    const float a = y.x + __shfl_xor_sync(kFull, y.z, 4);
    const float b = y.y + __shfl_xor_sync(kFull, y.w, 4);
    float c = a + __shfl_xor_sync(kFull, b, 2);
    c += __shfl_xor_sync(kFull, c, 1);
    return c;
}

// The four columns' values to every lane of the row-group set, in lane order, from x held
// for column quad_col(rq) (lanes rq and rq ^ 1 hold the same column).
__device__ __forceinline__ float4 quad_gather(float x) {
    const float xo = __shfl_xor_sync(kFull, x, 2);  // the pair partner column
    return make_float4(x, xo, __shfl_xor_sync(kFull, x, 4), __shfl_xor_sync(kFull, xo, 4));
}

}  // namespace quads
}  // namespace kda
