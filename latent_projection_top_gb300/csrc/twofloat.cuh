// Two-float (hi + lo) arithmetic for sums that must not lose what FP32
// rounding drops: Knuth's error-free addition (TwoSum) and a fixed-order
// warp reduction, so that results are bitwise reproducible.
#pragma once

#include "sm103_ptx.cuh"

namespace route {

// Error-free addition (Knuth's TwoSum): hi + x = s + e exactly; e joins lo.
__device__ __forceinline__ void two_sum_acc(float &hi, float &lo, float x) {
    const float s = hi + x;
    const float bp = s - hi;
    const float e = (hi - (s - bp)) + (x - bp);
    hi = s;
    lo += e;
}

// TwoSum on two independent two-floats at once, in packed FP32 pairs
// (hi, lo and x each hold one pair; the explicit rounding of every packed
// operation keeps the steps from being fused or reordered).
__device__ __forceinline__ void two_sum_acc_x2(uint64_t &hi, uint64_t &lo, uint64_t x) {
    const uint64_t s = ptx::f32x2_add(hi, x);
    const uint64_t bp = ptx::f32x2_sub(s, hi);
    const uint64_t e =
        ptx::f32x2_add(ptx::f32x2_sub(hi, ptx::f32x2_sub(s, bp)), ptx::f32x2_sub(x, bp));
    hi = s;
    lo = ptx::f32x2_add(lo, e);
}

// The value of a two-float sum.  An infinite high part is the value itself:
// once a sum reaches +-Inf its error term is Inf - Inf = NaN and must not be
// added (a NaN high part stays NaN).
__device__ __forceinline__ float two_float_value(float hi, float lo) {
    return fabsf(hi) == __int_as_float(0x7F800000) ? hi : hi + lo;
}

// Sum of the warp's 32 two-floats into lane 0, in a fixed tree order.
__device__ __forceinline__ void warp_two_sum(float &hi, float &lo) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float o_hi = __shfl_down_sync(0xFFFFFFFFu, hi, off);
        const float o_lo = __shfl_down_sync(0xFFFFFFFFu, lo, off);
        two_sum_acc(hi, lo, o_hi);
        lo += o_lo;
    }
}

}  // namespace route
