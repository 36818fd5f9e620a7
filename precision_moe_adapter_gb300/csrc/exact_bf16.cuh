// exact_bf16.cuh -- correctly rounded BF16 results of short dot products
// (the rotated activations x~ = bf16(x R) and h~ = bf16(h R_down) of the
// OFT adapter, "Orbit：把万亿模型 RL 后训练改写成部署一致性问题", 机制拆解).
//
// A rotation output is a sum of b <= 64 products of BF16 values.  The
// tensor cores give it in FP32 together with an error bound; when the FP32
// value lies farther than the bound from the midpoint between its two BF16
// neighbours, bf16_rne(value) is already the rounding of the exact sum.
// Otherwise the warp recomputes that sum error-free: every lane holds some
// of the products (exact in FP32: BF16 x BF16), TwoSum steps carry every
// addition's rounding error (a chain inside the lane, then a butterfly over
// the lanes), so s + e is the sum to about 2^-44 of the sum of magnitudes;
// rounding s decides unless s is a BF16 midpoint itself, where the sign of
// e breaks the tie.
#pragma once

#include "common.cuh"

namespace pmoe {

__device__ __forceinline__ bool near_bf16_midpoint(float v, float bound)
{
    const float mid = __uint_as_float((__float_as_uint(v) & 0xFFFF0000u) | 0x8000u);
    return fabsf(v - mid) <= bound;
}

// Knuth's TwoSum: s + t = a + b exactly, s = fl(a + b)
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &t)
{
    s = __fadd_rn(a, b);
    const float z = __fsub_rn(s, a);
    t = __fadd_rn(__fsub_rn(a, __fsub_rn(s, z)), __fsub_rn(b, z));
}

// BF16 rounding of the exact sum s + e (|e| small against s): s + t = s + e
// after one more TwoSum, and when s is a BF16 midpoint the sign of t decides
__device__ __forceinline__ uint16_t round_sum_bf16(float s, float e)
{
    float t;
    two_sum(s, e, s, t);
    const uint32_t sb = __float_as_uint(s);
    if ((sb & 0xFFFFu) == 0x8000u && t != 0.f) {
        const bool away = (t > 0.f) == ((sb >> 31) == 0u);
        return (uint16_t)((sb >> 16) + (away ? 1u : 0u));
    }
    return f2bf(s);
}

// Whole converged warp: the exact sum of p0 + p1 over all lanes (each an
// exact product), rounded to BF16 (nearest, ties to even); every lane
// returns the same value.
__device__ __forceinline__ uint16_t warp_sum_round_bf16(float p0, float p1)
{
    float s, e;
    two_sum(p0, p1, s, e);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const float so = __shfl_xor_sync(0xffffffffu, s, off);
        const float eo = __shfl_xor_sync(0xffffffffu, e, off);
        float t;
        two_sum(s, so, s, t);
        e = __fadd_rn(__fadd_rn(e, eo), t);
    }
    return round_sum_bf16(s, e);
}

// Whole converged warp in aligned groups of 8 lanes: each group's exact sum
// of its lanes' 8 products each, rounded to BF16; the group's lanes return
// the same value.  Four sums per warp at once.
__device__ __forceinline__ uint16_t group8_sum_round_bf16(const float (&p)[8])
{
    float s = p[0], e = 0.f;
#pragma unroll
    for (int k = 1; k < 8; ++k) {
        float t;
        two_sum(s, p[k], s, t);
        e = __fadd_rn(e, t);
    }
#pragma unroll
    for (int off = 4; off >= 1; off >>= 1) {
        const float so = __shfl_xor_sync(0xffffffffu, s, off);
        const float eo = __shfl_xor_sync(0xffffffffu, e, off);
        float t;
        two_sum(s, so, s, t);
        e = __fadd_rn(__fadd_rn(e, eo), t);
    }
    return round_sum_bf16(s, e);
}

}  // namespace pmoe
