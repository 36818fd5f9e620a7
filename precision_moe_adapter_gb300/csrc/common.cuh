// common.cuh -- shared device helpers of libpmoe (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>

#include "pmoe.h"

namespace pmoe {

// ------------------------------------------------------------------ errors
// The first 256 bytes of every workspace hold the device error word.
struct DevErr {
    int code;      // first pmoe_status recorded, 0 = none
    int info[3];   // diagnostic payload of the first error
};
constexpr size_t kHdrBytes = 256;

__device__ __forceinline__ void record_error(DevErr *err, int code, int a = 0, int b = 0)
{
    if (err && atomicCAS(&err->code, 0, code) == 0) {
        err->info[0] = a;
        err->info[1] = b;
    }
}

// Host-side launch accounting (pmoe_launch_count).
void note_launch(int n = 1);

// ------------------------------------------------------------------ bf16
__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
__device__ __forceinline__ uint16_t f2bf(float f)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi)
{
    return (uint32_t)f2bf(lo) | ((uint32_t)f2bf(hi) << 16);
}

__host__ __device__ constexpr int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ------------------------------------------------------------------ formats
// Element value of each frozen-base format, computed exactly in FP32 and
// rounded once to BF16 (see pmoe.h for the definitions).

// INT4 nibble (two's complement) times a BF16 scale: the product has at
// most 12 significant bits, so the FP32 product is exact.
__device__ __forceinline__ float int4_times(uint32_t nib, float s)
{
    int q = (int)nib - ((int)(nib & 8) << 1);
    return __fmul_rn((float)q, s);
}

// E2M1 magnitude codes 0..7 -> {0, .5, 1, 1.5, 2, 3, 4, 6} by bit fields:
// exponent field 0 is subnormal (m/2), else (1 + m/2) * 2^(e-1).
__device__ __forceinline__ float e2m1_value(uint32_t nib)
{
    uint32_t e = (nib >> 1) & 3u, m = nib & 1u;
    float mag = e == 0 ? 0.5f * (float)m : (1.0f + 0.5f * (float)m) * (float)(1u << (e - 1));
    return (nib & 8u) ? -mag : mag;
}

// E8M0 scale 2^(u-127) as an FP32 value; u = 255 is NaN.
__device__ __forceinline__ float e8m0_value(uint32_t u)
{
    if (u == 255u) return __uint_as_float(0x7FC00000u);
    if (u == 0u) return __uint_as_float(0x00400000u);   // 2^-127, subnormal in FP32
    return __uint_as_float(u << 23);
}

// E4M3 (FN) code to FP32 by bit fields: bias 7, exponent 0 subnormal,
// S.1111.111 NaN.
__device__ __forceinline__ float e4m3_value(uint32_t c)
{
    uint32_t s = (c >> 7) & 1u, e = (c >> 3) & 15u, m = c & 7u;
    float v;
    if (e == 15u && m == 7u)
        v = __uint_as_float(0x7FC00000u);
    else if (e == 0u)
        v = (float)m * 0.001953125f;                       // m * 2^-9
    else
        v = __uint_as_float(((e + 120u) << 23) | (m << 20)); // (1 + m/8) 2^(e-7)
    return s ? -v : v;
}

// Dequantized BF16 value (as float) of element (n, c) of an [N, K] matrix
// stored in `fmt` (storage coordinates: n = output row, c = input column).
__device__ __forceinline__ float dequant_elem(int fmt, const uint8_t *q, const void *s, int64_t K,
                                              int64_t n, int64_t c)
{
    if (fmt == PMOE_W_INT4_G32_BF16) {
        uint32_t byte = q[n * (K >> 1) + (c >> 1)];
        uint32_t nib = (c & 1) ? (byte >> 4) : (byte & 15u);
        float sc = bf2f(((const uint16_t *)s)[n * (K >> 5) + (c >> 5)]);
        return bf2f(f2bf(int4_times(nib, sc)));
    }
    if (fmt == PMOE_W_MXFP4_G32_E8M0) {
        uint32_t byte = q[n * (K >> 1) + (c >> 1)];
        uint32_t nib = (c & 1) ? (byte >> 4) : (byte & 15u);
        float sc = e8m0_value(((const uint8_t *)s)[n * (K >> 5) + (c >> 5)]);
        return bf2f(f2bf(__fmul_rn(e2m1_value(nib), sc)));
    }
    float v = e4m3_value(q[n * K + c]);
    float sc = ((const float *)s)[(n >> 7) * (K >> 7) + (c >> 7)];
    return bf2f(f2bf(__fmul_rn(v, sc)));
}

// Bytes of one expert's packed weights / scales for an [N, K] matrix.
__host__ __device__ inline int64_t wq_bytes(int fmt, int64_t N, int64_t K)
{
    return fmt == PMOE_W_FP8_B128_F32 ? N * K : N * K / 2;
}
__host__ __device__ inline int64_t ws_bytes_of(int fmt, int64_t N, int64_t K)
{
    if (fmt == PMOE_W_INT4_G32_BF16) return N * (K / 32) * 2;
    if (fmt == PMOE_W_MXFP4_G32_E8M0) return N * (K / 32);
    return (N / 128) * (K / 128) * 4;
}

// ------------------------------------------------------------------ work list
// A tile of consecutive expert-sorted pair rows of one expert.
struct Tile {
    int expert;
    int row0;
    int nrows;
    int chunk;
};

}  // namespace pmoe
