// dequant.cu -- the temporary dequantization step (Orbit announcement, 技艺细节): frozen INT4 /
// MXFP4 / FP8 weights to BF16, for one matrix or for the experts of one
// chunk into the bounded global scratch that the next chunk reuses.
#include "common.cuh"
#include "launch.h"

namespace pmoe {

// Eight consecutive elements (n, c..c+7) of an [N, K] matrix -> 16 bytes.
__device__ __forceinline__ uint4 dequant8(int fmt, const uint8_t *__restrict__ q,
                                          const void *__restrict__ s, int64_t K, int64_t n,
                                          int64_t c)
{
    float v[8];
    if (fmt == PMOE_W_INT4_G32_BF16 || fmt == PMOE_W_MXFP4_G32_E8M0) {
        uint32_t word = *(const uint32_t *)(q + n * (K >> 1) + (c >> 1));
        if (fmt == PMOE_W_INT4_G32_BF16) {
            float sc = bf2f(((const uint16_t *)s)[n * (K >> 5) + (c >> 5)]);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = int4_times((word >> (4 * i)) & 15u, sc);
        } else {
            float sc = e8m0_value(((const uint8_t *)s)[n * (K >> 5) + (c >> 5)]);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(e2m1_value((word >> (4 * i)) & 15u), sc);
        }
    } else {
        uint2 codes = *(const uint2 *)(q + n * K + c);
        float sc = ((const float *)s)[(n >> 7) * (K >> 7) + (c >> 7)];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t code = ((i < 4 ? codes.x : codes.y) >> (8 * (i & 3))) & 255u;
            v[i] = __fmul_rn(e4m3_value(code), sc);
        }
    }
    uint4 r;
    r.x = pack_bf2(v[0], v[1]);
    r.y = pack_bf2(v[2], v[3]);
    r.z = pack_bf2(v[4], v[5]);
    r.w = pack_bf2(v[6], v[7]);
    return r;
}

__global__ void k_dequant(int fmt, const uint8_t *__restrict__ q, const void *__restrict__ s,
                          int64_t N, int64_t K, uint16_t *__restrict__ out)
{
    int64_t groups = N * (K / 8);
    for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < groups;
         g += (int64_t)gridDim.x * blockDim.x) {
        int64_t n = g / (K / 8), c = (g % (K / 8)) * 8;
        *(uint4 *)(out + n * K + c) = dequant8(fmt, q, s, K, n, c);
    }
}

void launch_dequant(int fmt, const void *q, const void *s, int64_t N, int64_t K, uint16_t *out,
                    cudaStream_t st)
{
    int64_t groups = N * (K / 8);
    if (groups <= 0) return;
    int blocks = (int)std::min<int64_t>(cdiv(groups, 256), 152 * 16);
    k_dequant<<<blocks, 256, 0, st>>>(fmt, (const uint8_t *)q, s, N, K, out);
    note_launch();
}

// grid.y = slot within the chunk; slots past num_active exit.
__global__ void k_dequant_chunk(int fmt, int d, int I, int C, int chunk,
                                const int32_t *__restrict__ active,
                                const int32_t *__restrict__ num_active,
                                const uint8_t *__restrict__ w13, const uint8_t *__restrict__ s13,
                                const uint8_t *__restrict__ w2, const uint8_t *__restrict__ s2,
                                uint16_t *__restrict__ scratch)
{
    int slot = blockIdx.y;
    int a = chunk * C + slot;
    if (a >= *num_active) return;
    int e = active[a];
    int64_t n13 = 2 * (int64_t)I, slot_elems = 3 * (int64_t)I * d;
    const uint8_t *q13 = w13 + e * wq_bytes(fmt, n13, d);
    const uint8_t *sc13 = s13 + e * ws_bytes_of(fmt, n13, d);
    const uint8_t *q2 = w2 + e * wq_bytes(fmt, d, I);
    const uint8_t *sc2 = s2 + e * ws_bytes_of(fmt, d, I);
    uint16_t *dst = scratch + slot * slot_elems;
    int64_t g13 = n13 * (d / 8), g2 = (int64_t)d * (I / 8);
    for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < g13 + g2;
         g += (int64_t)gridDim.x * blockDim.x) {
        if (g < g13) {
            int64_t n = g / (d / 8), c = (g % (d / 8)) * 8;
            *(uint4 *)(dst + n * d + c) = dequant8(fmt, q13, sc13, d, n, c);
        } else {
            int64_t h = g - g13;
            int64_t n = h / (I / 8), c = (h % (I / 8)) * 8;
            *(uint4 *)(dst + n13 * d + n * I + c) = dequant8(fmt, q2, sc2, I, n, c);
        }
    }
}

void launch_dequant_chunk(int fmt, int d, int I, int C, int chunk, const int32_t *active,
                          const int32_t *num_active, const void *w13, const void *s13,
                          const void *w2, const void *s2, uint16_t *scratch, cudaStream_t st)
{
    int64_t per_slot = 3 * (int64_t)I * d / 8;
    int bx = (int)std::max<int64_t>(1, std::min<int64_t>(cdiv(per_slot, 256), (152 * 16 + C - 1) / C));
    dim3 grid(bx, C);
    k_dequant_chunk<<<grid, 256, 0, st>>>(fmt, d, I, C, chunk, active, num_active,
                                          (const uint8_t *)w13, (const uint8_t *)s13,
                                          (const uint8_t *)w2, (const uint8_t *)s2, scratch);
    note_launch();
}

}  // namespace pmoe
