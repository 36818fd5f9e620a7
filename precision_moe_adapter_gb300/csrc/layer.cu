// layer.cu -- the row-wise steps of the layer around the grouped GEMMs:
// the weighted un-permute (combine) and the slot sum of dX, row gathers,
// and the fixed-order d_topk_w reduction.
#include "common.cuh"
#include "launch.h"

namespace pmoe {

// Y[t] = bf16(sum_j w[t,j] o[inv_perm[t*k + j]]), slots in order, over the
// FP32 pair outputs o (w NULL: unit weights, the slot sum of the backward).
__global__ void __launch_bounds__(128) k_combine(int T, int d, int k, const float *__restrict__ o,
                                                 const int32_t *__restrict__ inv_perm,
                                                 const float *__restrict__ w,
                                                 uint16_t *__restrict__ Y)
{
    // CTA (t, y): columns 1024 y .. of token t (8 per thread)
    int t = blockIdx.x;
    for (int c = blockIdx.y * 1024 + threadIdx.x * 8; c < d; c += gridDim.y * 1024) {
        float acc[8] = {};
        for (int j = 0; j < k; ++j) {
            int r = inv_perm[(int64_t)t * k + j];
            if (r < 0) continue;
            float wj = w ? w[(int64_t)t * k + j] : 1.f;
            const float4 v0 = *(const float4 *)(o + (int64_t)r * d + c);
            const float4 v1 = *(const float4 *)(o + (int64_t)r * d + c + 4);
            const float hv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, hv[i], acc[i]);
        }
        uint4 out;
        out.x = pack_bf2(acc[0], acc[1]);
        out.y = pack_bf2(acc[2], acc[3]);
        out.z = pack_bf2(acc[4], acc[5]);
        out.w = pack_bf2(acc[6], acc[7]);
        *(uint4 *)(Y + (int64_t)t * d + c) = out;
    }
}

void launch_combine(int T, int d, int k, const float *o, const int32_t *inv_perm,
                    const float *w, uint16_t *Y, cudaStream_t st)
{
    if (T <= 0) return;
    k_combine<<<dim3(T, (d + 1023) / 1024), 128, 0, st>>>(T, d, k, o, inv_perm, w, Y);
    note_launch();
}

// out[r] = src[perm[r] / k] for the grouped rows r < *nvalid (the rows past
// it, pairs left out of the grouping, are not touched).  One CTA per row;
// every thread issues its (up to four) 16-byte loads before its stores.
__global__ void __launch_bounds__(256) k_gather_rows(int d, int k, const uint16_t *__restrict__ src,
                                                     const int32_t *__restrict__ perm,
                                                     const int32_t *__restrict__ nvalid,
                                                     uint16_t *__restrict__ out)
{
    const int r = blockIdx.x;
    if (r >= *nvalid) return;
    const uint4 *s = (const uint4 *)(src + (int64_t)(perm[r] / k) * d);
    uint4 *o = (uint4 *)(out + (int64_t)r * d);
    const int n = d / 8;
    for (int c0 = threadIdx.x; c0 < n; c0 += 4 * 256) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (c0 + u * 256 < n) v[u] = __ldg(s + c0 + u * 256);
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (c0 + u * 256 < n) o[c0 + u * 256] = v[u];
    }
}

void launch_gather_rows(int P, int d, int k, const uint16_t *src, const int32_t *perm,
                        const int32_t *nvalid, uint16_t *out, cudaStream_t st)
{
    if (P <= 0) return;
    k_gather_rows<<<P, 256, 0, st>>>(d, k, src, perm, nvalid, out);
    note_launch();
}

// d_topk_w[p] = sum of the I/32 partials of pair p's expert-sorted row, in
// order; a pair left out of the grouping (inv_perm[p] < 0: an expert id out
// of range) gets 0.  One thread per pair, so every write stays in [0, P).
__global__ void k_dtw_reduce(int P, int nparts, const float *__restrict__ part,
                             const int32_t *__restrict__ inv_perm, float *__restrict__ dtw)
{
    int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= P) return;
    const int r = inv_perm[p];
    float s = 0.f;
    if (r >= 0)
        for (int q = 0; q < nparts; ++q) s += part[(int64_t)r * nparts + q];
    dtw[p] = s;
}

void launch_dtw_reduce(int P, int nparts, const float *part, const int32_t *inv_perm, float *dtw,
                       cudaStream_t st)
{
    if (P <= 0) return;
    k_dtw_reduce<<<(int)cdiv(P, 256), 256, 0, st>>>(P, nparts, part, inv_perm, dtw);
    note_launch();
}

__global__ void k_adapter_snapshot(const uint64_t *ctrl, uint64_t *snap, uint32_t *version_out)
{
    if (threadIdx.x == 0) {
        const uint64_t v = atomicAdd((unsigned long long *)ctrl, 0ull);
        *snap = v;
        if (version_out) *version_out = (uint32_t)(v >> 32);
    }
}

void launch_adapter_snapshot(const uint64_t *ctrl, uint64_t *snap, uint32_t *version_out,
                             cudaStream_t st)
{
    k_adapter_snapshot<<<1, 32, 0, st>>>(ctrl, snap, version_out);
    note_launch();
}

__global__ void k_adapter_publish(uint64_t *ctrl, uint64_t word)
{
    if (threadIdx.x == 0) {
        __threadfence();   // earlier writes of this stream (the new slot) come first
        atomicExch((unsigned long long *)ctrl, (unsigned long long)word);
    }
}

void launch_adapter_publish(uint64_t *ctrl, uint32_t slot, uint32_t version, cudaStream_t st)
{
    k_adapter_publish<<<1, 32, 0, st>>>(ctrl, ((uint64_t)version << 32) | (slot & 1u));
    note_launch();
}

__global__ void k_set_offsets(int32_t *offsets, int rows)
{
    if (threadIdx.x == 0) {
        offsets[0] = 0;
        offsets[1] = rows;
    }
}

void launch_set_offsets(int32_t *offsets, int rows, cudaStream_t st)
{
    k_set_offsets<<<1, 32, 0, st>>>(offsets, rows);
    note_launch();
}

}  // namespace pmoe
