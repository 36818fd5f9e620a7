// layer.cu -- the row-wise steps of the layer around the grouped GEMMs:
// weighted un-permute (combine), row gathers, and the elementwise parts of
// the backward-data pass (SwiGLU backward, the down-adapter rotation and
// its adjoint, the d_topk_w reduction, the slot sum of dX).
#include "common.cuh"
#include "launch.h"

namespace pmoe {

__device__ __forceinline__ float silu_f(float g) { return g / (1.f + expf(-g)); }

// Y[t] = bf16(sum_j w[t,j] o[inv_perm[t*k + j]]), slots in order.
__global__ void __launch_bounds__(256) k_combine(int T, int d, int k, const uint16_t *__restrict__ o,
                                                 const int32_t *__restrict__ inv_perm,
                                                 const float *__restrict__ w,
                                                 uint16_t *__restrict__ Y)
{
    int t = blockIdx.x;
    for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
        float acc[8] = {};
        for (int j = 0; j < k; ++j) {
            int r = inv_perm[(int64_t)t * k + j];
            if (r < 0) continue;
            float wj = w[(int64_t)t * k + j];
            uint4 v = *(const uint4 *)(o + (int64_t)r * d + c);
            const uint16_t *hv = (const uint16_t *)&v;
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, bf2f(hv[i]), acc[i]);
        }
        uint4 out;
        out.x = pack_bf2(acc[0], acc[1]);
        out.y = pack_bf2(acc[2], acc[3]);
        out.z = pack_bf2(acc[4], acc[5]);
        out.w = pack_bf2(acc[6], acc[7]);
        *(uint4 *)(Y + (int64_t)t * d + c) = out;
    }
}

void launch_combine(int T, int d, int k, const uint16_t *o, const int32_t *inv_perm,
                    const float *w, uint16_t *Y, cudaStream_t st)
{
    if (T <= 0) return;
    k_combine<<<T, 256, 0, st>>>(T, d, k, o, inv_perm, w, Y);
    note_launch();
}

__global__ void k_gather_rows(int P, int d, int k, const uint16_t *__restrict__ src,
                              const int32_t *__restrict__ perm, uint16_t *__restrict__ out)
{
    int r = blockIdx.x;
    const uint16_t *s = src + (int64_t)(perm[r] / k) * d;
    for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8)
        *(uint4 *)(out + (int64_t)r * d + c) = *(const uint4 *)(s + c);
}

void launch_gather_rows(int P, int d, int k, const uint16_t *src, const int32_t *perm,
                        uint16_t *out, cudaStream_t st)
{
    if (P <= 0) return;
    k_gather_rows<<<P, 256, 0, st>>>(P, d, k, src, perm, out);
    note_launch();
}

// From the saved [g | u] of a row: h = bf16(silu(g) u), h~ = bf16(h R_down).
__global__ void __launch_bounds__(256) k_bwd_prep(int I, int b, const uint16_t *__restrict__ ctx,
                                                  const int32_t *__restrict__ perm,
                                                  const int32_t *__restrict__ idx_flat,
                                                  const uint16_t *__restrict__ R, int64_t stride,
                                                  uint16_t *__restrict__ h,
                                                  uint16_t *__restrict__ ht)
{
    extern __shared__ float hs[];
    int64_t r = blockIdx.x;
    const uint16_t *c = ctx + r * 2 * I;
    for (int n = threadIdx.x; n < I; n += blockDim.x) {
        float hv = bf2f(f2bf(silu_f(bf2f(c[n])) * bf2f(c[I + n])));
        hs[n] = hv;
        h[r * I + n] = f2bf(hv);
    }
    __syncthreads();
    const uint16_t *Re = R ? R + (stride ? (int64_t)idx_flat[perm[r]] * stride : 0) : nullptr;
    for (int n = threadIdx.x; n < I; n += blockDim.x) {
        if (!Re) {
            ht[r * I + n] = f2bf(hs[n]);
            continue;
        }
        int beta = n / b, j = n % b;
        const uint16_t *Rb = Re + (int64_t)beta * b * b;
        float acc = 0.f;
        for (int i = 0; i < b; ++i) acc = fmaf(hs[beta * b + i], bf2f(Rb[i * b + j]), acc);
        ht[r * I + n] = f2bf(acc);
    }
}

void launch_bwd_prep(int P, int I, int b, const uint16_t *ctx, const int32_t *perm,
                     const int32_t *idx_flat, const uint16_t *R_down, int64_t stride,
                     uint16_t *h, uint16_t *ht, cudaStream_t st)
{
    if (P <= 0) return;
    k_bwd_prep<<<P, 256, I * sizeof(float), st>>>(I, b, ctx, perm, idx_flat, R_down, stride, h, ht);
    note_launch();
}

// dh = dh~ R_down^T; dg = dh u s(g)(1 + g(1 - s(g))); du = dh silu(g).
__global__ void __launch_bounds__(256) k_bwd_mid(int I, int b, const uint16_t *__restrict__ ctx,
                                                 const uint16_t *__restrict__ dht,
                                                 const int32_t *__restrict__ perm,
                                                 const int32_t *__restrict__ idx_flat,
                                                 const uint16_t *__restrict__ R, int64_t stride,
                                                 uint16_t *__restrict__ dgu)
{
    extern __shared__ float ds[];
    int64_t r = blockIdx.x;
    for (int n = threadIdx.x; n < I; n += blockDim.x) ds[n] = bf2f(dht[r * I + n]);
    __syncthreads();
    const uint16_t *Re = R ? R + (stride ? (int64_t)idx_flat[perm[r]] * stride : 0) : nullptr;
    const uint16_t *c = ctx + r * 2 * I;
    for (int n = threadIdx.x; n < I; n += blockDim.x) {
        float dh;
        if (Re) {
            int beta = n / b, j = n % b;
            const uint16_t *Rb = Re + (int64_t)beta * b * b + (int64_t)j * b;
            dh = 0.f;
            for (int i = 0; i < b; ++i) dh = fmaf(ds[beta * b + i], bf2f(Rb[i]), dh);
        } else {
            dh = ds[n];
        }
        float g = bf2f(c[n]), u = bf2f(c[I + n]);
        float sg = 1.f / (1.f + expf(-g));
        dgu[r * 2 * I + n] = f2bf(dh * u * sg * (1.f + g * (1.f - sg)));
        dgu[r * 2 * I + I + n] = f2bf(dh * g * sg);
    }
}

void launch_bwd_mid(int P, int I, int b, const uint16_t *ctx, const uint16_t *dht,
                    const int32_t *perm, const int32_t *idx_flat, const uint16_t *R_down,
                    int64_t stride, uint16_t *dgu, cudaStream_t st)
{
    if (P <= 0) return;
    k_bwd_mid<<<P, 256, I * sizeof(float), st>>>(I, b, ctx, dht, perm, idx_flat, R_down, stride, dgu);
    note_launch();
}

__global__ void k_dtw_reduce(int P, int nparts, const float *__restrict__ part,
                             const int32_t *__restrict__ perm, float *__restrict__ dtw)
{
    int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= P) return;
    float s = 0.f;
    for (int q = 0; q < nparts; ++q) s += part[(int64_t)r * nparts + q];
    dtw[perm[r]] = s;
}

void launch_dtw_reduce(int P, int nparts, const float *part, const int32_t *perm, float *dtw,
                       cudaStream_t st)
{
    if (P <= 0) return;
    k_dtw_reduce<<<(int)cdiv(P, 256), 256, 0, st>>>(P, nparts, part, perm, dtw);
    note_launch();
}

// dX[t] = bf16(sum_j dx~_(t,j) R_up[e_j]^T), slots in order.
__global__ void __launch_bounds__(256) k_combine_bwd(int d, int k, int b,
                                                     const uint16_t *__restrict__ dxt,
                                                     const int32_t *__restrict__ inv_perm,
                                                     const int32_t *__restrict__ idx_flat,
                                                     const uint16_t *__restrict__ R, int64_t stride,
                                                     uint16_t *__restrict__ dX)
{
    extern __shared__ float xs[];
    int t = blockIdx.x;
    const int per = (d + blockDim.x - 1) / blockDim.x;   // <= 32 for d <= 8192
    float acc[32];
    for (int q = 0; q < per; ++q) acc[q] = 0.f;
    for (int j = 0; j < k; ++j) {
        int r = inv_perm[(int64_t)t * k + j];
        if (r < 0) continue;
        __syncthreads();
        for (int c = threadIdx.x; c < d; c += blockDim.x) xs[c] = bf2f(dxt[(int64_t)r * d + c]);
        __syncthreads();
        const uint16_t *Re = R ? R + (stride ? (int64_t)idx_flat[(int64_t)t * k + j] * stride : 0)
                               : nullptr;
        for (int q = 0; q < per; ++q) {
            int c = threadIdx.x + q * blockDim.x;
            if (c >= d) break;
            float v;
            if (Re) {
                int beta = c / b, rr = c % b;
                const uint16_t *Rb = Re + (int64_t)beta * b * b + (int64_t)rr * b;
                v = 0.f;
                for (int i = 0; i < b; ++i) v = fmaf(xs[beta * b + i], bf2f(Rb[i]), v);
            } else {
                v = xs[c];
            }
            acc[q] += v;
        }
    }
    for (int q = 0; q < per; ++q) {
        int c = threadIdx.x + q * blockDim.x;
        if (c < d) dX[(int64_t)t * d + c] = f2bf(acc[q]);
    }
}

void launch_combine_bwd(int T, int d, int k, int b, const uint16_t *dxt, const int32_t *inv_perm,
                        const int32_t *idx_flat, const uint16_t *R_up, int64_t stride,
                        uint16_t *dX, cudaStream_t st)
{
    if (T <= 0) return;
    k_combine_bwd<<<T, 256, d * sizeof(float), st>>>(d, k, b, dxt, inv_perm, idx_flat, R_up, stride,
                                                     dX);
    note_launch();
}

}  // namespace pmoe
