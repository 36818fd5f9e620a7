// adapter.cu -- the block-diagonal orthogonal (OFT-style) adapter: rotation
// of activation rows by blockdiag(R), its adjoint, the per-block gradient
// reduction, and the Cayley map R = (I + S)(I - S)^{-1} with its gradient
// (page 2, 机制拆解: the adapter is a local orthogonal transform).
#include "common.cuh"
#include "launch.h"

namespace pmoe {

// One CTA per row.  out[beta*b + j] = sum_i x[beta*b + i] * R[beta][i][j]
// (or R[beta][j][i] when `trans`), FP32 accumulate, one BF16 rounding.
template <bool kTrans>
__global__ void __launch_bounds__(256) k_rotate_rows(int nrows_max, int dim, int b,
                                                     const uint16_t *__restrict__ src,
                                                     bool gather,
                                                     const int32_t *__restrict__ perm, int k,
                                                     const int32_t *__restrict__ idx_flat,
                                                     const uint16_t *__restrict__ R, int64_t stride,
                                                     uint16_t *__restrict__ out,
                                                     const int32_t *__restrict__ rows_dev)
{
    extern __shared__ float xs[];
    int r0 = rows_dev ? rows_dev[0] : 0;
    int r1 = rows_dev ? rows_dev[1] : nrows_max;
    int r = r0 + blockIdx.x;
    if (r >= r1) return;
    int64_t srow = (gather && perm) ? perm[r] / k : r;
    const uint16_t *x = src + srow * dim;
    uint16_t *o = out + (int64_t)r * dim;
    if (!R) {
        for (int c = threadIdx.x * 8; c < dim; c += blockDim.x * 8)
            *(uint4 *)(o + c) = *(const uint4 *)(x + c);
        return;
    }
    const uint16_t *Re = R + (stride ? (int64_t)idx_flat[perm[r]] * stride : 0);
    for (int c = threadIdx.x; c < dim; c += blockDim.x) xs[c] = bf2f(x[c]);
    __syncthreads();
    for (int c = threadIdx.x; c < dim; c += blockDim.x) {
        int beta = c / b, j = c % b;
        const uint16_t *Rb = Re + (int64_t)beta * b * b;
        const float *xb = xs + beta * b;
        float acc = 0.f;
        for (int i = 0; i < b; ++i)
            acc = fmaf(xb[i], bf2f(kTrans ? Rb[j * b + i] : Rb[i * b + j]), acc);
        o[c] = f2bf(acc);
    }
}

void launch_rotate_rows(int nrows_max, int dim, int b, const uint16_t *src, bool gather,
                        const int32_t *perm, int k, const int32_t *idx_flat, const uint16_t *R,
                        int64_t stride, uint16_t *out, const int32_t *rows_dev, cudaStream_t st)
{
    if (nrows_max <= 0) return;
    k_rotate_rows<false><<<nrows_max, 256, dim * sizeof(float), st>>>(
        nrows_max, dim, b, src, gather, perm, k, idx_flat, R, stride, out, rows_dev);
    note_launch();
}

void launch_adapter_grad_dx(int rows, int dim, int b, const uint16_t *dXr, const uint16_t *R,
                            uint16_t *dX, cudaStream_t st)
{
    if (rows <= 0) return;
    k_rotate_rows<true><<<rows, 256, dim * sizeof(float), st>>>(rows, dim, b, dXr, false, nullptr,
                                                                 1, nullptr, R, 0, dX, nullptr);
    note_launch();
}

// dR[s][beta][i][j] = sum over the rows of set s, in row order, of
// a[arow][beta*b + i] * g[row][beta*b + j].  One CTA per (set, block).
__global__ void __launch_bounds__(256) k_block_outer(int nrows, int dim, int b,
                                                     const uint16_t *__restrict__ a,
                                                     const int32_t *__restrict__ perm, int k,
                                                     const uint16_t *__restrict__ g,
                                                     const int32_t *__restrict__ offsets,
                                                     float *__restrict__ dR)
{
    extern __shared__ float sm[];
    const int RB = 32;
    float *as = sm, *gs = sm + RB * b;
    int nb = dim / b;
    int s = blockIdx.x / nb, beta = blockIdx.x % nb;
    int r0 = offsets ? offsets[s] : 0, r1 = offsets ? offsets[s + 1] : nrows;
    int nout = b * b;
    int per = (nout + blockDim.x - 1) / blockDim.x;   // <= 64
    float acc[64];
    for (int q = 0; q < per; ++q) acc[q] = 0.f;
    for (int rb = r0; rb < r1; rb += RB) {
        int n = min(RB, r1 - rb);
        __syncthreads();
        for (int i = threadIdx.x; i < RB * b; i += blockDim.x) {
            int rr = i / b, c = i % b;
            float av = 0.f, gv = 0.f;
            if (rr < n) {
                int row = rb + rr;
                int64_t arow = perm ? perm[row] / k : row;
                av = bf2f(a[arow * dim + beta * b + c]);
                gv = bf2f(g[(int64_t)row * dim + beta * b + c]);
            }
            as[i] = av;
            gs[i] = gv;
        }
        __syncthreads();
        for (int q = 0; q < per; ++q) {
            int o = threadIdx.x + q * blockDim.x;
            if (o >= nout) break;
            int i = o / b, j = o % b;
            float v = acc[q];
            for (int rr = 0; rr < n; ++rr) v = fmaf(as[rr * b + i], gs[rr * b + j], v);
            acc[q] = v;
        }
    }
    float *D = dR + ((int64_t)s * nb + beta) * nout;
    for (int q = 0; q < per; ++q) {
        int o = threadIdx.x + q * blockDim.x;
        if (o < nout) D[o] = acc[q];
    }
}

void launch_block_outer(int nsets, int nrows, int dim, int b, const uint16_t *a,
                        const int32_t *perm, int k, const uint16_t *g, const int32_t *offsets,
                        float *dR, cudaStream_t st)
{
    int grid = nsets * (dim / b);
    if (grid <= 0) return;
    k_block_outer<<<grid, 256, 2 * 32 * b * sizeof(float), st>>>(nrows, dim, b, a, perm, k, g,
                                                                  offsets, dR);
    note_launch();
}

// ------------------------------------------------------------------ Cayley
// Gauss-Jordan with partial pivoting on the augmented [A | B] (b x 2b) in
// shared memory; on return the right half holds A^{-1} B.
__device__ void gauss_jordan(float *aug, int b, float *colbuf, int *piv)
{
    int w = 2 * b;
    for (int col = 0; col < b; ++col) {
        if (threadIdx.x == 0) {
            int p = col;
            float best = fabsf(aug[col * w + col]);
            for (int r = col + 1; r < b; ++r) {
                float v = fabsf(aug[r * w + col]);
                if (v > best) { best = v; p = r; }
            }
            *piv = p;
        }
        __syncthreads();
        int p = *piv;
        if (p != col)
            for (int j = threadIdx.x; j < w; j += blockDim.x) {
                float t = aug[col * w + j];
                aug[col * w + j] = aug[p * w + j];
                aug[p * w + j] = t;
            }
        __syncthreads();
        float pv = aug[col * w + col];
        __syncthreads();
        for (int j = threadIdx.x; j < w; j += blockDim.x) aug[col * w + j] /= pv;
        __syncthreads();
        for (int r = threadIdx.x; r < b; r += blockDim.x) colbuf[r] = aug[r * w + col];
        __syncthreads();
        for (int i = threadIdx.x; i < b * w; i += blockDim.x) {
            int r = i / w, j = i % w;
            if (r != col) aug[i] = fmaf(-colbuf[r], aug[col * w + j], aug[i]);
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(256) k_cayley(int b, const float *__restrict__ S,
                                                uint16_t *__restrict__ Rb, float *__restrict__ Rf)
{
    extern __shared__ float aug[];
    __shared__ float colbuf[128];
    __shared__ int piv;
    const float *Sb = S + (int64_t)blockIdx.x * b * b;
    int w = 2 * b;
    for (int i = threadIdx.x; i < b * b; i += blockDim.x) {
        int r = i / b, c = i % b;
        float s = Sb[i], id = r == c ? 1.f : 0.f;
        aug[r * w + c] = id - s;
        aug[r * w + b + c] = id + s;
    }
    __syncthreads();
    gauss_jordan(aug, b, colbuf, &piv);
    for (int i = threadIdx.x; i < b * b; i += blockDim.x) {
        float v = aug[(i / b) * w + b + i % b];
        if (Rf) Rf[(int64_t)blockIdx.x * b * b + i] = v;
        if (Rb) Rb[(int64_t)blockIdx.x * b * b + i] = f2bf(v);
    }
}

// M = (I + R)^T dR A^T with A = (I - S)^{-1}:  Z = A dR^T from
// Gauss-Jordan on [I - S | dR^T], then M[i][j] = sum_m (I+R)[m][i] Z[j][m],
// dS = M - M^T.
__global__ void __launch_bounds__(256) k_cayley_grad(int b, const float *__restrict__ S,
                                                     const float *__restrict__ Rf,
                                                     const float *__restrict__ dR,
                                                     float *__restrict__ dS)
{
    extern __shared__ float aug[];
    __shared__ float colbuf[128];
    __shared__ int piv;
    int64_t off = (int64_t)blockIdx.x * b * b;
    int w = 2 * b;
    for (int i = threadIdx.x; i < b * b; i += blockDim.x) {
        int r = i / b, c = i % b;
        aug[r * w + c] = (r == c ? 1.f : 0.f) - S[off + i];
        aug[r * w + b + c] = dR[off + c * b + r];
    }
    __syncthreads();
    gauss_jordan(aug, b, colbuf, &piv);
    // left half is now the identity: reuse it for M
    for (int i = threadIdx.x; i < b * b; i += blockDim.x) {
        int r = i / b, c = i % b;
        float acc = aug[c * w + b + r];   // m = r term of the identity part
        for (int m = 0; m < b; ++m) acc = fmaf(Rf[off + m * b + r], aug[c * w + b + m], acc);
        aug[r * w + c] = acc;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < b * b; i += blockDim.x) {
        int r = i / b, c = i % b;
        dS[off + i] = aug[r * w + c] - aug[c * w + r];
    }
}

void launch_cayley(int nblk, int b, const float *S, uint16_t *Rb, float *Rf, cudaStream_t st)
{
    if (nblk <= 0) return;
    size_t sm = (size_t)b * 2 * b * sizeof(float);
    cudaFuncSetAttribute(k_cayley, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    k_cayley<<<nblk, 256, sm, st>>>(b, S, Rb, Rf);
    note_launch();
}

void launch_cayley_grad(int nblk, int b, const float *S, const float *Rf, const float *dR,
                        float *dS, cudaStream_t st)
{
    if (nblk <= 0) return;
    size_t sm = (size_t)b * 2 * b * sizeof(float);
    cudaFuncSetAttribute(k_cayley_grad, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    k_cayley_grad<<<nblk, 256, sm, st>>>(b, S, Rf, dR, dS);
    note_launch();
}

}  // namespace pmoe
