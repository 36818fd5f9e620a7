// adapter.cu -- the Cayley parameterisation of the orthogonal adapter
// blocks, R = (I + S)(I - S)^{-1}, and its gradient (page 2, 机制拆解: the
// adapter is a local orthogonal transform; S skew-symmetric makes each
// block orthogonal).
#include "common.cuh"
#include "launch.h"

namespace pmoe {

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
