// adapter.cu -- the Cayley parameterisation of the orthogonal adapter
// blocks, R = (I + S)(I - S)^{-1}, and its gradient (page 2, 机制拆解: the
// adapter is a local orthogonal transform; S skew-symmetric makes each
// block orthogonal).
#include "common.cuh"
#include "launch.h"

namespace pmoe {

// ------------------------------------------------------------------ Cayley
// R = (I + S)(I - S)^{-1} = 2 (I - S)^{-1} - I.  The inverse comes from
// Gauss-Jordan elimination on [I - S | I] without row exchanges: the
// symmetric part of I - S is I (S is skew), so every leading minor is
// nonzero and elimination without pivoting is stable (its growth is bounded
// by 1 + |S|^2).  4*B threads per block matrix; thread (row r, quarter q)
// keeps the 2B/4 entries of row r's quarter q in registers; the pivot row
// goes through shared memory (double-buffered: one barrier per column).
template <int B>
__global__ void __launch_bounds__(4 * B) k_cayley(const float *__restrict__ S,
                                                  uint16_t *__restrict__ Rb, float *__restrict__ Rf)
{
    constexpr int W = 2 * B, Q = W / 4;   // row width, entries per thread
    __shared__ float prow[2][W];
    const int r = threadIdx.x >> 2, q = threadIdx.x & 3;
    const int64_t off = (int64_t)blockIdx.x * B * B;
    float v[Q];
#pragma unroll
    for (int i = 0; i < Q; ++i) {
        const int c = q * Q + i;
        v[i] = c < B ? (r == c ? 1.f : 0.f) - S[off + r * B + c] : (r == c - B ? 1.f : 0.f);
    }
    for (int col = 0; col < B; ++col) {
        const int oq = col / Q, oi = col % Q;   // owner quarter and slot of column col
        // value of column col in this row (lane of quarter oq of the same row)
        float mine = 0.f;
#pragma unroll
        for (int i = 0; i < Q; ++i)
            if (i == oi) mine = v[i];
        constexpr unsigned kMask = 4 * B >= 32 ? 0xffffffffu : (1u << (4 * B)) - 1u;
        const float colv = __shfl_sync(kMask, mine, (threadIdx.x & 31 & ~3) | oq);
        float *pr = prow[col & 1];
        if (r == col) {
            const float inv = 1.f / colv;
#pragma unroll
            for (int i = 0; i < Q; ++i) {
                v[i] *= inv;
                pr[q * Q + i] = v[i];
            }
        }
        __syncthreads();
        if (r != col) {
#pragma unroll
            for (int i = 0; i < Q; ++i) v[i] = fmaf(-colv, pr[q * Q + i], v[i]);
        }
    }
    // right half holds A = (I - S)^{-1}; R = 2A - I
#pragma unroll
    for (int i = 0; i < Q; ++i) {
        const int c = q * Q + i - B;
        if (c < 0) continue;
        const float rv = 2.f * v[i] - (r == c ? 1.f : 0.f);
        if (Rf) Rf[off + r * B + c] = rv;
        if (Rb) Rb[off + r * B + c] = f2bf(rv);
    }
}

// dL/dS for S skew: with A = (I - S)^{-1} = (I + R)/2, a perturbation dS
// moves R by (I + R) dS A, so M = (I + R)^T G A^T = (I + R)^T G (I + R)^T / 2
// and dS = M - M^T.  Two B x B products per block in shared memory.
template <int B>
__global__ void __launch_bounds__(256) k_cayley_grad(const float *__restrict__ Rf,
                                                     const float *__restrict__ G,
                                                     float *__restrict__ dS)
{
    extern __shared__ float sm[];
    constexpr int P = B + 1;   // padded pitch
    float *Ip = sm, *Gs = sm + B * P, *T = sm + 2 * B * P;
    const int64_t off = (int64_t)blockIdx.x * B * B;
    for (int i = threadIdx.x; i < B * B; i += blockDim.x) {
        const int r = i / B, c = i % B;
        Ip[r * P + c] = Rf[off + i] + (r == c ? 1.f : 0.f);
        Gs[r * P + c] = G[off + i];
    }
    __syncthreads();
    // T = (I + R)^T G
    for (int i = threadIdx.x; i < B * B; i += blockDim.x) {
        const int r = i / B, c = i % B;
        float acc = 0.f;
        for (int m = 0; m < B; ++m) acc = fmaf(Ip[m * P + r], Gs[m * P + c], acc);
        T[r * P + c] = acc;
    }
    __syncthreads();
    // M = T (I + R)^T / 2, stored over Gs
    for (int i = threadIdx.x; i < B * B; i += blockDim.x) {
        const int r = i / B, c = i % B;
        float acc = 0.f;
        for (int m = 0; m < B; ++m) acc = fmaf(T[r * P + m], Ip[c * P + m], acc);
        Gs[r * P + c] = 0.5f * acc;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < B * B; i += blockDim.x) {
        const int r = i / B, c = i % B;
        dS[off + i] = Gs[r * P + c] - Gs[c * P + r];
    }
}

template <int B>
static void cayley_b(int nblk, const float *S, uint16_t *Rb, float *Rf, cudaStream_t st)
{
    k_cayley<B><<<nblk, 4 * B, 0, st>>>(S, Rb, Rf);
}

template <int B>
static void cayley_grad_b(int nblk, const float *Rf, const float *dR, float *dS, cudaStream_t st)
{
    const size_t sm = 3 * (size_t)B * (B + 1) * sizeof(float);
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_cayley_grad<B>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        attr = true;
    }
    k_cayley_grad<B><<<nblk, 256, sm, st>>>(Rf, dR, dS);
}

bool cayley_block_ok(int b) { return b == 2 || b == 4 || b == 8 || b == 16 || b == 32 || b == 64 || b == 128; }

void launch_cayley(int nblk, int b, const float *S, uint16_t *Rb, float *Rf, cudaStream_t st)
{
    if (nblk <= 0) return;
    switch (b) {
    case 2: cayley_b<2>(nblk, S, Rb, Rf, st); break;
    case 4: cayley_b<4>(nblk, S, Rb, Rf, st); break;
    case 8: cayley_b<8>(nblk, S, Rb, Rf, st); break;
    case 16: cayley_b<16>(nblk, S, Rb, Rf, st); break;
    case 32: cayley_b<32>(nblk, S, Rb, Rf, st); break;
    case 64: cayley_b<64>(nblk, S, Rb, Rf, st); break;
    default: cayley_b<128>(nblk, S, Rb, Rf, st); break;
    }
    note_launch();
}

void launch_cayley_grad(int nblk, int b, const float *S, const float *Rf, const float *dR,
                        float *dS, cudaStream_t st)
{
    (void)S;
    if (nblk <= 0) return;
    switch (b) {
    case 2: cayley_grad_b<2>(nblk, Rf, dR, dS, st); break;
    case 4: cayley_grad_b<4>(nblk, Rf, dR, dS, st); break;
    case 8: cayley_grad_b<8>(nblk, Rf, dR, dS, st); break;
    case 16: cayley_grad_b<16>(nblk, Rf, dR, dS, st); break;
    case 32: cayley_grad_b<32>(nblk, Rf, dR, dS, st); break;
    case 64: cayley_grad_b<64>(nblk, Rf, dR, dS, st); break;
    default: cayley_grad_b<128>(nblk, Rf, dR, dS, st); break;
    }
    note_launch();
}

}  // namespace pmoe
