// adapter.cu -- the Cayley parameterisation of the orthogonal adapter
// blocks, R = (I + S)(I - S)^{-1}, and its gradient ("Orbit：把万亿模型 RL 后训练改写成部署一致性问题", 机制拆解: the
// adapter is a local orthogonal transform; S skew-symmetric makes each
// block orthogonal).
#include "common.cuh"
#include "mma_sync.cuh"
#include "launch.h"

namespace pmoe {

// ------------------------------------------------------------------ Cayley
// R = (I + S)(I - S)^{-1} = 2 (I - S)^{-1} - I.  The inverse comes from
// in-place Gauss-Jordan elimination of I - S without row exchanges: the
// symmetric part of I - S is I (S is skew), so every leading minor is
// nonzero and elimination without pivoting is stable (its growth is bounded
// by 1 + |S|^2).  4*B threads per block matrix; thread (row r, quarter q)
// keeps columns q*B/4 .. q*B/4 + B/4 - 1 of row r in registers.  Columns
// are visited quarter by quarter with the inner loop unrolled, so every
// register index is static; the pivot row goes through shared memory
// (double-buffered: one barrier per column).
template <int B>
__global__ void __launch_bounds__(4 * B) k_cayley(const float *__restrict__ S,
                                                  uint16_t *__restrict__ Rb, float *__restrict__ Rf)
{
    constexpr int Q = B / 4;
    constexpr unsigned kMask = 4 * B >= 32 ? 0xffffffffu : (1u << (4 * B)) - 1u;
    __shared__ __align__(16) float prow[2][B];
    const int r = threadIdx.x >> 2, q = threadIdx.x & 3;
    const int lane0 = threadIdx.x & 31 & ~3;   // lane of quarter 0 of this row
    const int64_t off = (int64_t)blockIdx.x * B * B;
    float v[Q];
#pragma unroll
    for (int i = 0; i < Q; ++i) {
        const int c = q * Q + i;
        v[i] = (r == c ? 1.f : 0.f) - S[off + r * B + c];
    }
    for (int oq = 0; oq < 4; ++oq) {
#pragma unroll
        for (int i = 0; i < Q; ++i) {
            const int col = oq * Q + i;
            const float colv = __shfl_sync(kMask, v[i], lane0 | oq);
            float *pr = prow[col & 1];
            const bool mine_col = q == oq;
            if (r == col) {
                // pivot row: a[col][:] /= a[col][col], with a[col][col] <- 1 / a[col][col]
                const float p = 1.f / colv;
                if (mine_col) v[i] = 1.f;
#pragma unroll
                for (int j = 0; j < Q; ++j) v[j] *= p;
#pragma unroll
                for (int j = 0; j < Q; j += 4)
                    *(float4 *)(pr + q * Q + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            }
            __syncthreads();
            if (r != col) {
                // a[r][:] -= a[r][col] * a[col][:], with a[r][col] <- -a[r][col] / pivot
                if (mine_col) v[i] = 0.f;
#pragma unroll
                for (int j = 0; j < Q; j += 4) {
                    const float4 pv = *(const float4 *)(pr + q * Q + j);
                    v[j] = fmaf(-colv, pv.x, v[j]);
                    v[j + 1] = fmaf(-colv, pv.y, v[j + 1]);
                    v[j + 2] = fmaf(-colv, pv.z, v[j + 2]);
                    v[j + 3] = fmaf(-colv, pv.w, v[j + 3]);
                }
            }
        }
    }
    // v holds row r of A = (I - S)^{-1}; R = 2A - I
#pragma unroll
    for (int i = 0; i < Q; ++i) {
        const int c = q * Q + i;
        const float rv = 2.f * v[i] - (r == c ? 1.f : 0.f);
        if (Rf) Rf[off + r * B + c] = rv;
        if (Rb) Rb[off + r * B + c] = f2bf(rv);
    }
}

// The same elimination with one warp per block matrix (b = 16, 32, 64), so
// no block-wide barrier is needed: lane (row group rg = lane / 8, column
// group cg = lane % 8) keeps rows rg*b/4 .. +b/4-1 and columns cg*b/8 ..
// +b/8-1 in registers.  For pivot k the lanes fetch, by shuffles, the old
// column k for their rows, the pivot row for their columns and the pivot
// itself; every element then takes one fused multiply-add.  Operation for
// operation this is the elimination above, so the results are identical.
template <int B>
__global__ void __launch_bounds__(128) k_cayley_warp(int nblk, const float *__restrict__ S,
                                                     uint16_t *__restrict__ Rb, float *__restrict__ Rf)
{
    constexpr int RL = B / 4, CL = B / 8;
    static_assert(RL == 2 * CL && CL >= 2, "b = 16, 32 or 64");
    const int lane = threadIdx.x & 31;
    const int blk = blockIdx.x * 4 + (threadIdx.x >> 5);
    if (blk >= nblk) return;
    const int rg = lane >> 3, cg = lane & 7;
    const int64_t off = (int64_t)blk * B * B;
    float v[RL][CL];
#pragma unroll
    for (int i = 0; i < RL; ++i) {
        const int row = rg * RL + i;
#pragma unroll
        for (int j = 0; j < CL; j += 2) {
            const int col = cg * CL + j;
            const float2 sv = *(const float2 *)(S + off + row * B + col);
            v[i][j] = (row == col ? 1.f : 0.f) - sv.x;
            v[i][j + 1] = (row == col + 1 ? 1.f : 0.f) - sv.y;
        }
    }
    for (int g = 0; g < 4; ++g) {
        const bool in_g = rg == g;   // this lane holds part of the pivot rows
#pragma unroll
        for (int kk = 0; kk < RL; ++kk) {
            const int jj = kk % CL;               // pivot column inside its group
            const int h = 2 * g + kk / CL;        // column group of pivot k
            const bool in_h = cg == h;
            float f[RL], ps[CL];
#pragma unroll
            for (int i = 0; i < RL; ++i) f[i] = __shfl_sync(0xffffffffu, v[i][jj], (lane & ~7) | h);
#pragma unroll
            for (int j = 0; j < CL; ++j) ps[j] = __shfl_sync(0xffffffffu, v[kk][j], (g << 3) | cg);
            const float p = 1.f / __shfl_sync(0xffffffffu, v[kk][jj], (g << 3) | h);
#pragma unroll
            for (int j = 0; j < CL; ++j) ps[j] *= p;
            if (in_g) f[kk] = 0.f;   // the pivot row is only rescaled
#pragma unroll
            for (int i = 0; i < RL; ++i)
#pragma unroll
                for (int j = 0; j < CL; ++j) v[i][j] = fmaf(-f[i], ps[j], v[i][j]);
            if (in_g) {
#pragma unroll
                for (int j = 0; j < CL; ++j) v[kk][j] = ps[j];
            }
            if (in_h) {   // column k becomes column k of the inverse
#pragma unroll
                for (int i = 0; i < RL; ++i) v[i][jj] = fmaf(-f[i], p, 0.f);   // +0, never -0
                if (in_g) v[kk][jj] = p;
            }
        }
    }
    // v holds A = (I - S)^{-1}; R = 2A - I
#pragma unroll
    for (int i = 0; i < RL; ++i) {
        const int row = rg * RL + i;
#pragma unroll
        for (int j = 0; j < CL; j += 2) {
            const int col = cg * CL + j;
            const float r0 = 2.f * v[i][j] - (row == col ? 1.f : 0.f);
            const float r1 = 2.f * v[i][j + 1] - (row == col + 1 ? 1.f : 0.f);
            if (Rf) *(float2 *)(Rf + off + row * B + col) = make_float2(r0, r1);
            if (Rb) *(uint32_t *)(Rb + off + row * B + col) = pack_bf2(r0, r1);
        }
    }
}

// b = 64 with two warps per block matrix (32 rows each), so a lane keeps
// 8 x 8 elements (about 140 registers instead of 255) and three times as
// many warps fit an SM.  Lane (row group rg = lane / 8, column group
// cg = lane % 8) of warp half h keeps rows 32h + 8rg .. +7, columns
// 8cg .. +7.  For pivot k the warp holding row k scales it and puts it in
// shared memory (double-buffered, one 64-thread barrier per pivot); the
// column-k values come by shuffles inside each warp.  Operation for
// operation this is the same elimination as above (identical results).
__global__ void __launch_bounds__(128) k_cayley_pair64(int nblk, const float *__restrict__ S,
                                                       uint16_t *__restrict__ Rb,
                                                       float *__restrict__ Rf)
{
    constexpr int B = 64;
    __shared__ __align__(16) float prow[2][2][B + 4];   // [matrix][buffer][64 + p]
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int mloc = w >> 1, half = w & 1;
    const int blk = blockIdx.x * 2 + mloc;
    const bool live = blk < nblk;   // both warps of a matrix agree
    const int rg = lane >> 3, cg = lane & 7;
    const int64_t off = (int64_t)(live ? blk : 0) * B * B;
    float v[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = 32 * half + 8 * rg + i;
#pragma unroll
        for (int j = 0; j < 8; j += 4) {
            const int col = 8 * cg + j;
            const float4 sv = live ? *(const float4 *)(S + off + row * B + col) : make_float4(0, 0, 0, 0);
            v[i][j] = (row == col ? 1.f : 0.f) - sv.x;
            v[i][j + 1] = (row == col + 1 ? 1.f : 0.f) - sv.y;
            v[i][j + 2] = (row == col + 2 ? 1.f : 0.f) - sv.z;
            v[i][j + 3] = (row == col + 3 ? 1.f : 0.f) - sv.w;
        }
    }
    // Software-pipelined over pivots: while pivot k is applied, row k+1 and
    // column k+1 are finished first, so pivot k+1's multipliers (shuffles)
    // and scaled row (shared memory) are on their way while the other 49
    // updates of pivot k issue.  Each element still takes the same operations
    // in the same order.
    float f[8];
    {   // pivot 0: multipliers and scaled row
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = __shfl_sync(0xffffffffu, v[i][0], lane & ~7);
        if (half == 0) {
            const float piv = __shfl_sync(0xffffffffu, v[0][0], 0);
            const float p = 1.f / piv;
            if (rg == 0) {
                float *pr = prow[mloc][0];
                *(float4 *)(pr + 8 * cg) = make_float4(v[0][0] * p, v[0][1] * p, v[0][2] * p, v[0][3] * p);
                *(float4 *)(pr + 8 * cg + 4) = make_float4(v[0][4] * p, v[0][5] * p, v[0][6] * p, v[0][7] * p);
                if (cg == 0) pr[B] = p;
            }
        }
        asm volatile("bar.sync %0, 64;" ::"r"(1 + mloc) : "memory");
    }
    for (int kb = 0; kb < 8; ++kb) {       // pivots k = 8 kb .. 8 kb + 7
        const int owner = kb >> 2, g = kb & 3;
        const bool in_g = half == owner && rg == g;
        const bool in_h = cg == kb;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            const int k = 8 * kb + jj;
            const int j1 = (jj + 1) & 7;                      // local index of pivot k+1
            const int kb1 = kb + (jj == 7);
            const float *pr = prow[mloc][k & 1];
            const float4 q0 = *(const float4 *)(pr + 8 * cg), q1 = *(const float4 *)(pr + 8 * cg + 4);
            const float p = pr[B];
            const float ps[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
            if (in_g) f[jj] = 0.f;   // the pivot row is only rescaled
            // 1. row j1 and column j1 of pivot k's result
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j1][j] = fmaf(-f[j1], ps[j], v[j1][j]);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i != j1) v[i][j1] = fmaf(-f[i], ps[j1], v[i][j1]);
            if (in_g) v[jj][j1] = ps[j1];
            if (in_h) v[j1][jj] = fmaf(-f[j1], p, 0.f);
            // 2. pivot k+1: multipliers, and the owner's scaled row
            float fn[8];
            if (kb1 < 8) {
                const int owner1 = kb1 >> 2, g1 = kb1 & 3;
#pragma unroll
                for (int i = 0; i < 8; ++i) fn[i] = __shfl_sync(0xffffffffu, v[i][j1], (lane & ~7) | kb1);
                if (half == owner1) {
                    const float piv = __shfl_sync(0xffffffffu, v[j1][j1], (g1 << 3) | kb1);
                    const float p1 = 1.f / piv;
                    if (rg == g1) {
                        float *pn = prow[mloc][(k + 1) & 1];
                        *(float4 *)(pn + 8 * cg) =
                            make_float4(v[j1][0] * p1, v[j1][1] * p1, v[j1][2] * p1, v[j1][3] * p1);
                        *(float4 *)(pn + 8 * cg + 4) =
                            make_float4(v[j1][4] * p1, v[j1][5] * p1, v[j1][6] * p1, v[j1][7] * p1);
                        if (cg == kb1) pn[B] = p1;
                    }
                }
            }
            // 3. the rest of pivot k
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (i == j1) continue;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j != j1) v[i][j] = fmaf(-f[i], ps[j], v[i][j]);
            }
            if (in_g) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j != j1) v[jj][j] = ps[j];
            }
            if (in_h) {   // column k becomes column k of the inverse
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (i != j1) v[i][jj] = fmaf(-f[i], p, 0.f);
                if (in_g) v[jj][jj] = p;
            }
            if (kb1 < 8) {
#pragma unroll
                for (int i = 0; i < 8; ++i) f[i] = fn[i];
            }
            asm volatile("bar.sync %0, 64;" ::"r"(1 + mloc) : "memory");
        }
    }
    if (!live) return;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = 32 * half + 8 * rg + i;
        float r[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) r[j] = 2.f * v[i][j] - (row == 8 * cg + j ? 1.f : 0.f);
        if (Rf) {
            *(float4 *)(Rf + off + row * B + 8 * cg) = make_float4(r[0], r[1], r[2], r[3]);
            *(float4 *)(Rf + off + row * B + 8 * cg + 4) = make_float4(r[4], r[5], r[6], r[7]);
        }
        if (Rb)
            *(uint4 *)(Rb + off + row * B + 8 * cg) =
                make_uint4(pack_bf2(r[0], r[1]), pack_bf2(r[2], r[3]), pack_bf2(r[4], r[5]),
                           pack_bf2(r[6], r[7]));
    }
}

// Small blocks (b <= 8): one thread per block matrix, the same in-place
// elimination in registers.
template <int B>
__global__ void k_cayley_small(int nblk, const float *__restrict__ S, uint16_t *__restrict__ Rb,
                               float *__restrict__ Rf)
{
    const int blk = blockIdx.x * blockDim.x + threadIdx.x;
    if (blk >= nblk) return;
    const int64_t off = (int64_t)blk * B * B;
    float a[B][B];
#pragma unroll
    for (int r = 0; r < B; ++r)
#pragma unroll
        for (int c = 0; c < B; ++c) a[r][c] = (r == c ? 1.f : 0.f) - S[off + r * B + c];
#pragma unroll
    for (int k = 0; k < B; ++k) {
        const float p = 1.f / a[k][k];
        a[k][k] = 1.f;
#pragma unroll
        for (int j = 0; j < B; ++j) a[k][j] *= p;
#pragma unroll
        for (int r = 0; r < B; ++r) {
            if (r == k) continue;
            const float f = a[r][k];
            a[r][k] = 0.f;
#pragma unroll
            for (int j = 0; j < B; ++j) a[r][j] = fmaf(-f, a[k][j], a[r][j]);
        }
    }
#pragma unroll
    for (int r = 0; r < B; ++r)
#pragma unroll
        for (int c = 0; c < B; ++c) {
            const float rv = 2.f * a[r][c] - (r == c ? 1.f : 0.f);
            if (Rf) Rf[off + r * B + c] = rv;
            if (Rb) Rb[off + r * B + c] = f2bf(rv);
        }
}

// dL/dS for S skew: with A = (I - S)^{-1} = (I + R)/2, a perturbation dS
// moves R by (I + R) dS A, so M = (I + R)^T G A^T = (I + R)^T G (I + R)^T / 2
// and dS = M - M^T.  Two B x B products per block in shared memory, each
// thread computing a 4 x 4 tile of the output (B >= 8; smaller blocks use
// one thread per output).
template <int B>
__global__ void __launch_bounds__(256) k_cayley_grad(const float *__restrict__ Rf,
                                                     const float *__restrict__ G,
                                                     float *__restrict__ dS)
{
    extern __shared__ float sm[];
    constexpr int P = B + 4;   // padded pitch, keeps float4 alignment
    constexpr int TS = B >= 8 ? 4 : 1;   // output tile side per thread
    constexpr int NT = (B / TS) * (B / TS);
    float *Ip = sm, *Gs = sm + B * P, *T = sm + 2 * B * P;
    const int64_t off = (int64_t)blockIdx.x * B * B;
    for (int i = threadIdx.x; i < B * B; i += blockDim.x) {
        const int r = i / B, c = i % B;
        Ip[r * P + c] = Rf[off + i] + (r == c ? 1.f : 0.f);
        Gs[r * P + c] = G[off + i];
    }
    __syncthreads();
    // T[r][c] = sum_m Ip[m][r] Gs[m][c]
    for (int t = threadIdx.x; t < NT; t += blockDim.x) {
        const int r0 = (t / (B / TS)) * TS, c0 = (t % (B / TS)) * TS;
        float acc[TS][TS] = {};
        for (int m = 0; m < B; ++m) {
            float x[TS], y[TS];
#pragma unroll
            for (int u = 0; u < TS; ++u) {
                x[u] = Ip[m * P + r0 + u];
                y[u] = Gs[m * P + c0 + u];
            }
#pragma unroll
            for (int u = 0; u < TS; ++u)
#pragma unroll
                for (int w = 0; w < TS; ++w) acc[u][w] = fmaf(x[u], y[w], acc[u][w]);
        }
#pragma unroll
        for (int u = 0; u < TS; ++u)
#pragma unroll
            for (int w = 0; w < TS; ++w) T[(r0 + u) * P + c0 + w] = acc[u][w];
    }
    __syncthreads();
    // M[r][c] = 1/2 sum_m T[r][m] Ip[c][m], written over Gs
    for (int t = threadIdx.x; t < NT; t += blockDim.x) {
        const int r0 = (t / (B / TS)) * TS, c0 = (t % (B / TS)) * TS;
        float acc[TS][TS] = {};
        for (int m = 0; m < B; ++m) {
            float x[TS], y[TS];
#pragma unroll
            for (int u = 0; u < TS; ++u) {
                x[u] = T[(r0 + u) * P + m];
                y[u] = Ip[(c0 + u) * P + m];
            }
#pragma unroll
            for (int u = 0; u < TS; ++u)
#pragma unroll
                for (int w = 0; w < TS; ++w) acc[u][w] = fmaf(x[u], y[w], acc[u][w]);
        }
#pragma unroll
        for (int u = 0; u < TS; ++u)
#pragma unroll
            for (int w = 0; w < TS; ++w) Gs[(r0 + u) * P + c0 + w] = 0.5f * acc[u][w];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < B * B; i += blockDim.x) {
        const int r = i / B, c = i % B;
        dS[off + i] = Gs[r * P + c] - Gs[c * P + r];
    }
}

// The same gradient for b >= 8 with every operand read as row segments:
// I + R, its transpose and G are staged in shared memory (pitch b + 4,
// float4-aligned), each thread computes 4 x 4 output tiles as sums of outer
// products, T = (I+R)^T G goes back transposed over G, and
// M = T (I+R)^T / 2 over I + R, so dS = M - M^T reads M twice.
template <int B>
__global__ void __launch_bounds__(256) k_cayley_grad4(const float *__restrict__ Rf,
                                                      const float *__restrict__ G,
                                                      float *__restrict__ dS)
{
    extern __shared__ __align__(16) float sm[];
    constexpr int P = B + 4;
    constexpr int NT = (B / 4) * (B / 4);          // 4 x 4 tiles
    constexpr int NTT = (NT + 255) / 256;          // tiles per thread
    float *Ip = sm, *IpT = sm + B * P, *W = sm + 2 * B * P;
    const int64_t off = (int64_t)blockIdx.x * B * B;
    for (int i = threadIdx.x; i < B * B; i += blockDim.x) {
        const int r = i / B, c = i % B;
        const float x = Rf[off + i] + (r == c ? 1.f : 0.f);
        Ip[r * P + c] = x;
        IpT[c * P + r] = x;
        W[r * P + c] = G[off + i];
    }
    __syncthreads();
    // C[r][c] = sum_m L[m][r] Q[m][c] for the thread's tiles
    auto outer = [&](const float *L, const float *Q, float (&acc)[NTT][4][4]) {
#pragma unroll
        for (int u = 0; u < NTT; ++u) {
            const int t = threadIdx.x + 256 * u;
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) acc[u][a][b] = 0.f;
            if (t >= NT) continue;
            const int r0 = (t / (B / 4)) * 4, c0 = (t % (B / 4)) * 4;
#pragma unroll 8
            for (int m = 0; m < B; ++m) {
                const float4 x = *(const float4 *)(L + m * P + r0);
                const float4 y = *(const float4 *)(Q + m * P + c0);
                const float xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) acc[u][a][b] = fmaf(xs[a], ys[b], acc[u][a][b]);
            }
        }
    };
    float acc[NTT][4][4];
    outer(Ip, W, acc);              // T = (I+R)^T G
    __syncthreads();
#pragma unroll
    for (int u = 0; u < NTT; ++u) {  // W <- T^T
        const int t = threadIdx.x + 256 * u;
        if (t >= NT) continue;
        const int r0 = (t / (B / 4)) * 4, c0 = (t % (B / 4)) * 4;
#pragma unroll
        for (int b = 0; b < 4; ++b)
            *(float4 *)(W + (c0 + b) * P + r0) =
                make_float4(acc[u][0][b], acc[u][1][b], acc[u][2][b], acc[u][3][b]);
    }
    __syncthreads();
    outer(W, IpT, acc);             // 2M = T (I+R)^T: L[m][r] = T[r][m], Q[m][c] = (I+R)[c][m]
#pragma unroll
    for (int u = 0; u < NTT; ++u) {  // Ip <- M (no longer read)
        const int t = threadIdx.x + 256 * u;
        if (t >= NT) continue;
        const int r0 = (t / (B / 4)) * 4, c0 = (t % (B / 4)) * 4;
#pragma unroll
        for (int a = 0; a < 4; ++a)
            *(float4 *)(Ip + (r0 + a) * P + c0) = make_float4(0.5f * acc[u][a][0], 0.5f * acc[u][a][1],
                                                              0.5f * acc[u][a][2], 0.5f * acc[u][a][3]);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < B * B; i += blockDim.x) {
        const int r = i / B, c = i % B;
        dS[off + i] = Ip[r * P + c] - Ip[c * P + r];
    }
}

// The same gradient for b = 32, 64 on the tensor cores: both products are
// B x B x B contractions, so they run on mma.sync with every FP32 operand
// split into three BF16 terms x = hi + mid + lo (hi = bf16(x), mid =
// bf16(x - hi), lo = bf16(x - hi - mid): together within 2^-24 |x|).  The
// six products whose terms sum to at most 2^-16 of the leading one are
// accumulated in FP32 (smallest first), which keeps FP32 accuracy.
// Warp w computes output rows 16 w .. 16 w + 15, all B columns.
//   T  = (I+R)^T G         A(m, k) = (I+R)[k][m], B(k, n) = G[k][n]
//   2M = T (I+R)^T         A(m, k) = T[m][k],     B(k, n) = (I+R)[n][k]
//   dS = M - M^T
__device__ __forceinline__ void split3(float x, uint16_t &h, uint16_t &m, uint16_t &l)
{
    h = f2bf(x);
    const float r1 = x - bf2f(h);
    m = f2bf(r1);
    l = f2bf(r1 - bf2f(m));
}

template <int B>
struct CgMma {
    static constexpr int kWarps = B / 16;
    static constexpr int kNT = B / 8;          // 8-wide output column tiles
    static constexpr int kPB = B + 8;          // BF16 plane pitch (conflict-free ldmatrix)
    static constexpr int kPF = B + 4;          // FP32 pitch of M
    static constexpr int kPlane = B * kPB;     // elements per plane
    static constexpr int kBytes = 2 * 3 * kPlane * 2;   // planes of I + R, of G then T (M over the first)
    static_assert(B * kPF * 4 <= 3 * kPlane * 2, "M fits over the I + R planes");
};

template <int B>
__global__ void __launch_bounds__(B * 2) k_cayley_grad_mma(const float *__restrict__ Rf,
                                                           const float *__restrict__ G,
                                                           float *__restrict__ dS)
{
    using C = CgMma<B>;
    extern __shared__ __align__(16) uint8_t cgsm[];
    uint16_t *Pp = (uint16_t *)cgsm, *Qp = Pp + 3 * C::kPlane;
    const uint32_t P_a = (uint32_t)__cvta_generic_to_shared(Pp), Q_a = P_a + 3 * C::kPlane * 2;
    const int64_t off = (int64_t)blockIdx.x * B * B;
    for (int i = threadIdx.x * 4; i < B * B; i += blockDim.x * 4) {
        const int r = i / B, c = i % B;
        const float4 rv = *(const float4 *)(Rf + off + i), gv = *(const float4 *)(G + off + i);
        const float x[4] = {rv.x + (r == c ? 1.f : 0.f), rv.y + (r == c + 1 ? 1.f : 0.f),
                            rv.z + (r == c + 2 ? 1.f : 0.f), rv.w + (r == c + 3 ? 1.f : 0.f)};
        const float y[4] = {gv.x, gv.y, gv.z, gv.w};
        uint16_t xs[3][4], ys[3][4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            split3(x[q], xs[0][q], xs[1][q], xs[2][q]);
            split3(y[q], ys[0][q], ys[1][q], ys[2][q]);
        }
#pragma unroll
        for (int pl = 0; pl < 3; ++pl) {
            *(uint2 *)(Pp + pl * C::kPlane + r * C::kPB + c) =
                make_uint2((uint32_t)xs[pl][0] | ((uint32_t)xs[pl][1] << 16), (uint32_t)xs[pl][2] | ((uint32_t)xs[pl][3] << 16));
            *(uint2 *)(Qp + pl * C::kPlane + r * C::kPB + c) =
                make_uint2((uint32_t)ys[pl][0] | ((uint32_t)ys[pl][1] << 16), (uint32_t)ys[pl][2] | ((uint32_t)ys[pl][3] << 16));
        }
    }
    __syncthreads();
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    // the six term pairs (a, b) with a + b <= 2, smallest first
    constexpr int kTa[6] = {2, 1, 0, 1, 0, 0}, kTb[6] = {0, 1, 2, 0, 1, 0};
    float acc[C::kNT][4];
#pragma unroll
    for (int n = 0; n < C::kNT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    // T = (I+R)^T G
#pragma unroll
    for (int kk = 0; kk < B / 16; ++kk) {
        uint32_t a[3][4];
        const int krow = kk * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int mcol = 16 * w + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int pa = 0; pa < 3; ++pa)
            ldsm_x4_t(P_a + (pa * C::kPlane + krow * C::kPB + mcol) * 2, a[pa][0], a[pa][1], a[pa][2], a[pa][3]);
#pragma unroll
        for (int n = 0; n < C::kNT; n += 2) {
            uint32_t bq[3][4];
            const int brow = kk * 16 + (lane & 15), bcol = n * 8 + (lane >> 4) * 8;
#pragma unroll
            for (int pb = 0; pb < 3; ++pb)
                ldsm_x4_t(Q_a + (pb * C::kPlane + brow * C::kPB + bcol) * 2, bq[pb][0], bq[pb][1], bq[pb][2], bq[pb][3]);
#pragma unroll
            for (int u = 0; u < 6; ++u) {
                const uint32_t *A = a[kTa[u]], *Bv = bq[kTb[u]];
                mma16816(acc[n], A[0], A[1], A[2], A[3], Bv[0], Bv[1]);
                mma16816(acc[n + 1], A[0], A[1], A[2], A[3], Bv[2], Bv[3]);
            }
        }
    }
    __syncthreads();   // every warp is done with the planes of G
#pragma unroll
    for (int n = 0; n < C::kNT; ++n)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = 16 * w + g + 8 * h, col = n * 8 + 2 * t;
            uint16_t h0, m0, l0, h1, m1, l1;
            split3(acc[n][2 * h], h0, m0, l0);
            split3(acc[n][2 * h + 1], h1, m1, l1);
            uint32_t *q = (uint32_t *)(Qp + row * C::kPB + col);
            q[0] = (uint32_t)h0 | ((uint32_t)h1 << 16);
            q[C::kPlane / 2] = (uint32_t)m0 | ((uint32_t)m1 << 16);
            q[C::kPlane] = (uint32_t)l0 | ((uint32_t)l1 << 16);
            acc[n][2 * h] = acc[n][2 * h + 1] = 0.f;
        }
    __syncthreads();
    // 2M = T (I+R)^T
#pragma unroll
    for (int kk = 0; kk < B / 16; ++kk) {
        uint32_t a[3][4];
        const int arow = 16 * w + (lane & 15), acol = kk * 16 + (lane >> 4) * 8;
#pragma unroll
        for (int pa = 0; pa < 3; ++pa)
            ldsm_x4(Q_a + (pa * C::kPlane + arow * C::kPB + acol) * 2, a[pa][0], a[pa][1], a[pa][2], a[pa][3]);
#pragma unroll
        for (int n = 0; n < C::kNT; n += 2) {
            uint32_t bq[3][4];
            const int nrow = n * 8 + (lane & 7) + ((lane >> 4) << 3);
            const int kcol = kk * 16 + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int pb = 0; pb < 3; ++pb)
                ldsm_x4(P_a + (pb * C::kPlane + nrow * C::kPB + kcol) * 2, bq[pb][0], bq[pb][1], bq[pb][2], bq[pb][3]);
#pragma unroll
            for (int u = 0; u < 6; ++u) {
                const uint32_t *A = a[kTa[u]], *Bv = bq[kTb[u]];
                mma16816(acc[n], A[0], A[1], A[2], A[3], Bv[0], Bv[1]);
                mma16816(acc[n + 1], A[0], A[1], A[2], A[3], Bv[2], Bv[3]);
            }
        }
    }
    __syncthreads();   // every warp is done with the planes of I + R: M goes over them
    float *Mf = (float *)cgsm;
#pragma unroll
    for (int n = 0; n < C::kNT; ++n)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = 16 * w + g + 8 * h, col = n * 8 + 2 * t;
            *(float2 *)(Mf + row * C::kPF + col) = make_float2(0.5f * acc[n][2 * h], 0.5f * acc[n][2 * h + 1]);
        }
    __syncthreads();
    for (int i = threadIdx.x; i < B * B; i += blockDim.x) {
        const int r = i / B, c = i % B;
        dS[off + i] = Mf[r * C::kPF + c] - Mf[c * C::kPF + r];
    }
}

template <int B>
static void cayley_b(int nblk, const float *S, uint16_t *Rb, float *Rf, cudaStream_t st)
{
    if constexpr (B < 16)
        k_cayley_small<B><<<(int)cdiv(nblk, 128), 128, 0, st>>>(nblk, S, Rb, Rf);
    else if constexpr (B == 64)
        k_cayley_pair64<<<(int)cdiv(nblk, 2), 128, 0, st>>>(nblk, S, Rb, Rf);
    else if constexpr (B <= 32)
        k_cayley_warp<B><<<(int)cdiv(nblk, 4), 128, 0, st>>>(nblk, S, Rb, Rf);
    else
        k_cayley<B><<<nblk, 4 * B, 0, st>>>(S, Rb, Rf);
}

template <int B>
static void cayley_grad_b(int nblk, const float *Rf, const float *dR, float *dS, cudaStream_t st)
{
    const size_t sm = 3 * (size_t)B * (B + 4) * sizeof(float);
    static bool attr = false;
    if constexpr (B == 32 || B == 64) {
        if (!attr) {
            cudaFuncSetAttribute(k_cayley_grad_mma<B>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 CgMma<B>::kBytes);
            attr = true;
        }
        k_cayley_grad_mma<B><<<nblk, 2 * B, CgMma<B>::kBytes, st>>>(Rf, dR, dS);
    } else if constexpr (B >= 8) {
        if (!attr) {
            cudaFuncSetAttribute(k_cayley_grad4<B>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
            attr = true;
        }
        k_cayley_grad4<B><<<nblk, 256, sm, st>>>(Rf, dR, dS);
    } else {
        if (!attr) {
            cudaFuncSetAttribute(k_cayley_grad<B>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
            attr = true;
        }
        k_cayley_grad<B><<<nblk, 256, sm, st>>>(Rf, dR, dS);
    }
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
