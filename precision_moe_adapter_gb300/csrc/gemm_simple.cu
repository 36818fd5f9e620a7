// gemm_simple.cu -- grouped GEMM over expert-sorted pair rows on CUDA
// cores with the frozen weights dequantized on the fly ("临时反量化后实行
// grouped GEMM", page 1, 技艺细节) and the layer's epilogues fused:
//   GK_FWD_GU   g, u = A W_gate^T, A W_up^T -> h = bf16(silu(g) u) (+ ctx g|u)
//   GK_FWD_DOWN o = A W_down^T              -> bf16
//   GK_BWD_G    G = A W_down (A = gathered dY) -> dh~ = bf16(w G), partial G.h~
//   GK_BWD_DX   dx~ = A W13 (A = [dg du])   -> bf16
// CTA tile: 64 rows x 64 output features, K step 32, 4 x 4 per thread.
#include "common.cuh"
#include "launch.h"

namespace pmoe {

__device__ __forceinline__ float wval(int fmt, const uint8_t *q, const uint8_t *s, int64_t Kst,
                                      int64_t row, int64_t col)
{
    if (fmt == kFmtBF16) return bf2f(((const uint16_t *)q)[row * Kst + col]);
    return dequant_elem(fmt, q, s, Kst, row, col);
}

__global__ void __launch_bounds__(256) k_gemm_simple(GemmArgs a)
{
    __shared__ float As[32][64 + 4];
    __shared__ float Bs[2][32][64 + 4];
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const int tbeg = a.chunk_tiles[a.c0], tend = a.chunk_tiles[a.c1];
    const int nft = a.Nout / 64;
    const int64_t items = (int64_t)(tend - tbeg) * nft;
    const bool dual = a.kind == GK_FWD_GU;
    const bool fwd = a.kind == GK_FWD_GU || a.kind == GK_FWD_DOWN;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const Tile tl = a.tiles[tbeg + it / nft];
        const int f0 = (int)(it % nft) * 64;
        const int slot = tl.chunk & 0xffff;
        const int64_t widx = a.slot_index ? slot : tl.expert;
        const uint8_t *wq = a.wq + widx * a.wq_stride;
        const uint8_t *wsc = a.ws ? a.ws + widx * a.ws_stride : nullptr;
        if (a.fmt == kFmtBF16) wq += a.w_off_elems * 2;
        float acc[2][4][4] = {};
        for (int k0 = 0; k0 < a.K; k0 += 32) {
            __syncthreads();
            for (int i = tid; i < 64 * 32; i += 256) {
                int r = i / 32, kk = i % 32;
                As[kk][r] = r < tl.nrows ? bf2f(a.A[(int64_t)(tl.row0 + r) * a.K + k0 + kk]) : 0.f;
                if (fwd) {
                    int n = i / 32;
                    Bs[0][kk][n] = wval(a.fmt, wq, wsc, a.Kst, f0 + n, k0 + kk);
                    if (dual) Bs[1][kk][n] = wval(a.fmt, wq, wsc, a.Kst, a.I + f0 + n, k0 + kk);
                } else {
                    int kb = i / 64, n = i % 64;
                    Bs[0][kb][n] = wval(a.fmt, wq, wsc, a.Kst, k0 + kb, f0 + n);
                }
            }
            __syncthreads();
#pragma unroll 4
            for (int kk = 0; kk < 32; ++kk) {
                float av[4], b0[4], b1[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
                for (int j = 0; j < 4; ++j) b0[j] = Bs[0][kk][tx * 4 + j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[0][i][j] = fmaf(av[i], b0[j], acc[0][i][j]);
                if (dual) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) b1[j] = Bs[1][kk][tx * 4 + j];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[1][i][j] = fmaf(av[i], b1[j], acc[1][i][j]);
                }
            }
        }
        // epilogue
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rl = ty * 4 + i;
            const bool live = rl < tl.nrows;
            const int64_t r = tl.row0 + rl;
            float part = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int f = f0 + tx * 4 + j;
                const float v = acc[0][i][j];
                if (!live) continue;
                if (a.kind == GK_FWD_GU) {
                    const float g = v, u = acc[1][i][j];
                    const float h = g / (1.f + expf(-g)) * u;
                    a.out[r * a.I + f] = f2bf(h);
                    if (a.ctx) {
                        a.ctx[r * 2 * a.I + f] = f2bf(g);
                        a.ctx[r * 2 * a.I + a.I + f] = f2bf(u);
                    }
                } else if (a.kind == GK_BWD_G) {
                    const float wr = a.w[a.perm[r]];
                    a.out[r * a.Nout + f] = f2bf(wr * v);
                    part = fmaf(v, bf2f(a.ht[r * a.Nout + f]), part);
                } else {
                    a.out[r * a.Nout + f] = f2bf(v);
                }
            }
            if (a.kind == GK_BWD_G) {
#pragma unroll
                for (int o = 8; o; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
                if (live && tx == 0) a.dtw_part[r * (a.Nout / 64) + f0 / 64] = part;
            }
        }
    }
}

void launch_gemm_simple(const GemmArgs &a, int max_tiles, cudaStream_t st)
{
    int64_t items = (int64_t)max_tiles * (a.Nout / 64);
    if (items <= 0) return;
    int grid = (int)std::min<int64_t>(items, 152 * 8);
    k_gemm_simple<<<grid, 256, 0, st>>>(a);
    note_launch();
}

}  // namespace pmoe
