// launch.h -- host-side launchers shared between the translation units of
// libpmoe (internal; the public interface is include/pmoe.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace pmoe {

// route_permute.cu
void launch_logits_f32(int T, int d, int E, const uint16_t *X, const float *Wr, float *out,
                       cudaStream_t st);
void launch_route_topk(int T, int E, int k, const float *logits, const float *bias, int32_t *idx,
                       float *w, float *logits_out, cudaStream_t st);
size_t permute_ws_bytes(int P, int E);
void launch_permute(int P, int E, const int32_t *idx, int32_t *counts, int32_t *offsets,
                    int32_t *perm, int32_t *inv_perm, int32_t *active, int32_t *num_active,
                    int32_t *hist, DevErr *err, cudaStream_t st);
void launch_build_tiles(int E, int C, int max_rows, int align, const int32_t *counts,
                        const int32_t *offsets, const int32_t *active, const int32_t *num_active,
                        Tile *tiles, int32_t *chunk_tiles, int32_t *chunk_rows, cudaStream_t st);

// dequant.cu
void launch_dequant(int fmt, const void *q, const void *s, int64_t N, int64_t K, uint16_t *out,
                    cudaStream_t st);
// Dequantize the experts of chunk `chunk` (active positions chunk*C ..) into
// scratch slots: slot j = [W13 (2I x d) | W2 (d x I)] BF16.
void launch_dequant_chunk(int fmt, int d, int I, int C, int chunk, const int32_t *active,
                          const int32_t *num_active, const void *w13, const void *s13,
                          const void *w2, const void *s2, uint16_t *scratch, cudaStream_t st);

// adapter.cu
// out[r] = bf16(src[row(r)] blockdiag(R[e(r)])) for r in [r0, r1) where the
// row range may come from device memory (rows_dev[0..1]) when non-NULL.
// row(r) = perm[r] / k when `gather` else r; e(r) = idx_flat[perm[r]] when
// R is per expert (stride != 0).  R == NULL copies (gathers) the rows.
void launch_rotate_rows(int nrows_max, int dim, int b, const uint16_t *src, bool gather,
                        const int32_t *perm, int k, const int32_t *idx_flat, const uint16_t *R,
                        int64_t stride, uint16_t *out, const int32_t *rows_dev, cudaStream_t st);
void launch_adapter_grad_dx(int rows, int dim, int b, const uint16_t *dXr, const uint16_t *R,
                            uint16_t *dX, cudaStream_t st);
// dR[s][beta] = sum over rows of set s of a_blk^T g_blk (fixed order).
// a rows: a[arow(i)] with arow(i) = perm[i]/k if perm (gather) else i.
// Sets: per expert (offsets given: rows offsets[s]..offsets[s+1]) or one
// set over rows [0, nrows) when offsets == NULL.
void launch_block_outer(int nsets, int nrows, int dim, int b, const uint16_t *a,
                        const int32_t *perm, int k, const uint16_t *g, const int32_t *offsets,
                        float *dR, cudaStream_t st);
void launch_cayley(int nblk, int b, const float *S, uint16_t *Rb, float *Rf, cudaStream_t st);
void launch_cayley_grad(int nblk, int b, const float *S, const float *Rf, const float *dR,
                        float *dS, cudaStream_t st);

// gemm_simple.cu
enum GemmKind { GK_FWD_GU = 0, GK_FWD_DOWN = 1, GK_BWD_G = 2, GK_BWD_DX = 3 };
constexpr int kFmtBF16 = 3;  // weights already dequantized (scratch mode)
struct GemmArgs {
    int kind;
    int fmt;                 // PMOE_W_* or kFmtBF16
    const uint8_t *wq;       // weights of expert 0 (or scratch slot 0)
    const uint8_t *ws;       // scales of expert 0
    int64_t wq_stride, ws_stride;  // bytes between experts (or slots)
    int64_t Nst, Kst;        // storage shape [Nst, Kst] of one expert's matrix
    int64_t w_off_elems;     // element offset of the matrix inside a scratch slot
    const uint16_t *A;       // activations [P, K] bf16, expert-sorted rows
    int K;                   // contraction length
    int Nout;                // output features
    const Tile *tiles;
    const int32_t *chunk_tiles;  // tile range [chunk_tiles[c0], chunk_tiles[c1])
    int c0, c1;
    bool slot_index;         // weights indexed by chunk slot (scratch) instead of expert
    uint16_t *out;           // [P, Nout] bf16
    uint16_t *ctx;           // FWD_GU: [P, 2I] g|u or NULL
    int I;
    const float *w;          // BWD_G: routing weights by pair id
    const int32_t *perm;
    const uint16_t *ht;      // BWD_G: h~ [P, I]
    float *dtw_part;         // BWD_G: [P, I/64]
};
void launch_gemm_simple(const GemmArgs &a, int max_tiles, cudaStream_t st);

// gemm_tc.cu: tcgen05 grouped GEMM (returns false if the request cannot be
// launched, e.g. the TMA descriptor could not be encoded)
bool launch_gemm_tc(const GemmArgs &g, int64_t P, DevErr *err, cudaStream_t st);
// counts / active / num_active of experts from row offsets [E+1]
void launch_offsets_to_active(int E, int rows, const int32_t *offsets, int32_t *counts,
                              int32_t *active, int32_t *num_active, DevErr *err, cudaStream_t st);

// layer.cu
void launch_combine(int T, int d, int k, const uint16_t *o, const int32_t *inv_perm,
                    const float *w, uint16_t *Y, cudaStream_t st);
void launch_gather_rows(int P, int d, int k, const uint16_t *src, const int32_t *perm,
                        uint16_t *out, cudaStream_t st);
void launch_bwd_prep(int P, int I, int b, const uint16_t *ctx, const int32_t *perm,
                     const int32_t *idx_flat, const uint16_t *R_down, int64_t stride,
                     uint16_t *h, uint16_t *ht, cudaStream_t st);
void launch_bwd_mid(int P, int I, int b, const uint16_t *ctx, const uint16_t *dht,
                    const int32_t *perm, const int32_t *idx_flat, const uint16_t *R_down,
                    int64_t stride, uint16_t *dgu, cudaStream_t st);
void launch_dtw_reduce(int P, int nparts, const float *part, const int32_t *perm, float *dtw,
                       cudaStream_t st);
void launch_combine_bwd(int T, int d, int k, int b, const uint16_t *dxt, const int32_t *inv_perm,
                        const int32_t *idx_flat, const uint16_t *R_up, int64_t stride,
                        uint16_t *dX, cudaStream_t st);

}  // namespace pmoe
