// launch.h -- host-side launchers shared between the translation units of
// libpmoe (internal; the public interface is include/pmoe.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace pmoe {

// api.cu: the shape checks every entry point applies
bool dims_ok(const pmoe_dims &d);

// route_permute.cu
// Wr [d, E] f32 -> WrT3 [E, 3d] bf16 with WrT3[e][s*d + c] the s-th term of
// the exact three-term BF16 split of Wr[c][e]; and the router's token tiles.
// Router K splits: the length-3d contraction runs as router_splits(d) parts
// of 3d / router_splits(d) columns each (a function of d alone, so a token's
// logits do not depend on the batch); their partials are summed in order.
int router_splits(int d);
void launch_router_reduce(int T, int E, int splits, const float *part, float *logits, cudaStream_t st);
void launch_router_prep(int T, int d, int E, const float *Wr, uint16_t *WrT3, Tile *tiles,
                        int32_t *chunk_tiles, int tile_rows, cudaStream_t st);
int router_tile_rows(int T, int E, int splits, int num_sms);
// Canonical router mode: FP32 logits (without bias) in one fixed summation
// order (32 lane-strided fmaf chains, then a pairwise tree); d % 64 == 0.
void launch_router_exact(int T, int d, int E, const uint16_t *X, const float *Wr, float *logits,
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
bool cayley_block_ok(int b);
void launch_cayley(int nblk, int b, const float *S, uint16_t *Rb, float *Rf, cudaStream_t st);
void launch_cayley_grad(int nblk, int b, const float *S, const float *Rf, const float *dR,
                        float *dS, cudaStream_t st);

// grouped GEMM (gemm_tc*.cu)
// GK_ROUTER: FP32 logits X Wr with Wr split into three BF16 terms stacked
// along K (A = [E, 3d]); the token operand X [T, d] is read three times.
// GK_BWD_DX_F16: GK_BWD_DX with FP16 operands (the token operand A is FP16;
// the weights' BF16 values are used in FP16 encoding).
enum GemmKind { GK_FWD_GU = 0, GK_FWD_DOWN = 1, GK_BWD_G = 2, GK_BWD_DX = 3, GK_ROUTER = 4,
                GK_BWD_DX_F16 = 5 };
constexpr int kFmtBF16 = 3;  // weights already dequantized (scratch mode)
struct GemmArgs {
    int kind;
    int fmt;                 // PMOE_W_* or kFmtBF16
    const uint8_t *wq;       // weights of expert 0 (or scratch slot 0)
    const uint8_t *ws;       // scales of expert 0
    int64_t wq_stride, ws_stride;  // bytes between experts (or slots)
    int64_t Nst, Kst;        // storage shape [Nst, Kst] of one expert's matrix
    int64_t nmat;            // number of stored matrices (experts, or scratch slots)
    int64_t w_off_elems;     // element offset of the matrix inside a scratch slot
    const uint16_t *A;       // activations [P, K] bf16, expert-sorted rows
    int K;                   // contraction length
    int Kb;                  // columns of A (the token operand); 0: K
    int Nout;                // output features
    const Tile *tiles;
    const int32_t *chunk_tiles;  // tile range [chunk_tiles[c0], chunk_tiles[c1])
    int c0, c1;
    bool slot_index;         // weights indexed by chunk slot (scratch) instead of expert
    uint16_t *out;           // [P, Nout] bf16 (when outf is NULL)
    float *ctxf;             // FWD_GU: saved g | u [P, 2I] f32, or NULL
    int I;
    const float *w;          // BWD_G: routing weights by pair id
    const int32_t *perm;
    const uint16_t *ht;      // BWD_G: h~ [P, I]
    float *dtw_part;         // BWD_G: [P, I/32]
    float *outf;             // ROUTER: [splits][P, Nout] f32 partials; DOWN, BWD_G,
                             // BWD_DX*: [P, Nout] f32 output in place of out
    int64_t outf_split;      // ROUTER: P * Nout (elements between two splits' partials)
};
// tcgen05 grouped GEMM (returns false if the request cannot be
// launched, e.g. the TMA descriptor could not be encoded)
bool launch_gemm_tc(const GemmArgs &g, int64_t P, DevErr *err, cudaStream_t st);
int gemm_num_sms();   // SMs of the current device (cached)
// counts / active / num_active of experts from row offsets [E+1]
void launch_offsets_to_active(int E, int rows, const int32_t *offsets, int32_t *counts,
                              int32_t *active, int32_t *num_active, DevErr *err, cudaStream_t st);

// rotate_tc.cu: block-diagonal rotation on mma.sync.  Tiles: 128-row tiles
// of one expert (indices *tbeg .. *tend-1), or NULL for rows 0..nrows-1 of
// one shared rotation.
struct RotCall {
    int b;
    bool trans;               // R^T
    bool swiglu_bwd;          // out = FP16 [dg | du] (out_ld = 2*dim) from ctxf
    const void *src;          // BF16 rows, or FP32 rows (src_f32)
    bool src_f32;
    int64_t src_ld;
    const int32_t *perm;      // gather source row perm[r] / k (NULL: row r)
    int k;
    const uint16_t *R;        // NULL: identity
    int64_t stride;
    int dim;
    void *out;                // BF16 rows, or FP32 rows (out_f32)
    bool out_f32;
    int64_t out_ld;
    const Tile *tiles;
    const int32_t *tbeg, *tend;
    int max_tiles;
    int rows_ub;              // tiles: upper bound on the rows they hold (0: unknown)
    int nrows;
    const float *ctxf;        // swiglu_bwd: saved [g | u] rows, FP32
    const uint16_t *R_alt;
    const uint64_t *sel;
};
void launch_rotate_tc(const RotCall &c, cudaStream_t st);
// dR[s][beta] = sum over rows of set s of a_blk^T g_blk on mma.sync (g BF16,
// or FP32 when g_f32)
void launch_outer_tc(int nsets, int nrows, int dim, int b, const uint16_t *a, int64_t a_ld,
                     bool gather, const int32_t *perm, int k, const void *g, bool g_f32, int64_t g_ld,
                     const int32_t *offsets, float *dR, cudaStream_t st);
// Fused backward of the adapter for b = 64 (adapter_bwd_fused_ok): per (set,
// block), out = g R^T (FP32 rows, or with swiglu the FP16 [dg | du] from
// ctxf) and dR[set][block] = sum a^T g, reading the FP32 g once
bool adapter_bwd_fused_ok(int b);
void launch_adapter_bwd_tc(int nsets, int nrows, int dim, const float *g, const uint16_t *a, int64_t a_ld,
                           bool gather, const int32_t *perm, int k, const uint16_t *R, int64_t stride,
                           const int32_t *offsets, void *out, bool swiglu, const float *ctxf, float *dR,
                           cudaStream_t st);
constexpr int kRotTileRows = 128;

// layer.cu
// Y[t] = bf16(sum_j w[t, j] o[inv_perm[t*k + j]]) over FP32 pair rows o
void launch_combine(int T, int d, int k, const float *o, const int32_t *inv_perm,
                    const float *w, uint16_t *Y, cudaStream_t st);
// adapter slots: snap = *ctrl (one atomic 64-bit read), *version_out =
// snap >> 32 when given; publish: *ctrl = version << 32 | slot (atomic)
void launch_adapter_snapshot(const uint64_t *ctrl, uint64_t *snap, uint32_t *version_out,
                             cudaStream_t st);
void launch_adapter_publish(uint64_t *ctrl, uint32_t slot, uint32_t version, cudaStream_t st);
// offsets = [0, rows] (a single-matrix work list)
void launch_set_offsets(int32_t *offsets, int rows, cudaStream_t st);
void launch_gather_rows(int P, int d, int k, const uint16_t *src, const int32_t *perm,
                        const int32_t *nvalid, uint16_t *out, cudaStream_t st);
// d_topk_w[p] = sum of pair p's partials (row inv_perm[p]); 0 for a pair
// left out of the grouping
void launch_dtw_reduce(int P, int nparts, const float *part, const int32_t *inv_perm, float *dtw,
                       cudaStream_t st);
}  // namespace pmoe
