// rotate_tc.cu -- the block-diagonal orthogonal adapter on the tensor cores
// (page 2, 机制拆解: OFT, a local orthogonal transform of the activations).
//
//   out[r, beta] = bf16( src[row(r), beta] R_e[beta] )      (or R_e[beta]^T)
//
// for expert-sorted pair rows r of one expert e per tile, each b-wide
// block beta separately.  The rotation is a dense contraction of b
// multiply-adds per element (b = 64: 32 FLOP per byte moved), so it runs
// on mma.sync m16n8k16 (BF16 in, FP32 accumulate); the kernel is bound by
// moving the rows.  One CTA = 4 warps x 16 rows = a 64-row tile of one
// expert; work items are (tile, group of blocks).
//
// Epilogues: plain BF16 store, or the SwiGLU backward (dh = dh~ R^T, then
// dg = dh u s(g)(1 + g(1 - s(g))), du = dh silu(g) from the saved g, u).
//
// Also: the per-block adapter gradient dR[e][beta] = sum_r a_blk^T g_blk
// over the rows of expert e, in a fixed order (deterministic).
#include "common.cuh"
#include "launch.h"

namespace pmoe {

constexpr int kRotRows = 64;      // rows per tile
constexpr int kRotBlocks = 8;     // b-blocks per work item

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &a, uint32_t &b, uint32_t &c,
                                        uint32_t &d)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &a, uint32_t &b, uint32_t &c,
                                          uint32_t &d)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool pred)
{
    int sz = pred ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(sz)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

enum RotEpi { ROT_STORE = 0, ROT_SWIGLU_BWD = 1 };

struct RotArgs {
    const uint16_t *src;       // source rows
    int64_t src_ld;            // elements between source rows
    int gather;                // source row = perm[r] / k (else r)
    const int32_t *perm;
    int k;
    const int32_t *idx_flat;   // expert of pair p (per-expert R)
    const uint16_t *R;         // rotation blocks [dim/b, b, b] of expert 0, or NULL (identity)
    int64_t stride;            // elements between experts' block sets (0 = shared)
    int dim;
    uint16_t *out;             // [P, out_ld] bf16
    int64_t out_ld;
    const Tile *tiles;         // 64-row tiles of one expert, or NULL: rows 64i.. of one set
    const int32_t *tbeg, *tend;   // device range of tiles to process
    int nrows;                 // rows when tiles == NULL
    const uint16_t *ctx;       // ROT_SWIGLU_BWD: [g | u | h] rows of 3*dim
    const uint16_t *R_alt;     // second adapter slot (NULL: none)
    const uint64_t *sel;       // adapter snapshot: low bit of the low word picks R_alt
};

// smem row pitch (elements): b + 8 keeps ldmatrix rows on distinct banks
template <int B>
struct RotSmem {
    static constexpr int kPitch = B + 8;
    static constexpr int kX = kRotRows * kPitch;   // x tile
    static constexpr int kR = (B > kRotRows ? B : kRotRows) * kPitch;   // rotation block / du tile
    static constexpr int kBytes = (kX + kR) * 2;
};

template <int B, bool TRANS, int EPI>
__global__ void __launch_bounds__(128) k_rotate_mma(RotArgs a)
{
    using S = RotSmem<B>;
    extern __shared__ __align__(16) uint16_t rsm[];
    uint16_t *xs = rsm, *rs = rsm + S::kX;
    const uint32_t xs_a = (uint32_t)__cvta_generic_to_shared(xs);
    const uint32_t rs_a = (uint32_t)__cvta_generic_to_shared(rs);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nblk = a.dim / B;
    const int ngroups = (nblk + kRotBlocks - 1) / kRotBlocks;
    const int t0 = a.tiles ? *a.tbeg : 0;
    const int nt = a.tiles ? *a.tend - t0 : (a.nrows + kRotRows - 1) / kRotRows;
    const int64_t items = (int64_t)nt * ngroups;
    constexpr int CPR = B / 8;   // 16-byte chunks per block row

    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        Tile tl;
        if (a.tiles) {
            tl = a.tiles[t0 + it / ngroups];
        } else {
            tl.expert = 0;
            tl.row0 = (int)(it / ngroups) * kRotRows;
            tl.nrows = min(kRotRows, a.nrows - tl.row0);
        }
        const int bg = (int)(it % ngroups);
        const uint16_t *Re = (a.sel && (*a.sel & 1u)) ? a.R_alt : a.R;
        if (Re && a.stride) Re += (int64_t)tl.expert * a.stride;
        for (int beta = bg * kRotBlocks; beta < min(nblk, (bg + 1) * kRotBlocks); ++beta) {
            __syncthreads();
            // stage the x tile (64 rows x B) and the rotation block (B x B)
            for (int i = threadIdx.x; i < kRotRows * CPR; i += 128) {
                const int rr = i / CPR, c = i % CPR;
                const bool live = rr < tl.nrows;
                const int r = tl.row0 + (live ? rr : 0);
                const int64_t srow = a.gather ? (int64_t)(a.perm[r] / a.k) : r;
                cp_async16(xs_a + (rr * S::kPitch + c * 8) * 2,
                           a.src + srow * a.src_ld + beta * B + c * 8, live);
            }
            if (Re)
                for (int i = threadIdx.x; i < B * CPR; i += 128) {
                    const int rr = i / CPR, c = i % CPR;
                    cp_async16(rs_a + (rr * S::kPitch + c * 8) * 2,
                               Re + (int64_t)beta * B * B + rr * B + c * 8, true);
                }
            cp_async_wait_all();
            __syncthreads();

            // warp w: rows 16w .. 16w+15, all B output columns
            float acc[B / 8][4];
#pragma unroll
            for (int n = 0; n < B / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
            if (Re) {
#pragma unroll
                for (int kk = 0; kk < B / 16; ++kk) {
                    uint32_t a0, a1, a2, a3;
                    {
                        const int row = 16 * warp + (lane & 15);
                        const int col = kk * 16 + (lane >> 4) * 8;
                        ldsm_x4(xs_a + (row * S::kPitch + col) * 2, a0, a1, a2, a3);
                    }
#pragma unroll
                    for (int n = 0; n < B / 8; n += 2) {
                        uint32_t b0, b1, b2, b3;
                        if (!TRANS) {
                            // B(k, n) = R[k][n], row-major [k][n]: transposed 8x8 loads
                            const int krow = kk * 16 + (lane & 15);
                            const int ncol = n * 8 + (lane >> 4) * 8;
                            ldsm_x4_t(rs_a + (krow * S::kPitch + ncol) * 2, b0, b1, b2, b3);
                            mma16816(acc[n], a0, a1, a2, a3, b0, b1);
                            mma16816(acc[n + 1], a0, a1, a2, a3, b2, b3);
                        } else {
                            // B(k, n) = R[n][k]: row-major [n][k] is the col layout
                            const int nrow = n * 8 + (lane & 7) + ((lane >> 4) << 3);
                            const int kcol = kk * 16 + ((lane >> 3) & 1) * 8;
                            ldsm_x4(rs_a + (nrow * S::kPitch + kcol) * 2, b0, b1, b2, b3);
                            mma16816(acc[n], a0, a1, a2, a3, b0, b1);
                            mma16816(acc[n + 1], a0, a1, a2, a3, b2, b3);
                        }
                    }
                }
            } else {
                // identity: C = A
                const int g = lane >> 2, t = lane & 3;
#pragma unroll
                for (int n = 0; n < B / 8; ++n)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int row = 16 * warp + g + 8 * h;
                        const uint32_t v = *(const uint32_t *)(xs + row * S::kPitch + n * 8 + 2 * t);
                        acc[n][2 * h] = bf2f(v & 0xFFFFu);
                        acc[n][2 * h + 1] = bf2f(v >> 16);
                    }
            }
            __syncthreads();   // x tile reads done: reuse it for the output tile
            {
                const int g = lane >> 2, t = lane & 3;
#pragma unroll
                for (int n = 0; n < B / 8; ++n)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int rl = 16 * warp + g + 8 * h;
                        const int col = n * 8 + 2 * t;
                        float v0 = acc[n][2 * h], v1 = acc[n][2 * h + 1];
                        uint32_t packed;
                        if (EPI == ROT_SWIGLU_BWD) {
                            packed = 0;
                            if (rl < tl.nrows) {
                                const int64_t r = tl.row0 + rl;
                                const uint16_t *c = a.ctx + r * 3 * a.dim + beta * B + col;
                                const uint32_t gg = *(const uint32_t *)c;
                                const uint32_t uu = *(const uint32_t *)(c + a.dim);
                                const float g0 = bf2f(gg & 0xFFFFu), g1 = bf2f(gg >> 16);
                                const float u0 = bf2f(uu & 0xFFFFu), u1 = bf2f(uu >> 16);
                                const float s0 = 1.f / (1.f + expf(-g0)), s1 = 1.f / (1.f + expf(-g1));
                                // dg into the x tile, du into the rotation block region
                                const uint32_t dg = pack_bf2(v0 * u0 * s0 * (1.f + g0 * (1.f - s0)),
                                                             v1 * u1 * s1 * (1.f + g1 * (1.f - s1)));
                                const uint32_t du = pack_bf2(v0 * g0 * s0, v1 * g1 * s1);
                                *(uint32_t *)(rs + rl * S::kPitch + col) = du;
                                packed = dg;
                            }
                        } else {
                            packed = pack_bf2(v0, v1);
                        }
                        *(uint32_t *)(xs + rl * S::kPitch + col) = packed;
                    }
            }
            __syncthreads();
            for (int i = threadIdx.x; i < kRotRows * CPR; i += 128) {
                const int rr = i / CPR, c = i % CPR;
                if (rr >= tl.nrows) continue;
                const int64_t r = tl.row0 + rr;
                const uint4 v = *(const uint4 *)(xs + rr * S::kPitch + c * 8);
                *(uint4 *)(a.out + r * a.out_ld + beta * B + c * 8) = v;
                if (EPI == ROT_SWIGLU_BWD) {
                    const uint4 du = *(const uint4 *)(rs + rr * S::kPitch + c * 8);
                    *(uint4 *)(a.out + r * a.out_ld + a.dim + beta * B + c * 8) = du;
                }
            }
        }
    }
}

template <int B, bool TRANS, int EPI>
static void rot_launch(const RotArgs &a, int max_tiles, cudaStream_t st)
{
    using S = RotSmem<B>;
    const int ngroups = (a.dim / B + kRotBlocks - 1) / kRotBlocks;
    int64_t items = (int64_t)max_tiles * ngroups;
    int grid = (int)std::min<int64_t>(items, 152 * 8);
    if (grid <= 0) return;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_rotate_mma<B, TRANS, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             S::kBytes);
        attr = true;
    }
    k_rotate_mma<B, TRANS, EPI><<<grid, 128, S::kBytes, st>>>(a);
    note_launch();
}

template <bool TRANS, int EPI>
static void rot_dispatch(int b, const RotArgs &a, int max_tiles, cudaStream_t st)
{
    switch (b) {
    case 16: rot_launch<16, TRANS, EPI>(a, max_tiles, st); break;
    case 32: rot_launch<32, TRANS, EPI>(a, max_tiles, st); break;
    case 64: rot_launch<64, TRANS, EPI>(a, max_tiles, st); break;
    default: rot_launch<128, TRANS, EPI>(a, max_tiles, st); break;
    }
}

void launch_rotate_tc(int b, bool trans, bool swiglu_bwd, const uint16_t *src, int64_t src_ld,
                      bool gather, const int32_t *perm, int k, const int32_t *idx_flat,
                      const uint16_t *R, int64_t stride, int dim, uint16_t *out, int64_t out_ld,
                      const Tile *tiles, const int32_t *tbeg, const int32_t *tend, int max_tiles,
                      int nrows, const uint16_t *ctx, cudaStream_t st, const uint16_t *R_alt,
                      const uint64_t *sel)
{
    RotArgs a{src, src_ld, gather ? 1 : 0, perm, k, idx_flat, R, stride, dim, out, out_ld, tiles,
              tbeg, tend, nrows, ctx, R_alt, sel};
    if (!tiles) max_tiles = (nrows + kRotRows - 1) / kRotRows;
    if (swiglu_bwd) rot_dispatch<true, ROT_SWIGLU_BWD>(b, a, max_tiles, st);
    else if (trans) rot_dispatch<true, ROT_STORE>(b, a, max_tiles, st);
    else rot_dispatch<false, ROT_STORE>(b, a, max_tiles, st);
}

// ------------------------------------------------------------------ dR
// dR[s][beta] = sum over the rows of set s (fixed order) of a_blk^T g_blk,
// on mma.sync: A(m = i, k = row) = a[row][i] and B(k = row, n = j) =
// g[row][j] both come from row-major [rows x b] tiles through transposed
// 8x8 loads.  One CTA per (set, block); warp w owns output rows
// i = 16w .. 16w+15 (b = 64: 4 warps; b = 128: 8 warps; b = 16, 32: one
// warp per 16 rows, the rest idle).
struct OuterArgs {
    const uint16_t *a;         // rows of a (gathered: perm[r] / k)
    int64_t a_ld;
    int gather;
    const int32_t *perm;
    int k;
    const uint16_t *g;         // rows of g, expert-sorted
    int64_t g_ld;
    const int32_t *offsets;    // rows of set s: offsets[s] .. offsets[s+1] (NULL: all rows)
    int nrows;
    int dim;
    float *dR;
};

template <int B>
__global__ void __launch_bounds__(256) k_outer_mma(OuterArgs p)
{
    constexpr int RB = 64;              // rows per K stage
    constexpr int PITCH = B + 8;
    __shared__ __align__(16) uint16_t as[RB * PITCH], gs[RB * PITCH];
    const uint32_t as_a = (uint32_t)__cvta_generic_to_shared(as);
    const uint32_t gs_a = (uint32_t)__cvta_generic_to_shared(gs);
    const int nb = p.dim / B;
    const int s = blockIdx.x / nb, beta = blockIdx.x % nb;
    const int r0 = p.offsets ? p.offsets[s] : 0, r1 = p.offsets ? p.offsets[s + 1] : p.nrows;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int CPR = B / 8;
    const bool active = warp < B / 16;
    float acc[B / 8][4];
#pragma unroll
    for (int n = 0; n < B / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    for (int rb = r0; rb < r1; rb += RB) {
        const int n_live = min(RB, r1 - rb);
        __syncthreads();
        for (int i = threadIdx.x; i < RB * CPR; i += 256) {
            const int rr = i / CPR, c = i % CPR;
            const bool live = rr < n_live;
            const int r = rb + (live ? rr : 0);
            const int64_t arow = p.gather ? (int64_t)(p.perm[r] / p.k) : r;
            cp_async16(as_a + (rr * PITCH + c * 8) * 2, p.a + arow * p.a_ld + beta * B + c * 8, live);
            cp_async16(gs_a + (rr * PITCH + c * 8) * 2, p.g + (int64_t)r * p.g_ld + beta * B + c * 8,
                       live);
        }
        cp_async_wait_all();
        __syncthreads();
        if (active) {
#pragma unroll
            for (int kk = 0; kk < RB / 16; ++kk) {
                // A(m, k) = a[k][m]: transposed 8x8 loads of the [rows x b] tile
                uint32_t a0, a1, a2, a3;
                {
                    const int krow = kk * 16 + (lane & 7) + ((lane >> 4) << 3);
                    const int mcol = 16 * warp + ((lane >> 3) & 1) * 8;
                    ldsm_x4_t(as_a + (krow * PITCH + mcol) * 2, a0, a1, a2, a3);
                }
#pragma unroll
                for (int n = 0; n < B / 8; n += 2) {
                    uint32_t b0, b1, b2, b3;
                    const int krow = kk * 16 + (lane & 15);
                    const int ncol = n * 8 + (lane >> 4) * 8;
                    ldsm_x4_t(gs_a + (krow * PITCH + ncol) * 2, b0, b1, b2, b3);
                    mma16816(acc[n], a0, a1, a2, a3, b0, b1);
                    mma16816(acc[n + 1], a0, a1, a2, a3, b2, b3);
                }
            }
        }
    }
    if (active) {
        float *D = p.dR + ((int64_t)s * nb + beta) * B * B;
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int n = 0; n < B / 8; ++n)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int i = 16 * warp + g + 8 * h, j = n * 8 + 2 * t;
                *(float2 *)(D + i * B + j) = make_float2(acc[n][2 * h], acc[n][2 * h + 1]);
            }
    }
}

void launch_outer_tc(int nsets, int nrows, int dim, int b, const uint16_t *a, int64_t a_ld,
                     bool gather, const int32_t *perm, int k, const uint16_t *g, int64_t g_ld,
                     const int32_t *offsets, float *dR, cudaStream_t st)
{
    OuterArgs p{a, a_ld, gather ? 1 : 0, perm, k, g, g_ld, offsets, nrows, dim, dR};
    int grid = nsets * (dim / b);
    if (grid <= 0) return;
    switch (b) {
    case 16: k_outer_mma<16><<<grid, 256, 0, st>>>(p); break;
    case 32: k_outer_mma<32><<<grid, 256, 0, st>>>(p); break;
    case 64: k_outer_mma<64><<<grid, 256, 0, st>>>(p); break;
    default: k_outer_mma<128><<<grid, 256, 0, st>>>(p); break;
    }
    note_launch();
}

}  // namespace pmoe
