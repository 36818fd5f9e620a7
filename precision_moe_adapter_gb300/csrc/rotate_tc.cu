// rotate_tc.cu -- the block-diagonal orthogonal adapter on the tensor cores
// ("Orbit：把万亿模型 RL 后训练改写成部署一致性问题", 机制拆解: the OFT
// adapter is a local orthogonal transform of the activations).
//
//   out[r, beta] = src[row(r), beta] R_e[beta]      (or R_e[beta]^T)
//
// for expert-sorted pair rows r of one expert e per tile, each b-wide
// block beta separately.  The rotation is a dense contraction of b
// multiply-adds per element (b = 64: 32 FLOP per BF16 byte moved), so it
// runs on mma.sync m16n8k16 (BF16 in, FP32 accumulate); the kernel is bound
// by moving the rows.  One CTA = 8 warps x 16 rows = a 128-row tile of one
// expert; a work item is (tile, group of blocks), and the next block's rows
// and rotation block are fetched by cp.async while the current one is
// multiplied (two stages).
//
// Sources are BF16, or FP32: an FP32 row is split into hi = bf16(x) and
// lo = bf16(x - hi) (together within 2^-16 of x) and both parts go through
// the MMA, so an FP32 tensor is rotated at FP32 accuracy.
// Outputs: BF16 or FP32 rows, or the SwiGLU backward (dh = dh~ R^T, then
// dg = dh u s(g)(1 + g(1 - s(g))), du = dh silu(g) from the saved FP32 g,
// u) written as FP16 [dg | du] (11 significant bits: the operand of the
// FP16 dx~ GEMM).
//
// Also: the per-block adapter gradient dR[e][beta] = sum_r a_blk^T g_blk
// over the rows of expert e, in a fixed order (deterministic), with g BF16
// or FP32 (split the same way).
#include <cuda_fp16.h>

#include "common.cuh"
#include "exact_bf16.cuh"
#include "launch.h"
#include "mma_sync.cuh"

namespace pmoe {

constexpr int kRotRows = kRotTileRows;   // rows per tile (8 warps x 16)
constexpr int kRotBlocks = 8;            // b-blocks per work item (fewer when few tiles exist)
constexpr int kRotThreads = 256;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool pred)
{
    int sz = pred ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(sz)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

// hi = bf16(x), lo = bf16(x - hi) for two FP32 values (one BF16 pair each)
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo)
{
    hi = pack_bf2(x0, x1);
    lo = pack_bf2(x0 - bf2f(hi & 0xFFFFu), x1 - bf2f(hi >> 16));
}

// Whole warp: the exact sum over r < B of x[r] * rc[r * rstride], rounded to
// BF16 (x and rc in shared memory; every lane returns the same value).
template <int B>
__device__ __forceinline__ uint16_t warp_exact_dot_bf16(const uint16_t *x, const uint16_t *rc, int rstride,
                                                        int lane)
{
    float p0 = 0.f, p1 = 0.f;
    if (lane < B) p0 = __fmul_rn(bf2f(x[lane]), bf2f(rc[lane * rstride]));
    if (lane + 32 < B) p1 = __fmul_rn(bf2f(x[lane + 32]), bf2f(rc[(lane + 32) * rstride]));
    return warp_sum_round_bf16(p0, p1);
}

enum RotEpi { ROT_STORE = 0, ROT_SWIGLU_BWD = 1 };

struct RotArgs {
    const void *src;           // source rows, BF16 or FP32
    int64_t src_ld;            // elements between source rows
    int gather;                // source row = perm[r] / k (else r)
    const int32_t *perm;
    int k;
    const uint16_t *R;         // rotation blocks [dim/b, b, b] of expert 0, or NULL (identity)
    int64_t stride;            // elements between experts' block sets (0 = shared)
    int dim;
    void *out;                 // rows [*, out_ld], BF16 or FP32; SWIGLU: FP16 [dg | du]
    int64_t out_ld;
    const Tile *tiles;         // 128-row tiles of one expert, or NULL: rows 128i.. of one set
    const int32_t *tbeg, *tend;   // device range of tiles to process
    int nrows;                 // rows when tiles == NULL
    const float *ctxf;         // SWIGLU: saved [g | u] rows of 2*dim FP32
    const uint16_t *R_alt;     // second adapter slot (NULL: none)
    const uint64_t *sel;       // adapter snapshot: low bit of the low word picks R_alt
    int gblk;                  // b-blocks per work item
};

// Shared memory of one stage: the source tile (BF16 rows of b + 8
// elements for conflict-free ldmatrix, or FP32 rows of b + 8 floats for
// conflict-free float2 fragment loads) and the rotation block.
template <int B, bool F32IN>
struct RotSmem {
    static constexpr int kPitchX = B + 8;                   // elements per source row
    static constexpr int kXBytes = kRotRows * kPitchX * (F32IN ? 4 : 2);
    static constexpr int kPitchR = B + 8;
    static constexpr int kRBytes = B * kPitchR * 2;
    static constexpr int kStage = kXBytes + kRBytes;
    static constexpr int kBytes = 2 * kStage;
};

template <int B, bool TRANS, int EPI, bool F32IN, bool F32OUT>
__global__ void __launch_bounds__(kRotThreads, F32IN ? 2 : 3) k_rotate_mma(RotArgs a)
{
    using S = RotSmem<B, F32IN>;
    extern __shared__ __align__(16) uint8_t rsm[];
    const uint32_t sm0 = (uint32_t)__cvta_generic_to_shared(rsm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nblk = a.dim / B;
    const int ngroups = (nblk + a.gblk - 1) / a.gblk;
    const int t0 = a.tiles ? *a.tbeg : 0;
    const int nt = a.tiles ? *a.tend - t0 : (a.nrows + kRotRows - 1) / kRotRows;
    const int64_t items = (int64_t)nt * ngroups;
    constexpr int kEsz = F32IN ? 4 : 2;
    constexpr int CPR = B * kEsz / 16;   // 16-byte chunks per source block row
    constexpr int CPRR = B / 8;          // 16-byte chunks per rotation block row
    const int g = lane >> 2, t = lane & 3;

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
        const int b0 = bg * a.gblk, b1 = min(nblk, b0 + a.gblk);

        // stage block beta (source tile and rotation block) into buffer buf
        auto stage = [&](int beta, int buf) {
            const uint32_t xs = sm0 + buf * S::kStage, rs = xs + S::kXBytes;
            for (int i = threadIdx.x; i < kRotRows * CPR; i += kRotThreads) {
                const int rr = i / CPR, c = i % CPR;
                const bool live = rr < tl.nrows;
                const int r = tl.row0 + (live ? rr : 0);
                const int64_t srow = a.gather ? (int64_t)(a.perm[r] / a.k) : r;
                const uint8_t *src = (const uint8_t *)a.src + (srow * a.src_ld + (int64_t)beta * B) * kEsz + c * 16;
                cp_async16(xs + rr * S::kPitchX * kEsz + c * 16, src, live);
            }
            if (Re)
                for (int i = threadIdx.x; i < B * CPRR; i += kRotThreads) {
                    const int rr = i / CPRR, c = i % CPRR;
                    cp_async16(rs + (rr * S::kPitchR + c * 8) * 2,
                               Re + (int64_t)beta * B * B + rr * B + c * 8, true);
                }
            cp_async_commit();
        };

        stage(b0, 0);
        for (int beta = b0; beta < b1; ++beta) {
            const int buf = (beta - b0) & 1;
            // one barrier per block: after it, block beta's copies are visible
            // and every warp is done with block beta - 1, whose buffer then
            // takes block beta + 1
            cp_async_wait<0>();
            __syncthreads();
            if (beta + 1 < b1) stage(beta + 1, buf ^ 1);
            const uint32_t xs_a = sm0 + buf * S::kStage, rs_a = xs_a + S::kXBytes;
            const uint8_t *xs_p = rsm + buf * S::kStage;

            // warp w: rows 16w .. 16w+15, the B output columns in NS slices
            // of NB column groups of 8 (fewer live accumulators: more CTAs
            // per SM).  kExact: BF16 results rounded as the exact sum would
            // be (accabs = |x| |R| bounds the FP32 error; see
            // warp_exact_dot_bf16)
            constexpr bool kExact = EPI == ROT_STORE && !F32IN && !F32OUT && B <= 64;
            constexpr int NS = (B >= 32 && !F32IN) ? 2 : 1;   // FP32 sources: split once per block
            constexpr int NB = B / 8 / NS;
#pragma unroll 1
            for (int ns = 0; ns < NS; ++ns) {
                float acc[NB][4];
                float accabs[kExact ? NB : 1][4];
#pragma unroll
                for (int n = 0; n < NB; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
                for (int n = 0; n < (kExact ? NB : 1); ++n)
                    accabs[n][0] = accabs[n][1] = accabs[n][2] = accabs[n][3] = 0.f;
                if (Re) {
#pragma unroll
                    for (int kk = 0; kk < B / 16; ++kk) {
                        uint32_t a0, a1, a2, a3, l0 = 0, l1 = 0, l2 = 0, l3 = 0;
                        if constexpr (F32IN) {
                            const float *x0 = (const float *)xs_p + (16 * warp + g) * S::kPitchX + kk * 16 + 2 * t;
                            const float *x1 = x0 + 8 * S::kPitchX;
                            const float2 v00 = *(const float2 *)x0, v02 = *(const float2 *)(x0 + 8);
                            const float2 v10 = *(const float2 *)x1, v12 = *(const float2 *)(x1 + 8);
                            split2(v00.x, v00.y, a0, l0);
                            split2(v10.x, v10.y, a1, l1);
                            split2(v02.x, v02.y, a2, l2);
                            split2(v12.x, v12.y, a3, l3);
                        } else {
                            const int row = 16 * warp + (lane & 15);
                            const int col = kk * 16 + (lane >> 4) * 8;
                            ldsm_x4(xs_a + (row * S::kPitchX + col) * 2, a0, a1, a2, a3);
                        }
#pragma unroll
                        for (int n = 0; n < NB; n += 2) {
                            const int nn = ns * NB + n;   // column group in the block
                            uint32_t b0r, b1r, b2r, b3r;
                            if (!TRANS) {
                                // B(k, n) = R[k][n], row-major [k][n]: transposed 8x8 loads
                                const int krow = kk * 16 + (lane & 15);
                                const int ncol = nn * 8 + (lane >> 4) * 8;
                                ldsm_x4_t(rs_a + (krow * S::kPitchR + ncol) * 2, b0r, b1r, b2r, b3r);
                            } else {
                                // B(k, n) = R[n][k]: row-major [n][k] is the col layout
                                const int nrow = nn * 8 + (lane & 7) + ((lane >> 4) << 3);
                                const int kcol = kk * 16 + ((lane >> 3) & 1) * 8;
                                ldsm_x4(rs_a + (nrow * S::kPitchR + kcol) * 2, b0r, b1r, b2r, b3r);
                            }
                            mma16816(acc[n], a0, a1, a2, a3, b0r, b1r);
                            mma16816(acc[n + 1], a0, a1, a2, a3, b2r, b3r);
                            if constexpr (kExact) {
                                constexpr uint32_t m = 0x7FFF7FFFu;   // |.| of both BF16 halves
                                mma16816(accabs[n], a0 & m, a1 & m, a2 & m, a3 & m, b0r & m, b1r & m);
                                mma16816(accabs[n + 1], a0 & m, a1 & m, a2 & m, a3 & m, b2r & m, b3r & m);
                            }
                            if constexpr (F32IN) {
                                mma16816(acc[n], l0, l1, l2, l3, b0r, b1r);
                                mma16816(acc[n + 1], l0, l1, l2, l3, b2r, b3r);
                            }
                        }
                    }
                } else {
                    // identity: C = A.  An FP32 source passes as hi + lo, exactly
                    // what the two MMAs give with R = I (hi + lo is exact in
                    // FP32), so a unit rotation and no rotation agree bit for bit
#pragma unroll
                    for (int n = 0; n < NB; ++n)
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int row = 16 * warp + g + 8 * h;
                            const int col = (ns * NB + n) * 8 + 2 * t;
                            if constexpr (F32IN) {
                                const float2 v = *(const float2 *)((const float *)xs_p + row * S::kPitchX + col);
                                uint32_t hi, lo;
                                split2(v.x, v.y, hi, lo);
                                acc[n][2 * h] = bf2f(hi & 0xFFFFu) + bf2f(lo & 0xFFFFu);
                                acc[n][2 * h + 1] = bf2f(hi >> 16) + bf2f(lo >> 16);
                            } else {
                                const uint32_t v = *(const uint32_t *)((const uint16_t *)xs_p + row * S::kPitchX + col);
                                acc[n][2 * h] = bf2f(v & 0xFFFFu);
                                acc[n][2 * h + 1] = bf2f(v >> 16);
                            }
                        }
                }
                // epilogue straight from the fragments: each quad of lanes
                // writes 2 consecutive columns of one row.  kExact: bit
                // (n * 4 + h * 2 + q) of cand marks a result that may sit near
                // a rounding midpoint; the warp recomputes those afterwards
                uint32_t cand = 0;
#pragma unroll
                for (int n = 0; n < NB; ++n)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int rl = 16 * warp + g + 8 * h;
                        if (rl >= tl.nrows) continue;
                        const int64_t r = tl.row0 + rl;
                        const int col = beta * B + (ns * NB + n) * 8 + 2 * t;
                        const float v0 = acc[n][2 * h], v1 = acc[n][2 * h + 1];
                        if constexpr (EPI == ROT_SWIGLU_BWD) {
                            const float *c = a.ctxf + r * 2 * a.dim + col;
                            const float2 gg = *(const float2 *)c;
                            const float2 uu = *(const float2 *)(c + a.dim);
                            const float s0 = 1.f / (1.f + expf(-gg.x)), s1 = 1.f / (1.f + expf(-gg.y));
                            const float dg0 = v0 * uu.x * s0 * (1.f + gg.x * (1.f - s0));
                            const float dg1 = v1 * uu.y * s1 * (1.f + gg.y * (1.f - s1));
                            const float du0 = v0 * (gg.x * s0), du1 = v1 * (gg.y * s1);
                            __half2 *o = (__half2 *)((uint16_t *)a.out + r * a.out_ld + col);
                            o[0] = __floats2half2_rn(dg0, dg1);
                            o[a.dim / 2] = __floats2half2_rn(du0, du1);
                        } else if constexpr (F32OUT) {
                            *(float2 *)((float *)a.out + r * a.out_ld + col) = make_float2(v0, v1);
                        } else {
                            if constexpr (kExact) {
                                // the FP32 sum of b <= 64 products over four
                                // MMAs is within 2^-21 of the sum of their
                                // magnitudes; 2^-20 of it decides which
                                // results may sit near a rounding midpoint
                                if (Re) {
                                    const int bit = n * 4 + h * 2;
                                    cand |= (uint32_t)near_bf16_midpoint(v0, accabs[n][2 * h] * 9.5367431640625e-07f) << bit;
                                    cand |= (uint32_t)near_bf16_midpoint(v1, accabs[n][2 * h + 1] * 9.5367431640625e-07f) << (bit + 1);
                                }
                            }
                            *(uint32_t *)((uint16_t *)a.out + r * a.out_ld + col) = pack_bf2(v0, v1);
                        }
                    }
                if constexpr (kExact) {
                    // one candidate at a time, in a rolled loop (a single copy
                    // of the warp-wide exact sum): the owning lane rewrites
                    // its element after the pair store above
                    const uint16_t *rs = (const uint16_t *)(xs_p + S::kXBytes);
#pragma unroll 1
                    while (true) {
                        const uint32_t any = __ballot_sync(0xffffffffu, cand != 0u);
                        if (!any) break;
                        const int src = __ffs(any) - 1;
                        const int bit = __shfl_sync(0xffffffffu, __ffs(cand) - 1, src);
                        if (lane == src) cand &= cand - 1u;
                        const int n = bit >> 2, h = (bit >> 1) & 1, q = bit & 1;
                        const int srow = 16 * warp + (src >> 2) + 8 * h;
                        const int scol = (ns * NB + n) * 8 + 2 * (src & 3) + q;   // column in the block
                        // column scol of R (x R), or row scol (x R^T)
                        const uint16_t *rc = TRANS ? rs + scol * S::kPitchR : rs + scol;
                        const uint16_t ex = warp_exact_dot_bf16<B>((const uint16_t *)xs_p + srow * S::kPitchX, rc,
                                                                   TRANS ? 1 : S::kPitchR, lane);
                        if (lane == src)
                            ((uint16_t *)a.out)[(tl.row0 + srow) * a.out_ld + beta * B + scol] = ex;
                    }
                }
            }
        }
        __syncthreads();   // the next item restages buffer 0
    }
}

template <int B, bool TRANS, int EPI, bool F32IN, bool F32OUT>
static void rot_launch(const RotArgs &a, int max_tiles, cudaStream_t st)
{
    using S = RotSmem<B, F32IN>;
    auto kern = k_rotate_mma<B, TRANS, EPI, F32IN, F32OUT>;
    static int per_sm = 0;
    if (!per_sm) {
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kRotThreads, S::kBytes);
        if (per_sm <= 0) per_sm = 1;
    }
    // work items of kRotBlocks blocks, or fewer when the tiles are too few to
    // fill the GPU (decode: a handful of one-row tiles)
    const int nblk = a.dim / B, cap = gemm_num_sms() * per_sm;
    RotArgs ar = a;
    ar.gblk = kRotBlocks;
    while (ar.gblk > 1 && (int64_t)max_tiles * ((nblk + ar.gblk - 1) / ar.gblk) < cap) ar.gblk >>= 1;
    const int64_t items = (int64_t)max_tiles * ((nblk + ar.gblk - 1) / ar.gblk);
    const int grid = (int)std::min<int64_t>(items, (int64_t)cap);
    if (grid <= 0) return;
    kern<<<grid, kRotThreads, S::kBytes, st>>>(ar);
    note_launch();
}

template <bool TRANS, int EPI, bool F32IN, bool F32OUT>
static void rot_dispatch(int b, const RotArgs &a, int max_tiles, cudaStream_t st)
{
    switch (b) {
    case 16: rot_launch<16, TRANS, EPI, F32IN, F32OUT>(a, max_tiles, st); break;
    case 32: rot_launch<32, TRANS, EPI, F32IN, F32OUT>(a, max_tiles, st); break;
    case 64: rot_launch<64, TRANS, EPI, F32IN, F32OUT>(a, max_tiles, st); break;
    default: rot_launch<128, TRANS, EPI, F32IN, F32OUT>(a, max_tiles, st); break;
    }
}

void launch_rotate_tc(const RotCall &c, cudaStream_t st)
{

    RotArgs a{c.src, c.src_ld, c.perm ? 1 : 0, c.perm, c.k, c.R, c.stride, c.dim, c.out, c.out_ld,
              c.tiles, c.tbeg, c.tend, c.nrows, c.ctxf, c.R_alt, c.sel, kRotBlocks};
    // tiles hold at least one row each: at most rows_ub of them
    const int max_tiles = c.tiles ? (c.rows_ub > 0 ? std::min(c.max_tiles, c.rows_ub) : c.max_tiles)
                                  : (c.nrows + kRotRows - 1) / kRotRows;
    if (c.swiglu_bwd) {
        rot_dispatch<true, ROT_SWIGLU_BWD, true, false>(c.b, a, max_tiles, st);
    } else if (c.trans) {
        if (c.src_f32 && c.out_f32) rot_dispatch<true, ROT_STORE, true, true>(c.b, a, max_tiles, st);
        else if (c.src_f32) rot_dispatch<true, ROT_STORE, true, false>(c.b, a, max_tiles, st);
        else rot_dispatch<true, ROT_STORE, false, false>(c.b, a, max_tiles, st);
    } else {
        rot_dispatch<false, ROT_STORE, false, false>(c.b, a, max_tiles, st);
    }
}

// ------------------------------------------------------------------ dR
// dR[s][beta] = sum over the rows of set s (fixed order) of a_blk^T g_blk,
// on mma.sync: A(m = i, k = row) = a[row][i] and B(k = row, n = j) =
// g[row][j] both come from row-major [rows x b] BF16 tiles through
// transposed 8x8 loads; an FP32 g is split into hi and lo tiles on the way
// into shared memory, both multiplied.  One CTA per (set, block); warp w
// owns output rows i = 16w .. 16w+15 (b = 64: 4 warps; b = 128: 8 warps;
// b = 16, 32: one warp per 16 rows, the rest idle).
struct OuterArgs {
    const uint16_t *a;         // rows of a (gathered: perm[r] / k)
    int64_t a_ld;
    int gather;
    const int32_t *perm;
    int k;
    const void *g;             // rows of g, expert-sorted, BF16 or FP32
    int64_t g_ld;
    const int32_t *offsets;    // rows of set s: offsets[s] .. offsets[s+1] (NULL: all rows)
    int nrows;
    int dim;
    float *dR;
};

constexpr int kOuterRows = 64;   // rows per K stage
template <int B, bool F32G>
struct OuterSmem {
    static constexpr int kPitch = B + 8;
    static constexpr int kTile = kOuterRows * kPitch * 2;
    static constexpr int kBytes = kTile * (F32G ? 3 : 2);   // a, g (hi), g lo
};

template <int B, bool F32G>
__global__ void __launch_bounds__(256) k_outer_mma(OuterArgs p)
{
    using S = OuterSmem<B, F32G>;
    constexpr int RB = kOuterRows;
    constexpr int PITCH = S::kPitch;
    extern __shared__ __align__(16) uint8_t osm[];
    uint16_t *as = (uint16_t *)osm, *gs = as + RB * PITCH, *gl = gs + RB * PITCH;
    const uint32_t as_a = (uint32_t)__cvta_generic_to_shared(as);
    const uint32_t gs_a = (uint32_t)__cvta_generic_to_shared(gs);
    const uint32_t gl_a = (uint32_t)__cvta_generic_to_shared(gl);
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
            if constexpr (!F32G)
                cp_async16(gs_a + (rr * PITCH + c * 8) * 2,
                           (const uint16_t *)p.g + (int64_t)r * p.g_ld + beta * B + c * 8, live);
        }
        if constexpr (F32G) {
            // 8 FP32 values per step -> 8 BF16 hi and 8 lo
            for (int i = threadIdx.x; i < RB * CPR; i += 256) {
                const int rr = i / CPR, c = i % CPR;
                uint4 hv = make_uint4(0, 0, 0, 0), lv = hv;
                if (rr < n_live) {
                    const float *src = (const float *)p.g + (int64_t)(rb + rr) * p.g_ld + beta * B + c * 8;
                    const float4 x0 = *(const float4 *)src, x1 = *(const float4 *)(src + 4);
                    split2(x0.x, x0.y, hv.x, lv.x);
                    split2(x0.z, x0.w, hv.y, lv.y);
                    split2(x1.x, x1.y, hv.z, lv.z);
                    split2(x1.z, x1.w, hv.w, lv.w);
                }
                *(uint4 *)(gs + rr * PITCH + c * 8) = hv;
                *(uint4 *)(gl + rr * PITCH + c * 8) = lv;
            }
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
                    if constexpr (F32G) {
                        ldsm_x4_t(gl_a + (krow * PITCH + ncol) * 2, b0, b1, b2, b3);
                        mma16816(acc[n], a0, a1, a2, a3, b0, b1);
                        mma16816(acc[n + 1], a0, a1, a2, a3, b2, b3);
                    }
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

template <int B, bool F32G>
static void outer_launch(const OuterArgs &p, int grid, cudaStream_t st)
{
    using S = OuterSmem<B, F32G>;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_outer_mma<B, F32G>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes);
        attr = true;
    }
    k_outer_mma<B, F32G><<<grid, 256, S::kBytes, st>>>(p);
}

template <bool F32G>
static void outer_dispatch(int b, const OuterArgs &p, int grid, cudaStream_t st)
{
    switch (b) {
    case 16: outer_launch<16, F32G>(p, grid, st); break;
    case 32: outer_launch<32, F32G>(p, grid, st); break;
    case 64: outer_launch<64, F32G>(p, grid, st); break;
    default: outer_launch<128, F32G>(p, grid, st); break;
    }
}

void launch_outer_tc(int nsets, int nrows, int dim, int b, const uint16_t *a, int64_t a_ld,
                     bool gather, const int32_t *perm, int k, const void *g, bool g_f32, int64_t g_ld,
                     const int32_t *offsets, float *dR, cudaStream_t st)
{
    OuterArgs p{a, a_ld, gather ? 1 : 0, perm, k, g, g_ld, offsets, nrows, dim, dR};
    int grid = nsets * (dim / b);
    if (grid <= 0) return;
    if (g_f32) outer_dispatch<true>(b, p, grid, st);
    else outer_dispatch<false>(b, p, grid, st);
    note_launch();
}

// ------------------------------------------------------------------ fused backward, b = 64
// One pass over an FP32 gradient g (dx~ or dh~, expert-sorted rows) per
// (set s, block beta), in 64-row batches of the set:
//   out  = g_blk R_beta^T         (FP32 dx rows; or, SWIGLU, the SwiGLU
//                                  backward from the saved g, u into FP16
//                                  [dg | du])
//   dR[s][beta] = sum_r a_blk^T g_blk   (a = x gathered by perm / k, or h)
// g is read once for both products (the separate kernels read it twice).
// g is split into hi = bf16(g) and lo = bf16(g - hi), both multiplied.
// Warp w: rows (rotation) or i (dR) 16 (w % 4) .., columns 32 (w / 4) ..
struct AdapterBwdArgs {
    const float *g;            // [rows, dim] FP32, expert-sorted
    const uint16_t *a;         // [*, a_ld] BF16 (gathered rows: perm[r] / k)
    int64_t a_ld;
    int gather;
    const int32_t *perm;
    int k;
    const uint16_t *R;         // [sets][dim/64][64][64] BF16 (stride elements per set)
    int64_t stride;
    const int32_t *offsets;    // rows of set s (NULL: all rows, one set)
    int nrows;
    int dim;
    void *out;                 // FP32 [rows, dim], or SWIGLU: FP16 [rows, 2 dim]
    const float *ctxf;         // SWIGLU: saved g | u rows [rows, 2 dim]
    float *dR;                 // [sets][dim/64][64][64]
};

constexpr int kAbB = 64, kAbRows = 64, kAbPitch = kAbB + 8;
struct AbSmem {
    static constexpr int kG = kAbRows * kAbB * 4;       // FP32 staging
    static constexpr int kA = kAbRows * kAbPitch * 2;   // a tile
    static constexpr int kStage = kG + kA;
    static constexpr int kT = kAbRows * kAbPitch * 2;   // hi, lo tiles
    static constexpr int kR = kAbB * kAbPitch * 2;
    static constexpr int kBytes = 2 * kStage + 2 * kT + kR;
};

template <int EPI>
__global__ void __launch_bounds__(256, 2) k_adapter_bwd(AdapterBwdArgs p)
{
    using S = AbSmem;
    extern __shared__ __align__(16) uint8_t absm[];
    const uint32_t sm0 = (uint32_t)__cvta_generic_to_shared(absm);
    const uint32_t hi_a = sm0 + 2 * S::kStage, lo_a = hi_a + S::kT, r_a = lo_a + S::kT;
    uint16_t *hi_p = (uint16_t *)(absm + 2 * S::kStage), *lo_p = hi_p + kAbRows * kAbPitch;
    const int nb = p.dim / kAbB;
    const int s = blockIdx.x / nb, beta = blockIdx.x % nb;
    const int r0 = p.offsets ? p.offsets[s] : 0, r1 = p.offsets ? p.offsets[s + 1] : p.nrows;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rg = warp & 3, ch = warp >> 2, gq = lane >> 2, tq = lane & 3;
    const uint16_t *Rb = p.R + (int64_t)s * p.stride + (int64_t)beta * kAbB * kAbB;

    // the rotation block (once), then batch staging: g FP32 rows and a rows
    for (int i = threadIdx.x; i < kAbB * 8; i += 256)
        cp_async16(r_a + ((i >> 3) * kAbPitch + (i & 7) * 8) * 2, Rb + (i >> 3) * kAbB + (i & 7) * 8, true);
    // source rows of thread t's two a-chunks (rows t/8 and t/8 + 32 of a
    // batch), read one batch ahead so that the gather's index loads do not
    // stall the batch being multiplied
    auto rows_of = [&](int rb, int (&ar)[2]) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = rb + (threadIdx.x >> 3) + 32 * h;
            ar[h] = r < r1 ? (p.gather ? p.perm[r] / p.k : r) : 0;
        }
    };
    auto stage = [&](int rb, int buf, const int (&ar)[2]) {
        const uint32_t ga = sm0 + buf * S::kStage, aa = ga + S::kG;
        const int n_live = min(kAbRows, r1 - rb);
        for (int i = threadIdx.x; i < kAbRows * 16; i += 256) {   // 16 chunks of 4 floats per row
            const int rr = i >> 4, c = i & 15;
            const bool live = rr < n_live;
            const int64_t r = rb + (live ? rr : 0);
            cp_async16(ga + (rr * kAbB + c * 4) * 4, p.g + r * p.dim + (int64_t)beta * kAbB + c * 4, live);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = threadIdx.x + 256 * h;
            const int rr = i >> 3, c = i & 7;
            cp_async16(aa + (rr * kAbPitch + c * 8) * 2, p.a + (int64_t)ar[h] * p.a_ld + (int64_t)beta * kAbB + c * 8,
                       rr < n_live);
        }
        cp_async_commit();
    };

    float dacc[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n) dacc[n][0] = dacc[n][1] = dacc[n][2] = dacc[n][3] = 0.f;
    int ar[2], ar_next[2];
    rows_of(r0, ar);
    if (r0 < r1) stage(r0, 0, ar);
    else cp_async_commit();
    rows_of(r0 + kAbRows, ar_next);
    for (int rb = r0, it = 0; rb < r1; rb += kAbRows, ++it) {
        const int buf = it & 1;
        if (rb + kAbRows < r1) {
            stage(rb + kAbRows, buf ^ 1, ar_next);
            rows_of(rb + 2 * kAbRows, ar_next);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        // split the FP32 rows into the hi and lo BF16 tiles
        {
            const float *gs = (const float *)(absm + buf * S::kStage);
            for (int i = threadIdx.x; i < kAbRows * 16; i += 256) {
                const int rr = i >> 4, c = i & 15;
                const float4 v = *(const float4 *)(gs + rr * kAbB + c * 4);
                uint32_t h0, l0, h1, l1;
                split2(v.x, v.y, h0, l0);
                split2(v.z, v.w, h1, l1);
                *(uint2 *)(hi_p + rr * kAbPitch + c * 4) = make_uint2(h0, h1);
                *(uint2 *)(lo_p + rr * kAbPitch + c * 4) = make_uint2(l0, l1);
            }
        }
        __syncthreads();
        const uint32_t aa = sm0 + buf * S::kStage + S::kG;
        const int n_live = min(kAbRows, r1 - rb);

        // SWIGLU: the saved g, u of this thread's outputs, loaded before the
        // MMAs so that their latency overlaps them
        float2 cg[4][2], cu[4][2];
        if constexpr (EPI == ROT_SWIGLU_BWD) {
#pragma unroll
            for (int n = 0; n < 4; ++n)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int rl = min(16 * rg + gq + 8 * h, n_live - 1);
                    const float *c = p.ctxf + (int64_t)(rb + rl) * 2 * p.dim + beta * kAbB + 32 * ch + n * 8 + 2 * tq;
                    cg[n][h] = *(const float2 *)c;
                    cu[n][h] = *(const float2 *)(c + p.dim);
                }
        }
        // out rows 16 rg .., columns 32 ch ..: g (hi + lo) R^T
        float acc[4][4];
#pragma unroll
        for (int n = 0; n < 4; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < kAbB / 16; ++kk) {
            uint32_t a0, a1, a2, a3, l0, l1, l2, l3;
            const int row = 16 * rg + (lane & 15), col = kk * 16 + (lane >> 4) * 8;
            ldsm_x4(hi_a + (row * kAbPitch + col) * 2, a0, a1, a2, a3);
            ldsm_x4(lo_a + (row * kAbPitch + col) * 2, l0, l1, l2, l3);
#pragma unroll
            for (int n = 0; n < 4; n += 2) {
                // B(k, n) = R[n][k]: row-major [n][k] is the col layout
                const int nrow = 32 * ch + n * 8 + (lane & 7) + ((lane >> 4) << 3);
                const int kcol = kk * 16 + ((lane >> 3) & 1) * 8;
                uint32_t b0, b1, b2, b3;
                ldsm_x4(r_a + (nrow * kAbPitch + kcol) * 2, b0, b1, b2, b3);
                mma16816(acc[n], a0, a1, a2, a3, b0, b1);
                mma16816(acc[n + 1], a0, a1, a2, a3, b2, b3);
                mma16816(acc[n], l0, l1, l2, l3, b0, b1);
                mma16816(acc[n + 1], l0, l1, l2, l3, b2, b3);
            }
        }
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int rl = 16 * rg + gq + 8 * h;
                if (rl >= n_live) continue;
                const int64_t r = rb + rl;
                const int col = beta * kAbB + 32 * ch + n * 8 + 2 * tq;
                const float v0 = acc[n][2 * h], v1 = acc[n][2 * h + 1];
                if constexpr (EPI == ROT_SWIGLU_BWD) {
                    const float2 gg = cg[n][h], uu = cu[n][h];
                    const float s0 = 1.f / (1.f + expf(-gg.x)), s1 = 1.f / (1.f + expf(-gg.y));
                    const float dg0 = v0 * uu.x * s0 * (1.f + gg.x * (1.f - s0));
                    const float dg1 = v1 * uu.y * s1 * (1.f + gg.y * (1.f - s1));
                    const float du0 = v0 * (gg.x * s0), du1 = v1 * (gg.y * s1);
                    __half2 *o = (__half2 *)((uint16_t *)p.out + r * 2 * p.dim + col);
                    o[0] = __floats2half2_rn(dg0, dg1);
                    o[p.dim / 2] = __floats2half2_rn(du0, du1);
                } else {
                    *(float2 *)((float *)p.out + r * p.dim + col) = make_float2(v0, v1);
                }
            }

        // dR rows i = 16 rg .., columns j = 32 ch ..: += a^T (hi + lo) over
        // the batch's rows (dead rows are zero in both tiles)
#pragma unroll
        for (int kk = 0; kk < kAbRows / 16; ++kk) {
            uint32_t a0, a1, a2, a3;
            {
                // A(m = i, k = row) = a[row][i]: transposed 8x8 loads
                const int krow = kk * 16 + (lane & 7) + ((lane >> 4) << 3);
                const int mcol = 16 * rg + ((lane >> 3) & 1) * 8;
                ldsm_x4_t(aa + (krow * kAbPitch + mcol) * 2, a0, a1, a2, a3);
            }
#pragma unroll
            for (int n = 0; n < 4; n += 2) {
                const int krow = kk * 16 + (lane & 15);
                const int ncol = 32 * ch + n * 8 + (lane >> 4) * 8;
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(hi_a + (krow * kAbPitch + ncol) * 2, b0, b1, b2, b3);
                mma16816(dacc[n], a0, a1, a2, a3, b0, b1);
                mma16816(dacc[n + 1], a0, a1, a2, a3, b2, b3);
                ldsm_x4_t(lo_a + (krow * kAbPitch + ncol) * 2, b0, b1, b2, b3);
                mma16816(dacc[n], a0, a1, a2, a3, b0, b1);
                mma16816(dacc[n + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        __syncthreads();   // the tiles and this stage are refilled next
    }
    cp_async_wait<0>();   // (an empty set still loaded its rotation block)
    float *D = p.dR + ((int64_t)s * nb + beta) * kAbB * kAbB;
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = 16 * rg + gq + 8 * h, j = 32 * ch + n * 8 + 2 * tq;
            *(float2 *)(D + i * kAbB + j) = make_float2(dacc[n][2 * h], dacc[n][2 * h + 1]);
        }
}

bool adapter_bwd_fused_ok(int b) { return b == kAbB; }

void launch_adapter_bwd_tc(int nsets, int nrows, int dim, const float *g, const uint16_t *a, int64_t a_ld,
                           bool gather, const int32_t *perm, int k, const uint16_t *R, int64_t stride,
                           const int32_t *offsets, void *out, bool swiglu, const float *ctxf, float *dR,
                           cudaStream_t st)
{
    AdapterBwdArgs p{g, a, a_ld, gather ? 1 : 0, perm, k, R, stride, offsets, nrows, dim, out, ctxf, dR};
    const int grid = nsets * (dim / kAbB);
    if (grid <= 0) return;
    auto kern = swiglu ? k_adapter_bwd<ROT_SWIGLU_BWD> : k_adapter_bwd<ROT_STORE>;
    static bool attr[2] = {false, false};
    if (!attr[swiglu]) {
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, AbSmem::kBytes);
        attr[swiglu] = true;
    }
    kern<<<grid, 256, AbSmem::kBytes, st>>>(p);
    note_launch();
}

}  // namespace pmoe
