// gemm_tc.cuh -- grouped GEMM of the layer on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA), with the frozen weights dequantized tile by
// tile into shared memory (Orbit announcement, 技艺细节: the active experts'
// weights are dequantized to BF16 only while their grouped GEMM runs).
//
// Orientation: the weights are the MMA's M operand (128 output features per
// tile) and the tokens of one expert are the N operand (16..256 rows per
// tile), so an expert with a few hundred routed tokens fills one tile with
// little padding and every weight tile is dequantized once per token tile.
//
//   D[f, t] = sum_k W~[f, k] * B[t, k]      (FP32 in TMEM: lanes = f, columns = t)
//
// Roles (800 threads, one CTA per SM, persistent over the work list):
//   warps 0-3   epilogue: TMEM -> registers -> fused epilogue -> global
//   warps 4, 7  TMA producers of the packed weight tiles and their scales,
//               taking alternate K steps (raw ring)
//   warp  5     TMEM allocator and MMA issuer (one elected lane per K step)
//   warps 6, 8  TMA producers of the token tiles B (128B swizzle), alternate
//               K steps; BF16 weights (scratch mode, router) come the same way
//   warps 9-24  converters in two groups taking alternate K steps: packed
//               weights -> BF16 A tiles, 128B-swizzled.  Forward kinds
//               contract over the stored matrix's columns and write A
//               K-major; backward kinds contract over its rows and write A
//               MN-major (each stored row segment lands as one swizzle row,
//               and the MMA reads the tile transposed).
// Pipeline: a raw ring of packed tiles, an A ring of converted tiles (16 KB)
// and a B ring of token tiles (up to 32 KB), with full/empty mbarriers; two
// TMEM accumulators of 256 columns so the epilogue of one tile overlaps the
// main loop of the next.  Every wait is bounded.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "launch.h"

namespace pmoe {
namespace tc {

constexpr int kBK = 64;                      // K per stage: one 128-byte swizzle row of BF16
constexpr int kM = 128;                      // MMA M (weight rows per tile)
constexpr int kNmax = 256;                   // largest token tile (MMA N)
constexpr int kABytes = kM * kBK * 2;        // 16 KB
constexpr int kBBytes = kNmax * kBK * 2;     // 32 KB
constexpr int kBoxRows = 32;                 // smallest TMA box: 32 token rows x 64 K
constexpr int kEpiWarps = 4;
#ifndef PMOE_PROD_SPLIT
#define PMOE_PROD_SPLIT 2
#endif
// producers: kProd warps for the weight tiles and kProd for the token tiles;
// producer warp p of a kind takes the K steps g = p (mod kProd)
constexpr int kProd = PMOE_PROD_SPLIT;
constexpr int kRawWarp = 4;                  // packed weight tiles + scale words: warps 4, 7, ...
constexpr int kMmaWarp = 5;
constexpr int kBWarp = 6;                    // token tiles (and BF16 weight tiles): warps 6, 8, ...
constexpr int kDqWarp0 = 5 + 2 * kProd;
#ifndef PMOE_DQ_WARPS
#define PMOE_DQ_WARPS 16
#endif
constexpr int kDqWarps = PMOE_DQ_WARPS;
#ifndef PMOE_CONV_GROUPS
#define PMOE_CONV_GROUPS 2
#endif
constexpr int kConvGroups = PMOE_CONV_GROUPS;   // converter groups taking alternate stages
constexpr int kThreads = (kDqWarp0 + kDqWarps) * 32;
constexpr int kTmemCols = 512;
constexpr unsigned long long kWaitNs = 2000000000ull;   // bounded waits: 2 s (default)

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: gives up after limit_ns, records PMOE_ERR_TIMEOUT with the
// waiting role and returns false (the caller then leaves its loop).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, DevErr *err, int where,
                                          uint64_t limit_ns)
{
    if (mbar_try(bar, parity)) return true;
    uint64_t t0 = globaltimer();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try(bar, parity)) return true;
        if (globaltimer() - t0 > limit_ns) {
            record_error(err, PMOE_ERR_TIMEOUT, where, (int)blockIdx.x);
            return false;
        }
    }
}
__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *tm, int x, int y,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"((uint64_t)tm), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (SBO), version 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;             // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset
    d |= (uint64_t)1 << 46;             // descriptor version
    d |= (uint64_t)2 << 61;             // 128-byte swizzle
    return d;
}
// MN-major A tile (128 M x 64 K, 128-byte swizzle): the swizzle atom is 64
// M-elements x 8 K-rows (1024 B); the two M halves sit 1024 B apart (LBO),
// consecutive 8-row K groups 2048 B apart (SBO).
__device__ __forceinline__ uint64_t sdesc_mn(uint32_t saddr)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(1024 >> 4) << 16;   // leading byte offset: next 64 M-elements
    d |= (uint64_t)(2048 >> 4) << 32;   // stride byte offset: next 8 K-rows
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}
// Instruction descriptor, kind::f16: BF16 (or, f16, FP16) A and B, FP32 D,
// M x N; B K-major, A K-major or (a_mn) MN-major.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N, bool a_mn = false, bool f16 = false)
{
    const uint32_t ab = f16 ? 0u : 1u;   // operand format: 0 FP16, 1 BF16
    return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)a_mn << 15) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// A BF16 pair re-encoded as an FP16 pair (exact for values in the FP16
// normal range and zero)
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t p)
{
    uint32_t h;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(__uint_as_float(p & 0xFFFF0000u)),
        "f"(__uint_as_float(p << 16)));
    return h;
}
// Called by a whole converged warp, so the issue loop's operands stay
// uniform: one K step of 64, i.e. four MMAs of K = 16 (descriptors a0..a3,
// b0..b3) and the commit of `bar`, issued by one elected lane.
__device__ __forceinline__ void umma_step_warp(uint32_t d_tmem, const uint64_t (&a)[4], const uint64_t (&b)[4],
                                               uint32_t idesc, uint32_t accum, uint32_t bar)
{
    asm volatile(
        "{ .reg .pred e, p, t; elect.sync _|e, 0xffffffff; setp.ne.b32 p, %9, 0; setp.eq.b32 t, %9, %9;\n"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %10, p;\n"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %6, %10, t;\n"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %7, %10, t;\n"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %8, %10, t;\n"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%11]; }" ::"r"(d_tmem),
        "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]),
        "r"(accum), "r"(idesc), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void umma_commit_warp(uint32_t bar)
{
    asm volatile(
        "{ .reg .pred e; elect.sync _|e, 0xffffffff;\n"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0]; }" ::"r"(bar)
        : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// total += partial over one warp's 32 TMEM lanes, columns [0, ncols): 16
// columns of each buffer per step under one wait (a wider step needs more
// registers than the kernel has), FP32 additions (round to nearest)
__device__ __forceinline__ void tmem_drain(uint32_t part, uint32_t total, int ncols)
{
    for (int c0 = 0; c0 < ncols; c0 += 16) {
        uint32_t p[16], t[16];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n"
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n"
            "tcgen05.wait::ld.sync.aligned;"
            : "=r"(p[0]), "=r"(p[1]), "=r"(p[2]), "=r"(p[3]), "=r"(p[4]), "=r"(p[5]), "=r"(p[6]),
              "=r"(p[7]), "=r"(p[8]), "=r"(p[9]), "=r"(p[10]), "=r"(p[11]), "=r"(p[12]), "=r"(p[13]),
              "=r"(p[14]), "=r"(p[15]), "=r"(t[0]), "=r"(t[1]), "=r"(t[2]), "=r"(t[3]), "=r"(t[4]),
              "=r"(t[5]), "=r"(t[6]), "=r"(t[7]), "=r"(t[8]), "=r"(t[9]), "=r"(t[10]), "=r"(t[11]),
              "=r"(t[12]), "=r"(t[13]), "=r"(t[14]), "=r"(t[15])
            : "r"(part + c0), "r"(total + c0)
            : "memory");
#pragma unroll
        for (int i = 0; i < 16; ++i) t[i] = __float_as_uint(__fadd_rn(__uint_as_float(t[i]), __uint_as_float(p[i])));
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
                total + c0),
            "r"(t[0]), "r"(t[1]), "r"(t[2]), "r"(t[3]), "r"(t[4]), "r"(t[5]), "r"(t[6]), "r"(t[7]),
            "r"(t[8]), "r"(t[9]), "r"(t[10]), "r"(t[11]), "r"(t[12]), "r"(t[13]), "r"(t[14]), "r"(t[15])
            : "memory");
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint32_t x, uint32_t y)
{
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ uint4 ldg_nc_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t lop3_and_xor(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;   // (a & b) ^ c
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
__device__ __forceinline__ uint32_t bf2_sub(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bf2_mul(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// 8 INT4 elements of one u32 (element j in nibble j) -> BF16 q*s, returned
// as the four pairs (e0,e4), (e1,e5), (e2,e6), (e3,e7).  A nibble n becomes
// the BF16 value 128 + (n ^ 8) by bit placement (0x4300 | (n ^ 8)); the
// subtraction of 136 is exact and gives the two's-complement value q; one
// BF16 multiply by the scale rounds q*s once (nearest even).
__device__ __forceinline__ void int4x8_pairs(uint32_t w, uint32_t s2, uint32_t (&p)[4])
{
    const uint32_t k136 = 0x43084308u;   // bf16x2 (136, 136)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t t = lop3_and_xor(w >> (4 * j), 0x000F000Fu, 0x43084308u);
        p[j] = bf2_mul(bf2_sub(t, k136), s2);
    }
}

// ------------------------------------------------------------------ arguments
struct TcArgs {
    const uint8_t *wq;          // packed weights of expert 0 (or BF16 scratch slot 0)
    const uint8_t *ws;          // scales of expert 0
    int64_t wq_stride, ws_stride;
    int64_t Kst;                // columns of one expert's stored [N, K] matrix
    int64_t Nst;                // rows of one expert's stored matrix
    int64_t w_off_elems;        // BF16 scratch: element offset of the matrix in a slot
    int K;                      // contraction length
    int Kb;                     // columns of the token operand (K, or d for the router)
    int Mtot;                   // output features
    int m_tile;                 // output features per tile (64 gate/up pairs, else 128)
    const Tile *tiles;
    const int32_t *chunk_tiles;
    int c0, c1;
    int slot_index;
    int scale_tma;              // backward kinds: scales by TMA (tmS) instead of cp.async
    uint16_t *out;              // BF16 output (when outf is NULL)
    float *ctxf;                // GU: saved g | u rows [P, 2I] f32 (or NULL)
    int I;
    const float *w;
    const int32_t *perm;
    const uint16_t *ht;
    float *dtw_part;
    float *outf;                // FP32 output: router partials, o, dh~ or dx~
    int64_t outf_split;         // router: elements between the partials of two K splits
    DevErr *err;
    uint64_t wait_ns;           // limit of every bounded wait
    int skip_commit_item;       // test hook: work item whose accumulator-full signal the
                                // MMA issuer withholds (-1: none)
};

#ifndef PMOE_GU_CHUNK
#define PMOE_GU_CHUNK 16
#endif
// ------------------------------------------------------------------ pipeline sizes
// Per kind and weight format.  Packed weight tiles come by TMA into a raw
// ring of kRawTma stages, each followed by the tile's scale words, which the
// producer warp's lanes fetch with cp.async:
//   forward kinds:  128 stored rows x 64 columns (kRowBytes each), no
//                   swizzle; one 4-byte scale word per row
//   backward kinds: 64 stored rows x 128 columns (kRowBytes each), 64- or
//                   128-byte TMA swizzle (conflict-free converter reads);
//                   per row the 16 aligned scale bytes around the tile's
//                   columns, by one TMA box with the tile when the scale
//                   rows are whole 16-byte units (no per-lane copies to
//                   compete with the epilogue's loads), else the words the
//                   lanes copy
// BF16 scratch weights come by TMA straight into the swizzled A stage.
template <int KIND, int FMT>
struct Pipe {
    // backward kinds: the contraction runs over the stored matrix's rows
    static constexpr bool kTrans = KIND == GK_BWD_G || KIND == GK_BWD_DX || KIND == GK_BWD_DX_F16;
    // FP16 operands: the converters write the weights' BF16 values in FP16
    // encoding and the token operand is FP16 (11 significant bits)
    static constexpr bool kF16 = KIND == GK_BWD_DX_F16;
    static constexpr int kTileN = kNmax;
    static constexpr int kBStage = kTileN * kBK * 2;
    // Chunked accumulation (gate/up, whose sums are rounded to BF16 in h):
    // the tensor cores' FP32 accumulation loses about one bit per 16-long K
    // step, so over thousands of steps g and u drift far beyond FP32 rounding
    // and flip the BF16 rounding of h.  Each run of kChunk K steps is summed
    // in its own TMEM buffer and added into the tile's total by the epilogue
    // warps in FP32, which bounds the drift by the chunk length.
    static constexpr int kChunk = KIND == GK_FWD_GU ? PMOE_GU_CHUNK : 1 << 30;
    static constexpr bool kBf16 = FMT == kFmtBF16;
    static constexpr bool kTmaRaw = !kBf16;
    static constexpr bool kFp8 = FMT == PMOE_W_FP8_B128_F32;
    // A (converted weights, 16 KB) and B (token tiles, up to 32 KB) rings of
    // different depths: the converters may run kStagesA steps ahead of the
    // MMA, the token producer kStagesB steps (kStagesB <= kStagesA)
#ifdef PMOE_A_STAGES
    static constexpr int kStagesA = kFp8 ? 3 : PMOE_A_STAGES;
#else
    static constexpr int kStagesA = kFp8 ? 3 : 4;
#endif
    static constexpr int kASmem = kABytes;                  // shared memory per A stage
    static constexpr int kAccCols = kTileN;                 // columns per accumulator buffer
    static_assert(2 * kAccCols <= 512, "tensor memory budget");
#ifdef PMOE_B_STAGES
    static constexpr int kStagesB = kFp8 ? 3 : PMOE_B_STAGES;
#else
    static constexpr int kStagesB = kFp8 ? 3 : 4;
#endif
    static_assert(kStagesB <= kStagesA, "token ring no deeper than the weight ring");
    static constexpr int kRawRows = kTrans ? 64 : 128;
    static constexpr int kRowBytes = kTrans ? (kFp8 ? 128 : 64) : (kFp8 ? 64 : 32);
    static constexpr int kScaleOff = kRawRows * kRowBytes;   // scale words after the data
    static constexpr int kRawTile = kTrans ? (kScaleOff + 64 * 16 + 1023) & ~1023 : kScaleOff + 128 * 4;
#ifdef PMOE_RAW_STAGES
    static constexpr int kRawTma = kFp8 ? 8 : PMOE_RAW_STAGES;
#else
    static constexpr int kRawTma = kFp8 ? 8 : 6;   // raw ring stages
#endif
    static constexpr int kRawBytes = kTmaRaw ? kRawTma * kRawTile : 0;
    // With kProd weight-producer warps taking alternate K steps, each warp
    // must always reuse its own raw slots: then a warp waiting on a slot's
    // release barrier is never more than one phase behind it.  With an odd
    // ring two warps share a slot, one can wait for a phase two completions
    // ahead, and the parity test passes early (it re-arms the slot's
    // transaction barrier while the tile is in use).
    static_assert(kRawTma % kProd == 0, "raw ring size must be a multiple of the producer warps");
    static constexpr int kNumBars = 2 * kStagesA + 4 + 2 * kRawTma;
    static constexpr int kBarOff = kStagesA * kASmem + kStagesB * kBStage;
    static constexpr int kBarBytes = 8 * kNumBars + 16;
    static constexpr int kRawOff = (kBarOff + kBarBytes + 1023) & ~1023;
    static constexpr size_t kSmem = (size_t)kRawOff + kRawBytes + 1024;
    static_assert(kSmem <= 232448, "shared memory budget");
};

__device__ __forceinline__ void cpa16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cpa8(uint32_t dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cpa4(uint32_t dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// arrive on `bar` once this thread's earlier cp.async copies have landed
__device__ __forceinline__ void cpa_mbar_arrive(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *tm, int x, int y, int z,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            dst),
        "l"((uint64_t)tm), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}
template <int N>
__device__ __forceinline__ void cpa_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ converters
// The converters turn one raw tile (TMA-fetched packed weights plus scale
// words) into one BF16 A stage.  compute_*() leaves the converted 16-byte
// chunks in registers; store_*() writes them, so a converter group can
// overlap the stores of one stage with the conversion of the next.
template <int KIND, int FMT>
struct Dequant {
    // raw-tile row of A row m: GU tiles hold [gate rows | up rows] (64 each)
    __device__ static int raw_row(int m)
    {
        if (KIND != GK_FWD_GU) return m;
        const int q = m >> 5, r = m & 31;
        return r < 16 ? 16 * q + r : 64 + 16 * q + r - 16;
    }
    // stored row of raw-tile row rr
    __device__ static int64_t stored_row(const TcArgs &a, int f0, int rr)
    {
        if (KIND == GK_FWD_GU) return rr < 64 ? (int64_t)(f0 + rr) : (int64_t)(a.I + f0 + rr - 64);
        return f0 + rr;
    }
    // byte offset of the aligned scale word of stored row `row` for step ks
    // (forward kinds: the two groups of 32 columns ks*64 .. ks*64+63)
    __device__ static int64_t scale_word(const TcArgs &a, int64_t row, int ks)
    {
        if (FMT == PMOE_W_INT4_G32_BF16) return 2 * (row * (a.Kst >> 5) + 2 * ks);
        if (FMT == PMOE_W_MXFP4_G32_E8M0) return (row * (a.Kst >> 5) + 2 * ks) & ~(int64_t)3;
        return 4 * ((row >> 7) * (a.Kst >> 7) + ((int64_t)ks * kBK >> 7));
    }
    // backward kinds: byte offset of the first aligned scale word covering
    // columns f0 .. f0+127 of stored row `row` (two consecutive words hold
    // the four groups of 32: INT4 4 x BF16; MXFP4 4 bytes starting at byte
    // (row * Kst/32) & 3 of the first word; FP8 the block's f32 scale)
    __device__ static int64_t scale_word_t(const TcArgs &a, int64_t row, int f0)
    {
        if (FMT == PMOE_W_INT4_G32_BF16) return 2 * (row * (a.Kst >> 5) + (f0 >> 5));
        if (FMT == PMOE_W_MXFP4_G32_E8M0) return (row * (a.Kst >> 5) + (f0 >> 5)) & ~(int64_t)3;
        return 4 * ((row >> 7) * (a.Kst >> 7) + (f0 >> 7));
    }

    // 8 packed elements (one u32 of 4-bit codes, or a uint2 of FP8 codes)
    // and their scale -> one 16-byte chunk of 8 BF16 in element order
    __device__ static uint4 chunk4(uint32_t w, uint32_t sbits)
    {
        uint4 o;
        if (FMT == PMOE_W_INT4_G32_BF16) {
            uint32_t p[4];
            int4x8_pairs(w, sbits | (sbits << 16), p);
            o.x = prmt(p[0], p[1], 0x5410);
            o.y = prmt(p[2], p[3], 0x5410);
            o.z = prmt(p[0], p[1], 0x7632);
            o.w = prmt(p[2], p[3], 0x7632);
        } else {
            // E2M1 by table: the BF16 pattern of |code| (0, 0.5, 1, 1.5, 2,
            // 3, 4, 6) as two 8-entry byte tables (high and low byte) looked
            // up by prmt with the 3 magnitude bits, the code's sign bit moved
            // to bit 7 of the high byte, then one BF16 multiply by the E8M0
            // scale 2^(u-127) (a power of two: a single rounding of the exact
            // product)
            const uint32_t sb = sbits == 0u ? 0x0040u : sbits == 255u ? 0x7FC0u : sbits << 7;
            const uint32_t s2 = sb | (sb << 16);
            const uint32_t ws = w << 4;   // bit 7 of byte k: sign of element 2k
            uint32_t r[4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {   // elements 4h .. 4h+3
                const uint32_t sel = (h ? w >> 16 : w) & 0x7777u;
                const uint32_t hi = prmt(0x3F3F3F00u, 0x40404040u, sel);
                const uint32_t lo = prmt(0xC0800000u, 0xC0804000u, sel);
                const uint32_t sg = prmt(ws, w, h ? 0x7362u : 0x5140u);
                const uint32_t hs = hi | (sg & 0x80808080u);
                r[2 * h] = bf2_mul(prmt(lo, hs, 0x5140u), s2);
                r[2 * h + 1] = bf2_mul(prmt(lo, hs, 0x7362u), s2);
            }
            o = make_uint4(r[0], r[1], r[2], r[3]);
        }
        return o;
    }
    __device__ static uint4 chunk8(uint2 w2, float sc)
    {
        uint32_t o[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t w = h ? w2.y : w2.x;
            __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFFu), __NV_E4M3);
            __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
            const float2 fl = __half22float2(*(const __half2 *)&lo);
            const float2 fh = __half22float2(*(const __half2 *)&hi);
            o[2 * h] = pack_bf2(__fmul_rn(fl.x, sc), __fmul_rn(fl.y, sc));
            o[2 * h + 1] = pack_bf2(__fmul_rn(fh.x, sc), __fmul_rn(fh.y, sc));
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    }

    // Forward kinds (K-major A).  A converter group of 8192 / EPT threads:
    // thread tg takes A row m = tg / (64 / EPT) and EPT consecutive K
    // elements of it (EPT / 8 chunks of the swizzled row).
    template <int EPT>
    __device__ static void compute_tma(const TcArgs &a, int f0, int ks, int tg, const uint8_t *rawt,
                                       uint4 (&out)[EPT / 8])
    {
        using PP = Pipe<KIND, FMT>;
        constexpr int P = 64 / EPT;
        const int m = tg / P, e0 = (tg % P) * EPT;
        const int rr = raw_row(m);
        const bool lv = KIND == GK_FWD_GU || f0 + m < a.Mtot;
        const uint8_t *row = rawt + rr * PP::kRowBytes;
        const uint32_t sw = *(const uint32_t *)(rawt + PP::kScaleOff + 4 * rr);
        // the thread's packed bytes are contiguous: load them as vectors
        constexpr int kB = FMT == PMOE_W_FP8_B128_F32 ? EPT : EPT / 2;
        uint32_t wv[kB / 4];
        const uint8_t *src = row + (FMT == PMOE_W_FP8_B128_F32 ? e0 : e0 / 2);
        if constexpr (kB >= 16) {
#pragma unroll
            for (int v = 0; v < kB / 16; ++v) {
                const uint4 q = *(const uint4 *)(src + 16 * v);
                wv[4 * v] = q.x, wv[4 * v + 1] = q.y, wv[4 * v + 2] = q.z, wv[4 * v + 3] = q.w;
            }
        } else {
            const uint2 q = *(const uint2 *)src;
            wv[0] = q.x, wv[1] = q.y;
        }
#pragma unroll
        for (int c = 0; c < EPT / 8; ++c) {
            const int e = e0 + 8 * c, grp = e >> 5;
            if (!lv) {
                out[c] = make_uint4(0, 0, 0, 0);
            } else if (FMT == PMOE_W_INT4_G32_BF16) {
                out[c] = chunk4(wv[c], grp ? sw >> 16 : sw & 0xFFFFu);
            } else if (FMT == PMOE_W_MXFP4_G32_E8M0) {
                const int64_t gi = stored_row(a, f0, rr) * (a.Kst >> 5) + 2 * ks + grp;
                out[c] = chunk4(wv[c], (sw >> (8 * (gi & 3))) & 0xFFu);
            } else {
                out[c] = chunk8(make_uint2(wv[2 * c], wv[2 * c + 1]), __uint_as_float(sw));
            }
        }
    }
    template <int EPT>
    __device__ static void store_tma(int tg, const uint4 (&out)[EPT / 8], uint32_t sA)
    {
        constexpr int P = 64 / EPT;
        const int m = tg / P, c0 = (tg % P) * (EPT / 8);
        const uint32_t rowaddr = sA + m * 128;
#pragma unroll
        for (int j = 0; j < EPT / 8; ++j) st_shared_v4(rowaddr + (((c0 + j) ^ (m & 7)) << 4), out[j]);
    }

    // Backward kinds (MN-major A): A[m][k] = W[ks*64 + k][f0 + m].  A group
    // of 256 threads; thread tg takes stored row k = 8*(tg >> 5) + (tg & 7)
    // of the step and the 32 columns 32*mq .. 32*mq+31, mq = (tg >> 3) & 3
    // (one scale group).  The 8 lanes of a quarter-warp take 8 consecutive
    // rows, so their raw reads and swizzled stores fall in distinct banks.
    __device__ static void compute_t(const TcArgs &a, int f0, int ks, int tg, const uint8_t *rawt,
                                     uint4 (&out)[4])
    {
        using PP = Pipe<KIND, FMT>;
        const int k = 8 * (tg >> 5) + (tg & 7), mq = (tg >> 3) & 3;
        if (f0 + 32 * mq >= a.Mtot) {
#pragma unroll
            for (int j = 0; j < 4; ++j) out[j] = make_uint4(0, 0, 0, 0);
            return;
        }
        const uint8_t *row = rawt + k * PP::kRowBytes;
        const uint8_t *sw = rawt + PP::kScaleOff + 16 * k;   // stored row k's 16 scale bytes
        if (FMT == PMOE_W_FP8_B128_F32) {
            // 128-byte rows, 128-byte swizzle: chunk c sits at c ^ (k & 7)
            const uint4 q0 = *(const uint4 *)(row + (((2 * mq) ^ (k & 7)) << 4));
            const uint4 q1 = *(const uint4 *)(row + (((2 * mq + 1) ^ (k & 7)) << 4));
            const float sc = *(const float *)sw;
            out[0] = chunk8(make_uint2(q0.x, q0.y), sc);
            out[1] = chunk8(make_uint2(q0.z, q0.w), sc);
            out[2] = chunk8(make_uint2(q1.x, q1.y), sc);
            out[3] = chunk8(make_uint2(q1.z, q1.w), sc);
        } else {
            // 64-byte rows, 64-byte swizzle: chunk c sits at c ^ ((k >> 1) & 3)
            const uint4 q = *(const uint4 *)(row + ((mq ^ ((k >> 1) & 3)) << 4));
            // scale group f0/32 + mq: BF16 index (f0/32 & 7) + mq (INT4); byte
            // (f0/32 & 15) + mq (MXFP4 by TMA), or ((row * Kst/32 + f0/32) & 3)
            // + mq of the two aligned words the lanes copied
            uint32_t sb;
            if (FMT == PMOE_W_INT4_G32_BF16) {
                sb = *(const uint16_t *)(sw + 2 * (((f0 >> 5) & 7) + mq));
            } else {
                const int64_t srow = (int64_t)ks * kBK + k;
                const int byte = a.scale_tma ? ((f0 >> 5) & 15) + mq
                                             : (int)((srow * (a.Kst >> 5) + (f0 >> 5)) & 3) + mq;
                sb = sw[byte];
            }
            out[0] = chunk4(q.x, sb);
            out[1] = chunk4(q.y, sb);
            out[2] = chunk4(q.z, sb);
            out[3] = chunk4(q.w, sb);
        }
    }
    __device__ static void store_t(int tg, const uint4 (&out)[4], uint32_t sA)
    {
        const int r = tg & 7, mq = (tg >> 3) & 3, kg = tg >> 5;
        const uint32_t base = sA + kg * 2048 + (mq >> 1) * 1024 + r * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint4 v = out[j];
            if (KIND == GK_BWD_DX_F16)   // the same values in FP16 encoding
                v = make_uint4(bf2_to_h2(v.x), bf2_to_h2(v.y), bf2_to_h2(v.z), bf2_to_h2(v.w));
            st_shared_v4(base + (((4 * (mq & 1) + j) ^ r) << 4), v);
        }
    }
};

// SiLU for the SwiGLU epilogue with the accurate exponential and an IEEE
// division: h = bf16(silu(g) u) is a BF16 rounding decision, and an error of
// a few ulp in silu flips it near a rounding midpoint
__device__ __forceinline__ float silu_f(float g) { return g / (1.f + expf(-g)); }

// A work item's token rows, at most the kind's tile width: a longer tile
// (a work list built for another width) is cut and reported, so no role
// writes past its stage or accumulator.
template <int W>
__device__ __forceinline__ Tile clamp_tile(Tile t, DevErr *err)
{
    if (t.nrows > W) {
        record_error(err, PMOE_ERR_INVALID_ARG, t.row0, t.nrows);
        t.nrows = W;
    }
    return t;
}

// ------------------------------------------------------------------ kernel
template <int KIND, int FMT>
__global__ void __launch_bounds__(kThreads, 1) k_gemm_tc(const __grid_constant__ CUtensorMap tmB256,
                                                         const __grid_constant__ CUtensorMap tmB128,
                                                         const __grid_constant__ CUtensorMap tmB64,
                                                         const __grid_constant__ CUtensorMap tmB32,
                                                         const __grid_constant__ CUtensorMap tmA,
                                                         const __grid_constant__ CUtensorMap tmS,
                                                         const TcArgs a)
{
    using PP = Pipe<KIND, FMT>;
    constexpr int kStages = PP::kStagesA;    // weight ring; step g uses A slot g % kStages
    constexpr int kStagesB = PP::kStagesB;   // token ring; step g uses B slot g % kStagesB
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sA0 = smem_u32(smem);
    const uint32_t sB0 = sA0 + kStages * PP::kASmem;
    const uint32_t bar0 = sB0 + kStagesB * PP::kBStage;
    uint32_t *tmem_slot = (uint32_t *)(smem + PP::kBarOff + 8 * PP::kNumBars);
    // full_a(s): step g's A and B are in place (s = g % kStages); empty(s):
    // the MMAs of the step that last used A slot s have completed
    auto full_a = [&](int s) { return bar0 + 8 * s; };
    auto empty = [&](int s) { return bar0 + 8 * (kStages + s); };
    auto tfull = [&](int c) { return bar0 + 8 * (2 * kStages + c); };
    auto tempty = [&](int c) { return bar0 + 8 * (2 * kStages + 2 + c); };
    auto raw_full = [&](int r) { return bar0 + 8 * (2 * kStages + 4 + r); };
    auto raw_empty = [&](int r) { return bar0 + 8 * (2 * kStages + 4 + PP::kRawTma + r); };
    const uint32_t raw0 = smem_u32(smem + PP::kRawOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tbeg = a.chunk_tiles[a.c0], tend = a.chunk_tiles[a.c1];
    const int nft = (a.Mtot + a.m_tile - 1) / a.m_tile;
    const int n_items = (tend - tbeg) * nft;
    const int nk = a.K / kBK;
    // barrier of K step g (one per A slot) and the parity of its use
    auto fb = [&](uint32_t g) { return (int)(g % (uint32_t)kStages); };
    auto fph = [&](uint32_t g) { return (uint32_t)((g / (uint32_t)kStages) & 1u); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            // one barrier per stage: the converter warps of the stage's group
            // and the token producer's arrive with the stage's TMA bytes
            mbar_init(full_a(s), PP::kBf16 ? 1 : kDqWarps / kConvGroups + 1);
            mbar_init(empty(s), 1);
        }
        for (int c = 0; c < 2; ++c) {
            mbar_init(tfull(c), 1);
            mbar_init(tempty(c), kEpiWarps);
        }
        for (int r = 0; r < PP::kRawTma; ++r) {
            mbar_init(raw_full(r), 1 + 32);   // TMA transaction + the 32 lanes' scale copies
            mbar_init(raw_empty(r), kDqWarps / kConvGroups);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *(volatile uint32_t *)tmem_slot;

    const bool raw_prod = warp == kRawWarp || (kProd > 1 && warp == 7);
    const bool b_prod = warp == kBWarp || (kProd > 1 && warp == 8);
    const uint32_t prod_part = (kProd > 1 && (warp == 7 || warp == 8)) ? 1u : 0u;
    if (raw_prod) {
        // ---------------- weight producer: packed weight tiles (TMA) with
        // their scale words (cp.async by the 32 lanes).  It runs ahead of
        // the token producer by up to the depth of the raw ring, so HBM
        // latency of the weights overlaps the conversion of earlier tiles.
        if constexpr (PP::kTmaRaw) {
            uint32_t g = 0;
            bool ok = true;
            for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
                const Tile tl = clamp_tile<PP::kTileN>(a.tiles[tbeg + item / nft], a.err);
                const int f0 = (item % nft) * a.m_tile;
                const int64_t widx = a.slot_index ? (tl.chunk & 0xffff) : tl.expert;
                for (int ks = 0; ks < nk; ++ks, ++g) {
                    if (kProd > 1 && g % kProd != prod_part) continue;
                    const int r = g % PP::kRawTma;
                    if (!(ok = mbar_wait(raw_empty(r), ((g / PP::kRawTma) & 1) ^ 1, a.err, 7, a.wait_ns))) break;
                    const uint32_t dst = raw0 + r * PP::kRawTile;
                    const uint8_t *ws = a.ws + widx * a.ws_stride;
                    if constexpr (PP::kTrans) {
                        // 64 stored rows ks*64 .. +63, columns f0 .. f0+127
                        if (lane == 0) {
                            mbar_expect_tx(raw_full(r), 64 * PP::kRowBytes + (a.scale_tma ? 64 * 16 : 0));
                            tma_load_2d(dst, &tmA, PP::kFp8 ? f0 : f0 >> 1,
                                        (int)(widx * a.Nst) + ks * kBK, raw_full(r));
                            if (a.scale_tma) {
                                // 16 aligned bytes of scale groups around f0/32, 64 stored rows
                                const int x = FMT == PMOE_W_INT4_G32_BF16 ? ((f0 >> 5) & ~7) * 2 : (f0 >> 5) & ~15;
                                tma_load_2d(dst + PP::kScaleOff, &tmS, x, (int)(widx * a.Nst) + ks * kBK,
                                            raw_full(r));
                            }
                        }
                        // columns past Mtot (a 64-wide last tile) get no scales
                        const bool full = f0 + 128 <= a.Mtot;
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            if (a.scale_tma) break;
                            const int k = lane + 32 * i;
                            const int64_t row = (int64_t)ks * kBK + k;
                            const uint8_t *src = ws + Dequant<KIND, FMT>::scale_word_t(a, row, f0);
                            // INT4: the 4 BF16 at index f0/32 & 7 of the row's 16 bytes
                            const uint32_t sd = dst + PP::kScaleOff + 16 * k +
                                                (FMT == PMOE_W_INT4_G32_BF16 ? 2 * ((f0 >> 5) & 7) : 0);
                            cpa4(sd, src);
                            const bool second = FMT == PMOE_W_INT4_G32_BF16 ? full
                                              : FMT == PMOE_W_MXFP4_G32_E8M0
                                                  ? full && ((row * (a.Kst >> 5)) & 3) != 0
                                                  : false;
                            if (second) cpa4(sd + 4, src + 4);
                        }
                    } else {
                        if (lane == 0) {
                            mbar_expect_tx(raw_full(r), 128 * PP::kRowBytes);
                            const int x = ks * PP::kRowBytes;
                            const int y = (int)(widx * a.Nst) + f0;
                            if (KIND == GK_FWD_GU) {
                                tma_load_2d(dst, &tmA, x, y, raw_full(r));
                                tma_load_2d(dst + 64 * PP::kRowBytes, &tmA, x, y + a.I, raw_full(r));
                            } else {
                                tma_load_2d(dst, &tmA, x, y, raw_full(r));
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int rr = lane + 32 * i;
                            const bool lv = KIND == GK_FWD_GU || f0 + rr < a.Mtot;
                            if (lv)
                                cpa4(dst + PP::kScaleOff + 4 * rr,
                                     ws + Dequant<KIND, FMT>::scale_word(
                                              a, Dequant<KIND, FMT>::stored_row(a, f0, rr), ks));
                        }
                    }
                    cpa_mbar_arrive(raw_full(r));
                }
            }
        }
    } else if (b_prod) {
        // ---------------- token producer: token tiles (TMA), or BF16 weight
        // tiles (TMA into the swizzled A stage)
        uint32_t g = 0;
        bool ok = true;
        for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
            const Tile tl = clamp_tile<PP::kTileN>(a.tiles[tbeg + item / nft], a.err);
            // token rows covered: round up to 32, in boxes of 256/128/64/32 rows
            const int brows = (tl.nrows + kBoxRows - 1) & ~(kBoxRows - 1);
            const int f0 = (item % nft) * a.m_tile;
            const int64_t widx = a.slot_index ? (tl.chunk & 0xffff) : tl.expert;
            (void)f0;
            (void)widx;
            for (int ks = 0; ks < nk; ++ks, ++g) {
                if (kProd > 1 && g % kProd != prod_part) continue;
                const int s = g % kStages, sb = g % kStagesB;
                // B slot sb was last read by step g - kStagesB: wait for its
                // MMAs (which also frees A slot s for the BF16 weight tiles)
                if (g >= (uint32_t)kStagesB) {
                    const uint32_t gp = g - kStagesB;
                    if (!(ok = mbar_wait(empty(fb(gp)), fph(gp), a.err, 1, a.wait_ns))) break;
                }
                const uint32_t fbar = full_a(fb(g));
                if (lane == 0) {
                    mbar_expect_tx(fbar, brows * kBK * 2 + (PP::kBf16 ? kABytes : 0));
                    for (int r0 = 0; r0 < brows;) {
                        const int left = brows - r0;
                        const CUtensorMap *tm = left >= 256 ? &tmB256 : left >= 128 ? &tmB128
                                              : left >= 64 ? &tmB64 : &tmB32;
                        const int rows = left >= 256 ? 256 : left >= 128 ? 128 : left >= 64 ? 64 : 32;
                        // router: split widx covers K steps widx*nk .. of the
                        // [X | X | X] operand of length 3d
                        const int xb = KIND == GK_ROUTER ? (int)((((int64_t)widx * nk + ks) * kBK) % a.Kb) : ks * kBK;
                        tma_load_3d(sB0 + sb * PP::kBStage + r0 * kBK * 2, tm, xb, tl.row0 + r0, 0, fbar);
                        r0 += rows;
                    }
                    if constexpr (PP::kBf16) {
                        const int slot = (int)widx;
                        if (KIND == GK_FWD_GU) {
                            // A rows 32q .. 32q+15: gate f0+16q ..; 32q+16 .. 32q+31: up
#pragma unroll
                            for (int qq = 0; qq < 4; ++qq) {
                                tma_load_3d(sA0 + s * kABytes + (32 * qq) * 128, &tmA, ks * kBK,
                                            f0 + 16 * qq, slot, fbar);
                                tma_load_3d(sA0 + s * kABytes + (32 * qq + 16) * 128, &tmA, ks * kBK,
                                            a.I + f0 + 16 * qq, slot, fbar);
                            }
                        } else {
                            tma_load_3d(sA0 + s * kABytes, &tmA, ks * kBK, f0, slot, fbar);
                        }
                    }
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer (the whole warp runs the loop; one
        // elected lane issues each MMA and commit)
        {
            uint32_t g = 0, li = 0;
            bool ok = true;
            // descriptors of stage 0; a stage or K step moves only the start
            // address field (address / 16, bits 0-13), so they are plain adds
            const uint64_t adesc0 = PP::kTrans ? sdesc_mn(sA0) : sdesc(sA0);
            const uint64_t bdesc0 = sdesc(sB0);
            constexpr uint32_t kAStep = PP::kTrans ? 4096 >> 4 : 32 >> 4;   // per K step of 16
            // The two 256-column TMEM buffers: item li sums into buffer li & 1
            // (its total) and, when its K loop is chunked, runs every chunk
            // after the first in the other buffer (a partial the epilogue adds
            // into the total).  fills0/1 count each buffer's fills; a fill
            // waits until the epilogue has consumed the previous one.
            uint32_t fills0 = 0u, fills1 = 0u;   // (scalars: no local-memory array)
            for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++li) {
                const Tile tl = clamp_tile<PP::kTileN>(a.tiles[tbeg + item / nft], a.err);
                const int N = (tl.nrows + 15) & ~15;
                const uint32_t idesc = idesc_bf16(kM, N, PP::kTrans, PP::kF16);
                const int tot = li & 1, par = tot ^ 1;
                for (int ks = 0; ks < nk; ++ks, ++g) {
                    const int s = g % kStages;
                    const bool first = ks % PP::kChunk == 0;
                    const int buf = ks < PP::kChunk ? tot : par;
                    if (first) {
                        // every lane waits; the outcome is made warp-uniform so
                        // that the lanes stay converged for the elected issue
                        const uint32_t u = buf ? fills1++ : fills0++;
                        if (!(ok = __all_sync(0xffffffffu, mbar_wait(tempty(buf), (u & 1) ^ 1, a.err, 2, a.wait_ns))))
                            break;
                        tc_fence_after();
                    }
                    if (!(ok = __all_sync(0xffffffffu, mbar_wait(full_a(fb(g)), fph(g), a.err, 3, a.wait_ns)))) break;
                    tc_fence_after();
                    // K step of 16: +32 B inside the K-major swizzle row, or two
                    // 8-row K groups (2 x 2048 B) of the MN-major tile
                    const uint64_t bd = bdesc0 + (uint32_t)((g % kStagesB) * (PP::kBStage >> 4));
                    static_assert(kBK == 64, "four MMAs of K = 16 per step");
                    const uint64_t bv[4] = {bd, bd + 2, bd + 4, bd + 6};
                    const uint32_t dacc = tmem + buf * PP::kAccCols;
                    const uint64_t ad = adesc0 + (uint32_t)(s * (kABytes >> 4));
                    const uint64_t av[4] = {ad, ad + kAStep, ad + 2 * kAStep, ad + 3 * kAStep};
                    umma_step_warp(dacc, av, bv, idesc, !first, empty(fb(g)));
                    // a partial chunk is complete: hand it to the epilogue
                    if (buf == par && ((ks + 1) % PP::kChunk == 0 || ks + 1 == nk)) umma_commit_warp(tfull(par));
                }
                // (the test hook withholds one accumulator-full signal: the
                // epilogue's bounded wait for it then runs out)
                if (ok && item != a.skip_commit_item) umma_commit_warp(tfull(tot));
            }
        }
    } else if (warp >= kDqWarp0) {
        const int td = threadIdx.x - kDqWarp0 * 32;
        if constexpr (PP::kTmaRaw) {
            // ---------------- converters: TMA raw tile -> BF16 A stage.  The
            // converter warps form kConvGroups groups; group G takes the steps
            // g = G (mod kConvGroups), so several stages are in conversion at
            // once.  Within a group the loop is software-pipelined: step g+G
            // is converted in registers while the stores of step g drain.
            constexpr int kTPG = kDqWarps * 32 / kConvGroups;   // threads per group
            constexpr int kEPT = 8192 / kTPG;                   // elements per thread
            const int grp = td / kTPG, tg = td % kTPG;
            const int my_items = n_items > (int)blockIdx.x ? (n_items - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
            const uint32_t total = (uint32_t)my_items * nk;
            static_assert(!PP::kTrans || kEPT == 32, "backward converters take 32 elements each");
            // position of a step in this CTA's work: K step ks of the item's
            // feature tile f0, advanced incrementally (no divisions per step)
            struct Cur {
                uint32_t j;
                int ks, li, f0;
            };
            auto at = [&](uint32_t j) {
                Cur c;
                c.j = j;
                c.li = (int)(j / nk);
                c.ks = (int)(j - (uint32_t)c.li * nk);
                c.f0 = (((int)blockIdx.x + c.li * (int)gridDim.x) % nft) * a.m_tile;
                return c;
            };
            auto advance = [&](Cur &c) {
                c.j += kConvGroups;
                c.ks += kConvGroups;
                if (c.ks >= nk) c = at(c.j);
            };
            auto compute = [&](const Cur &c, uint4 (&o)[kEPT / 8]) -> bool {
                const int r = c.j % PP::kRawTma;
                if (!mbar_wait(raw_full(r), (c.j / PP::kRawTma) & 1, a.err, 8, a.wait_ns)) return false;
                const uint8_t *rawt = smem + PP::kRawOff + r * PP::kRawTile;
                if constexpr (PP::kTrans)
                    Dequant<KIND, FMT>::compute_t(a, c.f0, c.ks, tg, rawt, o);
                else
                    Dequant<KIND, FMT>::template compute_tma<kEPT>(a, c.f0, c.ks, tg, rawt, o);
                __syncwarp();
                if (lane == 0) mbar_arrive(raw_empty(r));
                return true;
            };
            uint4 bufa[kEPT / 8], bufb[kEPT / 8];
            Cur nc = at((uint32_t)grp);
            bool ok = (uint32_t)grp >= total || compute(nc, bufa);
            // one step of the group: store step g's chunks (cur), convert the
            // group's next step into nxt, publish step g
            auto body = [&](uint32_t g, const uint4 (&cur)[kEPT / 8], uint4 (&nxt)[kEPT / 8]) -> bool {
                const int s = g % kStages;
                if (!mbar_wait(empty(fb(g)), fph(g) ^ 1, a.err, 5, a.wait_ns)) return false;
                if constexpr (PP::kTrans)
                    Dequant<KIND, FMT>::store_t(tg, cur, sA0 + s * kABytes);
                else
                    Dequant<KIND, FMT>::template store_tma<kEPT>(tg, cur, sA0 + s * kABytes);
                advance(nc);
                // converting the next step before publishing this one lets
                // the stores drain meanwhile (publishing first measured slower)
                const bool okc = nc.j >= total || compute(nc, nxt);
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive(full_a(fb(g)));
                return okc;
            };
            // unrolled by two so the converted chunks alternate between two
            // buffers instead of being copied
            for (uint32_t g = grp; ok && g < total; g += 2 * kConvGroups) {
                ok = body(g, bufa, bufb);
                if (!ok || g + kConvGroups >= total) break;
                ok = body(g + kConvGroups, bufb, bufa);
            }
        }
    } else {
        // ---------------- epilogue (warps 0-3: TMEM lanes 32*warp .. +31)
        uint32_t li = 0;
        const int q = warp;
        uint32_t cons0 = 0u, cons1 = 0u;   // fills of each TMEM buffer consumed so far
        const int nchunks = (nk + PP::kChunk - 1) / PP::kChunk;
        const uint32_t lanes = (uint32_t)(32 * q) << 16;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++li) {
            const Tile tl = clamp_tile<PP::kTileN>(a.tiles[tbeg + item / nft], a.err);
            const int f0 = (item % nft) * a.m_tile;
            const int tot = li & 1, par = tot ^ 1;
            const int ncols = (tl.nrows + 15) & ~15;
            // chunked K loop: add each partial into the total (the MMA warp
            // fills the partial buffer again once it is released)
            bool ok = true;
            for (int j = 1; j < nchunks && ok; ++j) {
                const uint32_t u = par ? cons1++ : cons0++;
                if (!(ok = mbar_wait(tfull(par), u & 1, a.err, 9, a.wait_ns))) break;
                tc_fence_after();
                tmem_drain(tmem + lanes + par * PP::kAccCols, tmem + lanes + tot * PP::kAccCols, ncols);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty(par));
            }
            if (!ok) break;
            const uint32_t ut = tot ? cons1++ : cons0++;
            if (!mbar_wait(tfull(tot), ut & 1, a.err, 6, a.wait_ns)) break;
            tc_fence_after();
            const uint32_t taddr = tmem + lanes + tot * PP::kAccCols;
            for (int c0 = 0; c0 < ncols; c0 += 16) {
                float v[16];
                tmem_ld16(taddr + c0, v);
                if (KIND == GK_FWD_GU) {
                    // lanes 0-15 gate, 16-31 up of features f0 + 16q + (lane & 15)
                    const int f = f0 + 16 * q + (lane & 15);
                    const bool up = lane >= 16;
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        const float send = up ? v[j] : v[j + 1];
                        const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
                        const float g = up ? recv : v[j];
                        const float u = up ? v[j + 1] : recv;
                        const int col = c0 + j + (up ? 1 : 0);
                        if (col < tl.nrows) {
                            const int64_t r = tl.row0 + col;
                            const uint16_t h = f2bf(silu_f(g) * u);
                            a.out[r * a.I + f] = h;
                            if (a.ctxf) {   // saved for the backward: g, u in FP32
                                a.ctxf[r * 2 * a.I + f] = g;
                                a.ctxf[r * 2 * a.I + a.I + f] = u;
                            }
                        }
                    }
                } else if (KIND == GK_BWD_G) {
                    const int f = f0 + 32 * q + lane;
                    const bool fl = f < a.Mtot;
                    const int ncol = min(16, tl.nrows - c0);
                    // routing weight of column `lane` (one load per lane, then broadcast)
                    const float w_lane = lane < ncol ? a.w[a.perm[tl.row0 + c0 + lane]] : 0.f;
#pragma unroll
                    for (int j8 = 0; j8 < 16; j8 += 8) {
                        uint16_t hts[8];   // h~ of 8 columns, loaded together
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            hts[j] = (fl && j8 + j < ncol)
                                         ? a.ht[(int64_t)(tl.row0 + c0 + j8 + j) * a.Mtot + f]
                                         : 0;
                        float part[8];   // G * h~ of the lane's feature, per column
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int jj = j8 + j;
                            const float wr = __shfl_sync(0xffffffffu, w_lane, jj);
                            const int64_t r = tl.row0 + c0 + jj;
                            part[j] = fl ? v[jj] * bf2f(hts[j]) : 0.f;
                            if (fl && jj < ncol) a.outf[r * a.Mtot + f] = wr * v[jj];   // dh~ = w G, FP32
                        }
                        // sum over the warp's 32 features for the 8 columns at once
                        // (reduce-scatter over lane distances 16, 8, 4): lane l then
                        // holds column (l >> 2) & 7 over the lanes sharing bits 2-4
#pragma unroll
                        for (int h = 4; h >= 1; h >>= 1) {
                            const bool up = lane & (4 * h);
#pragma unroll
                            for (int i = 0; i < h; ++i) {
                                const float send = up ? part[i] : part[i + h];
                                const float keep = up ? part[i + h] : part[i];
                                part[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4 * h);
                            }
                        }
                        float sum = part[0] + __shfl_xor_sync(0xffffffffu, part[0], 1);
                        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                        const int jj = j8 + ((lane >> 2) & 7);
                        if ((lane & 3) == 0 && jj < ncol && f0 + 32 * q < a.Mtot)
                            a.dtw_part[(int64_t)(tl.row0 + c0 + jj) * (a.Mtot / 32) + (f0 + 32 * q) / 32] = sum;
                    }
                } else if (KIND == GK_ROUTER) {
                    const int f = f0 + 32 * q + lane;
                    if (f < a.Mtot) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int col = c0 + j;
                            if (col < tl.nrows)
                                a.outf[(int64_t)tl.expert * a.outf_split + (int64_t)(tl.row0 + col) * a.Mtot + f] = v[j];
                        }
                    }
                } else {
                    // FP32 store (the layer's o and dx~: a warp writes 128 contiguous
                    // bytes per column), or BF16
                    const int f = f0 + 32 * q + lane;
                    if (f < a.Mtot) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int col = c0 + j;
                            if (col >= tl.nrows) continue;
                            const int64_t o = (int64_t)(tl.row0 + col) * a.Mtot + f;
                            if (a.outf) a.outf[o] = v[j];
                            else a.out[o] = f2bf(v[j]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty(tot));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

}  // namespace tc
}  // namespace pmoe
