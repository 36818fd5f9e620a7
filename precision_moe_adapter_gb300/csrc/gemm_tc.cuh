// gemm_tc.cuh -- grouped GEMM of the layer on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA), with the frozen weights dequantized tile by
// tile into shared memory ("临时反量化后实行 grouped GEMM", page 1, 技艺细节).
//
// Orientation: the weights are the MMA's M operand (128 output features per
// tile) and the tokens of one expert are the N operand (16..256 rows per
// tile), so an expert with a few hundred routed tokens fills one tile with
// little padding and every weight tile is dequantized once per token tile.
//
//   D[f, t] = sum_k W~[f, k] * B[t, k]      (FP32 in TMEM: lanes = f, columns = t)
//
// Roles (448 threads, one CTA per SM, persistent over the work list):
//   warps 0-3  epilogue: TMEM -> registers -> fused epilogue -> global
//   warp  4    TMA producer of the activation tiles B (128B swizzle)
//   warp  5    TMEM allocator and MMA issuer (one elected thread)
//   warps 6-13 dequant producers: packed weights -> BF16 A tiles in the
//              canonical K-major 128B-swizzled layout
// Pipeline: kStages shared-memory stages (A 16 KB + B 32 KB) with full/empty
// mbarriers; two TMEM accumulators of 256 columns so the epilogue of one
// tile overlaps the main loop of the next.  Every wait is bounded.
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
constexpr int kNmax = 256;                   // tokens per tile (MMA N)
constexpr int kABytes = kM * kBK * 2;        // 16 KB
constexpr int kBBytes = kNmax * kBK * 2;     // 32 KB
constexpr int kBoxRows = 32;                 // smallest TMA box: 32 token rows x 64 K
constexpr int kEpiWarps = 4;
constexpr int kProdWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kDqWarp0 = 6;
constexpr int kDqWarps = 16;
#ifndef PMOE_CONV_GROUPS
#define PMOE_CONV_GROUPS 2
#endif
constexpr int kConvGroups = PMOE_CONV_GROUPS;   // converter groups taking alternate stages
constexpr int kThreads = (kDqWarp0 + kDqWarps) * 32;
constexpr int kTmemCols = 512;
constexpr unsigned long long kWaitNs = 2000000000ull;   // bounded waits: 2 s

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
// Bounded wait: gives up after kWaitNs, records PMOE_ERR_TIMEOUT with the
// waiting role and returns false (the caller then leaves its loop).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, DevErr *err, int where)
{
    if (mbar_try(bar, parity)) return true;
    uint64_t t0 = globaltimer();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try(bar, parity)) return true;
        if (globaltimer() - t0 > kWaitNs) {
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
// Instruction descriptor, kind::f16: BF16 A and B (K-major), FP32 D, M x N.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                     uint32_t accum)
{
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(
            d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accum)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
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
    int Mtot;                   // output features
    int m_tile;                 // output features per tile (64 gate/up pairs, else 128)
    const Tile *tiles;
    const int32_t *chunk_tiles;
    int c0, c1;
    int slot_index;
    uint16_t *out;
    uint16_t *ctx;
    int I;
    const float *w;
    const int32_t *perm;
    const uint16_t *ht;
    float *dtw_part;
    DevErr *err;
};

template <int KIND>
struct KindTraits {
    // transposed: the contraction runs over the stored matrix's rows
    static constexpr bool kTrans = (KIND == GK_BWD_G || KIND == GK_BWD_DX);
};

// ------------------------------------------------------------------ pipeline sizes
// Per kind and weight format.  Non-transposed kinds get their packed weight
// tile by TMA (raw ring of kRawTma stages: 128 rows of kRowBytes, then 128
// scale words fetched by the producer warp's lanes with cp.async).  BF16
// scratch weights come by TMA straight into the swizzled A stage.  The
// transposed kinds (contraction over the stored rows) prefetch per thread
// with cp.async (ring of kRawStages steps, kSlot bytes per thread).
template <int KIND, int FMT>
struct Pipe {
    static constexpr bool kTrans = KIND == GK_BWD_G || KIND == GK_BWD_DX;
    static constexpr bool kBf16 = FMT == kFmtBF16;
    static constexpr bool kTmaRaw = !kTrans && !kBf16;
    static constexpr bool kFp8 = FMT == PMOE_W_FP8_B128_F32;
    static constexpr int kStagesAB = kFp8 ? 3 : 4;
    static constexpr int kRowBytes = kFp8 ? 64 : 32;
    static constexpr int kRawTile = 128 * kRowBytes + 128 * 4;
    static constexpr int kRawTma = 4;      // raw ring stages
    static constexpr int kRawStages = 4;
    static constexpr int kSlot = kFp8 ? 48 : 32;
    static constexpr int kRawBytes =
        kTmaRaw ? kRawTma * kRawTile : (kTrans ? kRawStages * 256 * kSlot : 0);
    static constexpr int kNumBars = 3 * kStagesAB + 4 + 2 * kRawTma;
    static constexpr int kBarOff = kStagesAB * (kABytes + kBBytes);
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

// ------------------------------------------------------------------ dequant producers
// Thread task per stage (256 threads):
//   non-transposed: smem row m = td >> 1, K half = td & 1 (32 elements)
//   transposed:     rows m = 8*(td & 15) .. +7, K = 4*(td >> 4) .. +3
// issue() copies the thread's packed bytes (and the aligned 4-byte word
// holding its scale) into the ring stage; convert() turns them into BF16 in
// the A stage.  A ring stage is laid out by piece, not by thread: piece j of
// thread td sits at j * 256 * size + td * size, so a warp reading its
// pieces touches consecutive words (no bank conflicts).  Pieces:
//   4-bit, non-transposed: q (16 B), scale word (4 B)
//   FP8,   non-transposed: q0, q1 (16 B each), scale (4 B)
//   BF16 (scratch):        4 x 16 B
//   4-bit, transposed:     4 q words, 4 scale words (4 B each)
//   FP8,   transposed:     4 x q (8 B), 4 scales (4 B)
template <int KIND, int FMT>
struct Dequant {
    static constexpr bool T = KindTraits<KIND>::kTrans;
    // storage row of smem row m (non-transposed kinds)
    __device__ static int64_t row_of(const TcArgs &a, int f0, int m)
    {
        if (KIND == GK_FWD_GU) {
            int q = m >> 5, r = m & 31;
            return r < 16 ? (int64_t)(f0 + 16 * q + r) : (int64_t)(a.I + f0 + 16 * q + r - 16);
        }
        return f0 + m;
    }
    __device__ static bool live(const TcArgs &a, int f0, int td)
    {
        if (T) return f0 + 8 * (td >> 4) < a.Mtot;
        return KIND == GK_FWD_GU || f0 + (td >> 1) < a.Mtot;
    }
    // byte offset of the aligned 4-byte word holding scale index gi
    __device__ static int64_t sword(int64_t gi)
    {
        return FMT == PMOE_W_INT4_G32_BF16 ? 2 * (gi & ~(int64_t)1) : (gi & ~(int64_t)3);
    }
    __device__ static uint32_t spick(uint32_t word, int64_t gi)
    {
        if (FMT == PMOE_W_INT4_G32_BF16) return (gi & 1) ? word >> 16 : word & 0xFFFFu;
        return (word >> (8 * (gi & 3))) & 0xFFu;
    }

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
    __device__ static int64_t scale_word(const TcArgs &a, int64_t row, int ks)
    {
        if (FMT == PMOE_W_INT4_G32_BF16) return 2 * (row * (a.Kst >> 5) + 2 * ks);
        if (FMT == PMOE_W_MXFP4_G32_E8M0) return (row * (a.Kst >> 5) + 2 * ks) & ~(int64_t)3;
        return 4 * ((row >> 7) * (a.Kst >> 7) + ((int64_t)ks * kBK >> 7));
    }

    // Convert one TMA raw tile (non-transposed kinds) for the A stage.
    // A converter group of 8192 / EPT threads: thread tg takes A row
    // m = tg / (64 / EPT) and EPT consecutive K elements of it (EPT / 8
    // 16-byte chunks of the swizzled row).  The converted chunks stay in
    // registers; store_tma() writes them.
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
        const uint32_t sw = *(const uint32_t *)(rawt + 128 * PP::kRowBytes + 4 * rr);
#pragma unroll
        for (int c = 0; c < EPT / 8; ++c) {
            const int e = e0 + 8 * c, grp = e >> 5;
            if (!lv) {
                out[c] = make_uint4(0, 0, 0, 0);
            } else if (FMT == PMOE_W_INT4_G32_BF16) {
                const uint32_t w = *(const uint32_t *)(row + (e >> 1));
                const uint32_t sb = grp ? sw >> 16 : sw & 0xFFFFu;
                uint32_t p[4];
                int4x8_pairs(w, sb | (sb << 16), p);
                out[c].x = prmt(p[0], p[1], 0x5410);
                out[c].y = prmt(p[2], p[3], 0x5410);
                out[c].z = prmt(p[0], p[1], 0x7632);
                out[c].w = prmt(p[2], p[3], 0x7632);
            } else if (FMT == PMOE_W_MXFP4_G32_E8M0) {
                const uint32_t w = *(const uint32_t *)(row + (e >> 1));
                const int64_t gi = stored_row(a, f0, rr) * (a.Kst >> 5) + 2 * ks + grp;
                const float sc = e8m0_value((sw >> (8 * (gi & 3))) & 0xFFu);
                uint32_t o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    o[j] = pack_bf2(__fmul_rn(e2m1_value((w >> (8 * j)) & 15u), sc),
                                    __fmul_rn(e2m1_value((w >> (8 * j + 4)) & 15u), sc));
                out[c] = make_uint4(o[0], o[1], o[2], o[3]);
            } else {
                const uint2 w2 = *(const uint2 *)(row + e);
                const float sc = __uint_as_float(sw);
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
                out[c] = make_uint4(o[0], o[1], o[2], o[3]);
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

    // byte offsets of a thread's pieces inside a ring stage (256 threads)
    __device__ static uint32_t p16(int j, int td) { return (uint32_t)(j * 256 + td) * 16; }
    __device__ static uint32_t p8(int j, int td) { return (uint32_t)(j * 256 + td) * 8; }
    __device__ static uint32_t p4(int j, int td) { return (uint32_t)(j * 256 + td) * 4; }

    __device__ static void issue(const TcArgs &a, const uint8_t *wq, const uint8_t *ws, int f0,
                                 int ks, int td, uint32_t slot)
    {
        if (!live(a, f0, td)) return;
        if (!T) {
            const int m = td >> 1, half = td & 1;
            const int64_t row = row_of(a, f0, m);
            const int64_t k0 = (int64_t)ks * kBK + 32 * half;
            if (FMT == PMOE_W_INT4_G32_BF16 || FMT == PMOE_W_MXFP4_G32_E8M0) {
                cpa16(slot + p16(0, td), wq + row * (a.Kst >> 1) + (k0 >> 1));
                cpa4(slot + 256 * 16 + p4(0, td), ws + sword(row * (a.Kst >> 5) + (k0 >> 5)));
            } else if (FMT == PMOE_W_FP8_B128_F32) {
                const uint8_t *src = wq + row * a.Kst + k0;
                cpa16(slot + p16(0, td), src);
                cpa16(slot + p16(1, td), src + 16);
                cpa4(slot + 2 * 256 * 16 + p4(0, td), ws + 4 * ((row >> 7) * (a.Kst >> 7) + (k0 >> 7)));
            } else {
                const uint8_t *src = wq + 2 * (row * a.Kst + k0);
#pragma unroll
                for (int j = 0; j < 4; ++j) cpa16(slot + p16(j, td), src + 16 * j);
            }
        } else {
            const int mg0 = f0 + 8 * (td >> 4);
            const int64_t n0 = (int64_t)ks * kBK + 4 * (td & 15);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t n = n0 + j;
                if (FMT == PMOE_W_FP8_B128_F32) {
                    cpa8(slot + p8(j, td), wq + n * a.Kst + mg0);
                    cpa4(slot + 4 * 256 * 8 + p4(j, td), ws + 4 * ((n >> 7) * (a.Kst >> 7) + (mg0 >> 7)));
                } else {
                    cpa4(slot + p4(j, td), wq + n * (a.Kst >> 1) + (mg0 >> 1));
                    cpa4(slot + 4 * 256 * 4 + p4(j, td), ws + sword(n * (a.Kst >> 5) + (mg0 >> 5)));
                }
            }
        }
    }

    // Convert the slot into the A stage (zeros for rows past a ragged tile).
    __device__ static void convert(const TcArgs &a, int f0, int ks, int td, const uint8_t *slot,
                                   uint32_t sA)
    {
        const bool lv = live(a, f0, td);
        if (!T) {
            const int m = td >> 1, half = td & 1;
            const int64_t row = row_of(a, f0, m);
            const int64_t k0 = (int64_t)ks * kBK + 32 * half;
            uint4 out[4];
            if (!lv) {
#pragma unroll
                for (int j = 0; j < 4; ++j) out[j] = make_uint4(0, 0, 0, 0);
            } else if (FMT == PMOE_W_INT4_G32_BF16) {
                const uint4 q = *(const uint4 *)(slot + p16(0, td));
                const uint32_t sb = spick(*(const uint32_t *)(slot + 256 * 16 + p4(0, td)),
                                          row * (a.Kst >> 5) + (k0 >> 5));
                const uint32_t s2 = sb | (sb << 16);
                const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t p[4];
                    int4x8_pairs(words[j], s2, p);
                    out[j].x = prmt(p[0], p[1], 0x5410);
                    out[j].y = prmt(p[2], p[3], 0x5410);
                    out[j].z = prmt(p[0], p[1], 0x7632);
                    out[j].w = prmt(p[2], p[3], 0x7632);
                }
            } else if (FMT == PMOE_W_MXFP4_G32_E8M0) {
                const uint4 q = *(const uint4 *)(slot + p16(0, td));
                const float sc = e8m0_value(spick(*(const uint32_t *)(slot + 256 * 16 + p4(0, td)),
                                                  row * (a.Kst >> 5) + (k0 >> 5)));
                const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t w = words[j], o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        o[e] = pack_bf2(__fmul_rn(e2m1_value((w >> (8 * e)) & 15u), sc),
                                        __fmul_rn(e2m1_value((w >> (8 * e + 4)) & 15u), sc));
                    out[j] = make_uint4(o[0], o[1], o[2], o[3]);
                }
            } else if (FMT == PMOE_W_FP8_B128_F32) {
                const uint4 q0 = *(const uint4 *)(slot + p16(0, td));
                const uint4 q1 = *(const uint4 *)(slot + p16(1, td));
                const float sc = *(const float *)(slot + 2 * 256 * 16 + p4(0, td));
                const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t o[4];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t w = words[2 * j + h];
                        __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFFu), __NV_E4M3);
                        __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
                        const float2 fl = __half22float2(*(const __half2 *)&lo);
                        const float2 fh = __half22float2(*(const __half2 *)&hi);
                        o[2 * h] = pack_bf2(__fmul_rn(fl.x, sc), __fmul_rn(fl.y, sc));
                        o[2 * h + 1] = pack_bf2(__fmul_rn(fh.x, sc), __fmul_rn(fh.y, sc));
                    }
                    out[j] = make_uint4(o[0], o[1], o[2], o[3]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) out[j] = *(const uint4 *)(slot + p16(j, td));
            }
            const uint32_t rowaddr = sA + m * 128;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = 4 * half + j;
                st_shared_v4(rowaddr + ((c ^ (m & 7)) << 4), out[j]);
            }
        } else {
            // transposed: A[m][k] = W[k0 + k][f0 + m] (contraction over stored rows)
            // lanes vary kb (K chunks of one row m): the 8-byte stores of a warp
            // cover whole 128-byte rows, conflict-free
            const int kb = td & 15, mb = td >> 4;
            const int mg0 = f0 + 8 * mb;
            const int64_t n0 = (int64_t)ks * kBK + 4 * kb;
            uint32_t v[8][2];   // for each m: (k0,k1), (k2,k3)
            if (!lv) {
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i][0] = v[i][1] = 0;
            } else if (FMT == PMOE_W_INT4_G32_BF16) {
                uint32_t p[4][4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t w = *(const uint32_t *)(slot + p4(j, td));
                    const uint32_t sb = spick(*(const uint32_t *)(slot + 4 * 256 * 4 + p4(j, td)),
                                              (n0 + j) * (a.Kst >> 5) + (mg0 >> 5));
                    int4x8_pairs(w, sb | (sb << 16), p[j]);
                }
                // p[j][i & 3] holds (m = i, m = i + 4) of row j
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t sel = i < 4 ? 0x5410u : 0x7632u;
                    v[i][0] = prmt(p[0][i & 3], p[1][i & 3], sel);
                    v[i][1] = prmt(p[2][i & 3], p[3][i & 3], sel);
                }
            } else {
                float f[4][8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (FMT == PMOE_W_MXFP4_G32_E8M0) {
                        const uint32_t w = *(const uint32_t *)(slot + p4(j, td));
                        const float sc = e8m0_value(spick(*(const uint32_t *)(slot + 4 * 256 * 4 + p4(j, td)),
                                                          (n0 + j) * (a.Kst >> 5) + (mg0 >> 5)));
#pragma unroll
                        for (int i = 0; i < 8; ++i) f[j][i] = __fmul_rn(e2m1_value((w >> (4 * i)) & 15u), sc);
                    } else {
                        const uint2 w = *(const uint2 *)(slot + p8(j, td));
                        const float sc = *(const float *)(slot + 4 * 256 * 8 + p4(j, td));
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            f[j][i] = __fmul_rn(e4m3_value(((i < 4 ? w.x : w.y) >> (8 * (i & 3))) & 255u), sc);
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    v[i][0] = pack_bf2(f[0][i], f[1][i]);
                    v[i][1] = pack_bf2(f[2][i], f[3][i]);
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int m = 8 * mb + i;
                st_shared_v2(sA + m * 128 + ((((kb >> 1)) ^ (m & 7)) << 4) + (kb & 1) * 8, v[i][0],
                             v[i][1]);
            }
        }
    }
};

__device__ __forceinline__ float silu_f(float g) { return g / (1.f + expf(-g)); }

// ------------------------------------------------------------------ kernel
template <int KIND, int FMT>
__global__ void __launch_bounds__(kThreads, 1) k_gemm_tc(const __grid_constant__ CUtensorMap tmB256,
                                                         const __grid_constant__ CUtensorMap tmB128,
                                                         const __grid_constant__ CUtensorMap tmB64,
                                                         const __grid_constant__ CUtensorMap tmB32,
                                                         const __grid_constant__ CUtensorMap tmA,
                                                         const TcArgs a)
{
    using PP = Pipe<KIND, FMT>;
    constexpr int kStages = PP::kStagesAB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sA0 = smem_u32(smem);
    const uint32_t sB0 = sA0 + kStages * kABytes;
    const uint32_t bar0 = sB0 + kStages * kBBytes;
    uint32_t *tmem_slot = (uint32_t *)(smem + PP::kBarOff + 8 * PP::kNumBars);
    auto full_a = [&](int s) { return bar0 + 8 * s; };
    auto full_b = [&](int s) { return bar0 + 8 * (kStages + s); };
    auto empty = [&](int s) { return bar0 + 8 * (2 * kStages + s); };
    auto tfull = [&](int c) { return bar0 + 8 * (3 * kStages + c); };
    auto tempty = [&](int c) { return bar0 + 8 * (3 * kStages + 2 + c); };
    auto raw_full = [&](int r) { return bar0 + 8 * (3 * kStages + 4 + r); };
    auto raw_empty = [&](int r) { return bar0 + 8 * (3 * kStages + 4 + PP::kRawTma + r); };
    const uint32_t raw0 = smem_u32(smem + PP::kRawOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tbeg = a.chunk_tiles[a.c0], tend = a.chunk_tiles[a.c1];
    const int nft = (a.Mtot + a.m_tile - 1) / a.m_tile;
    const int n_items = (tend - tbeg) * nft;
    const int nk = a.K / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_a(s), PP::kBf16 ? 1 : PP::kTmaRaw ? kDqWarps / kConvGroups : kDqWarps);
            mbar_init(full_b(s), 1);
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

    if (warp == kProdWarp) {
        // ---------------- producer: token tiles (TMA), packed weight tiles
        // (TMA) with their scale words (cp.async by the 32 lanes), or BF16
        // weight tiles (TMA into the swizzled A stage)
        uint32_t g = 0;
        bool ok = true;
        for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
            const Tile tl = a.tiles[tbeg + item / nft];
            // token rows covered: round up to 32, in boxes of 256/128/64/32 rows
            const int brows = (tl.nrows + kBoxRows - 1) & ~(kBoxRows - 1);
            const int f0 = (item % nft) * a.m_tile;
            const int64_t widx = a.slot_index ? (tl.chunk & 0xffff) : tl.expert;
            for (int ks = 0; ks < nk; ++ks, ++g) {
                if constexpr (PP::kTmaRaw) {
                    const int r = g % PP::kRawTma;
                    if (!(ok = mbar_wait(raw_empty(r), ((g / PP::kRawTma) & 1) ^ 1, a.err, 7))) break;
                    const uint32_t dst = raw0 + r * PP::kRawTile;
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
                    const uint8_t *ws = a.ws + widx * a.ws_stride;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int rr = lane + 32 * i;
                        const bool lv = KIND == GK_FWD_GU || f0 + rr < a.Mtot;
                        if (lv)
                            cpa4(dst + 128 * PP::kRowBytes + 4 * rr,
                                 ws + Dequant<KIND, FMT>::scale_word(
                                          a, Dequant<KIND, FMT>::stored_row(a, f0, rr), ks));
                    }
                    cpa_mbar_arrive(raw_full(r));
                }
                const int s = g % kStages;
                const uint32_t ph = (g / kStages) & 1;
                if (!(ok = mbar_wait(empty(s), ph ^ 1, a.err, 1))) break;
                if (lane == 0) {
                    mbar_expect_tx(full_b(s), brows * kBK * 2);
                    for (int r0 = 0; r0 < brows;) {
                        const int left = brows - r0;
                        const CUtensorMap *tm = left >= 256 ? &tmB256 : left >= 128 ? &tmB128
                                              : left >= 64 ? &tmB64 : &tmB32;
                        const int rows = left >= 256 ? 256 : left >= 128 ? 128 : left >= 64 ? 64 : 32;
                        tma_load_2d(sB0 + s * kBBytes + r0 * kBK * 2, tm, ks * kBK, tl.row0 + r0, full_b(s));
                        r0 += rows;
                    }
                    if constexpr (PP::kBf16) {
                        mbar_expect_tx(full_a(s), kABytes);
                        const int slot = (int)widx;
                        if (KIND == GK_FWD_GU) {
                            // A rows 32q .. 32q+15: gate f0+16q ..; 32q+16 .. 32q+31: up
#pragma unroll
                            for (int qq = 0; qq < 4; ++qq) {
                                tma_load_3d(sA0 + s * kABytes + (32 * qq) * 128, &tmA, ks * kBK,
                                            f0 + 16 * qq, slot, full_a(s));
                                tma_load_3d(sA0 + s * kABytes + (32 * qq + 16) * 128, &tmA, ks * kBK,
                                            a.I + f0 + 16 * qq, slot, full_a(s));
                            }
                        } else {
                            tma_load_3d(sA0 + s * kABytes, &tmA, ks * kBK, f0, slot, full_a(s));
                        }
                    }
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer
        if (lane == 0) {
            uint32_t g = 0, li = 0;
            bool ok = true;
            for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++li) {
                const Tile tl = a.tiles[tbeg + item / nft];
                const int N = (tl.nrows + 15) & ~15;
                const uint32_t idesc = idesc_bf16(kM, N);
                const int acc = li & 1;
                if (!(ok = mbar_wait(tempty(acc), ((li >> 1) & 1) ^ 1, a.err, 2))) break;
                tc_fence_after();
                const uint32_t d = tmem + acc * (kTmemCols / 2);
                for (int ks = 0; ks < nk; ++ks, ++g) {
                    const int s = g % kStages;
                    const uint32_t ph = (g / kStages) & 1;
                    if (!(ok = mbar_wait(full_a(s), ph, a.err, 3))) break;
                    if (!(ok = mbar_wait(full_b(s), ph, a.err, 4))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        umma(d, sdesc(sA0 + s * kABytes + kk * 32), sdesc(sB0 + s * kBBytes + kk * 32),
                             idesc, (ks | kk) != 0);
                    umma_commit(empty(s));
                }
                if (ok) umma_commit(tfull(acc));
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
            auto compute = [&](uint32_t j, uint4 (&o)[kEPT / 8]) -> bool {
                const int item = (int)blockIdx.x + (int)(j / nk) * (int)gridDim.x;
                const int r = j % PP::kRawTma;
                if (!mbar_wait(raw_full(r), (j / PP::kRawTma) & 1, a.err, 8)) return false;
                Dequant<KIND, FMT>::template compute_tma<kEPT>(a, (item % nft) * a.m_tile, (int)(j % nk),
                                                               tg, smem + PP::kRawOff + r * PP::kRawTile, o);
                __syncwarp();
                if (lane == 0) mbar_arrive(raw_empty(r));
                return true;
            };
            uint4 cur[kEPT / 8], nxt[kEPT / 8];
            bool ok = (uint32_t)grp >= total || compute(grp, cur);
            for (uint32_t g = grp; ok && g < total; g += kConvGroups) {
                const int s = g % kStages;
                if (!mbar_wait(empty(s), ((g / kStages) & 1) ^ 1, a.err, 5)) break;
                Dequant<KIND, FMT>::template store_tma<kEPT>(tg, cur, sA0 + s * kABytes);
                if (g + kConvGroups < total) ok = compute(g + kConvGroups, nxt);
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive(full_a(s));
#pragma unroll
                for (int c = 0; c < kEPT / 8; ++c) cur[c] = nxt[c];
            }
        } else if constexpr (PP::kTrans) {
            // transposed kinds: the first 256 converter threads convert, the
            // other warps only take part in the stage handshake
            const bool worker = td < 256;
        // ---------------- dequant producers: packed weights prefetched
        // kRawStages - 1 steps ahead with cp.async, converted into the A stage
        uint8_t *raw = smem + PP::kRawOff;
        const uint32_t raw_a = smem_u32(raw);
        const int my_items = n_items > (int)blockIdx.x ? (n_items - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
        const uint32_t total = (uint32_t)my_items * nk;
        constexpr uint32_t kRing = PP::kRawStages, kRingStride = 256 * PP::kSlot;
        // work-item context, reloaded only when a step starts a new item
        struct Ctx {
            int li = -1, f0 = 0;
            const uint8_t *wq = nullptr, *ws = nullptr;
        };
        auto load_ctx = [&](Ctx &c, int li) {
            if (c.li == li) return;
            const int item = (int)blockIdx.x + li * (int)gridDim.x;
            const Tile tl = a.tiles[tbeg + item / nft];
            c.li = li;
            c.f0 = (item % nft) * a.m_tile;
            const int64_t widx = a.slot_index ? (tl.chunk & 0xffff) : tl.expert;
            c.wq = a.wq + widx * a.wq_stride + (FMT == kFmtBF16 ? 2 * a.w_off_elems : 0);
            c.ws = a.ws ? a.ws + widx * a.ws_stride : nullptr;
        };
        Ctx cur, ahead;
        auto issue_step = [&](uint32_t j) {
            if (worker && j < total) {
                load_ctx(ahead, (int)(j / nk));
                Dequant<KIND, FMT>::issue(a, ahead.wq, ahead.ws, ahead.f0, (int)(j % nk), td,
                                          raw_a + (j % kRing) * kRingStride);
            }
            cpa_commit();
        };
        for (uint32_t j = 0; j + 1 < kRing; ++j) issue_step(j);
        for (uint32_t g = 0; g < total; ++g) {
            issue_step(g + kRing - 1);
            load_ctx(cur, (int)(g / nk));
            cpa_wait<kRing - 1>();
            const int s = g % kStages;
            const uint32_t ph = (g / kStages) & 1;
            if (!mbar_wait(empty(s), ph ^ 1, a.err, 5)) break;
            if (worker)
                Dequant<KIND, FMT>::convert(a, cur.f0, (int)(g % nk), td,
                                            raw + (g % kRing) * kRingStride, sA0 + s * kABytes);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(full_a(s));
        }
        cpa_wait<0>();
        }
    } else {
        // ---------------- epilogue (warps 0-3: TMEM lanes 32*warp .. +31)
        uint32_t li = 0;
        const int q = warp;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++li) {
            const Tile tl = a.tiles[tbeg + item / nft];
            const int f0 = (item % nft) * a.m_tile;
            const int acc = li & 1;
            if (!mbar_wait(tfull(acc), (li >> 1) & 1, a.err, 6)) break;
            tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + acc * (kTmemCols / 2);
            const int ncols = (tl.nrows + 15) & ~15;
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
                            if (a.ctx) {   // saved for the backward: [g | u | h]
                                uint16_t *c = a.ctx + r * 3 * a.I + f;
                                c[0] = f2bf(g);
                                c[a.I] = f2bf(u);
                                c[2 * a.I] = h;
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
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int jj = j8 + j;
                            const float wr = __shfl_sync(0xffffffffu, w_lane, jj);
                            const int64_t r = tl.row0 + c0 + jj;
                            float part = fl ? v[jj] * bf2f(hts[j]) : 0.f;
                            if (fl && jj < ncol) a.out[r * a.Mtot + f] = f2bf(wr * v[jj]);
#pragma unroll
                            for (int o = 16; o; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
                            if (fl && lane == 0 && jj < ncol)
                                a.dtw_part[r * (a.Mtot / 32) + (f0 + 32 * q) / 32] = part;
                        }
                    }
                } else {
                    const int f = f0 + 32 * q + lane;
                    if (f < a.Mtot) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int col = c0 + j;
                            if (col < tl.nrows) a.out[(int64_t)(tl.row0 + col) * a.Mtot + f] = f2bf(v[j]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty(acc));
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
