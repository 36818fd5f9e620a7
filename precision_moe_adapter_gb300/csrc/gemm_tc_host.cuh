// gemm_tc_host.cuh -- host launcher of the tcgen05 grouped GEMM for one
// weight format (instantiated once per format in its own translation unit).
#pragma once

#include <cstring>

#include "gemm_tc.cuh"

namespace pmoe {
namespace tc {

// 16-bit token operand [rows][cols] (as one plane of a 3-D map), box of
// box_rows x 64 columns, 128-byte swizzle
bool make_rows_tmap(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int box_rows);
// uint8 [rows, row_bytes] tensor, box of box_rows x box_bytes, swizzle of
// swizzle_bytes (0: none, 64 or 128; box_bytes must then equal it)
bool make_bytes_tmap(CUtensorMap *m, const void *base, int64_t rows, int64_t row_bytes,
                     int box_bytes, int box_rows, int swizzle_bytes, int l2_promote = 256);
// BF16 scratch slots [slots][rows][cols], box 64 cols x box_rows, 128-byte swizzle
bool make_slots_tmap(CUtensorMap *m, const void *base, int64_t slots, int64_t rows, int64_t cols,
                     int64_t slot_bytes, int box_rows);
int num_sms();
// The bounded-wait limit and withheld item of the next launch: the armed test
// hook (once), else the default limit and none.
void take_wait_hook(uint64_t &wait_ns, int &skip_item);

template <int KIND, int FMT>
bool launch_kind(const CUtensorMap (&tmB)[4], const TcArgs &a, int64_t nmat, cudaStream_t st)
{
    using PP = Pipe<KIND, FMT>;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_gemm_tc<KIND, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)PP::kSmem);
        attr = true;
    }
    CUtensorMap tmA;
    memset(&tmA, 0, sizeof tmA);
    if constexpr (PP::kTmaRaw) {
        // packed weights of all experts as one [nmat * Nst, row bytes] byte tensor
        const int64_t rb = FMT == PMOE_W_FP8_B128_F32 ? a.Kst : a.Kst / 2;
        const int box_rows = PP::kTrans ? 64 : KIND == GK_FWD_GU ? 64 : 128;
        if (!make_bytes_tmap(&tmA, a.wq, nmat * a.Nst, rb, PP::kRowBytes, box_rows,
                             PP::kTrans ? PP::kRowBytes : 0))
            return false;
    } else if constexpr (PP::kBf16) {
        if (!make_slots_tmap(&tmA, a.wq + 2 * a.w_off_elems, nmat, a.Nst, a.Kst, a.wq_stride,
                             KIND == GK_FWD_GU ? 16 : 128))
            return false;
    }
    // Backward kinds: the scales by TMA where their rows are whole 16-byte
    // units and one tensor spans every expert; FP8 (one word per block)
    // and other shapes go by cp.async.
    CUtensorMap tmS;
    memset(&tmS, 0, sizeof tmS);
    TcArgs b = a;
    b.scale_tma = 0;
    if constexpr (PP::kTrans && FMT != PMOE_W_FP8_B128_F32) {
        const int64_t srb = FMT == PMOE_W_INT4_G32_BF16 ? (a.Kst >> 5) * 2 : a.Kst >> 5;
        if (srb % 16 == 0 && ((uintptr_t)a.ws & 15) == 0 && a.ws_stride == a.Nst * srb &&
            make_bytes_tmap(&tmS, a.ws, nmat * a.Nst, srb, 16, kBK, 0))
            b.scale_tma = 1;
    }
    k_gemm_tc<KIND, FMT><<<num_sms(), kThreads, PP::kSmem, st>>>(tmB[0], tmB[1], tmB[2], tmB[3], tmA, tmS, b);
    note_launch();
    return true;
}

template <int FMT>
bool launch_fmt(const GemmArgs &g, int64_t P, DevErr *err, cudaStream_t st)
{
    if (P <= 0) return true;
    CUtensorMap tm[4];   // token tiles in boxes of 256, 128, 64 and 32 rows
    const int Kb = g.Kb ? g.Kb : g.K;
    for (int i = 0; i < 4; ++i)
        if (!make_rows_tmap(&tm[i], g.A, P, Kb, 256 >> i)) return false;
    TcArgs a{};
    a.wq = g.wq;
    a.ws = g.ws;
    a.wq_stride = g.wq_stride;
    a.ws_stride = g.ws_stride;
    a.Kst = g.Kst;
    a.Nst = g.Nst;
    a.w_off_elems = g.w_off_elems;
    a.K = g.K;
    a.Kb = Kb;
    a.Mtot = g.Nout;
    a.m_tile = g.kind == GK_FWD_GU ? 64 : 128;
    a.tiles = g.tiles;
    a.chunk_tiles = g.chunk_tiles;
    a.c0 = g.c0;
    a.c1 = g.c1;
    a.slot_index = g.slot_index;
    a.out = g.out;
    a.ctxf = g.ctxf;
    a.I = g.I;
    a.w = g.w;
    a.perm = g.perm;
    a.ht = g.ht;
    a.dtw_part = g.dtw_part;
    a.outf = g.outf;
    a.outf_split = g.outf_split;
    a.err = err;
    take_wait_hook(a.wait_ns, a.skip_commit_item);
    switch (g.kind) {
    case GK_FWD_GU: return launch_kind<GK_FWD_GU, FMT>(tm, a, g.nmat, st);
    case GK_FWD_DOWN: return launch_kind<GK_FWD_DOWN, FMT>(tm, a, g.nmat, st);
    case GK_BWD_G:
        if constexpr (FMT != kFmtBF16) return launch_kind<GK_BWD_G, FMT>(tm, a, g.nmat, st);
        return false;
    case GK_BWD_DX:
        if constexpr (FMT != kFmtBF16) return launch_kind<GK_BWD_DX, FMT>(tm, a, g.nmat, st);
        return false;
    case GK_BWD_DX_F16:
        if constexpr (FMT != kFmtBF16) return launch_kind<GK_BWD_DX_F16, FMT>(tm, a, g.nmat, st);
        return false;
    case GK_ROUTER:
        if constexpr (FMT == kFmtBF16) return launch_kind<GK_ROUTER, FMT>(tm, a, g.nmat, st);
        return false;
    }
    return false;
}

}  // namespace tc
}  // namespace pmoe
