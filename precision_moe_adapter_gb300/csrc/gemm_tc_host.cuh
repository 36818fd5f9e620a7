// gemm_tc_host.cuh -- host launcher of the tcgen05 grouped GEMM for one
// weight format (instantiated once per format in its own translation unit).
#pragma once

#include "gemm_tc.cuh"

namespace pmoe {
namespace tc {

bool make_rows_tmap(CUtensorMap *m, const void *base, int64_t rows, int64_t cols);
int num_sms();

template <int KIND, int FMT>
void launch_kind(const CUtensorMap &tm, const TcArgs &a, cudaStream_t st)
{
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_gemm_tc<KIND, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Pipe<FMT>::kSmem);
        attr = true;
    }
    k_gemm_tc<KIND, FMT><<<num_sms(), kThreads, Pipe<FMT>::kSmem, st>>>(tm, a);
    note_launch();
}

template <int FMT>
bool launch_fmt(const GemmArgs &g, int64_t P, DevErr *err, cudaStream_t st)
{
    if (P <= 0) return true;
    CUtensorMap tm;
    if (!make_rows_tmap(&tm, g.A, P, g.K)) return false;
    TcArgs a{};
    a.wq = g.wq;
    a.ws = g.ws;
    a.wq_stride = g.wq_stride;
    a.ws_stride = g.ws_stride;
    a.Kst = g.Kst;
    a.w_off_elems = g.w_off_elems;
    a.K = g.K;
    a.Mtot = g.Nout;
    a.m_tile = g.kind == GK_FWD_GU ? 64 : 128;
    a.tiles = g.tiles;
    a.chunk_tiles = g.chunk_tiles;
    a.c0 = g.c0;
    a.c1 = g.c1;
    a.slot_index = g.slot_index;
    a.out = g.out;
    a.ctx = g.ctx;
    a.I = g.I;
    a.w = g.w;
    a.perm = g.perm;
    a.ht = g.ht;
    a.dtw_part = g.dtw_part;
    a.err = err;
    switch (g.kind) {
    case GK_FWD_GU: launch_kind<GK_FWD_GU, FMT>(tm, a, st); break;
    case GK_FWD_DOWN: launch_kind<GK_FWD_DOWN, FMT>(tm, a, st); break;
    case GK_BWD_G:
        if constexpr (FMT != kFmtBF16) launch_kind<GK_BWD_G, FMT>(tm, a, st);
        else return false;
        break;
    case GK_BWD_DX:
        if constexpr (FMT != kFmtBF16) launch_kind<GK_BWD_DX, FMT>(tm, a, st);
        else return false;
        break;
    default: return false;
    }
    return true;
}

}  // namespace tc
}  // namespace pmoe
