// api.cu -- the extern "C" entry points of libpmoe (declared in pmoe.h):
// host-side validation, workspace layout and the order of launches.
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "launch.h"

namespace pmoe {

static std::atomic<uint64_t> g_launches{0};
void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

// ------------------------------------------------------------------ timer
// Event pairs around launches of the timed kernel classes (diagnostic).
struct TimerRec {
    int cls;
    cudaEvent_t a, b;
};
static std::mutex g_tmu;
static bool g_timing = false;
static std::vector<TimerRec> g_recs;
static std::vector<cudaEvent_t> g_pool;

static cudaEvent_t pool_event()
{
    if (!g_pool.empty()) {
        cudaEvent_t e = g_pool.back();
        g_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

struct ScopedTimer {
    bool on = false;
    TimerRec rec{};
    cudaStream_t st;
    ScopedTimer(int cls, cudaStream_t s) : st(s)
    {
        std::lock_guard<std::mutex> g(g_tmu);
        if (!g_timing) return;
        rec.cls = cls;
        rec.a = pool_event();
        rec.b = pool_event();
        on = rec.a && rec.b;
        if (on) cudaEventRecord(rec.a, st);
    }
    ~ScopedTimer()
    {
        if (!on) return;
        cudaEventRecord(rec.b, st);
        std::lock_guard<std::mutex> g(g_tmu);
        g_recs.push_back(rec);
    }
};

static void clear_records()
{
    for (auto &r : g_recs) {
        g_pool.push_back(r.a);
        g_pool.push_back(r.b);
    }
    g_recs.clear();
}

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
static size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

// Sequential carving of a workspace into 256-byte aligned regions.
struct Carver {
    uint8_t *base;
    size_t off = 0;
    explicit Carver(void *b) : base((uint8_t *)b) {}
    template <class T>
    T *take(size_t count)
    {
        T *p = base ? (T *)(base + off) : nullptr;
        off = up256(off + count * sizeof(T));
        return p;
    }
};

bool dims_ok(const pmoe_dims &d)
{
    if (d.T < 0 || d.d <= 0 || d.inter <= 0 || d.E <= 0 || d.k <= 0) return false;
    if (d.k > d.E || d.E > 4096 || d.k > 32) return false;
    if (d.d % 64 || d.inter % 64) return false;
    if (d.d > 8192 || d.inter > 8192) return false;   // row buffers live in shared memory
    if (!(d.block == 16 || d.block == 32 || d.block == 64 || d.block == 128)) return false;
    if (d.d % d.block || d.inter % d.block) return false;
    if ((int64_t)d.T * d.k > (int64_t)INT32_MAX / 2) return false;
    return true;
}

static bool fmt_ok(const pmoe_dims &d, int fmt)
{
    if (fmt == PMOE_W_INT4_G32_BF16 || fmt == PMOE_W_MXFP4_G32_E8M0) return true;
    if (fmt == PMOE_W_FP8_B128_F32) return d.d % 128 == 0 && d.inter % 128 == 0;
    return false;
}

static int nchunks_of(const pmoe_dims &d, int C) { return (int)cdiv(d.E, C); }
// Work-list sizes: GEMM token tiles (<= 256 rows, multiples of 16) and
// rotation tiles (<= 64 rows), each at most rows/16 (rows/64) + E.
static int max_tiles_of(const pmoe_dims &d) { return (int)(cdiv((int64_t)d.T * d.k, 16) + d.E); }
static int max_rot_tiles_of(const pmoe_dims &d)
{
    return (int)(cdiv((int64_t)d.T * d.k, kRotTileRows) + d.E);
}
constexpr int kGemmRows = 256, kGemmAlign = 16;   // token tile <= the GEMM tile width

static pmoe_status run_gemm(const GemmArgs &g, int64_t P, DevErr *err, cudaStream_t st)
{
    return launch_gemm_tc(g, P, err, st) ? PMOE_OK : PMOE_ERR_CUDA;
}

// Work lists of one call: GEMM tiles per chunk and rotation tiles per chunk.
struct Lists {
    Tile *tiles, *rtiles;
    int32_t *chunk_tiles, *chunk_rows, *chunk_rtiles, *chunk_rrows;
};
static Lists carve_lists(Carver &c, const pmoe_dims &d, int C)
{
    Lists l;
    l.tiles = c.take<Tile>(max_tiles_of(d));
    l.rtiles = c.take<Tile>(max_rot_tiles_of(d));
    l.chunk_tiles = c.take<int32_t>(nchunks_of(d, C) + 2);
    l.chunk_rows = c.take<int32_t>(nchunks_of(d, C) + 2);
    l.chunk_rtiles = c.take<int32_t>(nchunks_of(d, C) + 2);
    l.chunk_rrows = c.take<int32_t>(nchunks_of(d, C) + 2);
    return l;
}
static void build_lists(const Lists &l, const pmoe_dims &d, int C, const pmoe_routing *rt,
                        cudaStream_t st)
{
    launch_build_tiles(d.E, C, kGemmRows, kGemmAlign, rt->counts, rt->offsets, rt->active,
                       rt->num_active, l.tiles, l.chunk_tiles, l.chunk_rows, st);
    launch_build_tiles(d.E, C, kRotTileRows, 1, rt->counts, rt->offsets, rt->active,
                       rt->num_active, l.rtiles, l.chunk_rtiles, l.chunk_rrows, st);
}

struct FwdWs {
    DevErr *err;
    Lists l;
    uint16_t *xt, *h, *ht, *scratch;
    float *o;         // each pair's expert output, FP32 [P, d]
    uint64_t *snap;   // adapter-slot snapshot of this forward
};
static FwdWs carve_fwd(void *ws, const pmoe_dims &d, int C, int mode, size_t *bytes)
{
    Carver c(ws);
    FwdWs w;
    int64_t P = (int64_t)d.T * d.k;
    w.err = c.take<DevErr>(kHdrBytes / sizeof(DevErr));
    w.l = carve_lists(c, d, C);
    w.xt = c.take<uint16_t>(P * d.d);
    w.h = c.take<uint16_t>(P * d.inter);
    w.ht = c.take<uint16_t>(P * d.inter);
    w.o = c.take<float>(P * d.d);
    int64_t slots = mode == PMOE_MODE_SCRATCH ? std::min(C, d.E) : 0;
    w.scratch = c.take<uint16_t>(slots * 3 * (int64_t)d.inter * d.d);
    w.snap = c.take<uint64_t>(2);
    if (bytes) *bytes = c.off;
    return w;
}

struct BwdWs {
    DevErr *err;
    Lists l;
    uint16_t *dyp;
    uint16_t *dgu;          // [dg | du], FP16 [P, 2I]
    float *dht, *dxt, *dxp; // dh~ [P, I], dx~ [P, d], rotated dx [P, d], FP32
    float *dtw_part;
};
static BwdWs carve_bwd(void *ws, const pmoe_dims &d, int C, size_t *bytes)
{
    Carver c(ws);
    BwdWs w;
    int64_t P = (int64_t)d.T * d.k;
    w.err = c.take<DevErr>(kHdrBytes / sizeof(DevErr));
    w.l = carve_lists(c, d, C);
    w.dyp = c.take<uint16_t>(P * d.d);      // gathered dY rows
    w.dht = c.take<float>(P * d.inter);
    w.dgu = c.take<uint16_t>(P * 2 * d.inter);
    w.dxt = c.take<float>(P * d.d);
    w.dxp = c.take<float>(P * d.d);
    w.dtw_part = c.take<float>(P * (d.inter / 32));
    if (bytes) *bytes = c.off;
    return w;
}

struct PermWs {
    DevErr *err;
    int32_t *hist;
    float *logits;
    uint16_t *wr3;        // router weight split, [splits][E][3d / splits] bf16
    float *rpart;         // router partials [splits][T][E] f32
    Tile *rtiles;         // router token tiles of every split
    int32_t *rchunk;      // [2]
};
static PermWs carve_perm(void *ws, const pmoe_dims &d, size_t *bytes)
{
    Carver c(ws);
    PermWs w;
    w.err = c.take<DevErr>(kHdrBytes / sizeof(DevErr));
    w.hist = c.take<int32_t>(permute_ws_bytes(d.T * d.k, d.E) / sizeof(int32_t));
    w.logits = c.take<float>((int64_t)d.T * d.E);
    w.wr3 = c.take<uint16_t>((int64_t)d.E * 3 * d.d);
    w.rpart = c.take<float>((int64_t)router_splits(d.d) * d.T * d.E);
    w.rtiles = c.take<Tile>(cdiv(d.T > 0 ? d.T : 1, 16) * router_splits(d.d));
    w.rchunk = c.take<int32_t>(2);
    if (bytes) *bytes = c.off;
    return w;
}

static pmoe_status launched(cudaStream_t st)
{
    (void)st;
    return cudaPeekAtLastError() == cudaSuccess ? PMOE_OK : PMOE_ERR_CUDA;
}

}  // namespace pmoe

using namespace pmoe;

extern "C" {

const char *pmoe_status_string(pmoe_status s)
{
    switch (s) {
    case PMOE_OK: return "ok";
    case PMOE_ERR_INVALID_ARG: return "invalid argument";
    case PMOE_ERR_UNSUPPORTED: return "unsupported";
    case PMOE_ERR_WORKSPACE: return "workspace too small";
    case PMOE_ERR_CUDA: return "CUDA error";
    case PMOE_ERR_BAD_INDEX: return "expert index out of range";
    case PMOE_ERR_TIMEOUT: return "bounded wait timed out";
    }
    return "unknown status";
}

uint64_t pmoe_launch_count(void) { return g_launches.load(); }

pmoe_status pmoe_kernel_timing(int enable)
{
    std::lock_guard<std::mutex> g(g_tmu);
    clear_records();
    g_timing = enable != 0;
    return PMOE_OK;
}

pmoe_status pmoe_kernel_time(int which, double *ms_total, int *launches)
{
    if (which < 0 || which >= PMOE_KT_COUNT || !ms_total || !launches)
        return PMOE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(g_tmu);
    double tot = 0;
    int n = 0;
    for (auto &r : g_recs) {
        if (r.cls != which) continue;
        if (cudaEventSynchronize(r.b) != cudaSuccess) return PMOE_ERR_CUDA;
        float ms = 0;
        if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return PMOE_ERR_CUDA;
        tot += ms;
        ++n;
    }
    *ms_total = tot;
    *launches = n;
    return PMOE_OK;
}

size_t moe_workspace_bytes(pmoe_dims dims, int op, int32_t chunk_C, int mode)
{
    if (!dims_ok(dims)) return 0;
    int C = chunk_C < 1 ? 1 : std::min(chunk_C, dims.E);
    size_t b = 0;
    if (op == PMOE_OP_PERMUTE) carve_perm(nullptr, dims, &b);
    else if (op == PMOE_OP_FORWARD) carve_fwd(nullptr, dims, C, mode, &b);
    else if (op == PMOE_OP_BACKWARD) carve_bwd(nullptr, dims, C, &b);
    return b;
}

size_t moe_ctx_bytes(pmoe_dims dims)
{
    if (!dims_ok(dims)) return 0;
    return (size_t)dims.T * dims.k * dims.inter * (4 * 2 + 2 + 2);
}

size_t moe_scratch_bytes(pmoe_dims dims, int32_t chunk_C, int mode)
{
    if (!dims_ok(dims) || mode != PMOE_MODE_SCRATCH || chunk_C < 1) return 0;
    return (size_t)std::min(chunk_C, dims.E) * 3 * (size_t)dims.inter * dims.d * 2;
}

pmoe_status moe_clear_status(void *ws, cudaStream_t stream)
{
    if (!ws) return PMOE_ERR_INVALID_ARG;
    return cudaMemsetAsync(ws, 0, sizeof(DevErr), stream) == cudaSuccess ? PMOE_OK : PMOE_ERR_CUDA;
}

pmoe_status moe_query_status(void *ws, cudaStream_t stream)
{
    if (!ws) return PMOE_ERR_INVALID_ARG;
    DevErr e;
    if (cudaMemcpyAsync(&e, ws, sizeof e, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return PMOE_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return PMOE_ERR_CUDA;
    if (cudaMemsetAsync(ws, 0, sizeof e, stream) != cudaSuccess) return PMOE_ERR_CUDA;
    return (pmoe_status)e.code;
}

pmoe_status moe_route(pmoe_dims dims, const void *X, const float *Wr, const float *bias,
                      float *logits, int32_t *idx, float *w, int mode, void *ws, size_t ws_bytes,
                      cudaStream_t stream)
{
    if (!dims_ok(dims) || (mode != PMOE_ROUTE_FAST && mode != PMOE_ROUTE_EXACT))
        return PMOE_ERR_INVALID_ARG;
    if (dims.T > 0 && (!X || !Wr || !idx || !w)) return PMOE_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Wr) || !aligned16(idx) || !aligned16(w) || !aligned16(bias) ||
        !aligned16(logits))
        return PMOE_ERR_INVALID_ARG;
    size_t need;
    PermWs pw = carve_perm(ws, dims, &need);
    if (!ws || ws_bytes < need || !aligned16(ws)) return PMOE_ERR_WORKSPACE;
    if (dims.T == 0) return PMOE_OK;
    if (mode == PMOE_ROUTE_EXACT) {
        ScopedTimer tm(PMOE_KT_ROUTER, stream);
        launch_router_exact(dims.T, dims.d, dims.E, (const uint16_t *)X, Wr, pw.logits, stream);
    } else {
        ScopedTimer tm(PMOE_KT_ROUTER, stream);
        // K splits (a function of d alone): every split is one matrix of
        // [E, 3d / splits] and writes its own partial logits
        const int splits = router_splits(dims.d);
        const int ks = 3 * dims.d / splits;
        const int rows = router_tile_rows(dims.T, dims.E, splits, gemm_num_sms());
        launch_router_prep(dims.T, dims.d, dims.E, Wr, pw.wr3, pw.rtiles, pw.rchunk, rows, stream);
        GemmArgs g{};
        g.kind = GK_ROUTER;
        g.fmt = kFmtBF16;
        g.wq = (const uint8_t *)pw.wr3;
        g.wq_stride = (int64_t)dims.E * ks * 2;
        g.Nst = dims.E;
        g.Kst = ks;
        g.nmat = splits;
        g.A = (const uint16_t *)X;
        g.K = ks;
        g.Kb = dims.d;
        g.Nout = dims.E;
        g.tiles = pw.rtiles;
        g.chunk_tiles = pw.rchunk;
        g.c0 = 0;
        g.c1 = 1;
        g.outf = pw.rpart;
        g.outf_split = (int64_t)dims.T * dims.E;
        if (!launch_gemm_tc(g, dims.T, pw.err, stream)) return PMOE_ERR_CUDA;
        launch_router_reduce(dims.T, dims.E, splits, pw.rpart, pw.logits, stream);
    }
    launch_route_topk(dims.T, dims.E, dims.k, pw.logits, bias, idx, w, logits, stream);
    return launched(stream);
}

pmoe_status moe_permute(pmoe_dims dims, const int32_t *idx, const pmoe_routing *out, void *ws,
                        size_t ws_bytes, cudaStream_t stream)
{
    if (!dims_ok(dims) || !out) return PMOE_ERR_INVALID_ARG;
    if ((dims.T > 0 && (!idx || !out->perm || !out->inv_perm)) || !out->counts ||
        !out->offsets || !out->active || !out->num_active)
        return PMOE_ERR_INVALID_ARG;
    size_t need;
    PermWs pw = carve_perm(ws, dims, &need);
    if (!ws || ws_bytes < need || !aligned16(ws)) return PMOE_ERR_WORKSPACE;
    launch_permute(dims.T * dims.k, dims.E, idx, out->counts, out->offsets, out->perm,
                   out->inv_perm, out->active, out->num_active, pw.hist, pw.err, stream);
    return launched(stream);
}

static bool routing_ok(const pmoe_routing *rt, const pmoe_dims &d)
{
    if (!rt) return false;
    if (!rt->counts || !rt->offsets || !rt->active || !rt->num_active) return false;
    if (d.T > 0 && (!rt->idx || !rt->w || !rt->perm || !rt->inv_perm)) return false;
    return true;
}

static bool weights_ok(const pmoe_weights *wt, const pmoe_dims &d)
{
    if (!wt || !fmt_ok(d, wt->fmt)) return false;
    if (!wt->w13 || !wt->s13 || !wt->w2 || !wt->s2) return false;
    return aligned16(wt->w13) && aligned16(wt->w2) && aligned16(wt->s13) && aligned16(wt->s2);
}

static bool adapter_ok(const pmoe_adapter *ad)
{
    if (!ad) return true;
    if (!ad->R_up && ad->R_down) return false;
    if (ad->stride_up < 0 || ad->stride_down < 0) return false;
    return aligned16(ad->R_up) && aligned16(ad->R_down);
}

namespace pmoe {
// Plain rotation of BF16 rows (x R, or x R^T with trans) over a work list.
static RotCall rot_rows(int b, bool trans, const void *src, int64_t src_ld, const int32_t *gather_perm,
                        int k, const uint16_t *R, int64_t stride, int dim, void *out, int64_t out_ld,
                        const Tile *tiles, const int32_t *tbeg, const int32_t *tend, int max_tiles,
                        int nrows)
{
    RotCall c{};
    c.b = b;
    c.trans = trans;
    c.src = src;
    c.src_ld = src_ld;
    c.perm = gather_perm;
    c.k = k;
    c.R = R;
    c.stride = stride;
    c.dim = dim;
    c.out = out;
    c.out_ld = out_ld;
    c.tiles = tiles;
    c.tbeg = tbeg;
    c.tend = tend;
    c.max_tiles = max_tiles;
    // tile mode: nrows is the number of rows the tiles cover (an upper bound
    // on the tile count); otherwise the plain row count
    c.rows_ub = tiles ? nrows : 0;
    c.nrows = tiles ? 0 : nrows;
    return c;
}

// The forward for one adapter, or for two adapter slots picked on the device
// by a snapshot of the slot control word (slots: R_*_alt is slot 1).
static pmoe_status forward_impl(pmoe_dims dims, const pmoe_weights *wts, const uint16_t *R_up,
                                const uint16_t *R_up_alt, const uint16_t *R_dn,
                                const uint16_t *R_dn_alt, int64_t su, int64_t sd,
                                const uint64_t *ctrl, uint32_t *version_out,
                                const pmoe_routing *rt, const void *X, int32_t chunk_C, int mode,
                                void *Y, void *ctx, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    const int C = std::min(chunk_C, dims.E);
    size_t need;
    FwdWs w = carve_fwd(ws, dims, C, mode, &need);
    if (!ws || ws_bytes < need || !aligned16(ws)) return PMOE_ERR_WORKSPACE;
    if (dims.T == 0) return PMOE_OK;

    const int d = dims.d, I = dims.inter, b = dims.block, k = dims.k;
    const int P = dims.T * k;
    const int fmt = wts->fmt;
    const uint64_t *sel = nullptr;
    if (ctrl) {   // every rotation of this forward reads one snapshot of the slot word
        launch_adapter_snapshot(ctrl, w.snap, version_out, stream);
        sel = w.snap;
    }
    // the saved context: g | u rows (FP32, [P, 2I]), then h and h~ rows (BF16,
    // [P, I] each)
    float *ctx_gu = (float *)ctx;
    uint16_t *h = ctx ? (uint16_t *)(ctx_gu + (int64_t)P * 2 * I) : w.h;
    uint16_t *ht = ctx ? h + (int64_t)P * I : w.ht;
    const int nch = nchunks_of(dims, C);
    const int maxrt = max_rot_tiles_of(dims);
    const Lists &L = w.l;
    build_lists(L, dims, C, rt, stream);
    // x~ = bf16(x R_up[e]) for every pair, gathered into expert-sorted order
    {
        RotCall c = rot_rows(b, false, X, d, rt->perm, k, R_up, su, d, w.xt, d, L.rtiles,
                             L.chunk_rtiles, L.chunk_rtiles + nch, maxrt, (int)P);
        c.R_alt = R_up_alt;
        c.sel = sel;
        launch_rotate_tc(c, stream);
    }

    GemmArgs gu{};
    gu.kind = GK_FWD_GU;
    gu.A = w.xt;
    gu.K = d;
    gu.Nout = I;
    gu.Nst = 2 * (int64_t)I;
    gu.Kst = d;
    gu.tiles = L.tiles;
    gu.chunk_tiles = L.chunk_tiles;
    gu.out = h;
    gu.ctxf = ctx_gu;
    gu.I = I;
    gu.nmat = dims.E;
    GemmArgs dn{};
    dn.kind = GK_FWD_DOWN;
    dn.A = R_dn ? ht : h;
    dn.K = I;
    dn.Nout = d;
    dn.Nst = d;
    dn.Kst = I;
    dn.tiles = L.tiles;
    dn.chunk_tiles = L.chunk_tiles;
    dn.outf = w.o;
    dn.I = I;
    dn.nmat = dims.E;
    pmoe_status gs;
    auto rot_down = [&](const int32_t *tb, const int32_t *te) {
        RotCall c = rot_rows(b, false, h, I, nullptr, k, R_dn, sd, I, ht, I, L.rtiles, tb, te,
                             maxrt, (int)P);
        c.R_alt = R_dn_alt;
        c.sel = sel;
        launch_rotate_tc(c, stream);
    };

    if (mode == PMOE_MODE_FUSED) {
        gu.fmt = dn.fmt = fmt;
        gu.wq = (const uint8_t *)wts->w13;
        gu.ws = (const uint8_t *)wts->s13;
        gu.wq_stride = wq_bytes(fmt, 2 * (int64_t)I, d);
        gu.ws_stride = ws_bytes_of(fmt, 2 * (int64_t)I, d);
        dn.wq = (const uint8_t *)wts->w2;
        dn.ws = (const uint8_t *)wts->s2;
        dn.wq_stride = wq_bytes(fmt, d, I);
        dn.ws_stride = ws_bytes_of(fmt, d, I);
        gu.c0 = dn.c0 = 0;
        gu.c1 = dn.c1 = nch;
        {
            ScopedTimer tm(PMOE_KT_GEMM_GATE_UP, stream);
            if ((gs = run_gemm(gu, P, w.err, stream)) != PMOE_OK) return gs;
        }
        if (R_dn) rot_down(L.chunk_rtiles, L.chunk_rtiles + nch);
        {
            ScopedTimer tm(PMOE_KT_GEMM_DOWN, stream);
            if ((gs = run_gemm(dn, P, w.err, stream)) != PMOE_OK) return gs;
        }
    } else {
        // the pages' literal scheme: dequantize the chunk's experts into the
        // bounded BF16 scratch, run the chunk's GEMMs, reuse the scratch
        const int64_t slot_bytes = 3 * (int64_t)I * d * 2;
        gu.fmt = dn.fmt = kFmtBF16;
        gu.wq = dn.wq = (const uint8_t *)w.scratch;
        gu.ws = dn.ws = nullptr;
        gu.wq_stride = dn.wq_stride = slot_bytes;
        gu.w_off_elems = 0;
        dn.w_off_elems = 2 * (int64_t)I * d;
        gu.slot_index = dn.slot_index = true;
        gu.nmat = dn.nmat = C;
        for (int c = 0; c < nch; ++c) {
            launch_dequant_chunk(fmt, d, I, C, c, rt->active, rt->num_active, wts->w13, wts->s13,
                                 wts->w2, wts->s2, w.scratch, stream);
            gu.c0 = dn.c0 = c;
            gu.c1 = dn.c1 = c + 1;
            {
                ScopedTimer tm(PMOE_KT_GEMM_GATE_UP, stream);
                if ((gs = run_gemm(gu, P, w.err, stream)) != PMOE_OK) return gs;
            }
            if (R_dn) rot_down(L.chunk_rtiles + c, L.chunk_rtiles + c + 1);
            {
                ScopedTimer tm(PMOE_KT_GEMM_DOWN, stream);
                if ((gs = run_gemm(dn, P, w.err, stream)) != PMOE_OK) return gs;
            }
        }
    }
    launch_combine(dims.T, d, k, w.o, rt->inv_perm, rt->w, (uint16_t *)Y, stream);
    return launched(stream);
}
}  // namespace pmoe

pmoe_status moe_chunked_forward(pmoe_dims dims, const pmoe_weights *wts, const pmoe_adapter *adp,
                                const pmoe_routing *rt, const void *X, int32_t chunk_C, int mode,
                                void *Y, void *ctx, void *ws, size_t ws_bytes,
                                cudaStream_t stream)
{
    using namespace pmoe;
    if (!dims_ok(dims) || !weights_ok(wts, dims) || !adapter_ok(adp) || !routing_ok(rt, dims))
        return PMOE_ERR_INVALID_ARG;
    if (chunk_C < 1 || (mode != PMOE_MODE_FUSED && mode != PMOE_MODE_SCRATCH))
        return PMOE_ERR_INVALID_ARG;
    if (dims.T > 0 && (!X || !Y)) return PMOE_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Y) || !aligned16(ctx)) return PMOE_ERR_INVALID_ARG;
    const uint16_t *R_up = adp ? (const uint16_t *)adp->R_up : nullptr;
    const uint16_t *R_dn = adp && R_up ? (const uint16_t *)adp->R_down : nullptr;
    const int64_t su = adp ? adp->stride_up : 0, sd = adp ? adp->stride_down : 0;
    return forward_impl(dims, wts, R_up, nullptr, R_dn, nullptr, su, sd, nullptr, nullptr, rt, X,
                        chunk_C, mode, Y, ctx, ws, ws_bytes, stream);
}

pmoe_status moe_adapter_publish(uint64_t *ctrl, uint32_t slot, uint32_t version,
                                cudaStream_t stream)
{
    using namespace pmoe;
    if (!ctrl || slot > 1 || ((uintptr_t)ctrl & 7)) return PMOE_ERR_INVALID_ARG;
    launch_adapter_publish(ctrl, slot, version, stream);
    return launched(stream);
}

pmoe_status moe_chunked_forward_slots(pmoe_dims dims, const pmoe_weights *wts,
                                      const pmoe_adapter_slots *slots, const pmoe_routing *rt,
                                      const void *X, int32_t chunk_C, int mode, void *Y, void *ctx,
                                      uint32_t *version_out, void *ws, size_t ws_bytes,
                                      cudaStream_t stream)
{
    using namespace pmoe;
    if (!dims_ok(dims) || !weights_ok(wts, dims) || !routing_ok(rt, dims) || !slots || !slots->ctrl)
        return PMOE_ERR_INVALID_ARG;
    if (!slots->R_up[0] || !slots->R_up[1] || ((uintptr_t)slots->ctrl & 7) ||
        (!slots->R_down[0]) != (!slots->R_down[1]))
        return PMOE_ERR_INVALID_ARG;
    for (int i = 0; i < 2; ++i)
        if (!aligned16(slots->R_up[i]) || !aligned16(slots->R_down[i])) return PMOE_ERR_INVALID_ARG;
    if (slots->stride_up < 0 || slots->stride_down < 0) return PMOE_ERR_INVALID_ARG;
    if (chunk_C < 1 || (mode != PMOE_MODE_FUSED && mode != PMOE_MODE_SCRATCH))
        return PMOE_ERR_INVALID_ARG;
    if (dims.T > 0 && (!X || !Y)) return PMOE_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Y) || !aligned16(ctx)) return PMOE_ERR_INVALID_ARG;
    return forward_impl(dims, wts, (const uint16_t *)slots->R_up[0], (const uint16_t *)slots->R_up[1],
                        (const uint16_t *)slots->R_down[0], (const uint16_t *)slots->R_down[1],
                        slots->stride_up, slots->stride_down, slots->ctrl, version_out, rt, X,
                        chunk_C, mode, Y, ctx, ws, ws_bytes, stream);
}

pmoe_status moe_backward_data(pmoe_dims dims, const pmoe_weights *wts, const pmoe_adapter *adp,
                              const pmoe_routing *rt, const void *X, const void *dY,
                              const void *ctx, int32_t chunk_C, void *dX, float *d_topk_w,
                              float *dR_up, float *dR_down, void *ws, size_t ws_bytes,
                              cudaStream_t stream)
{
    if (!dims_ok(dims) || !weights_ok(wts, dims) || !adapter_ok(adp) || !routing_ok(rt, dims))
        return PMOE_ERR_INVALID_ARG;
    if (chunk_C < 1) return PMOE_ERR_INVALID_ARG;
    const uint16_t *R_up = adp ? (const uint16_t *)adp->R_up : nullptr;
    const uint16_t *R_dn = adp && R_up ? (const uint16_t *)adp->R_down : nullptr;
    if ((R_up && !dR_up) || (R_dn && !dR_down)) return PMOE_ERR_INVALID_ARG;
    if (dims.T > 0 && (!X || !dY || !ctx || !dX)) return PMOE_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(dY) || !aligned16(ctx) || !aligned16(dX) ||
        !aligned16(d_topk_w) || !aligned16(dR_up) || !aligned16(dR_down))
        return PMOE_ERR_INVALID_ARG;
    const int C = std::min(chunk_C, dims.E);
    size_t need;
    BwdWs w = carve_bwd(ws, dims, C, &need);
    if (!ws || ws_bytes < need || !aligned16(ws)) return PMOE_ERR_WORKSPACE;

    const int d = dims.d, I = dims.inter, b = dims.block, k = dims.k, E = dims.E;
    const int P = dims.T * k;
    const int fmt = wts->fmt;
    const int64_t su = adp ? adp->stride_up : 0, sd = adp ? adp->stride_down : 0;
    const int nch = nchunks_of(dims, C);
    const int maxrt = max_rot_tiles_of(dims);
    const int nsets_up = su ? E : 1, nsets_dn = sd ? E : 1;

    if (dims.T == 0) {
        // empty batch: adapter gradients are zero
        if (R_up && cudaMemsetAsync(dR_up, 0, (size_t)nsets_up * d * b * sizeof(float), stream))
            return PMOE_ERR_CUDA;
        if (R_dn && cudaMemsetAsync(dR_down, 0, (size_t)nsets_dn * I * b * sizeof(float), stream))
            return PMOE_ERR_CUDA;
        return PMOE_OK;
    }
    const Lists &L = w.l;
    // the forward's saved context: g | u rows (FP32, [P, 2I]), then h and h~
    // rows (BF16, [P, I] each; h~ = h without an adapter's R_down)
    const float *ctx_gu = (const float *)ctx;
    const uint16_t *h = (const uint16_t *)(ctx_gu + (int64_t)P * 2 * I);
    const uint16_t *ht = R_dn ? h + (int64_t)P * I : h;
    const int32_t *rtb = L.chunk_rtiles, *rte = L.chunk_rtiles + nch;
    build_lists(L, dims, C, rt, stream);
    // dY rows per pair (expert-sorted)
    launch_gather_rows(P, d, k, (const uint16_t *)dY, rt->perm, rt->offsets + E, w.dyp, stream);
    pmoe_status gs;
    GemmArgs g{};
    g.kind = GK_BWD_G;
    g.fmt = fmt;
    g.wq = (const uint8_t *)wts->w2;
    g.ws = (const uint8_t *)wts->s2;
    g.wq_stride = wq_bytes(fmt, d, I);
    g.ws_stride = ws_bytes_of(fmt, d, I);
    g.Nst = d;
    g.Kst = I;
    g.A = w.dyp;
    g.K = d;
    g.Nout = I;
    g.tiles = L.tiles;
    g.chunk_tiles = L.chunk_tiles;
    g.c0 = 0;
    g.c1 = nch;
    g.outf = w.dht;   // dh~ = w G in FP32
    g.I = I;
    g.w = rt->w;
    g.perm = rt->perm;
    g.ht = ht;
    g.dtw_part = w.dtw_part;
    g.nmat = E;
    {
        ScopedTimer tm(PMOE_KT_GEMM_BWD_G, stream);
        if ((gs = run_gemm(g, P, w.err, stream)) != PMOE_OK) return gs;
    }
    if (d_topk_w) launch_dtw_reduce(P, I / 32, w.dtw_part, rt->inv_perm, d_topk_w, stream);
    // dh = dh~ R_down^T (FP32 dh~ split into two BF16 parts), then the SwiGLU
    // backward from the saved FP32 g, u into FP16 [dg | du]; and dR_down.
    // Per-expert adapters of block 64 do both in one pass over dh~.
    if (R_dn && sd && adapter_bwd_fused_ok(b)) {
        launch_adapter_bwd_tc(E, P, I, w.dht, h, I, false, rt->perm, k, R_dn, sd, rt->offsets, w.dgu,
                              true, ctx_gu, dR_down, stream);
    } else {
        RotCall c = rot_rows(b, true, w.dht, I, nullptr, k, R_dn, sd, I, w.dgu, 2 * (int64_t)I,
                             L.rtiles, rtb, rte, maxrt, (int)P);
        c.src_f32 = true;
        c.swiglu_bwd = true;
        c.ctxf = ctx_gu;
        launch_rotate_tc(c, stream);
        if (R_dn)
            launch_outer_tc(nsets_dn, P, I, b, h, I, false, rt->perm, k, w.dht, true, I,
                            sd ? rt->offsets : nullptr, dR_down, stream);
    }

    // dx~ = [dg | du] W13 on FP16 operands (dg, du to 11 significant bits)
    GemmArgs x{};
    x.kind = GK_BWD_DX_F16;
    x.fmt = fmt;
    x.wq = (const uint8_t *)wts->w13;
    x.ws = (const uint8_t *)wts->s13;
    x.wq_stride = wq_bytes(fmt, 2 * (int64_t)I, d);
    x.ws_stride = ws_bytes_of(fmt, 2 * (int64_t)I, d);
    x.Nst = 2 * (int64_t)I;
    x.Kst = d;
    x.A = w.dgu;
    x.K = 2 * I;
    x.Nout = d;
    x.tiles = L.tiles;
    x.chunk_tiles = L.chunk_tiles;
    x.c0 = 0;
    x.c1 = nch;
    x.outf = w.dxt;
    x.I = I;
    x.nmat = E;
    {
        ScopedTimer tm(PMOE_KT_GEMM_BWD_DX, stream);
        if ((gs = run_gemm(x, P, w.err, stream)) != PMOE_OK) return gs;
    }
    // dR_up and dx_pair = dx~ R_up^T (FP32; without an adapter the same pass
    // as the identity, so that R = I and no adapter agree bit for bit), then
    // the slot sum per token.  Per-expert adapters of block 64: one pass.
    if (R_up && su && adapter_bwd_fused_ok(b)) {
        launch_adapter_bwd_tc(E, P, d, w.dxt, (const uint16_t *)X, d, true, rt->perm, k, R_up, su,
                              rt->offsets, w.dxp, false, nullptr, dR_up, stream);
    } else {
        if (R_up)
            launch_outer_tc(nsets_up, P, d, b, (const uint16_t *)X, d, true, rt->perm, k, w.dxt, true, d,
                            su ? rt->offsets : nullptr, dR_up, stream);
        RotCall c = rot_rows(b, true, w.dxt, d, nullptr, k, R_up, su, d, w.dxp, d, L.rtiles, rtb, rte,
                             maxrt, (int)P);
        c.src_f32 = c.out_f32 = true;
        launch_rotate_tc(c, stream);
    }
    launch_combine(dims.T, d, k, w.dxp, rt->inv_perm, nullptr, (uint16_t *)dX, stream);
    return launched(stream);
}

pmoe_status moe_dequant(pmoe_wfmt fmt, const void *q, const void *s, int64_t N, int64_t K,
                        void *out, cudaStream_t stream)
{
    if (N < 0 || K <= 0) return PMOE_ERR_INVALID_ARG;
    if (fmt == PMOE_W_FP8_B128_F32) {
        if (N % 128 || K % 128) return PMOE_ERR_INVALID_ARG;
    } else if (fmt == PMOE_W_INT4_G32_BF16 || fmt == PMOE_W_MXFP4_G32_E8M0) {
        if (K % 32) return PMOE_ERR_INVALID_ARG;
    } else {
        return PMOE_ERR_INVALID_ARG;
    }
    if (N == 0) return PMOE_OK;
    if (!q || !s || !out || !aligned16(q) || !aligned16(s) || !aligned16(out))
        return PMOE_ERR_INVALID_ARG;
    launch_dequant(fmt, q, s, N, K, (uint16_t *)out, stream);
    return launched(stream);
}

struct GgWs {
    DevErr *err;
    Tile *tiles;
    int32_t *chunk_tiles, *chunk_rows, *counts, *active, *num_active;
};
static GgWs carve_gg(void *ws, int E, int rows, size_t *bytes)
{
    Carver c(ws);
    GgWs w;
    w.err = c.take<DevErr>(kHdrBytes / sizeof(DevErr));
    w.tiles = c.take<Tile>(cdiv(rows, 16) + E);
    w.chunk_tiles = c.take<int32_t>(4);
    w.chunk_rows = c.take<int32_t>(4);
    w.counts = c.take<int32_t>(E);
    w.active = c.take<int32_t>(E);
    w.num_active = c.take<int32_t>(1);
    if (bytes) *bytes = c.off;
    return w;
}

size_t moe_grouped_gemm_ws_bytes(int32_t E, int32_t rows)
{
    if (E <= 0 || rows < 0) return 0;
    size_t b;
    carve_gg(nullptr, E, rows, &b);
    return b;
}

pmoe_status moe_grouped_gemm(pmoe_wfmt fmt, const void *q, const void *s, int32_t E, int32_t N,
                             int32_t K, int trans, const void *A, const int32_t *offsets,
                             int32_t rows, void *out, void *ws, size_t ws_bytes,
                             cudaStream_t stream)
{
    if (E <= 0 || E > 4096 || N <= 0 || K <= 0 || N % 64 || K % 64 || rows < 0)
        return PMOE_ERR_INVALID_ARG;
    if (fmt != PMOE_W_INT4_G32_BF16 && fmt != PMOE_W_MXFP4_G32_E8M0 && fmt != PMOE_W_FP8_B128_F32)
        return PMOE_ERR_INVALID_ARG;
    if (fmt == PMOE_W_FP8_B128_F32 && (N % 128 || K % 128)) return PMOE_ERR_INVALID_ARG;
    if (trans != 0 && trans != 1) return PMOE_ERR_INVALID_ARG;
    if (!q || !s || !offsets || (rows > 0 && (!A || !out))) return PMOE_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(s) || !aligned16(A) || !aligned16(out))
        return PMOE_ERR_INVALID_ARG;
    size_t need;
    GgWs w = carve_gg(ws, E, rows, &need);
    if (!ws || ws_bytes < need || !aligned16(ws)) return PMOE_ERR_WORKSPACE;
    if (rows == 0) return PMOE_OK;
    launch_offsets_to_active(E, rows, offsets, w.counts, w.active, w.num_active, w.err, stream);
    launch_build_tiles(E, E, kGemmRows, kGemmAlign, w.counts, offsets, w.active, w.num_active,
                       w.tiles, w.chunk_tiles, w.chunk_rows, stream);
    GemmArgs g{};
    g.kind = trans ? GK_BWD_DX : GK_FWD_DOWN;
    g.fmt = fmt;
    g.wq = (const uint8_t *)q;
    g.ws = (const uint8_t *)s;
    g.wq_stride = wq_bytes(fmt, N, K);
    g.ws_stride = ws_bytes_of(fmt, N, K);
    g.Nst = N;
    g.Kst = K;
    g.A = (const uint16_t *)A;
    g.K = trans ? N : K;
    g.Nout = trans ? K : N;
    g.tiles = w.tiles;
    g.chunk_tiles = w.chunk_tiles;
    g.c0 = 0;
    g.c1 = 1;
    g.out = (uint16_t *)out;
    g.I = N;
    g.nmat = E;
    pmoe_status gs = run_gemm(g, rows, w.err, stream);
    if (gs != PMOE_OK) return gs;
    return launched(stream);
}

static bool block_ok(int b) { return b == 16 || b == 32 || b == 64 || b == 128; }

pmoe_status adapter_apply(int32_t rows, int32_t dim, int32_t b, const void *X, const void *R,
                          void *Xr, cudaStream_t stream)
{
    if (rows < 0 || dim <= 0 || !block_ok(b) || dim % b || dim % 8) return PMOE_ERR_INVALID_ARG;
    if (rows == 0) return PMOE_OK;
    if (!X || !R || !Xr || X == Xr || !aligned16(X) || !aligned16(R) || !aligned16(Xr))
        return PMOE_ERR_INVALID_ARG;
    launch_rotate_tc(rot_rows(b, false, X, dim, nullptr, 1, (const uint16_t *)R, 0, dim, Xr, dim,
                              nullptr, nullptr, nullptr, 0, rows),
                     stream);
    return launched(stream);
}

pmoe_status adapter_grad(int32_t rows, int32_t dim, int32_t b, const void *X, const void *dXr,
                         const void *R, void *dX, float *dR, cudaStream_t stream)
{
    if (rows < 0 || dim <= 0 || !block_ok(b) || dim % b || dim % 8) return PMOE_ERR_INVALID_ARG;
    if (!dR || (rows > 0 && (!X || !dXr || !R))) return PMOE_ERR_INVALID_ARG;
    if (dX && dX == dXr) return PMOE_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(dXr) || !aligned16(R) || !aligned16(dX) || !aligned16(dR))
        return PMOE_ERR_INVALID_ARG;
    if (dX && rows > 0)
        launch_rotate_tc(rot_rows(b, true, dXr, dim, nullptr, 1, (const uint16_t *)R, 0, dim, dX, dim,
                                  nullptr, nullptr, nullptr, 0, rows),
                         stream);
    launch_outer_tc(1, rows, dim, b, (const uint16_t *)X, dim, false, nullptr, 1, dXr, false, dim,
                    nullptr, dR, stream);
    return launched(stream);
}

// ------------------------------------------------------------------ dense linear
namespace pmoe {
struct DenseWs {
    GgWs g;
    int32_t *offsets;
    void *buf;   // x~ (forward, BF16) or dx~ (backward, FP32), [rows, K]
};
static DenseWs carve_dense(void *ws, int rows, int K, size_t *bytes)
{
    size_t gb;
    DenseWs w;
    w.g = carve_gg(ws, 1, rows, &gb);
    Carver c(ws);
    c.off = gb;
    w.offsets = c.take<int32_t>(2);
    w.buf = c.take<float>((int64_t)(rows > 0 ? rows : 1) * K);
    if (bytes) *bytes = c.off;
    return w;
}
static bool dense_shape_ok(pmoe_wfmt fmt, int N, int K, int b, int rows)
{
    if (N <= 0 || K <= 0 || N % 64 || K % 64 || rows < 0 || N > 65536 || K > 65536) return false;
    if (fmt != PMOE_W_INT4_G32_BF16 && fmt != PMOE_W_MXFP4_G32_E8M0 && fmt != PMOE_W_FP8_B128_F32)
        return false;
    if (fmt == PMOE_W_FP8_B128_F32 && (N % 128 || K % 128)) return false;
    return block_ok(b) && K % b == 0;
}
// One frozen [N, K] matrix as a single-expert grouped GEMM over rows 0..rows-1.
static pmoe_status dense_gemm(pmoe_wfmt fmt, const void *q, const void *s, int N, int K, bool trans,
                              const void *A, int rows, void *out, bool out_f32, DenseWs &w,
                              cudaStream_t st)
{
    launch_set_offsets(w.offsets, rows, st);
    launch_offsets_to_active(1, rows, w.offsets, w.g.counts, w.g.active, w.g.num_active, w.g.err, st);
    launch_build_tiles(1, 1, kGemmRows, kGemmAlign, w.g.counts, w.offsets, w.g.active,
                       w.g.num_active, w.g.tiles, w.g.chunk_tiles, w.g.chunk_rows, st);
    GemmArgs g{};
    g.kind = trans ? GK_BWD_DX : GK_FWD_DOWN;
    g.fmt = fmt;
    g.wq = (const uint8_t *)q;
    g.ws = (const uint8_t *)s;
    g.wq_stride = wq_bytes(fmt, N, K);
    g.ws_stride = ws_bytes_of(fmt, N, K);
    g.Nst = N;
    g.Kst = K;
    g.A = (const uint16_t *)A;
    g.K = trans ? N : K;
    g.Nout = trans ? K : N;
    g.tiles = w.g.tiles;
    g.chunk_tiles = w.g.chunk_tiles;
    g.c0 = 0;
    g.c1 = 1;
    if (out_f32) g.outf = (float *)out;
    else g.out = (uint16_t *)out;
    g.I = N;
    g.nmat = 1;
    return run_gemm(g, rows, w.g.err, st);
}
}  // namespace pmoe

size_t dense_linear_ws_bytes(int32_t rows, int32_t N, int32_t K)
{
    if (rows < 0 || N <= 0 || K <= 0) return 0;
    size_t b;
    pmoe::carve_dense(nullptr, rows, K, &b);
    return b;
}

pmoe_status dense_linear_forward(pmoe_wfmt fmt, const void *q, const void *s, int32_t N, int32_t K,
                                 int32_t block, const void *R, int32_t rows, const void *X, void *Y,
                                 void *ws, size_t ws_bytes, cudaStream_t stream)
{
    using namespace pmoe;
    if (!dense_shape_ok(fmt, N, K, block, rows)) return PMOE_ERR_INVALID_ARG;
    if (!q || !s || (rows > 0 && (!X || !Y))) return PMOE_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(s) || !aligned16(R) || !aligned16(X) || !aligned16(Y))
        return PMOE_ERR_INVALID_ARG;
    size_t need;
    DenseWs w = carve_dense(ws, rows, K, &need);
    if (!ws || ws_bytes < need || !aligned16(ws)) return PMOE_ERR_WORKSPACE;
    if (rows == 0) return PMOE_OK;
    const void *A = X;
    if (R) {   // x~ = bf16(x blockdiag(R))
        launch_rotate_tc(rot_rows(block, false, X, K, nullptr, 1, (const uint16_t *)R, 0, K, w.buf, K,
                                  nullptr, nullptr, nullptr, 0, rows),
                         stream);
        A = w.buf;
    }
    pmoe_status st = dense_gemm(fmt, q, s, N, K, false, A, rows, Y, false, w, stream);
    if (st != PMOE_OK) return st;
    return launched(stream);
}

pmoe_status dense_linear_backward(pmoe_wfmt fmt, const void *q, const void *s, int32_t N, int32_t K,
                                  int32_t block, const void *R, int32_t rows, const void *X,
                                  const void *dY, void *dX, float *dR, void *ws, size_t ws_bytes,
                                  cudaStream_t stream)
{
    using namespace pmoe;
    if (!dense_shape_ok(fmt, N, K, block, rows)) return PMOE_ERR_INVALID_ARG;
    if (!q || !s || (R && !dR) || (rows > 0 && (!dY || !dX || (R && !X)))) return PMOE_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(s) || !aligned16(R) || !aligned16(X) || !aligned16(dY) ||
        !aligned16(dX) || !aligned16(dR))
        return PMOE_ERR_INVALID_ARG;
    size_t need;
    DenseWs w = carve_dense(ws, rows, K, &need);
    if (!ws || ws_bytes < need || !aligned16(ws)) return PMOE_ERR_WORKSPACE;
    if (rows == 0) {
        if (R && cudaMemsetAsync(dR, 0, (size_t)K * block * sizeof(float), stream) != cudaSuccess)
            return PMOE_ERR_CUDA;
        return PMOE_OK;
    }
    // dx~ = dY W (contraction over the stored rows); with an adapter dx~ is
    // kept in FP32, then dX = bf16(dx~ R^T) and dR = sum x^T dx~ (dx~ split
    // into two BF16 parts for the MMAs)
    pmoe_status st = dense_gemm(fmt, q, s, N, K, true, dY, rows, R ? w.buf : dX, R != nullptr, w,
                                stream);
    if (st != PMOE_OK) return st;
    if (R) {
        launch_outer_tc(1, rows, K, block, (const uint16_t *)X, K, false, nullptr, 1, w.buf, true, K,
                        nullptr, dR, stream);
        RotCall c = rot_rows(block, true, w.buf, K, nullptr, 1, (const uint16_t *)R, 0, K, dX, K,
                             nullptr, nullptr, nullptr, 0, rows);
        c.src_f32 = true;
        launch_rotate_tc(c, stream);
    }
    return launched(stream);
}

pmoe_status adapter_cayley(int32_t nblk, int32_t b, const float *S, void *R_bf16, float *R_f32,
                           cudaStream_t stream)
{
    if (nblk < 0 || !cayley_block_ok(b)) return PMOE_ERR_INVALID_ARG;
    if (nblk == 0) return PMOE_OK;
    if (!S || (!R_bf16 && !R_f32)) return PMOE_ERR_INVALID_ARG;
    launch_cayley(nblk, b, S, (uint16_t *)R_bf16, R_f32, stream);
    return launched(stream);
}

pmoe_status adapter_cayley_grad(int32_t nblk, int32_t b, const float *S, const float *R_f32,
                                const float *dR, float *dS, cudaStream_t stream)
{
    if (nblk < 0 || !cayley_block_ok(b)) return PMOE_ERR_INVALID_ARG;
    if (nblk == 0) return PMOE_OK;
    if (!R_f32 || !dR || !dS) return PMOE_ERR_INVALID_ARG;
    launch_cayley_grad(nblk, b, S, R_f32, dR, dS, stream);
    return launched(stream);
}

}  // extern "C"
