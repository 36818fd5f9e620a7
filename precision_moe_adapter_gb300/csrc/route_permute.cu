// route_permute.cu -- router top-k and the grouping of (token, slot) pairs
// by expert (Orbit announcement, 技艺细节, active-expert-chunked dequantization: the
// router's selected experts are gathered into fixed-size batches).
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace pmoe {

// ------------------------------------------------------------------ exact logits
// The canonical router mode: FP32 logits on the CUDA cores in one fixed
// summation order, independent of the batch and of the launch shape.  For
// token t and expert e, lane i of the token's warp forms the partial
// fmaf chain over the columns c = i, i + 32, ... in ascending order; the 32
// partials are then added by the tree s[i] += s[i + h], h = 16, 8, 4, 2, 1
// (shuffles down).  A CTA takes 8 tokens (one warp each) and 32 experts,
// staging 64 rows of those experts' router weights at a time in shared
// memory (row pitch 33: lanes reading different rows hit different banks).
constexpr int kRxTok = 8, kRxE = 32, kRxRows = 64;

__global__ void __launch_bounds__(kRxTok * 32) k_router_exact(int T, int d, int E,
                                                               const uint16_t *__restrict__ X,
                                                               const float *__restrict__ Wr,
                                                               float *__restrict__ logits)
{
    __shared__ float ws[kRxRows][kRxE + 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kRxTok + warp, e0 = blockIdx.y * kRxE;
    float acc[kRxE];
#pragma unroll
    for (int e = 0; e < kRxE; ++e) acc[e] = 0.f;
    for (int c0 = 0; c0 < d; c0 += kRxRows) {
        __syncthreads();
        for (int i = threadIdx.x; i < kRxRows * kRxE; i += kRxTok * 32) {
            const int r = i / kRxE, e = i % kRxE;
            ws[r][e] = e0 + e < E ? Wr[(int64_t)(c0 + r) * E + e0 + e] : 0.f;
        }
        __syncthreads();
        if (t < T) {
#pragma unroll
            for (int q = 0; q < kRxRows / 32; ++q) {
                const int r = lane + 32 * q;   // column c0 + r: c = lane (mod 32), ascending
                const float x = bf2f(X[(int64_t)t * d + c0 + r]);
#pragma unroll
                for (int e = 0; e < kRxE; ++e) acc[e] = fmaf(x, ws[r][e], acc[e]);
            }
        }
    }
#pragma unroll
    for (int h = 16; h >= 1; h >>= 1)
#pragma unroll
        for (int e = 0; e < kRxE; ++e) acc[e] += __shfl_down_sync(0xffffffffu, acc[e], h);
    if (t < T && lane == 0) {
#pragma unroll
        for (int e = 0; e < kRxE; ++e)
            if (e0 + e < E) logits[(int64_t)t * E + e0 + e] = acc[e];
    }
}

void launch_router_exact(int T, int d, int E, const uint16_t *X, const float *Wr, float *logits,
                         cudaStream_t st)
{
    if (T <= 0) return;
    dim3 grid((unsigned)cdiv(T, kRxTok), (unsigned)cdiv(E, kRxE));
    k_router_exact<<<grid, kRxTok * 32, 0, st>>>(T, d, E, X, Wr, logits);
    note_launch();
}

// ------------------------------------------------------------------ top-k
// One warp per token.  Selection j picks the best element strictly after
// selection j-1 in the total order (logit descending, id ascending), so no
// "taken" marks are needed and ties go to the lower id.
__global__ void k_route_topk(int T, int E, int k, const float *__restrict__ logits,
                             const float *__restrict__ bias, int32_t *__restrict__ idx,
                             float *__restrict__ w, float *__restrict__ logits_out)
{
    int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= T) return;
    const float *l = logits + (int64_t)warp * E;
    if (bias || logits_out) {
        for (int e = lane; e < E; e += 32) {
            float v = l[e] + (bias ? bias[e] : 0.f);
            if (logits_out) logits_out[(int64_t)warp * E + e] = v;
        }
    }
    float pv = __int_as_float(0x7f800000);  // previous selection (+inf, id -1)
    int pe = -1;
    float sel_v[32];
    int sel_e[32];
#pragma unroll 1
    for (int j = 0; j < k; ++j) {
        float bv = -__int_as_float(0x7f800000);
        int be = 0x7fffffff;
        for (int e = lane; e < E; e += 32) {
            float v = l[e] + (bias ? bias[e] : 0.f);
            bool after = (v < pv) || (v == pv && e > pe);
            bool better = (v > bv) || (v == bv && e < be);
            if (after && better) { bv = v; be = e; }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
        }
        pv = bv;
        pe = be;
        if (j < 32) { sel_v[j] = bv; sel_e[j] = be; }
    }
    if (lane == 0) {
        float den = 0.f;
        for (int j = 0; j < k; ++j) den += expf(sel_v[j] - sel_v[0]);
        for (int j = 0; j < k; ++j) {
            idx[(int64_t)warp * k + j] = sel_e[j];
            w[(int64_t)warp * k + j] = expf(sel_v[j] - sel_v[0]) / den;
        }
    }
}

void launch_route_topk(int T, int E, int k, const float *logits, const float *bias, int32_t *idx,
                       float *w, float *logits_out, cudaStream_t st)
{
    if (T <= 0) return;
    int threads = 256, blocks = (int)cdiv((int64_t)T * 32, threads);
    k_route_topk<<<blocks, threads, 0, st>>>(T, E, k, logits, bias, idx, w, logits_out);
    note_launch();
}

// ------------------------------------------------------------------ grouping
// Pairs are processed in blocks of kPB.  Pass 1: per-block histogram.
// Pass 2 (one CTA): counts, exclusive-scan offsets, per-(block, expert)
// base positions, active list.  Pass 3: stable scatter; within a block the
// rank of a pair among same-expert pairs comes from a warp match plus a
// warp-ordered running counter in shared memory.
constexpr int kPB = 1024;

__global__ void k_hist(int P, int E, const int32_t *__restrict__ idx, int32_t *__restrict__ hist,
                       DevErr *err)
{
    extern __shared__ int32_t sh[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) sh[e] = 0;
    __syncthreads();
    int p = blockIdx.x * kPB + threadIdx.x;
    if (p < P) {
        int e = idx[p];
        if (e >= 0 && e < E) atomicAdd(&sh[e], 1);
        else record_error(err, PMOE_ERR_BAD_INDEX, p, e);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(int64_t)blockIdx.x * E + e] = sh[e];
}

// Block-wide exclusive scan of one int per thread (blockDim = 1024).
__device__ int block_excl_scan(int v, int *total)
{
    __shared__ int warp_sums[32];
    int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int s = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        warp_sums[lane] = s;
    }
    __syncthreads();
    int base = wid ? warp_sums[wid - 1] : 0;
    if (total) *total = warp_sums[31];
    __syncthreads();
    return base + x - v;
}

__global__ void __launch_bounds__(1024) k_scan(int nb, int E, int32_t *__restrict__ hist,
                                               int32_t *__restrict__ counts,
                                               int32_t *__restrict__ offsets,
                                               int32_t *__restrict__ active,
                                               int32_t *__restrict__ num_active)
{
    // each thread owns experts [t*per, t*per + per)
    int per = (E + 1023) / 1024;
    int e0 = threadIdx.x * per;
    int my_cnt = 0, my_act = 0;
    for (int i = 0; i < per; ++i) {
        int e = e0 + i;
        if (e >= E) break;
        int c = 0;
        for (int b = 0; b < nb; ++b) c += hist[(int64_t)b * E + e];
        counts[e] = c;
        my_cnt += c;
        my_act += c > 0;
    }
    int tot_cnt, tot_act;
    int off = block_excl_scan(my_cnt, &tot_cnt);
    int apos = block_excl_scan(my_act, &tot_act);
    for (int i = 0; i < per; ++i) {
        int e = e0 + i;
        if (e >= E) break;
        int c = counts[e];
        offsets[e] = off;
        int run = off;
        for (int b = 0; b < nb; ++b) {
            int h = hist[(int64_t)b * E + e];
            hist[(int64_t)b * E + e] = run;   // base position of (block b, expert e)
            run += h;
        }
        off += c;
        if (c > 0) active[apos++] = e;
    }
    if (threadIdx.x == 0) {
        offsets[E] = tot_cnt;
        *num_active = tot_act;
    }
    for (int e = tot_act + threadIdx.x; e < E; e += blockDim.x) active[e] = -1;
}

__global__ void __launch_bounds__(kPB) k_scatter(int P, int E, const int32_t *__restrict__ idx,
                                                 const int32_t *__restrict__ base,
                                                 int32_t *__restrict__ perm,
                                                 int32_t *__restrict__ inv_perm)
{
    extern __shared__ int32_t cnt[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = base[(int64_t)blockIdx.x * E + e];
    int p = blockIdx.x * kPB + threadIdx.x;
    int e = p < P ? idx[p] : -1;
    bool valid = e >= 0 && e < E;
    int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    unsigned mask = __match_any_sync(0xffffffffu, valid ? e : -1);
    int rank = __popc(mask & ((1u << lane) - 1u));
    int leader = __ffs(mask) - 1;
    int pos = 0;
    for (int w = 0; w < kPB / 32; ++w) {
        __syncthreads();
        if (wid == w) {
            int old = 0;
            if (lane == leader && valid) {
                old = cnt[e];
                cnt[e] = old + __popc(mask);
            }
            old = __shfl_sync(0xffffffffu, old, leader);
            pos = old + rank;
        }
    }
    if (valid) {
        perm[pos] = p;
        inv_perm[p] = pos;
    } else if (p < P) {
        inv_perm[p] = -1;
    }
}

size_t permute_ws_bytes(int P, int E)
{
    int nb = (int)cdiv(P > 0 ? P : 1, kPB);
    return (size_t)nb * E * sizeof(int32_t);
}

void launch_permute(int P, int E, const int32_t *idx, int32_t *counts, int32_t *offsets,
                    int32_t *perm, int32_t *inv_perm, int32_t *active, int32_t *num_active,
                    int32_t *hist, DevErr *err, cudaStream_t st)
{
    int nb = (int)cdiv(P, kPB);
    size_t sm = (size_t)E * sizeof(int32_t);
    if (nb > 0) {
        k_hist<<<nb, kPB, sm, st>>>(P, E, idx, hist, err);
        note_launch();
    }
    k_scan<<<1, 1024, 0, st>>>(nb, E, hist, counts, offsets, active, num_active);
    note_launch();
    if (nb > 0) {
        k_scatter<<<nb, kPB, sm, st>>>(P, E, idx, hist, perm, inv_perm);
        note_launch();
    }
}

// ------------------------------------------------------------------ tiles
// Work list: for the active experts in ascending order, chunk c = active
// positions [c*C, c*C + C), each expert's rows cut into ceil(n / max_rows)
// tiles of near-equal size (multiples of `align` rows, last one ragged).
// Also writes chunk_tiles[c] (first tile of chunk c, nchunks + 1 entries)
// and chunk_rows[c] = first expert-sorted row of chunk c (nchunks + 1).
__global__ void __launch_bounds__(1024) k_build_tiles(int E, int C, int max_rows, int align,
                                                      const int32_t *__restrict__ counts,
                                                      const int32_t *__restrict__ offsets,
                                                      const int32_t *__restrict__ active,
                                                      const int32_t *__restrict__ num_active,
                                                      Tile *__restrict__ tiles,
                                                      int32_t *__restrict__ chunk_tiles,
                                                      int32_t *__restrict__ chunk_rows)
{
    int na = *num_active;
    int nchunks_max = (E + C - 1) / C;
    int per = (E + 1023) / 1024;
    int a0 = threadIdx.x * per;
    int my = 0;
    for (int i = 0; i < per; ++i) {
        int a = a0 + i;
        if (a >= na) break;
        int n = counts[active[a]];
        my += (n + max_rows - 1) / max_rows;
    }
    int total;
    int t = block_excl_scan(my, &total);
    for (int i = 0; i < per; ++i) {
        int a = a0 + i;
        if (a >= na) break;
        int e = active[a];
        int n = counts[e];
        int nt = (n + max_rows - 1) / max_rows;
        int sz = (n + nt - 1) / nt;
        sz = (sz + align - 1) / align * align;
        int chunk = a / C, slot = a % C;
        if (slot == 0) {
            chunk_tiles[chunk] = t;
            chunk_rows[chunk] = offsets[e];
        }
        for (int j = 0; j < nt; ++j) {
            int r0 = j * sz;
            Tile tl;
            tl.expert = e;
            tl.row0 = offsets[e] + r0;
            tl.nrows = min(sz, n - r0);
            tl.chunk = (chunk << 16) | slot;
            tiles[t++] = tl;
        }
    }
    __syncthreads();
    // chunks past the active experts are empty
    int nch = (na + C - 1) / C;
    for (int c = nch + threadIdx.x; c <= nchunks_max; c += blockDim.x) {
        chunk_tiles[c] = total;
        chunk_rows[c] = offsets[E];
    }
}

void launch_build_tiles(int E, int C, int max_rows, int align, const int32_t *counts,
                        const int32_t *offsets, const int32_t *active, const int32_t *num_active,
                        Tile *tiles, int32_t *chunk_tiles, int32_t *chunk_rows, cudaStream_t st)
{
    k_build_tiles<<<1, 1024, 0, st>>>(E, C, max_rows, align, counts, offsets, active, num_active,
                                      tiles, chunk_tiles, chunk_rows);
    note_launch();
}

// counts[e] = offsets[e+1] - offsets[e]; active = experts with rows, ascending.
// Offsets that are not a nondecreasing 0..rows sequence record
// PMOE_ERR_BAD_INDEX and leave every expert empty (nothing is read).
__global__ void __launch_bounds__(1024) k_offsets_to_active(int E, int rows,
                                                            const int32_t *__restrict__ offsets,
                                                            int32_t *__restrict__ counts,
                                                            int32_t *__restrict__ active,
                                                            int32_t *__restrict__ num_active,
                                                            DevErr *err)
{
    __shared__ int bad;
    if (threadIdx.x == 0) bad = (offsets[0] != 0 || offsets[E] != rows);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        if (offsets[e + 1] < offsets[e]) bad = 1;
    __syncthreads();
    if (bad && threadIdx.x == 0) record_error(err, PMOE_ERR_BAD_INDEX, -1, -1);
    int per = (E + 1023) / 1024;
    int e0 = threadIdx.x * per;
    int my = 0;
    for (int i = 0; i < per; ++i) {
        int e = e0 + i;
        if (e >= E) break;
        int c = bad ? 0 : offsets[e + 1] - offsets[e];
        counts[e] = c;
        my += c > 0;
    }
    int tot;
    int pos = block_excl_scan(my, &tot);
    for (int i = 0; i < per; ++i) {
        int e = e0 + i;
        if (e >= E) break;
        if (counts[e] > 0) active[pos++] = e;
    }
    if (threadIdx.x == 0) *num_active = tot;
    for (int e = tot + threadIdx.x; e < E; e += blockDim.x) active[e] = -1;
}

void launch_offsets_to_active(int E, int rows, const int32_t *offsets, int32_t *counts,
                              int32_t *active, int32_t *num_active, DevErr *err, cudaStream_t st)
{
    k_offsets_to_active<<<1, 1024, 0, st>>>(E, rows, offsets, counts, active, num_active, err);
    note_launch();
}

// ------------------------------------------------------------------ router logits
// On the tensor cores: Wr = hi + mid + lo exactly, with hi = bf16(Wr),
// mid = bf16(Wr - hi), lo = bf16(Wr - hi - mid) (each difference is exact in
// FP32, and the three terms hold all 24 bits of the FP32 value).  The
// logits X Wr = [X | X | X] [hi; mid; lo] are then one BF16 contraction of
// length 3d whose products are exact and whose sums are FP32.
// The split terms are stored split-major: K split s of the length-3d row of
// expert e is row e of matrix s, [splits][E][3d / splits].
__global__ void __launch_bounds__(256) k_router_split(int d, int E, int splits, const float *__restrict__ Wr,
                                                      uint16_t *__restrict__ WrS)
{
    __shared__ float t[32][33];
    const int c0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int ks = 3 * d / splits;
    for (int i = ty; i < 32; i += 8) {
        const int c = c0 + i, e = e0 + tx;
        t[i][tx] = (c < d && e < E) ? Wr[(int64_t)c * E + e] : 0.f;
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
        const int e = e0 + i, c = c0 + tx;
        if (e >= E || c >= d) continue;
        const float w = t[tx][i];
        const uint16_t hi = f2bf(w);
        const float r1 = w - bf2f(hi);
        const uint16_t mid = f2bf(r1);
        const uint16_t lo = f2bf(r1 - bf2f(mid));
        const uint16_t term[3] = {hi, mid, lo};
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            const int kk = q * d + c;   // column of the length-3d row
            WrS[((int64_t)(kk / ks) * E + e) * ks + kk % ks] = term[q];
        }
    }
}
// token tiles of every K split: tile i is split i / n, token rows (i % n) * rows ..
__global__ void k_router_tiles(int T, int rows, int splits, Tile *__restrict__ tiles,
                               int32_t *__restrict__ chunk_tiles)
{
    const int n = (T + rows - 1) / rows;
    for (int i = threadIdx.x; i < n * splits; i += blockDim.x) {
        Tile tl;
        tl.expert = i / n;
        tl.row0 = (i % n) * rows;
        tl.nrows = min(rows, T - (i % n) * rows);
        tl.chunk = 0;
        tiles[i] = tl;
    }
    if (threadIdx.x == 0) {
        chunk_tiles[0] = 0;
        chunk_tiles[1] = n * splits;
    }
}
// logits = the splits' partials summed in split order
__global__ void __launch_bounds__(256) k_router_reduce(int64_t n, int splits, const float *__restrict__ part,
                                                       float *__restrict__ logits)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        float s = part[i];
        for (int q = 1; q < splits; ++q) s += part[q * n + i];
        logits[i] = s;
    }
}
int router_splits(int d)
{
    const int steps = d / 64;   // K steps of one term
    return 3 * (steps % 4 == 0 ? 4 : steps % 2 == 0 ? 2 : 1);
}
// Token rows per tile: enough work items to give every SM one (feature
// tiles of 128 experts times the K splits), multiples of 16, at most 256.
int router_tile_rows(int T, int E, int splits, int num_sms)
{
    const int64_t nft = cdiv(E, 128);
    int64_t r = cdiv((int64_t)T * nft * splits, num_sms > 0 ? num_sms : 1);
    r = (r + 15) & ~(int64_t)15;
    return (int)std::min<int64_t>(192, std::max<int64_t>(16, r));   // at most the GEMM tile width
}
void launch_router_reduce(int T, int E, int splits, const float *part, float *logits, cudaStream_t st)
{
    const int64_t n = (int64_t)T * E;
    if (n <= 0) return;
    const int grid = (int)std::min<int64_t>(cdiv(n, 256), 152 * 8);
    k_router_reduce<<<grid, 256, 0, st>>>(n, splits, part, logits);
    note_launch();
}
void launch_router_prep(int T, int d, int E, const float *Wr, uint16_t *WrS, Tile *tiles,
                        int32_t *chunk_tiles, int tile_rows, cudaStream_t st)
{
    const int splits = router_splits(d);
    dim3 grid((unsigned)cdiv(d, 32), (unsigned)cdiv(E, 32));
    k_router_split<<<grid, 256, 0, st>>>(d, E, splits, Wr, WrS);
    note_launch();
    k_router_tiles<<<1, 256, 0, st>>>(T, tile_rows, splits, tiles, chunk_tiles);
    note_launch();
}
}  // namespace pmoe
