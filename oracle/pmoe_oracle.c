/*
 * pmoe_oracle.c -- plain, slow CPU oracle for the active-expert-chunked
 * low-precision MoE layer with a block-diagonal orthogonal adapter.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the smoke check and the timed CPU
 * baseline of the benchmark do.  It shares no code, header, table or
 * constant with the CUDA path.
 *
 * Sources (pages on adapter-first RL with a frozen low-precision base):
 *  - "Orbit ... 技艺细节", Active-expert-chunked dequantization: router
 *    selects experts, selected experts are grouped into fixed-size batches,
 *    dequantized temporarily, run through a grouped GEMM, then released.
 *  - same section, bypass-base-weight-grad GEMM backward: the backward
 *    computes no gradient for the frozen base, only what flows to the
 *    inputs and to the adapter.
 *  - "Orbit：把万亿模型 RL 后训练改写成部署一致性问题", 机制拆解 (OFT):
 *    the BF16 adapter is a local orthogonal transform; 术语 (reference
 *    policy): disabling the adapter recovers the frozen base.
 *  - NeMo RL FP8 blog, Table 1: FP8 E4M3 weights with an FP32 scale per
 *    [128,128] block.
 *  - Orbit announcement (Kimi-K2.6 / DeepSeek V4 Flash sections): INT4 base and FP4 base
 *    with a BF16 adapter.
 *
 * Everything accumulates in double precision.  The BF16 rounding points are
 * the tensors the method itself stores in BF16: the rotated activations x~
 * (input of the gate/up projection), the SwiGLU output h and the rotated h~
 * (input of the down projection), the layer output Y and the input gradient
 * dX.  Every other quantity -- the projections g and u, each pair's expert
 * output o and all the backward intermediates (G, dh~, dh, dg, du, dx~, the
 * rotated dx of each pair) -- keeps the full precision of the sum that
 * produced it.  The rounding is a round-to-nearest-even conversion written
 * out below; the flag OR_NO_ROUND turns it off so that finite differences
 * can check the backward against the forward.
 *
 * Where the pages are silent the plainest reading is taken (layouts,
 * rotation side, tie-breaking); each is stated beside the code that uses it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_NO_ROUND 1

enum { OR_INT4 = 0, OR_MXFP4 = 1, OR_FP8 = 2 };

/* ------------------------------------------------------------------ */
/* BF16 <-> double                                                      */
/* ------------------------------------------------------------------ */

/* BF16 is the upper half of an IEEE binary32: 1 sign, 8 exponent and
 * 7 fraction bits.  Widening is exact. */
double or_bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest BF16 value, ties to even, keeping
 * subnormals (quantum 2^-133) and overflowing to infinity. */
uint16_t or_bf16_round(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80;
    int e;
    frexp(a, &e);                 /* a = m * 2^e, m in [0.5, 1) */
    int q = e - 8;                /* 8 significant bits */
    if (q < -133)
        q = -133;                 /* smallest BF16 subnormal step */
    double r = nearbyint(ldexp(a, -q));   /* default mode: nearest, ties even */
    double res = ldexp(r, q);
    if (res >= 0x1p128)
        return sign | 0x7F80;
    float f = (float)res;         /* exact: res has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

static double rbf(double v, int flags)
{
    return (flags & OR_NO_ROUND) ? v : or_bf16_to_double(or_bf16_round(v));
}

/* ------------------------------------------------------------------ */
/* Element decoders (format definitions, no tables)                    */
/* ------------------------------------------------------------------ */

/* INT4, symmetric: a nibble is a two's-complement integer in [-8, 7]. */
static double int4_value(unsigned n)
{
    return (double)((int)n - 16 * (n >= 8));
}

/* E2M1 (OCP MX FP4): sign bit 3, exponent bits 2..1 with bias 1,
 * mantissa bit 0; exponent 0 is subnormal (0.m * 2^0). */
static double e2m1_value(unsigned n)
{
    unsigned s = (n >> 3) & 1, ex = (n >> 1) & 3, m = n & 1;
    double mag = ex == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, (int)ex - 1);
    return s ? -mag : mag;
}

/* E8M0 (OCP MX scale): 2^(u-127); u = 255 encodes NaN. */
static double e8m0_value(unsigned u)
{
    return u == 255 ? NAN : ldexp(1.0, (int)u - 127);
}

/* E4M3 "FN" (OCP FP8): sign bit 7, exponent bits 6..3 with bias 7,
 * mantissa bits 2..0; exponent 0 is subnormal (0.m * 2^-6); no
 * infinities; S.1111.111 is NaN; largest finite value 448. */
double or_e4m3_value(unsigned c)
{
    unsigned s = (c >> 7) & 1, ex = (c >> 3) & 15, m = c & 7;
    double mag;
    if (ex == 15 && m == 7)
        mag = NAN;
    else if (ex == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, (int)ex - 7);
    return s ? -mag : mag;
}

/* ------------------------------------------------------------------ */
/* Weight dequantization (the temporary dequantization step)         */
/* ------------------------------------------------------------------ */
/*
 * A weight matrix is stored in the linear convention [N_out, K_in].
 *   INT4  : q  u8 [N, K/2], element 2i in the low nibble of byte i and
 *           2i+1 in the high nibble; s bf16 [N, K/32] (group of 32 along K).
 *           W = bf16(q * s).
 *   MXFP4 : q  u8 [N, K/2] of E2M1 nibbles (same packing); s u8 [N, K/32]
 *           of E8M0 exponents.  W = bf16(e2m1 * 2^(u-127)).
 *   FP8   : q  u8 [N, K] of E4M3 codes; s f32 [N/128, K/128].
 *           W = bf16(fp32(e4m3 * s)): one rounding to FP32, then RNE to BF16.
 * Returns the dequantized BF16 value of element (n, c) as a double.
 */
static double dequant_elem(int fmt, const uint8_t *q, const void *s,
                           int64_t K, int64_t n, int64_t c)
{
    if (fmt == OR_INT4) {
        uint8_t byte = q[n * (K / 2) + c / 2];
        unsigned nib = (c & 1) ? (byte >> 4) : (byte & 15);
        double sc = or_bf16_to_double(((const uint16_t *)s)[n * (K / 32) + c / 32]);
        return or_bf16_to_double(or_bf16_round(int4_value(nib) * sc));
    }
    if (fmt == OR_MXFP4) {
        uint8_t byte = q[n * (K / 2) + c / 2];
        unsigned nib = (c & 1) ? (byte >> 4) : (byte & 15);
        double sc = e8m0_value(((const uint8_t *)s)[n * (K / 32) + c / 32]);
        return or_bf16_to_double(or_bf16_round(e2m1_value(nib) * sc));
    }
    /* FP8 */
    {
        double v = or_e4m3_value(q[n * K + c]);
        float sc = ((const float *)s)[(n / 128) * (K / 128) + c / 128];
        float p = (float)(v * (double)sc);   /* exact product, one rounding */
        return or_bf16_to_double(or_bf16_round((double)p));
    }
}

/* Dequantize a whole [N, K] matrix to BF16 bits (used by the format pins
 * and as the expected value of the GPU's bounded-scratch dequant). */
void or_dequant(int fmt, const uint8_t *q, const void *s, int64_t N, int64_t K,
                uint16_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t c = 0; c < K; ++c)
            out[n * K + c] = or_bf16_round(dequant_elem(fmt, q, s, K, n, c));
}

/* Byte sizes of one expert's packed weights and scales (for pointer
 * arithmetic over the expert axis). */
static int64_t q_bytes(int fmt, int64_t N, int64_t K)
{
    return fmt == OR_FP8 ? N * K : N * K / 2;
}
static int64_t s_bytes(int fmt, int64_t N, int64_t K)
{
    if (fmt == OR_INT4) return N * (K / 32) * 2;
    if (fmt == OR_MXFP4) return N * (K / 32);
    return (N / 128) * (K / 128) * 4;
}

/* ------------------------------------------------------------------ */
/* Router (top-k over the experts, softmax over the selected)          */
/* ------------------------------------------------------------------ */
/*
 * Selection and weights from given FP32 logits (bias already added): the k
 * largest by (logit descending, expert id ascending) fill the slots in that
 * order; w[t, j] = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the k
 * selected, in double, rounded to FP32.  Only the tokens in `toks` (n_toks
 * of them; NULL: 0 .. n_toks-1) are handled, at their own rows.
 */
void or_topk(int E, int k, const float *logits, const int32_t *toks, int n_toks, int32_t *idx,
             float *w)
{
#pragma omp parallel for schedule(static)
    for (int it = 0; it < n_toks; ++it) {
        int t = toks ? toks[it] : it;
        const float *l = logits + (int64_t)t * E;
        /* k passes of "best remaining", ties to the lower id */
        char *taken = calloc((size_t)E, 1);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;
            }
            taken[best] = 1;
            idx[(int64_t)t * k + j] = best;
        }
        free(taken);
        double lmax = l[idx[(int64_t)t * k]], den = 0.0;
        for (int j = 0; j < k; ++j)
            den += exp((double)l[idx[(int64_t)t * k + j]] - lmax);
        for (int j = 0; j < k; ++j)
            w[(int64_t)t * k + j] = (float)(exp((double)l[idx[(int64_t)t * k + j]] - lmax) / den);
    }
}

/*
 * logits[t, e] = fp32( sum_c x[t,c] * Wr[c,e] + bias[e] ), the sum in
 * double, then or_topk.  Only the tokens in `toks` are computed; outputs
 * are written at the token's own row.
 */
void or_route(int T, int d, int E, int k, const uint16_t *X, const float *Wr,
              const float *bias, const int32_t *toks, int n_toks,
              float *logits, int32_t *idx, float *w)
{
    (void)T;
#pragma omp parallel for schedule(dynamic, 1)
    for (int it = 0; it < n_toks; ++it) {
        int t = toks ? toks[it] : it;
        float *l = logits + (int64_t)t * E;
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += or_bf16_to_double(X[(int64_t)t * d + c]) * (double)Wr[(int64_t)c * E + e];
            if (bias)
                acc += (double)bias[e];
            l[e] = (float)acc;
        }
    }
    or_topk(E, k, logits, toks, n_toks, idx, w);
}

/*
 * The router logits in one fixed FP32 summation order (the library's
 * canonical router mode, so that its logits can be compared bit for bit):
 * 32 partial sums, partial i = fmaf chain over the columns c = i, i + 32,
 * i + 64, ... in ascending order starting from 0; then the pairwise tree
 * s[i] = s[i] + s[i + h] for i < h, h = 16, 8, 4, 2, 1; the logit is
 * s[0] + bias[e] (one FP32 addition; no bias: s[0]).  d % 32 == 0.
 */
void or_route_canonical(int d, int E, const uint16_t *X, const float *Wr, const float *bias,
                        const int32_t *toks, int n_toks, float *logits)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int it = 0; it < n_toks; ++it) {
        int t = toks ? toks[it] : it;
        for (int e = 0; e < E; ++e) {
            float s[32];
            for (int i = 0; i < 32; ++i) {
                float acc = 0.0f;
                for (int c = i; c < d; c += 32) {
                    uint32_t u = (uint32_t)X[(int64_t)t * d + c] << 16;
                    float x;
                    memcpy(&x, &u, sizeof x);
                    acc = fmaf(x, Wr[(int64_t)c * E + e], acc);
                }
                s[i] = acc;
            }
            for (int h = 16; h >= 1; h >>= 1)
                for (int i = 0; i < h; ++i)
                    s[i] = s[i] + s[i + h];
            logits[(int64_t)t * E + e] = bias ? s[0] + bias[e] : s[0];
        }
    }
}

/* ------------------------------------------------------------------ */
/* Grouping of the (token, slot) pairs by expert                       */
/* ------------------------------------------------------------------ */
/*
 * pairs p = t*k + j, P = T*k.  counts[e] = number of pairs routed to e;
 * offsets = exclusive prefix sum of counts (offsets[E] = P); perm lists
 * the pair ids ordered by (expert, pair id) -- a stable sort by expert;
 * inv_perm[perm[i]] = i; active = experts with a nonzero count, ascending;
 * num_active = their number.
 */
void or_permute(int P, int E, const int32_t *idx, int32_t *counts, int32_t *offsets,
                int32_t *perm, int32_t *inv_perm, int32_t *active, int32_t *num_active)
{
    for (int e = 0; e < E; ++e)
        counts[e] = 0;
    for (int p = 0; p < P; ++p)
        counts[idx[p]]++;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    /* insertion sort by expert id: stable, obviously so (slow on purpose) */
    int32_t *order = malloc(sizeof(int32_t) * (size_t)(P > 0 ? P : 1));
    for (int p = 0; p < P; ++p) {
        int i = p;
        while (i > 0 && idx[order[i - 1]] > idx[p]) {
            order[i] = order[i - 1];
            --i;
        }
        order[i] = p;
    }
    for (int i = 0; i < P; ++i) {
        perm[i] = order[i];
        inv_perm[order[i]] = i;
    }
    free(order);
    int na = 0;
    for (int e = 0; e < E; ++e)
        if (counts[e] > 0)
            active[na++] = e;
    for (int i = na; i < E; ++i)
        active[i] = -1;
    *num_active = na;
}

/* ------------------------------------------------------------------ */
/* Block-diagonal orthogonal adapter                                   */
/* ------------------------------------------------------------------ */
/*
 * A row vector v of length dim is rotated block by block:
 *   (v R)[beta*b + c] = sum_r v[beta*b + r] * R[beta][r][c],
 * R stored as [dim/b][b][b] BF16, row-major within a block.  This is the
 * "local orthogonal transform" of the OFT adapter applied on the input
 * side of a projection (x~ = x blockdiag(R)).
 */
static double relem(const uint16_t *R, const double *R64, int64_t i)
{
    return R64 ? R64[i] : or_bf16_to_double(R[i]);
}

static void rotate_row64(const double *v, const uint16_t *R, const double *R64, int dim, int b,
                         double *out)
{
    for (int beta = 0; beta < dim / b; ++beta) {
        int64_t o = (int64_t)beta * b * b;
        for (int c = 0; c < b; ++c) {
            double acc = 0.0;
            for (int r = 0; r < b; ++r)
                acc += v[beta * b + r] * relem(R, R64, o + r * b + c);
            out[beta * b + c] = acc;
        }
    }
}

static void rotate_row(const double *v, const uint16_t *R, int dim, int b, double *out)
{
    rotate_row64(v, R, NULL, dim, b, out);
}

/* v R^T: the adjoint of rotate_row. */
static void rotate_row_t64(const double *v, const uint16_t *R, const double *R64, int dim, int b,
                           double *out)
{
    for (int beta = 0; beta < dim / b; ++beta) {
        int64_t o = (int64_t)beta * b * b;
        for (int r = 0; r < b; ++r) {
            double acc = 0.0;
            for (int c = 0; c < b; ++c)
                acc += v[beta * b + c] * relem(R, R64, o + r * b + c);
            out[beta * b + r] = acc;
        }
    }
}

static void rotate_row_t(const double *v, const uint16_t *R, int dim, int b, double *out)
{
    rotate_row_t64(v, R, NULL, dim, b, out);
}

/* Standalone adapter application: Xr[i] = bf16(X[i] blockdiag(R)). */
void or_adapter_apply(int rows, int dim, int b, const uint16_t *X, const uint16_t *R,
                      uint16_t *Xr)
{
#pragma omp parallel for schedule(static)
    for (int i = 0; i < rows; ++i) {
        double *v = malloc(sizeof(double) * (size_t)dim * 2);
        for (int c = 0; c < dim; ++c)
            v[c] = or_bf16_to_double(X[(int64_t)i * dim + c]);
        rotate_row(v, R, dim, b, v + dim);
        for (int c = 0; c < dim; ++c)
            Xr[(int64_t)i * dim + c] = or_bf16_round(v[dim + c]);
        free(v);
    }
}

/* Adapter backward: dX = dXr blockdiag(R)^T (bf16), and
 * dR[beta] = sum_i X_blk[i]^T dXr_blk[i] (double), rows in order. */
void or_adapter_grad(int rows, int dim, int b, const uint16_t *X, const uint16_t *dXr,
                     const uint16_t *R, uint16_t *dX, double *dR)
{
    int nblk = dim / b;
    if (dX) {
#pragma omp parallel for schedule(static)
        for (int i = 0; i < rows; ++i) {
            double *v = malloc(sizeof(double) * (size_t)dim * 2);
            for (int c = 0; c < dim; ++c)
                v[c] = or_bf16_to_double(dXr[(int64_t)i * dim + c]);
            rotate_row_t(v, R, dim, b, v + dim);
            for (int c = 0; c < dim; ++c)
                dX[(int64_t)i * dim + c] = or_bf16_round(v[dim + c]);
            free(v);
        }
    }
#pragma omp parallel for schedule(static)
    for (int beta = 0; beta < nblk; ++beta) {
        double *D = dR + (int64_t)beta * b * b;
        for (int r = 0; r < b * b; ++r)
            D[r] = 0.0;
        for (int i = 0; i < rows; ++i)
            for (int r = 0; r < b; ++r) {
                double xr = or_bf16_to_double(X[(int64_t)i * dim + beta * b + r]);
                for (int c = 0; c < b; ++c)
                    D[r * b + c] += xr * or_bf16_to_double(dXr[(int64_t)i * dim + beta * b + c]);
            }
    }
}

/* ------------------------------------------------------------------ */
/* Cayley parameterisation of each orthogonal block                    */
/* ------------------------------------------------------------------ */

/* Inverse of an n x n matrix by Gauss-Jordan elimination with partial
 * pivoting.  A is destroyed.  Returns 0 on success. */
static int gj_inverse(double *A, double *Ainv, int n)
{
    for (int i = 0; i < n * n; ++i)
        Ainv[i] = 0.0;
    for (int i = 0; i < n; ++i)
        Ainv[i * n + i] = 1.0;
    for (int col = 0; col < n; ++col) {
        int piv = col;
        for (int r = col + 1; r < n; ++r)
            if (fabs(A[r * n + col]) > fabs(A[piv * n + col]))
                piv = r;
        if (A[piv * n + col] == 0.0)
            return -1;
        if (piv != col)
            for (int c = 0; c < n; ++c) {
                double t = A[col * n + c]; A[col * n + c] = A[piv * n + c]; A[piv * n + c] = t;
                t = Ainv[col * n + c]; Ainv[col * n + c] = Ainv[piv * n + c]; Ainv[piv * n + c] = t;
            }
        double p = A[col * n + col];
        for (int c = 0; c < n; ++c) {
            A[col * n + c] /= p;
            Ainv[col * n + c] /= p;
        }
        for (int r = 0; r < n; ++r) {
            if (r == col) continue;
            double f = A[r * n + col];
            if (f == 0.0) continue;
            for (int c = 0; c < n; ++c) {
                A[r * n + c] -= f * A[col * n + c];
                Ainv[r * n + c] -= f * Ainv[col * n + c];
            }
        }
    }
    return 0;
}

/* R = (I + S)(I - S)^{-1} for each skew-symmetric b x b block S. */
int or_cayley(int nblk, int b, const double *S, double *R)
{
    int rc = 0;
#pragma omp parallel for schedule(static) reduction(| : rc)
    for (int blk = 0; blk < nblk; ++blk) {
        const double *Sb = S + (int64_t)blk * b * b;
        double *A = malloc(sizeof(double) * (size_t)b * b * 2);
        double *Ai = A + (int64_t)b * b;
        for (int i = 0; i < b; ++i)
            for (int j = 0; j < b; ++j)
                A[i * b + j] = (i == j ? 1.0 : 0.0) - Sb[i * b + j];
        rc |= gj_inverse(A, Ai, b);
        double *Rb = R + (int64_t)blk * b * b;
        for (int i = 0; i < b; ++i)
            for (int j = 0; j < b; ++j) {
                double acc = 0.0;
                for (int m = 0; m < b; ++m)
                    acc += ((i == m ? 1.0 : 0.0) + Sb[i * b + m]) * Ai[m * b + j];
                Rb[i * b + j] = acc;
            }
        free(A);
    }
    return rc;
}

/*
 * Gradient through the Cayley map.  With A = (I - S)^{-1} and R = (I+S)A,
 * a perturbation dS gives dR = (I + R) dS A, so the gradient with respect
 * to S as an unconstrained matrix is M = (I + R)^T G A^T (G = dL/dR).
 * S is skew, parameterised by its upper triangle (S_ji = -S_ij), so the
 * gradient is returned as the skew matrix M - M^T; its (i, j) entry for
 * i < j is the derivative with respect to S_ij.
 */
int or_cayley_grad(int nblk, int b, const double *S, const double *G, double *dS)
{
    int rc = 0;
#pragma omp parallel for schedule(static) reduction(| : rc)
    for (int blk = 0; blk < nblk; ++blk) {
        const double *Sb = S + (int64_t)blk * b * b;
        const double *Gb = G + (int64_t)blk * b * b;
        size_t bb = (size_t)b * b;
        double *A = malloc(sizeof(double) * bb * 5);
        double *Ai = A + bb, *R = A + 2 * bb, *T1 = A + 3 * bb, *M = A + 4 * bb;
        for (int i = 0; i < b; ++i)
            for (int j = 0; j < b; ++j)
                A[i * b + j] = (i == j ? 1.0 : 0.0) - Sb[i * b + j];
        rc |= gj_inverse(A, Ai, b);
        for (int i = 0; i < b; ++i)
            for (int j = 0; j < b; ++j) {
                double acc = 0.0;
                for (int m = 0; m < b; ++m)
                    acc += ((i == m ? 1.0 : 0.0) + Sb[i * b + m]) * Ai[m * b + j];
                R[i * b + j] = acc;
            }
        /* T1 = (I + R)^T G */
        for (int i = 0; i < b; ++i)
            for (int j = 0; j < b; ++j) {
                double acc = 0.0;
                for (int m = 0; m < b; ++m)
                    acc += ((m == i ? 1.0 : 0.0) + R[m * b + i]) * Gb[m * b + j];
                T1[i * b + j] = acc;
            }
        /* M = T1 A^T */
        for (int i = 0; i < b; ++i)
            for (int j = 0; j < b; ++j) {
                double acc = 0.0;
                for (int m = 0; m < b; ++m)
                    acc += T1[i * b + m] * Ai[j * b + m];
                M[i * b + j] = acc;
            }
        double *D = dS + (int64_t)blk * b * b;
        for (int i = 0; i < b; ++i)
            for (int j = 0; j < b; ++j)
                D[i * b + j] = M[i * b + j] - M[j * b + i];
        free(A);
    }
    return rc;
}

/* ------------------------------------------------------------------ */
/* The MoE layer                                                        */
/* ------------------------------------------------------------------ */

typedef struct {
    int T, d, E, k, I, b;
    int fmt;
    const uint8_t *w13; const void *s13;  /* [E][2I, d]: gate rows 0..I-1, up rows I..2I-1 */
    const uint8_t *w2;  const void *s2;   /* [E][d, I] */
    const uint16_t *R_up;   int64_t stride_up;    /* elements between experts; 0 = shared; NULL = off */
    const uint16_t *R_down; int64_t stride_down;
    /* optional double-precision copies of the rotation blocks, used in
     * place of R_up / R_down when non-NULL (finite-difference checks) */
    const double *R_up64, *R_down64;
} or_layer;

static const uint8_t *wq(const or_layer *L, int which, int e)
{
    int64_t N = which == 13 ? 2 * (int64_t)L->I : L->d, K = which == 13 ? L->d : L->I;
    return (which == 13 ? L->w13 : L->w2) + (int64_t)e * q_bytes(L->fmt, N, K);
}
static const void *ws(const or_layer *L, int which, int e)
{
    int64_t N = which == 13 ? 2 * (int64_t)L->I : L->d, K = which == 13 ? L->d : L->I;
    return (const uint8_t *)(which == 13 ? L->s13 : L->s2) + (int64_t)e * s_bytes(L->fmt, N, K);
}

/* Per-pair forward state kept for the backward. */
typedef struct {
    double *x, *xt, *g, *u, *h, *ht, *o;
    double *hp, *htp;   /* nullable: h and h~ before their BF16 rounding */
} pair_buf;

static double silu(double g) { return g / (1.0 + exp(-g)); }
static double sigm(double g) { return 1.0 / (1.0 + exp(-g)); }

/* One (token, expert) pair through the expert, straight from the
 * definition: x~ = bf16(x R_up); g, u = x~ W_gate^T, x~ W_up^T;
 * h = bf16(silu(g) u); h~ = bf16(h R_down); o = h~ W_down^T.  g, u and o
 * keep the precision of their sums. */
static void expert_forward(const or_layer *L, int e, const uint16_t *xrow, const double *xrow64,
                           int flags, pair_buf *pb)
{
    int d = L->d, I = L->I;
    for (int c = 0; c < d; ++c)
        pb->x[c] = xrow64 ? xrow64[c] : or_bf16_to_double(xrow[c]);
    if (L->R_up) {
        int64_t o = (int64_t)e * L->stride_up;
        rotate_row64(pb->x, L->R_up + o, L->R_up64 ? L->R_up64 + o : NULL, d, L->b, pb->xt);
        for (int c = 0; c < d; ++c)
            pb->xt[c] = rbf(pb->xt[c], flags);
    } else {
        memcpy(pb->xt, pb->x, sizeof(double) * (size_t)d);
    }
    const uint8_t *q13 = wq(L, 13, e);
    const void *s13 = ws(L, 13, e);
    for (int n = 0; n < I; ++n) {
        double g = 0.0, u = 0.0;
        for (int c = 0; c < d; ++c) {
            g += pb->xt[c] * dequant_elem(L->fmt, q13, s13, d, n, c);
            u += pb->xt[c] * dequant_elem(L->fmt, q13, s13, d, I + n, c);
        }
        pb->g[n] = g;
        pb->u[n] = u;
        if (pb->hp) pb->hp[n] = silu(g) * u;
        pb->h[n] = rbf(silu(g) * u, flags);
    }
    if (L->R_down) {
        int64_t o = (int64_t)e * L->stride_down;
        rotate_row64(pb->h, L->R_down + o, L->R_down64 ? L->R_down64 + o : NULL, I, L->b, pb->ht);
        if (pb->htp) memcpy(pb->htp, pb->ht, sizeof(double) * (size_t)I);
        for (int n = 0; n < I; ++n)
            pb->ht[n] = rbf(pb->ht[n], flags);
    } else {
        memcpy(pb->ht, pb->h, sizeof(double) * (size_t)I);
    }
    const uint8_t *q2 = wq(L, 2, e);
    const void *s2 = ws(L, 2, e);
    for (int c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int n = 0; n < I; ++n)
            acc += pb->ht[n] * dequant_elem(L->fmt, q2, s2, I, c, n);
        pb->o[c] = acc;
    }
}

static pair_buf pb_alloc(int d, int I)
{
    pair_buf pb;
    double *m = malloc(sizeof(double) * (size_t)(3 * d + 5 * I));
    pb.x = m; pb.xt = m + d; pb.o = m + 2 * d;
    pb.g = m + 3 * d; pb.u = pb.g + I; pb.h = pb.u + I; pb.ht = pb.h + I;
    pb.hp = pb.htp = NULL;
    return pb;
}

/*
 * The values each BF16 rounding decision of the down path is taken on, per
 * pair p = it*k + j of the listed tokens (it = position in toks): hx[p][n]
 * = silu(g) u before it is rounded to h, and hx[p][I + n] = (h R_down)
 * before it is rounded to h~ (h~ = h without an adapter).  Lets a test see
 * which decisions lie near a BF16 rounding midpoint.
 */
void or_pre_round(const or_layer *L, const uint16_t *X, const int32_t *idx, const int32_t *toks,
                  int n_toks, double *hx)
{
    int d = L->d, I = L->I, k = L->k;
    int64_t np = (int64_t)n_toks * k;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t p = 0; p < np; ++p) {
        int t = toks ? toks[p / k] : (int)(p / k);
        int e = idx[(int64_t)t * k + p % k];
        pair_buf pb = pb_alloc(d, I);
        pb.hp = hx + p * 2 * I;
        pb.htp = hx + p * 2 * I + I;
        expert_forward(L, e, X + (int64_t)t * d, NULL, 0, &pb);
        if (!L->R_down) memcpy(pb.htp, pb.hp, sizeof(double) * (size_t)I);
        free(pb.x);
    }
}

/*
 * Forward of the layer for the tokens in toks[0..n_toks): for every slot j
 * of token t with e = idx[t, j], run the pair through expert e and return
 * Y[t] = bf16(sum_j w[t, j] o_j) (slots summed in order).  No permutation
 * and no chunking: the per-token definition.  Y is written at the token's
 * row; o_out (nullable) receives o for each pair p = t*k + j as doubles.
 */
void or_forward(const or_layer *L, const uint16_t *X, const double *X64, const int32_t *idx,
                const float *w, const int32_t *toks, int n_toks, int flags, uint16_t *Y,
                double *Y64, double *o_out)
{
    int d = L->d, k = L->k;
    int64_t np = (int64_t)n_toks * k;
    double *o_all = malloc(sizeof(double) * (size_t)(np > 0 ? np * d : 1));
    /* every (token, slot) pair independently */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t p = 0; p < np; ++p) {
        int t = toks ? toks[p / k] : (int)(p / k);
        int e = idx[(int64_t)t * k + p % k];
        pair_buf pb = pb_alloc(d, L->I);
        expert_forward(L, e, X + (int64_t)t * d, X64 ? X64 + (int64_t)t * d : NULL, flags, &pb);
        memcpy(o_all + p * d, pb.o, sizeof(double) * (size_t)d);
        free(pb.x);
    }
    /* Y_t = sum over the slots in order of w_tj o_j */
#pragma omp parallel for schedule(static)
    for (int it = 0; it < n_toks; ++it) {
        int t = toks ? toks[it] : it;
        double *acc = calloc((size_t)d, sizeof(double));
        for (int j = 0; j < k; ++j) {
            const double *o = o_all + ((int64_t)it * k + j) * d;
            for (int c = 0; c < d; ++c)
                acc[c] += (double)w[(int64_t)t * k + j] * o[c];
            if (o_out)
                memcpy(o_out + ((int64_t)t * k + j) * d, o, sizeof(double) * (size_t)d);
        }
        for (int c = 0; c < d; ++c) {
            if (Y) Y[(int64_t)t * d + c] = or_bf16_round(acc[c]);
            if (Y64) Y64[(int64_t)t * d + c] = acc[c];
        }
        free(acc);
    }
    free(o_all);
}

/*
 * Backward-data of the layer (routing and w held fixed; no gradient for
 * the frozen base weights).  For each listed token t and slot j, e = idx,
 * with g and u the forward's unrounded projections:
 *   G = dY_t W_down                      d_topk_w[t,j] = G . h~
 *   dh~ = w_tj G                         dR_down[e] += h_blk^T dh~_blk
 *   dh = dh~ R_down^T
 *   dg = dh u sigma(g)(1 + g(1 - sigma(g)))     du = dh silu(g)
 *   dx~ = dg W_gate + du W_up            dR_up[e] += x_blk^T dx~_blk
 *   dx_pair = dx~ R_up^T                 dX_t = bf16(sum_j dx_pair)
 * The adapter gradients accumulate over the listed tokens only, in token
 * then slot order; when the adapter is shared (stride 0) everything
 * accumulates into block set 0.  dX, d_topk_w, dR_up, dR_down nullable.
 */
void or_backward(const or_layer *L, const uint16_t *X, const double *X64, const uint16_t *dY,
                 const int32_t *idx,
                 const float *w, const int32_t *toks, int n_toks, int flags,
                 uint16_t *dX, double *dX64, float *d_topk_w, double *dR_up, double *dR_down)
{
    int d = L->d, I = L->I, k = L->k, b = L->b;
    int64_t np = (int64_t)n_toks * k;
    /* per-pair state needed by the ordered adapter-gradient reduction */
    double *xs = malloc(sizeof(double) * (size_t)(np * d));
    double *dxts = malloc(sizeof(double) * (size_t)(np * d));
    double *hs = malloc(sizeof(double) * (size_t)(np * I));
    double *dhts = malloc(sizeof(double) * (size_t)(np * I));
    double *dxps = malloc(sizeof(double) * (size_t)(np > 0 ? np * d : 1));
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t p = 0; p < np; ++p) {
        int t = toks ? toks[p / k] : (int)(p / k);
        int j = (int)(p % k);
        pair_buf pb = pb_alloc(d, I);
        double *G = malloc(sizeof(double) * (size_t)(2 * I + 2 * d + 2 * I));
        double *dh = G + I, *dxt = dh + I, *dxp = dxt + d, *dg = dxp + d, *du = dg + I;
        {
            int e = idx[(int64_t)t * k + j];
            double wt = (double)w[(int64_t)t * k + j];
            expert_forward(L, e, X + (int64_t)t * d, X64 ? X64 + (int64_t)t * d : NULL, flags, &pb);
            const uint8_t *q2 = wq(L, 2, e);
            const void *s2 = ws(L, 2, e);
            for (int n = 0; n < I; ++n) {
                double a = 0.0;
                for (int c = 0; c < d; ++c)
                    a += or_bf16_to_double(dY[(int64_t)t * d + c]) * dequant_elem(L->fmt, q2, s2, I, c, n);
                G[n] = a;
            }
            double dw = 0.0;
            for (int n = 0; n < I; ++n)
                dw += G[n] * pb.ht[n];
            if (d_topk_w)
                d_topk_w[(int64_t)t * k + j] = (float)dw;
            double *dht = dhts + p * I;
            for (int n = 0; n < I; ++n)
                dht[n] = wt * G[n];
            memcpy(hs + p * I, pb.h, sizeof(double) * (size_t)I);
            if (L->R_down) {
                int64_t o = (int64_t)e * L->stride_down;
                rotate_row_t64(dht, L->R_down + o, L->R_down64 ? L->R_down64 + o : NULL, I, b, dh);
            } else {
                memcpy(dh, dht, sizeof(double) * (size_t)I);
            }
            for (int n = 0; n < I; ++n) {
                double g = pb.g[n], u = pb.u[n], sg = sigm(g);
                dg[n] = dh[n] * u * sg * (1.0 + g * (1.0 - sg));
                du[n] = dh[n] * silu(g);
            }
            const uint8_t *q13 = wq(L, 13, e);
            const void *s13 = ws(L, 13, e);
            for (int c = 0; c < d; ++c) {
                double a = 0.0;
                for (int n = 0; n < I; ++n)
                    a += dg[n] * dequant_elem(L->fmt, q13, s13, d, n, c)
                       + du[n] * dequant_elem(L->fmt, q13, s13, d, I + n, c);
                dxt[c] = a;
            }
            memcpy(dxts + p * d, dxt, sizeof(double) * (size_t)d);
            memcpy(xs + p * d, pb.x, sizeof(double) * (size_t)d);
            if (L->R_up) {
                int64_t o = (int64_t)e * L->stride_up;
                rotate_row_t64(dxt, L->R_up + o, L->R_up64 ? L->R_up64 + o : NULL, d, b, dxp);
            } else {
                memcpy(dxp, dxt, sizeof(double) * (size_t)d);
            }
            memcpy(dxps + p * d, dxp, sizeof(double) * (size_t)d);
        }
        free(G);
        free(pb.x);
    }
    /* dX_t = bf16(sum over the slots in order of dx_pair) */
#pragma omp parallel for schedule(static)
    for (int it = 0; it < n_toks; ++it) {
        int t = toks ? toks[it] : it;
        double *acc = calloc((size_t)d, sizeof(double));
        for (int j = 0; j < k; ++j)
            for (int c = 0; c < d; ++c)
                acc[c] += dxps[((int64_t)it * k + j) * d + c];
        for (int c = 0; c < d; ++c) {
            if (dX) dX[(int64_t)t * d + c] = or_bf16_round(acc[c]);
            if (dX64) dX64[(int64_t)t * d + c] = acc[c];
        }
        free(acc);
    }
    free(dxps);
    /* ordered reduction of the adapter gradients: one expert (block set)
     * per task, pairs in token-list then slot order */
    int nset_up = L->stride_up ? L->E : 1, nset_dn = L->stride_down ? L->E : 1;
    if (dR_up && L->R_up) {
        int nb = d / b;
        memset(dR_up, 0, sizeof(double) * (size_t)nset_up * nb * b * b);
#pragma omp parallel for schedule(dynamic, 1)
        for (int s = 0; s < nset_up; ++s)
            for (int64_t p = 0; p < np; ++p) {
                int t = toks ? toks[p / k] : (int)(p / k);
                int e = idx[(int64_t)t * k + p % k];
                if ((L->stride_up ? e : 0) != s) continue;
                double *D = dR_up + (int64_t)s * nb * b * b;
                for (int beta = 0; beta < nb; ++beta)
                    for (int r = 0; r < b; ++r) {
                        double xr = xs[p * d + beta * b + r];
                        for (int c = 0; c < b; ++c)
                            D[(int64_t)beta * b * b + r * b + c] += xr * dxts[p * d + beta * b + c];
                    }
            }
    }
    if (dR_down && L->R_down) {
        int nb = I / b;
        memset(dR_down, 0, sizeof(double) * (size_t)nset_dn * nb * b * b);
#pragma omp parallel for schedule(dynamic, 1)
        for (int s = 0; s < nset_dn; ++s)
            for (int64_t p = 0; p < np; ++p) {
                int t = toks ? toks[p / k] : (int)(p / k);
                int e = idx[(int64_t)t * k + p % k];
                if ((L->stride_down ? e : 0) != s) continue;
                double *D = dR_down + (int64_t)s * nb * b * b;
                for (int beta = 0; beta < nb; ++beta)
                    for (int r = 0; r < b; ++r) {
                        double hr = hs[p * I + beta * b + r];
                        for (int c = 0; c < b; ++c)
                            D[(int64_t)beta * b * b + r * b + c] += hr * dhts[p * I + beta * b + c];
                    }
            }
    }
    free(xs); free(dxts); free(hs); free(dhts);
}

/*
 * Dense bypass-base-weight-grad linear with the OFT adapter: one frozen
 * low-precision projection outside the experts ("Orbit ... 技艺细节": the
 * frozen base needs no weight gradient; "Orbit：把万亿模型 RL 后训练改写成部署
 * 一致性问题", 机制拆解: the adapter is a local orthogonal transform of the
 * activations).  W is [N, K] in the packed format fmt, R (nullable) is one
 * block-diagonal rotation [K/b, b, b] (BF16 bits, or doubles in R64).
 *   forward:  x~ = bf16(x R);  y = x~ W^T;  Y = bf16(y)
 *   backward: dx~ = dY W;  dR = sum_rows x_blk^T dx~_blk;  dX = bf16(dx~ R^T)
 *             (without R: dX = bf16(dY W))
 * Rounding points as in the layer: x~, Y and dX (OR_NO_ROUND removes them);
 * X64 replaces the BF16 input for finite differences.
 */
void or_dense_forward(int rows, int N, int K, int b, int fmt, const uint8_t *q, const void *s,
                      const uint16_t *R, const double *R64, const uint16_t *X, const double *X64,
                      int flags, uint16_t *Y, double *Y64)
{
#pragma omp parallel for schedule(static)
    for (int i = 0; i < rows; ++i) {
        double *x = malloc(sizeof(double) * (size_t)K * 2), *xt = x + K;
        for (int c = 0; c < K; ++c)
            x[c] = X64 ? X64[(int64_t)i * K + c] : or_bf16_to_double(X[(int64_t)i * K + c]);
        if (R || R64) {
            rotate_row64(x, R, R64, K, b, xt);
            for (int c = 0; c < K; ++c)
                xt[c] = rbf(xt[c], flags);
        } else {
            memcpy(xt, x, sizeof(double) * (size_t)K);
        }
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int c = 0; c < K; ++c)
                acc += xt[c] * dequant_elem(fmt, q, s, K, n, c);
            if (Y) Y[(int64_t)i * N + n] = or_bf16_round(acc);
            if (Y64) Y64[(int64_t)i * N + n] = acc;
        }
        free(x);
    }
}

void or_dense_backward(int rows, int N, int K, int b, int fmt, const uint8_t *q, const void *s,
                       const uint16_t *R, const double *R64, const uint16_t *X, const double *X64,
                       const uint16_t *dY, int flags, uint16_t *dX, double *dX64, double *dR)
{
    const int has_r = R || R64;
    double *dxts = malloc(sizeof(double) * (size_t)(rows > 0 ? rows : 1) * K);
#pragma omp parallel for schedule(static)
    for (int i = 0; i < rows; ++i) {
        double *dxt = dxts + (int64_t)i * K;
        double *dx = malloc(sizeof(double) * (size_t)K);
        for (int c = 0; c < K; ++c) {
            double a = 0.0;
            for (int n = 0; n < N; ++n)
                a += or_bf16_to_double(dY[(int64_t)i * N + n]) * dequant_elem(fmt, q, s, K, n, c);
            dxt[c] = a;
        }
        if (has_r)
            rotate_row_t64(dxt, R, R64, K, b, dx);
        else
            memcpy(dx, dxt, sizeof(double) * (size_t)K);
        for (int c = 0; c < K; ++c) {
            if (dX) dX[(int64_t)i * K + c] = or_bf16_round(dx[c]);
            if (dX64) dX64[(int64_t)i * K + c] = dx[c];
        }
        free(dx);
    }
    if (dR && has_r) {
        int nblk = K / b;
#pragma omp parallel for schedule(static)
        for (int beta = 0; beta < nblk; ++beta) {
            double *D = dR + (int64_t)beta * b * b;
            for (int r = 0; r < b * b; ++r)
                D[r] = 0.0;
            for (int i = 0; i < rows; ++i)
                for (int r = 0; r < b; ++r) {
                    int64_t o = (int64_t)i * K + (int64_t)beta * b;
                    double xr = X64 ? X64[o + r] : or_bf16_to_double(X[o + r]);
                    for (int c = 0; c < b; ++c)
                        D[r * b + c] += xr * dxts[o + c];
                }
        }
    }
    free(dxts);
}

/* Number of OpenMP threads the oracle runs with. */
int or_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
