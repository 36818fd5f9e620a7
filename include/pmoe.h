/*
 * pmoe.h -- C ABI of libpmoe.so: the active-expert-chunked low-precision
 * MoE layer with a block-diagonal orthogonal (OFT-style) adapter, for one
 * GB300 (sm_103a).
 *
 * The operation follows the "Active-expert-chunked dequantization" and
 * "bypass-base-weight-grad GEMM backward" passages of the Orbit
 * announcement (section 技艺细节), the OFT adapter of the Orbit analysis
 * "Orbit：把万亿模型 RL 后训练改写成部署一致性问题" (sections 机制拆解 and
 * 术语和概念边界), and the block-scaled FP8 weight format of the NeMo RL FP8
 * article (section "RL 中线性层的 FP8", Table 1).
 *
 * Conventions for every entry point:
 *  - Ownership: the caller allocates every buffer.  The library never
 *    allocates device or pinned memory; scratch lives in the caller's
 *    workspace (see moe_workspace_bytes).
 *  - Pointers are DEVICE pointers unless stated otherwise; they must be
 *    16-byte aligned.  Matrices are row-major and dense.
 *  - Ordering: every call is asynchronous on `stream` (no host sync) except
 *    moe_query_status, which synchronizes the stream.
 *  - Errors: argument checks run on the host before anything is launched
 *    and return PMOE_ERR_INVALID_ARG / PMOE_ERR_UNSUPPORTED /
 *    PMOE_ERR_WORKSPACE with nothing enqueued.  A launch failure returns
 *    PMOE_ERR_CUDA.  Errors found on the device (an expert id out of range,
 *    a bounded wait that ran out) are recorded in the error word at the
 *    start of the workspace and read back by moe_query_status; the kernels
 *    never trap.
 *  - Threading: the library holds no state between calls; calls with
 *    distinct workspaces may run concurrently.
 *  - Numerics: inputs must be finite.  BF16 values are raw uint16 bit
 *    patterns (IEEE binary32 upper half).
 *
 * Notation: T tokens, d hidden size, E experts, k experts per token,
 * I = inter (expert hidden size), b adapter block size, P = T*k pairs,
 * a pair p = t*k + j is token t in slot j.
 */
#ifndef PMOE_H
#define PMOE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PMOE_OK = 0,
    PMOE_ERR_INVALID_ARG = 1,   /* bad shape, NULL pointer, misalignment */
    PMOE_ERR_UNSUPPORTED = 2,   /* valid request this build does not handle */
    PMOE_ERR_WORKSPACE = 3,     /* workspace missing or smaller than moe_workspace_bytes */
    PMOE_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    PMOE_ERR_BAD_INDEX = 5,     /* device: an expert id outside [0, E) */
    PMOE_ERR_TIMEOUT = 6        /* device: a bounded wait gave up */
} pmoe_status;

/* Frozen-base weight formats (the INT4 and FP4 bases of the Orbit
 * announcement; FP8 E4M3 with [128,128] FP32 block scales, NeMo RL FP8
 * article, Table 1).  Every weight matrix
 * is stored in the linear convention [N_out, K_in]:
 *   INT4  : q u8 [N, K/2] (element 2i = low nibble of byte i, two's
 *           complement in [-8, 7]); s bf16 [N, K/32].  W = bf16(q*s).
 *   MXFP4 : q u8 [N, K/2] of E2M1 nibbles (same packing); s u8 [N, K/32]
 *           of E8M0 exponents.  W = bf16(e2m1 * 2^(s-127)).
 *   FP8   : q u8 [N, K] of E4M3 codes; s f32 [N/128, K/128].
 *           W = bf16(fp32(e4m3 * s)). */
typedef enum {
    PMOE_W_INT4_G32_BF16 = 0,
    PMOE_W_MXFP4_G32_E8M0 = 1,
    PMOE_W_FP8_B128_F32 = 2
} pmoe_wfmt;

/* Layer shape.  Requirements: d % 64 == 0, inter % 64 == 0, d <= 8192,
 * inter <= 8192, d % block == 0, inter % block == 0, block in
 * {16, 32, 64, 128}, 1 <= k <= min(E, 32), E <= 4096, T >= 0; FP8
 * additionally needs d % 128 == 0 and inter % 128 == 0. */
typedef struct {
    int32_t T, d, E, k, inter, block;
} pmoe_dims;

/* The frozen experts.  w13 holds, per expert, the gate rows 0..I-1 then the
 * up rows I..2I-1 of the [2I, d] gate/up projection; w2 holds the [d, I]
 * down projection.  Experts are consecutive along the leading axis. */
typedef struct {
    pmoe_wfmt fmt;
    const void *w13, *s13;
    const void *w2, *s2;
} pmoe_weights;

/* The orthogonal adapter: per expert, R_up [d/b, b, b] rotates the input of
 * the gate/up projection (x~ = x blockdiag(R_up)) and R_down [I/b, b, b]
 * the input of the down projection (h~ = h blockdiag(R_down)), BF16.
 * stride_* = elements between consecutive experts' block sets; 0 means one
 * set shared by all experts.  R_up == NULL disables the whole adapter (the
 * reference policy: the frozen base alone); R_down may be NULL alone. */
typedef struct {
    const void *R_up, *R_down;
    int64_t stride_up, stride_down;
} pmoe_adapter;

/* Routing and its grouping by expert (all device int32 / float):
 * idx [T,k], w [T,k], counts [E], offsets [E+1], perm [P] (pair id at each
 * expert-sorted position), inv_perm [P], active [E] (active experts
 * ascending, -1 padded), num_active [1]. */
typedef struct {
    int32_t *idx;
    float *w;
    int32_t *counts, *offsets, *perm, *inv_perm, *active, *num_active;
} pmoe_routing;

/* Forward modes. */
enum {
    PMOE_MODE_FUSED = 0,   /* dequantize tile by tile in shared memory inside the GEMM */
    PMOE_MODE_SCRATCH = 1  /* dequantize C experts into a global BF16 scratch, GEMM, reuse */
};

/* Router modes. */
enum {
    PMOE_ROUTE_FAST = 0,   /* FP32 logits from an exact 3-term BF16 split of Wr on tensor cores */
    PMOE_ROUTE_EXACT = 1   /* FP32 logits on the CUDA cores in one fixed summation order */
};

/* Ops for moe_workspace_bytes. */
enum { PMOE_OP_PERMUTE = 0, PMOE_OP_FORWARD = 1, PMOE_OP_BACKWARD = 2 };

/*
 * moe_route -- router top-k (Orbit announcement, 技艺细节: the experts the
 * router selects).
 * logits = fp32(X Wr) + bias; the k experts with the largest logits are
 * selected (ties to the lower expert id), slots in descending logit order;
 * w = softmax over the k selected logits (FP32).
 *   X      bf16 [T, d]          Wr  f32 [d, E]       bias f32 [E] or NULL
 *   logits f32 [T, E] or NULL (written when given)
 *   idx    int32 [T, k] (out)   w   f32 [T, k] (out)
 *   ws     workspace of moe_workspace_bytes(dims, PMOE_OP_PERMUTE, 0, 0)
 *          bytes or more (holds the split router weights and the error word)
 * Requires E <= 4096 and k <= 32.
 * Modes (the logits before the bias; the bias is then one FP32 addition):
 *   PMOE_ROUTE_FAST  the tensor-core contraction in fixed K splits whose
 *                    FP32 partials are summed in order: within the FP32
 *                    summation error of the exact logits, and per token
 *                    independent of the batch.
 *   PMOE_ROUTE_EXACT the canonical order, reproducible bit for bit by a
 *                    plain CPU program: 32 partial sums, partial i the
 *                    fmaf chain over columns i, i+32, i+64, ... from 0;
 *                    then s[i] = s[i] + s[i+h] for i < h, h = 16, 8, 4, 2,
 *                    1; the logit is s[0] (+ bias).  Slower (CUDA cores).
 * The selection and the softmax are the same for both: the order (logit
 * descending, id ascending) over the FP32 logits, and w_j = exp(l_j - l_0)
 * / sum_i exp(l_i - l_0) in FP32.
 */
pmoe_status moe_route(pmoe_dims dims, const void *X, const float *Wr, const float *bias,
                      float *logits, int32_t *idx, float *w, int mode,
                      void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * moe_permute -- groups the (token, slot) pairs by expert (Orbit
 * announcement, 技艺细节:
 * the selected experts are gathered into batches): histogram of idx,
 * exclusive-scan offsets and a stable scatter.  Bit-exact and
 * deterministic: perm lists pair ids by (expert, pair id).
 *   idx    int32 [T, k] (device, in); out->idx may alias it
 *   out    host struct of device pointers (counts, offsets, perm, inv_perm,
 *          active, num_active written; idx and w untouched)
 *   ws     >= moe_workspace_bytes(dims, PMOE_OP_PERMUTE, 0, 0) bytes
 * An id outside [0, E) sets PMOE_ERR_BAD_INDEX in the error word and the
 * pair is left out of every count.
 */
pmoe_status moe_permute(pmoe_dims dims, const int32_t *idx, const pmoe_routing *out,
                        void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * moe_permute_noalloc -- moe_permute for callers that cannot provide a
 * workspace (an operator or plugin hook that is handed only its tensors, or
 * code running where it must not allocate).  The pages have no counterpart:
 * this is a convenience of the library, not a step of the method.
 *
 * Same arguments, outputs and results as moe_permute (bit-identical), but
 * the per-block histogram lives in a fixed buffer of
 * PMOE_PERMUTE_NOALLOC_SCRATCH_BYTES of device memory inside the library
 * image; nothing is allocated, on the device or through another library.
 *   Size limit: ceil(T*k / 1024) * E * 4 bytes must not exceed
 *   PMOE_PERMUTE_NOALLOC_SCRATCH_BYTES, else PMOE_ERR_WORKSPACE (checked on
 *   the host before any device work; e.g. E = 384 allows T*k <= 699392).
 *   Nothing has to be zeroed first: each call overwrites what it reads.
 *   There is no device error word: an id outside [0, E) is left out of
 *   counts and gets inv_perm = -1, so offsets[E] < T*k reveals it.
 *   The buffer is one per device for the whole process: calls that can
 *   overlap in time (different streams, or different host threads without
 *   ordering) race on it; order them.  The first call on a device looks up
 *   the buffer's device address (a runtime call); make that first call
 *   outside any stream capture.
 * Errors: PMOE_ERR_INVALID_ARG as moe_permute; PMOE_ERR_WORKSPACE when the
 * problem exceeds the buffer; PMOE_ERR_CUDA if the address lookup or the
 * launch fails.
 */
#define PMOE_PERMUTE_NOALLOC_SCRATCH_BYTES (1u << 20)
pmoe_status moe_permute_noalloc(pmoe_dims dims, const int32_t *idx, const pmoe_routing *out,
                                cudaStream_t stream);

/*
 * moe_chunked_forward -- the layer (Orbit announcement, 技艺细节): active
 * experts are
 * taken C at a time in ascending id order; each chunk's experts are
 * dequantized to BF16 (FUSED: tile by tile in shared memory, no global
 * scratch; SCRATCH: into a C-expert global BF16 buffer that the next chunk
 * reuses), then for every pair of expert e:
 *   x~ = bf16(x blockdiag(R_up[e]))             (adapter on the activations)
 *   g, u = x~ W_gate[e]^T, x~ W_up[e]^T          (FP32 accumulate)
 *   h  = bf16(silu(g) u);  h~ = bf16(h blockdiag(R_down[e]))
 *   o  = h~ W_down[e]^T                          (kept in FP32)
 * and finally Y_t = bf16(sum_j w[t,j] o_(t,j)), slots summed in order in
 * FP32.
 *   X   bf16 [T, d] (in)         Y bf16 [T, d] (out)
 *   ctx NULL, or moe_ctx_bytes(dims) bytes: when given, receives what
 *       moe_backward_data needs, per pair in expert-sorted order (row i =
 *       pair perm[i]): first g | u as f32 [P, 2I] (g in columns 0..I-1,
 *       u in I..2I-1), then h as bf16 [P, I], then h~ as bf16 [P, I]
 *   chunk_C >= 1 experts per chunk (>= E means one chunk)
 *   ws  >= moe_workspace_bytes(dims, PMOE_OP_FORWARD, chunk_C, mode)
 * The result does not depend on chunk_C or mode (bit-identical).
 */
pmoe_status moe_chunked_forward(pmoe_dims dims, const pmoe_weights *wts, const pmoe_adapter *adp,
                                const pmoe_routing *rt, const void *X, int32_t chunk_C, int mode,
                                void *Y, void *ctx, void *ws, size_t ws_bytes,
                                cudaStream_t stream);
/* Bytes of the forward's saved context: P * I * (8 + 2 + 2); 0 for invalid dims. */
size_t moe_ctx_bytes(pmoe_dims dims);

/*
 * Adapter slots for rollout while training publishes (the Orbit analysis:
 * the BF16 adapter is the only thing the trainer sends to the rollout side,
 * and the rollout engine must switch to a new adapter without tearing a
 * step).  Two device copies of the adapter and one control word:
 *   ctrl   device uint64, 8-byte aligned: (version << 32) | active_slot
 * moe_adapter_publish stores a new control word with one atomic 64-bit
 * write, ordered after the earlier work of its stream (so the new slot's
 * contents, copied on that stream, are in place first).
 * moe_chunked_forward_slots is moe_chunked_forward with the adapter taken
 * from the active slot: its first kernel reads the control word once and
 * every rotation of that forward uses the slot it names, so a forward
 * running while a publish lands uses one adapter throughout; the version it
 * used is written to *version_out (device uint32, may be NULL).
 * Protocol: write only the inactive slot, and rewrite a slot only after
 * every forward that reported that slot's version has completed.
 */
typedef struct {
    const void *R_up[2], *R_down[2];   /* bf16, as pmoe_adapter; R_down[] both NULL or both set */
    int64_t stride_up, stride_down;
    const uint64_t *ctrl;
} pmoe_adapter_slots;

pmoe_status moe_adapter_publish(uint64_t *ctrl, uint32_t slot, uint32_t version,
                                cudaStream_t stream);
pmoe_status moe_chunked_forward_slots(pmoe_dims dims, const pmoe_weights *wts,
                                      const pmoe_adapter_slots *slots, const pmoe_routing *rt,
                                      const void *X, int32_t chunk_C, int mode, void *Y, void *ctx,
                                      uint32_t *version_out, void *ws, size_t ws_bytes,
                                      cudaStream_t stream);

/*
 * moe_backward_data -- backward through the frozen experts with no base
 * weight gradient (Orbit announcement, 技艺细节: bypass-base-weight-grad GEMM
 * backward; the Orbit analysis, 机制拆解: the base takes no backward update
 * cost).  Routing and
 * w are held fixed.  Per pair (t, j), e = idx[t, j]:
 *   G = dY_t W_down[e]          d_topk_w[t,j] = G . h~
 *   dh~ = w[t,j] G              dR_down[e] += h_blk^T dh~_blk
 *   dh = dh~ R_down^T;  dg = dh u s(g)(1 + g(1 - s(g)));  du = dh silu(g)
 *   dx~ = dg W_gate + du W_up   dR_up[e] += x_blk^T dx~_blk
 *   dx_pair = dx~ R_up^T        dX_t = bf16(sum_j dx_pair), slots in order
 * with h and h~ = bf16(h blockdiag(R_down[e])) as the forward saved them.  Every
 * intermediate is FP32 (g, u from ctx; G, dh~, dh, dg, du, dx~, dx_pair),
 * except at the tensor cores: dh~ and dx~ enter the rotations and adapter
 * gradients as two BF16 parts hi = bf16(v), lo = bf16(v - hi), which carry
 * v to 2^-16; [dg | du] enters the dx~ GEMM in FP16 (11 significant bits),
 * with the weights' BF16 values in FP16 encoding (exact for weights in the
 * FP16 normal range [2^-14, 65504] and zero).  The only BF16 roundings are
 * h~ and dX.
 *   X, dY   bf16 [T, d] (in)    ctx from the forward (in, moe_ctx_bytes)
 *   dX      bf16 [T, d] (out)
 *   d_topk_w f32 [T, k] or NULL (out)
 *   dR_up   f32 shaped like R_up, dR_down f32 shaped like R_down (out,
 *           overwritten; NULL iff the matching rotation is NULL); with a
 *           shared adapter they hold the sum over all experts
 *   ws  >= moe_workspace_bytes(dims, PMOE_OP_BACKWARD, chunk_C, 0)
 * Reductions run in a fixed order: results are run-to-run identical.
 */
pmoe_status moe_backward_data(pmoe_dims dims, const pmoe_weights *wts, const pmoe_adapter *adp,
                              const pmoe_routing *rt, const void *X, const void *dY,
                              const void *ctx, int32_t chunk_C, void *dX, float *d_topk_w,
                              float *dR_up, float *dR_down, void *ws, size_t ws_bytes,
                              cudaStream_t stream);

/*
 * moe_dequant -- the dequantization step alone (Orbit announcement,
 * 技艺细节: temporary dequantization of the selected experts): one [N, K] weight matrix in `fmt` to BF16 [N, K].
 * Bit-exact with the format definitions above.  N >= 0, K % 32 == 0
 * (INT4 / MXFP4) or N % 128 == 0 and K % 128 == 0 (FP8).
 */
pmoe_status moe_dequant(pmoe_wfmt fmt, const void *q, const void *s, int64_t N, int64_t K,
                        void *out, cudaStream_t stream);

/*
 * moe_grouped_gemm -- the grouped GEMM step alone (Orbit announcement, 技艺细节:
 * "grouped GEMM" over the dequantized experts), on the tensor cores with
 * the weights dequantized tile by tile in shared memory.  Rows
 * offsets[e] .. offsets[e+1]-1 of A belong to expert e.
 *   trans == 0: out[r] = bf16(A[r] W_e^T), A bf16 [rows, K], out [rows, N]
 *   trans == 1: out[r] = bf16(A[r] W_e),   A bf16 [rows, N], out [rows, K]
 * with W_e the [N, K] matrix of expert e in `fmt` (q, s laid out as in
 * pmoe_wfmt, experts consecutive).  offsets: device int32 [E+1],
 * nondecreasing, offsets[0] = 0, offsets[E] = rows.  N % 64 == 0,
 * K % 64 == 0 (FP8: both % 128), rows >= 0, E <= 4096.
 *   ws  >= moe_grouped_gemm_ws_bytes(E, rows) bytes.
 */
pmoe_status moe_grouped_gemm(pmoe_wfmt fmt, const void *q, const void *s, int32_t E, int32_t N,
                             int32_t K, int trans, const void *A, const int32_t *offsets,
                             int32_t rows, void *out, void *ws, size_t ws_bytes,
                             cudaStream_t stream);
size_t moe_grouped_gemm_ws_bytes(int32_t E, int32_t rows);

/*
 * adapter_apply -- Xr = bf16(X blockdiag(R)) (the Orbit analysis, 机制拆解: the OFT
 * adapter as a local orthogonal transform).  X bf16 [rows, dim], R bf16
 * [dim/b, b, b], Xr bf16 [rows, dim] (must not alias X).  dim % b == 0,
 * b in {16, 32, 64, 128}.
 */
pmoe_status adapter_apply(int32_t rows, int32_t dim, int32_t b, const void *X, const void *R,
                          void *Xr, cudaStream_t stream);

/*
 * adapter_grad -- backward of adapter_apply: dX = bf16(dXr blockdiag(R)^T)
 * (skipped when dX is NULL) and dR[beta] = sum_i X_blk[i]^T dXr_blk[i]
 * (f32 [dim/b, b, b], overwritten, fixed summation order).
 */
pmoe_status adapter_grad(int32_t rows, int32_t dim, int32_t b, const void *X, const void *dXr,
                         const void *R, void *dX, float *dR, cudaStream_t stream);

/*
 * dense_linear_forward / dense_linear_backward -- one frozen low-precision
 * projection outside the experts, with the orthogonal adapter on its input
 * and no gradient for the frozen weight (the Orbit article, technical
 * details: bypass-base-weight-grad; the Orbit analysis, OFT section: a
 * local orthogonal transform of the activations).
 *   forward:  x~ = bf16(X blockdiag(R));  Y = bf16(x~ W^T)
 *   backward: dx~ = bf16(dY W);  dR = sum_rows x_blk^T dx~_blk (FP32);
 *             dX = bf16(dx~ blockdiag(R)^T)      (R NULL: dX = bf16(dY W))
 *   q, s   W [N, K] in the packed format fmt (as one expert of pmoe_weights)
 *   R      bf16 [K/block, block, block] or NULL (no adapter); block in
 *          {16, 32, 64, 128}, K % block == 0
 *   X      bf16 [rows, K] (in)          Y  bf16 [rows, N] (out)
 *   dY     bf16 [rows, N] (in)          dX bf16 [rows, K] (out)
 *   dR     f32 [K/block, block, block] (out, overwritten; required iff R)
 *   ws     >= dense_linear_ws_bytes(rows, N, K) bytes, 16-byte aligned
 * N % 64 == 0 and K % 64 == 0 (FP8: % 128).  All pointers 16-byte aligned.
 */
size_t dense_linear_ws_bytes(int32_t rows, int32_t N, int32_t K);
pmoe_status dense_linear_forward(pmoe_wfmt fmt, const void *q, const void *s, int32_t N, int32_t K,
                                 int32_t block, const void *R, int32_t rows, const void *X, void *Y,
                                 void *ws, size_t ws_bytes, cudaStream_t stream);
pmoe_status dense_linear_backward(pmoe_wfmt fmt, const void *q, const void *s, int32_t N, int32_t K,
                                  int32_t block, const void *R, int32_t rows, const void *X,
                                  const void *dY, void *dX, float *dR, void *ws, size_t ws_bytes,
                                  cudaStream_t stream);

/*
 * adapter_cayley -- R = (I + S)(I - S)^{-1} for nblk skew-symmetric b x b
 * blocks S (f32 [nblk, b, b]; only skew input is meaningful: the symmetric
 * part of I - S must be I); R written as bf16 (R_bf16, nullable) and f32
 * (R_f32, nullable).  b in {2, 4, 8, 16, 32, 64, 128}.
 */
pmoe_status adapter_cayley(int32_t nblk, int32_t b, const float *S, void *R_bf16, float *R_f32,
                           cudaStream_t stream);

/*
 * adapter_cayley_grad -- dS = M - M^T with M = (I + R)^T dR (I - S)^{-T},
 * the gradient with respect to the skew parameter of each block.  Since
 * (I - S)^{-1} = (I + R)/2, it is computed from R_f32 (the output of
 * adapter_cayley for the same S) alone; S is accepted for reference and
 * may be NULL.  R_f32, dR: f32 [nblk, b, b]; dS f32 out.
 */
pmoe_status adapter_cayley_grad(int32_t nblk, int32_t b, const float *S, const float *R_f32,
                                const float *dR, float *dS, cudaStream_t stream);

/* Bytes of device workspace an op needs (op = PMOE_OP_*).  Includes the
 * 256-byte error word at the start.  In SCRATCH mode this includes the
 * C-expert BF16 dequant buffer, reported separately by
 * moe_scratch_bytes. */
size_t moe_workspace_bytes(pmoe_dims dims, int op, int32_t chunk_C, int mode);

/* Bytes of the bounded dequant scratch of one chunk in SCRATCH mode:
 * min(C, E) experts x 3 x I x d BF16; 0 in FUSED mode. */
size_t moe_scratch_bytes(pmoe_dims dims, int32_t chunk_C, int mode);

/* Clear the device error word at the start of `ws` (asynchronous). */
pmoe_status moe_clear_status(void *ws, cudaStream_t stream);

/* Synchronize `stream`, read the device error word of `ws`, clear it and
 * return it (PMOE_OK when no device error was recorded). */
pmoe_status moe_query_status(void *ws, cudaStream_t stream);

/* Static description of a status code. */
const char *pmoe_status_string(pmoe_status s);

/* Number of kernels the library has enqueued since load (all entry
 * points, all streams); a diagnostic counter for launch accounting. */
uint64_t pmoe_launch_count(void);

/* Kernel classes of the diagnostic timer. */
enum {
    PMOE_KT_GEMM_GATE_UP = 0,   /* forward gate/up grouped GEMM (+ SwiGLU epilogue) */
    PMOE_KT_GEMM_DOWN = 1,      /* forward down grouped GEMM */
    PMOE_KT_GEMM_BWD_G = 2,     /* backward dY W_down grouped GEMM */
    PMOE_KT_GEMM_BWD_DX = 3,    /* backward [dg du] W13 grouped GEMM */
    PMOE_KT_ROUTER = 4,         /* router logits */
    PMOE_KT_COUNT = 5
};

/* Diagnostic per-kernel timing.  While enabled, every launch of a timed
 * kernel class is bracketed by two CUDA events recorded on the launch
 * stream (events come from a host-side pool; no device memory is
 * allocated).  Enabling or disabling clears the records. */
pmoe_status pmoe_kernel_timing(int enable);

/* Total device time (ms) and number of launches of kernel class `which`
 * recorded since timing was enabled; waits for the recorded events. */
pmoe_status pmoe_kernel_time(int which, double *ms_total, int *launches);

/*
 * pmoe_debug_expire_gemm_wait -- test hook for the bounded waits (no
 * counterpart in the pages).  Every wait inside the grouped-GEMM kernel is
 * bounded; this makes one of them run out without any fault: the NEXT
 * grouped-GEMM launch in the process (whichever entry point makes it) uses
 * wait_ns as the limit of its waits, and its MMA issuer withholds the
 * accumulator-full signal of CTA 0's first work item.  CTA 0's epilogue
 * then gives up after wait_ns, records PMOE_ERR_TIMEOUT in the call's error
 * word, and every role of that CTA leaves its loop after its own bounded
 * wait and frees its tensor memory; the call's outputs are incomplete.
 * One-shot: the launch consumes the hook.  wait_ns in [1e5, 2e9] (the
 * bound keeps every issued copy and MMA long finished before a role gives
 * up), else PMOE_ERR_INVALID_ARG.  Process-wide state: not for use while
 * other threads launch layer work.
 */
pmoe_status pmoe_debug_expire_gemm_wait(uint64_t wait_ns);

#ifdef __cplusplus
}
#endif
#endif /* PMOE_H */
