/*
 * fp8bs.h -- C ABI of the block-scaled FP8 (E4M3) library for GB300 (sm_103a).
 *
 * What the calls compute comes from three web pages, cited by title and
 * section:
 *  [SkyRL]  "Anyscale、SkyRL で FP8 学習・ロールアウトをサポートし一貫性を維持"
 *  [AIS]    "AIS: Adaptive Importance Sampling for Quantized RL" (explainer)
 *  [Jet-RL] "Jet-RL: Enabling On-Policy FP8 Reinforcement Learning with
 *            Unified Training and Rollout Precision Flow" (summary)
 *
 * Conventions shared by every call
 *  - Matrices are row-major.  A linear layer is Y = X W^T with X [M,K],
 *    W [N,K] (the torch nn.Linear convention).  "K-major" means the
 *    contraction index is contiguous.
 *  - E4M3 is the FN variant (bias 7, largest finite 448, no infinity);
 *    encoding rounds to nearest-even and saturates.  Blockwise scales are
 *    s = amax/448 in fp32 (1 for an all-zero group) and elements are encoded
 *    from the IEEE fp32 quotient x/s.  MX scales are E8M0 bytes e+127 with
 *    e = clamp(floor(log2 amax) - 8, -127, 127); elements are encoded from
 *    x * 2^-e.
 *  - Every pointer inside an fp8_tensor and every data pointer argument is
 *    DEVICE memory owned by the caller; the library never frees or keeps
 *    it.  Pointers must be 16-byte aligned, leading dimensions (ld, in
 *    elements) a multiple of 8.  The library's own device memory is one
 *    small status block per device, allocated on first use.
 *  - Every call is asynchronous on the given stream (NULL = the legacy
 *    default stream).  Argument checks happen before anything is enqueued
 *    and are reported by the return value; nothing is enqueued when the
 *    return value is not FP8_OK.  Errors found on the device (a bounded
 *    wait that expired, a checksum mismatch) are recorded in the device
 *    status block and returned by fp8_status_poll().
 *  - No call throws, traps, or allocates memory other than the status block.
 *  - Thread safety: calls may come from several host threads.  Calls that
 *    run concurrently on different streams of the same device share the
 *    status block: fp8_sync_install() calls must not overlap each other.
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FP8BS_ABI_VERSION 1

typedef struct CUstream_st* fp8_stream_t; /* identical to cudaStream_t */

typedef enum {
    FP8_OK = 0,
    FP8_ERR_INVALID_ARG = 1,  /* null pointer, negative size, wrong recipe/layout for the call */
    FP8_ERR_ALIGNMENT = 2,    /* pointer not 16-byte aligned or ld not a multiple of 8 */
    FP8_ERR_UNSUPPORTED = 3,  /* shape outside what the kernels handle (see each call) */
    FP8_ERR_BAD_PAYLOAD = 4,  /* sync payload header/table does not match the destinations */
    FP8_ERR_CHECKSUM = 5,     /* sync payload checksum mismatch (reported by fp8_status_poll) */
    FP8_ERR_TIMEOUT = 6,      /* a bounded on-chip wait expired; the kernel gave up cleanly */
    FP8_ERR_CUDA = 7,         /* a CUDA runtime/driver call failed; see fp8_last_error() */
    FP8_ERR_CAPACITY = 8      /* destination buffer too small */
} fp8_status;

typedef enum {
    FP8_RECIPE_BLOCKWISE_FP32 = 1, /* fp32 scales: 1x128 / 128x1 groups, 128x128 blocks */
    FP8_RECIPE_MXFP8 = 2,          /* E8M0 scales, 1x32 blocks */
    /* The blockwise groups with power-of-two scales ([SkyRL] "Deep dive:
     * FP8 quantization with FP32 and power-of-two block scales": Blackwell
     * tensor cores take only power-of-two block scales).  Scale 2^e with
     * e = ceil(log2(amax/448)) (amax/448 the fp32 recipe's IEEE quotient),
     * clamped to [-127, 127], e = 0 for an all-zero group; codes from the
     * exact product x * 2^-e.  Scales are E8M0 bytes (e + 127) in
     * FP8_LAYOUT_MX_1x32, each group's byte repeated in the 1x32 blocks it
     * covers, so the tensor is also a valid MXFP8 tensor and the GEMMs run
     * on the block-scaled MMA with no promotion. */
    FP8_RECIPE_BLOCKWISE_POW2 = 3
} fp8_recipe;

typedef enum {
    /* fp32 [cols/128][rows]: one scale per row per 128 consecutive columns,
     * stored group-major so a 128-row tile reads its scales contiguously. */
    FP8_LAYOUT_GROUP_1x128 = 1,
    /* fp32 [rows/128][cols/128]: one scale per 128x128 block. */
    FP8_LAYOUT_BLOCK_128x128 = 2,
    /* E8M0 bytes in the tensor-core scale-factor layout: atoms of 128 rows x
     * 4 blocks of 32 columns (512 bytes); atom (rt, ct) at byte
     * (rt * ceil(cols/128) + ct) * 512; row r, 32-block j inside it at
     * (r%32)*16 + ((r%128)/32)*4 + j%4.  Size fp8_mx_scale_bytes(rows, cols);
     * padding entries are 0. */
    FP8_LAYOUT_MX_1x32 = 3,
    /* E8M0, MX layout per group of rows (MoE experts): group g's rows start
     * at atom row P_g = sum_{h<g} ceil(M_h/128), so every group begins on a
     * 128-row atom boundary.  Size fp8_mx_grouped_scale_bytes(). */
    FP8_LAYOUT_MX_1x32_GROUPED = 4
} fp8_scale_layout;

typedef enum {
    FP8_AXIS_K = 0, /* 1x128 groups along the contiguous axis (activations, dY for DGrad) */
    FP8_AXIS_M = 1  /* 128x1 groups along the rows, written transposed (WGrad operands) */
} fp8_axis;

typedef enum {
    FP8_GEMM_FWD = 0,   /* Y  = X W^T:  A = X [M,K] 1x128,  B = W [N,K] 128x128 */
    FP8_GEMM_DGRAD = 1, /* dX = dY W:   A = dY [M,N] 1x128, B = W^T [K,N] 128x128 */
    FP8_GEMM_WGRAD = 2  /* dW = dY^T X: A = dY^T [N,M] 1x128 (from 128x1), B = X^T [K,M] 1x128 */
} fp8_gemm_op;

typedef enum { FP8_OUT_BF16 = 0, FP8_OUT_F32 = 1 } fp8_out_dtype;

/* Non-owning view of a quantized matrix: codes u8 [rows][cols] row-major,
 * scales in `layout`. */
typedef struct {
    void* codes;
    void* scales;
    int64_t rows;
    int64_t cols;
    int32_t recipe; /* fp8_recipe */
    int32_t layout; /* fp8_scale_layout */
} fp8_tensor;

typedef enum { FP8_SYNC_FP8 = 1, FP8_SYNC_BF16 = 2 } fp8_sync_kind;

/* One tensor of a weight-sync payload.  FP8: t.codes/t.scales/rows/cols/
 * recipe/layout describe the quantized tensor.  BF16 (tensors kept in high
 * precision, e.g. norms and embeddings): t.codes points to the bf16 data
 * [rows][cols], t.scales = NULL, recipe = layout = 0. */
typedef struct {
    uint64_t tag;     /* caller's identifier (e.g. a hash of the parameter name) */
    int32_t kind;     /* fp8_sync_kind */
    int32_t reserved; /* must be 0 */
    fp8_tensor t;
} fp8_sync_entry;

/* ---------------------------------------------------------------------- */
/* Quantizers                                                              */
/* ---------------------------------------------------------------------- */

/* Group quantization of a bf16 matrix x [M][ld] (first K columns used).
 * out->recipe selects the scales: FP8_RECIPE_BLOCKWISE_FP32 with the fp32
 * layouts below, or FP8_RECIPE_BLOCKWISE_POW2 with out->layout =
 * FP8_LAYOUT_MX_1x32 and a scale buffer of fp8_mx_scale_bytes(rows, cols)
 * of the output (K x M for FP8_AXIS_M); the codes are laid out the same.
 * [Jet-RL] "Kwantisatieschema": activations in 1x128 groups; for WGrad the
 * operands in 128x1 groups.  [AIS] equation Q(X): s = max|X| / qmax.
 *  axis = FP8_AXIS_K: out->codes [M][K], out->scales fp32 [K/128][M];
 *                     requires K % 128 == 0, any M >= 0.
 *  axis = FP8_AXIS_M: one scale per column per 128 rows, codes written
 *                     transposed: out->codes [K][M], out->scales fp32
 *                     [M/128][K] -- exactly the 1x128 quantization of x^T.
 *                     Requires M % 128 == 0, K % 8 == 0.
 * out->rows/cols must equal (M, K) for AXIS_K and (K, M) for AXIS_M;
 * out->recipe = FP8_RECIPE_BLOCKWISE_FP32, out->layout = FP8_LAYOUT_GROUP_1x128
 * (or FP8_RECIPE_BLOCKWISE_POW2 with FP8_LAYOUT_MX_1x32). */
fp8_status fp8_quantize_group(const void* x_bf16, int64_t M, int64_t K, int64_t ld,
                              fp8_axis axis, const fp8_tensor* out, fp8_stream_t stream);

/* The WGrad operand from a saved FP8 activation ([Jet-RL]
 * "Kwantisatieschema": activations kept for the backward pass are stored in
 * FP8, quantized 1x128; WGrad takes its operands in 128x1 groups along M),
 * without the bf16 tensor: every element of `in` is dequantized once in
 * fp32, x' = RN(dec(q) * s), and x' is quantized in 128x1 groups with the
 * codes transposed -- exactly fp8_quantize_group(AXIS_M) applied to x'.
 *  in:  FP8_RECIPE_BLOCKWISE_FP32, FP8_LAYOUT_GROUP_1x128, rows M, cols K.
 *  out: FP8_RECIPE_BLOCKWISE_FP32, FP8_LAYOUT_GROUP_1x128, rows K, cols M
 *       (codes [K][M], scales fp32 [M/128][K]).
 * Requires M % 128 == 0, K % 128 == 0.  Scales are IEEE fp32 divisions; the
 * codes are those of the IEEE fp32 quotients x' / s (x' has a full fp32
 * significand).  An E4M3 NaN code in `in` (0x7F, 0xFF; never written by the
 * quantizers here) gives a NaN code, of either sign, at its transposed
 * position, and does not enter its group's scale. */
fp8_status fp8_requantize_transposed(const fp8_tensor* in, const fp8_tensor* out, fp8_stream_t stream);

/* 128x128 block quantization of a bf16 weight w [N][ld] (first K columns).
 * [SkyRL] "なぜ強化学習に FP8 が重要なのか": one scale per 128x128 weight block;
 * [Jet-RL] "Kwantisatieschema".  Requires N % 128 == 0, K % 128 == 0.
 * out: codes [N][K], scales fp32 [N/128][K/128], layout BLOCK_128x128.
 * out_t (nullable): the same codes transposed [K][N] with the transposed
 * scale grid [K/128][N/128] (rows = K, cols = N), the DGrad B operand;
 * [SkyRL] "Performance analysis", トレーニング: the trainer keeps a row-wise and a
 * transposed copy.  FP8_RECIPE_BLOCKWISE_POW2 in out (and out_t):
 * power-of-two scales in FP8_LAYOUT_MX_1x32 instead, every byte of a block's
 * 512-byte atom holding its exponent. */
fp8_status fp8_quantize_block(const void* w_bf16, int64_t N, int64_t K, int64_t ld,
                              const fp8_tensor* out, const fp8_tensor* out_t,
                              fp8_stream_t stream);

/* fp8_param: recomputes the FP8 storage of a weight from its fp32 master,
 * optionally applying the optimizer step's final add first.  [SkyRL]
 * overview: FP8 parameters plus an FP32 master weight, with no BF16 copy;
 * "Deep dive: FP8 quantization with FP32 and power-of-two block scales":
 * the optimizer updates the FP32 master and re-quantizes it into the FP8
 * storage after every step, Q(W_t) from the current master.
 *  master: fp32 [N][ld] on the device (first K columns used), 16-byte
 *          aligned, ld % 4 == 0.  Written only when delta is non-NULL.
 *  delta:  NULL, or fp32 [N][ld] (same ld): master <- RN(master + delta)
 *          element by element before quantizing (the update is not kept).
 *  out:    codes [N][K] and 128x128 block scales of the (updated) master;
 *          FP8_RECIPE_BLOCKWISE_FP32 with FP8_LAYOUT_BLOCK_128x128 (fp32
 *          scales s = RN(amax/448), 1 for a block whose quotient is 0, codes
 *          from the IEEE quotient w/s), or FP8_RECIPE_BLOCKWISE_POW2 with
 *          FP8_LAYOUT_MX_1x32 (E8M0 exponents, codes from w * 2^-e).
 *  out_t:  NULL or the transposed copy [K][N] in the same recipe.
 * Requires N % 128 == 0, K % 128 == 0.  Errors: INVALID_ARG / ALIGNMENT /
 * UNSUPPORTED before anything is enqueued; the call is asynchronous. */
fp8_status fp8_param_requantize(float* master, const float* delta, int64_t N, int64_t K, int64_t ld,
                                const fp8_tensor* out, const fp8_tensor* out_t, fp8_stream_t stream);

/* Producers fused with the activation quantization.  [Jet-RL]
 * "Kwantisatieschema": the activations saved for the backward pass are
 * stored in FP8, fused with the operator that produces them;
 * "Implementatie": fused activation and RMSNorm kernels.  Each computes its
 * producer in fp32, rounds it to bf16 and quantizes those bf16 values, so
 * the codes equal fp8_quantize_group / fp8_quantize_mx applied to the bf16
 * output.  out->recipe selects the quantization: FP8_RECIPE_BLOCKWISE_FP32
 * (layout FP8_LAYOUT_GROUP_1x128, fp32 scales [cols/128][rows]),
 * FP8_RECIPE_BLOCKWISE_POW2 or FP8_RECIPE_MXFP8 (layout FP8_LAYOUT_MX_1x32,
 * fp8_mx_scale_bytes(rows, cols) bytes).
 *
 * RMSNorm: y = RN_bf16(RN(x * rstd) * gamma), rstd = 1/sqrt(mean_k x^2 +
 * eps) per row (fp32: the sum of squares in fp32, then the correctly
 * rounded reciprocal square root).
 *  x:     bf16 [M][ld]; gamma: bf16 [K] (16-byte aligned).
 *  y:     NULL or bf16 [M][ldy], the normalized rows.
 *  rstd:  NULL or fp32 [M], saved for the backward pass.
 *  out:   codes [M][K] of y.  Requires K % 128 == 0, K <= 8192. */
fp8_status fp8_rmsnorm_quantize(const void* x_bf16, const void* gamma_bf16, int64_t M, int64_t K, int64_t ld,
                                float eps, void* y_bf16, int64_t ldy, float* rstd, const fp8_tensor* out,
                                fp8_stream_t stream);

/* SwiGLU: h = RN_bf16(silu(g) * u), silu(g) = g / (1 + exp(-g)), with the
 * gate projection g in columns [0, F) and the up projection u in [F, 2F) of
 * each row of gu (bf16 [M][ld], ld >= 2F).
 *  h:     NULL or bf16 [M][ldh].
 *  out:   codes [M][F] of h.  Requires F % 128 == 0. */
fp8_status fp8_swiglu_quantize(const void* gu_bf16, int64_t M, int64_t F, int64_t ld, void* h_bf16, int64_t ldh,
                               const fp8_tensor* out, fp8_stream_t stream);

/* MXFP8 quantization of x [R][ld] (first K columns) in 1x32 blocks with E8M0
 * scales.  [SkyRL] "独立した量子化がポリシーの一貫性を崩す場合": one scale per
 * 1x32 block in the MXFP8 recipe; "Deep dive: FP8 quantization with FP32
 * and power-of-two block scales": Blackwell tensor cores take power-of-two
 * scales only.  Requires K % 32 == 0, any R >= 0.
 * out: codes [R][K], scales in FP8_LAYOUT_MX_1x32 (fp8_mx_scale_bytes(R, K)
 * bytes, padding entries written as 0), recipe MXFP8. */
fp8_status fp8_quantize_mx(const void* x_bf16, int64_t R, int64_t K, int64_t ld,
                           const fp8_tensor* out, fp8_stream_t stream);

/* MXFP8 operands of the backward GEMMs: 32x1 blocks along the rows of x
 * [R][ld] (first K columns), codes written transposed -- exactly the 1x32
 * quantization of x^T.  out: codes [K][R], scales FP8_LAYOUT_MX_1x32 of the
 * K x R output (fp8_mx_scale_bytes(K, R) bytes); out->rows/cols = (K, R),
 * recipe FP8_RECIPE_MXFP8.  Requires R % 128 == 0, K % 8 == 0.  DGrad:
 * B = W^T from W [N][K]; WGrad: A = dY^T, B = X^T. */
fp8_status fp8_quantize_mx_transposed(const void* x_bf16, int64_t R, int64_t K, int64_t ld,
                                      const fp8_tensor* out, fp8_stream_t stream);

/* Bytes of an FP8_LAYOUT_MX_1x32 scale buffer for a rows x cols matrix. */
int64_t fp8_mx_scale_bytes(int64_t rows, int64_t cols);
/* Upper bound of an FP8_LAYOUT_MX_1x32_GROUPED scale buffer. */
int64_t fp8_mx_grouped_scale_bytes(int64_t total_rows, int64_t cols, int32_t num_groups);

/* Row gather of MX-quantized rows into expert-contiguous groups (MoE
 * dispatch): dst row i = src row gather[i]; codes copied, scales moved into
 * the grouped layout, group padding entries set to 0.  Quantize-then-permute
 * equals permute-then-quantize exactly, because 1x32 blocks lie inside a row.
 * gather_dev: int32 [total_rows] device; m_offsets_dev: int32 [num_groups+1]
 * device, non-decreasing, m_offsets[0] = 0, m_offsets[num_groups] =
 * total_rows.  src: MXFP8, layout MX_1x32; dst: rows = total_rows, same cols,
 * layout MX_1x32_GROUPED with fp8_mx_grouped_scale_bytes() bytes of scales.
 * Requires cols % 128 == 0.  Out-of-range gather entries are skipped on the
 * device; rows whose group offsets break the rules above get their codes
 * row copied but no scale words.  Both are reported as FP8_ERR_INVALID_ARG by
 * fp8_status_poll().  After such a report dst is partly written (some code
 * rows copied, some scale words not), so its contents must not be used;
 * every write of the call stays inside dst. */
fp8_status fp8_permute_rows_mx(const fp8_tensor* src, const int32_t* gather_dev,
                               const int32_t* m_offsets_dev, int32_t num_groups,
                               const fp8_tensor* dst, fp8_stream_t stream);

/* MoE dispatch fused with the MX quantization ([Jet-RL] "Kwantisatieschema":
 * the activation quantization fused with the operator before it), token
 * major: each bf16 row t of x [T][ld] (first K columns) is read and
 * quantized (1x32 blocks, E8M0) once, and its codes and scales are written
 * to dst rows dst_index[t][j], j < top_k, in the expert-grouped layout -- the
 * same bytes as fp8_quantize_mx followed by fp8_permute_rows_mx with the
 * inverse index, without the intermediate FP8 copy or re-reading a token
 * once per expert.
 *  dst_index_dev: int32 [T][top_k] device; -1 drops the slot; each dst row
 *                 should be named at most once (rows named by no slot keep
 *                 their codes, their scales read 0).
 *  m_offsets_dev, num_groups, dst: as for fp8_permute_rows_mx (dst->cols = K).
 * Requires K % 128 == 0, 0 <= top_k <= 64.  Out-of-range entries are skipped
 * on the device and reported as FP8_ERR_INVALID_ARG by fp8_status_poll();
 * group offsets that break the rules of fp8_permute_rows_mx are reported
 * the same way and no codes are written (the scales read 0). */
fp8_status fp8_dispatch_quantize_mx(const void* x_bf16, int64_t T, int64_t K, int64_t ld, const int32_t* dst_index_dev,
                                    int32_t top_k, const int32_t* m_offsets_dev, int32_t num_groups,
                                    const fp8_tensor* dst, fp8_stream_t stream);

/* ---------------------------------------------------------------------- */
/* GEMMs                                                                   */
/* ---------------------------------------------------------------------- */

/* Block-scaled FP8 GEMM D[m][n] = sum_k A[m][k] B[n][k] with fp32
 * accumulation, both operands K-major (codes [rows][K]).
 *  Blockwise recipe ([SkyRL] "Performance analysis", トレーニング: FP8 linear-layer GEMMs; [Jet-RL]
 *  "Kwantisatieschema": forward, DGrad and WGrad in FP8):
 *    D = sum over 128-column blocks kb of sa(m,kb) sb(n,kb) (sum_{k in kb} qa qb)
 *    A: layout GROUP_1x128.  B: BLOCK_128x128 for FWD/DGRAD, GROUP_1x128
 *    for WGRAD (its 128x1 scales become per-column scales of D).
 *  MXFP8 recipe ([SkyRL] "Performance analysis": fp8_recipe=auto selects native
 *  MXFP8 on Blackwell): D = sum_k qa 2^ea(m,k/32) qb 2^eb(n,k/32); A and B
 *  in layout MX_1x32; FWD, DGRAD (B = W^T from fp8_quantize_mx_transposed)
 *  and WGRAD (A = dY^T, B = X^T, both from fp8_quantize_mx_transposed).
 *  Blockwise recipe with power-of-two scales (both operands
 *  FP8_RECIPE_BLOCKWISE_POW2, layout MX_1x32): the blockwise formula with
 *  sa, sb powers of two, computed by the block-scaled MMA; FWD, DGRAD and
 *  WGRAD (operands as for the fp32 recipe); bf16 D only.
 * Sizes: M = A->rows, K = A->cols = B->cols, N = B->rows.  K % 128 == 0,
 * N % 16 == 0 (blockwise: N % 128 == 0), any M >= 0.
 * D: [M][ldd] of d_dtype (FP8_OUT_F32 only for the blockwise recipe).
 * d_quant (nullable): also quantizes the bf16-rounded D for the next layer
 * inside the epilogue ([SkyRL] "Performance analysis", 生成: activation quantization folded into
 * the GEMM kernel; [Jet-RL] "Kwantisatieschema": fused with the previous
 * operator): blockwise -> 1x128 groups (GROUP_1x128, N % 128 == 0);
 * MXFP8 -> 1x32 (MX_1x32); power-of-two blockwise -> 1x128 groups with
 * power-of-two scales (MX_1x32, N % 128 == 0).  d_quant rows/cols =
 * (M, N); requires bf16 D.
 * The result equals fp8_quantize_group / fp8_quantize_mx applied to D. */
fp8_status fp8_gemm_blockscaled(const fp8_tensor* A, const fp8_tensor* B, void* D, int64_t ldd,
                                int32_t d_dtype, int32_t op, const fp8_tensor* d_quant,
                                fp8_stream_t stream);

/* Grouped MXFP8 GEMM for MoE experts: for each group g,
 * D[off_g + i][n] = sum_k A[off_g + i][k] B[g*N + n][k], 0 <= i < M_g.
 * [SkyRL] "メモリ削減効果": MoE routed experts hold most parameters.
 * A: MXFP8 rows = total_rows (= m_offsets[num_groups]), layout
 *    MX_1x32_GROUPED (from fp8_permute_rows_mx).
 * B_stack: MXFP8 rows = num_groups * N, layout MX_1x32 (fp8_quantize_mx of
 *    the [num_groups*N][K] weight stack).
 * m_offsets_dev: int32 [num_groups+1] on the device (see above).  The
 *    kernel checks them: offsets that are negative, decreasing, above
 *    total_rows, or that do not start at 0 are clamped to [0, total_rows]
 *    (no row outside A or D is touched) and fp8_status_poll() returns
 *    FP8_ERR_INVALID_ARG.
 * D: bf16 [total_rows][ldd].  Requires K % 128 == 0, N % 256 == 0,
 * 1 <= num_groups <= 1024. */
fp8_status fp8_grouped_gemm(const fp8_tensor* A, const fp8_tensor* B_stack,
                            const int32_t* m_offsets_dev, int32_t num_groups, int64_t N,
                            void* D, int64_t ldd, fp8_stream_t stream);

/* ---------------------------------------------------------------------- */
/* On-policy weight sync ([SkyRL] "On-Policy FP8 weight sync", Fig. 3:     */
/* quantized parameters travel as FP8 payloads with their block scales,    */
/* precision-sensitive tensors stay BF16, the receiver installs them       */
/* without a quantizer and the weights are bit-identical; "実践的な知見":    */
/* values, scales, exclusions and layouts come from one shared description */
/* rather than being inferred by each side).                               */
/*                                                                         */
/* Payload bytes (little-endian):                                          */
/*   header 64 B: u64 magic "FP8SYNC1", u32 version 2, u32 n_entries,      */
/*     u64 total_bytes, u64 data_offset, u64 checksum, 24 zero bytes;      */
/*   n entries of 128 B at byte 64: u64 tag, u32 kind, u32 recipe,         */
/*     i64 rows, i64 cols, u32 layout, u32 0, u64 data_offset,             */
/*     u64 data_bytes, u64 scales_offset, u64 scales_bytes, 56 zero bytes; */
/*   segments from data_offset = roundup(64 + 128 n, 256): each entry's    */
/*     data then scales, each 256-byte aligned, zero padded; total_bytes   */
/*     is a multiple of 256.                                               */
/*   checksum = sum over 8-byte words w_i at offsets 8i >= 64, lo_i and    */
/*     hi_i their 32-bit halves, of ((lo_i + i 0x9E3779B9) mod 2^32) *     */
/*     ((hi_i + i 0x85EBCA6B) mod 2^32), mod 2^64 (the NH inner product of */
/*     UMAC, Black et al., CRYPTO 1999, keyed by the word index).  Any     */
/*     change to one 32-bit half of one word is detected unless the        */
/*     word's other keyed half is 0 mod 2^32.                              */
/* ---------------------------------------------------------------------- */

/* Payload size for these entries (host-only computation). */
fp8_status fp8_sync_payload_size(const fp8_sync_entry* entries, int32_t n, uint64_t* bytes);

/* Packs the entries (device tensors) into payload_dev (device, capacity
 * bytes, 256-byte aligned).  *used_bytes (host) receives the payload size.
 * The segment copy and the checksum run on the device.  When the header and
 * table fit 3136 bytes (up to 23 entries) the pack kernel writes them too,
 * so the call is device work only and can be captured in a CUDA graph;
 * larger tables are copied from the host (a pageable copy, which waits for
 * the stream). */
fp8_status fp8_sync_pack(const fp8_sync_entry* entries, int32_t n, void* payload_dev,
                         uint64_t capacity, uint64_t* used_bytes, fp8_stream_t stream);

/* Installs a payload into the destination tensors described by dst (device
 * buffers of the rollout side).  Never quantizes: the bytes are copied.
 * Every header and table byte (the checksum field excepted) must equal what
 * dst implies, and the checksum must match; both are verified on the device
 * before any destination byte is written.  For up to 23 entries the header
 * check also runs on the device (the call does not synchronize `stream`): a
 * mismatch writes nothing and fp8_status_poll() returns FP8_ERR_BAD_PAYLOAD.
 * With more entries the header and table are read back and checked on the
 * host (this synchronizes `stream`) and a mismatch is returned at once.  A
 * checksum mismatch writes nothing and fp8_status_poll() returns
 * FP8_ERR_CHECKSUM.  Installs keep their verdict in per-device state, so the
 * library orders every install after the previous one on the device (its
 * stream waits on an event the previous install recorded), whatever streams
 * or host threads issue them; inside a stream capture that ordering is the
 * caller's. */
fp8_status fp8_sync_install(const void* payload_dev, uint64_t bytes, const fp8_sync_entry* dst,
                            int32_t n, fp8_stream_t stream);

/* Install for callers that cannot allocate device memory.  The pages have
 * no counterpart of this call; it exists for processes in which cudaMalloc
 * is off limits while weights are swapped in -- for example a rollout engine
 * whose memory pool has already claimed the device, or code running inside a
 * region where allocation is forbidden.  fp8_sync_install itself allocates a
 * small status block on first use; this variant allocates nothing.
 * Result: the same bytes in the destinations as fp8_sync_install.
 * Scratch: a fixed device array inside the library (about 10 KB, present on
 * every GPU that loads the library until the process exits) holds the
 * checksum accumulator, the verdict and the segment table, so at most 128
 * entries per call; more returns FP8_ERR_CAPACITY.  The first call on a
 * device looks up the array's device address; make that first call before
 * any stream capture.  Every call shares the array; calls are ordered on
 * the device as for fp8_sync_install (the same per-device event), so calls
 * from other streams or host threads do not overlap on the GPU; calls that
 * did overlap there would race on the array.
 * Unlike fp8_sync_install it waits for the copy to finish and reports a
 * checksum mismatch directly (FP8_ERR_CHECKSUM, nothing written); header or
 * table mismatches return FP8_ERR_BAD_PAYLOAD before anything is enqueued.
 * It allocates no device memory, and no host memory unless it fails. */
fp8_status fp8_sync_install_noalloc(const void* payload_dev, uint64_t bytes, const fp8_sync_entry* dst,
                                    int32_t n, fp8_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Status and diagnostics                                                  */
/* ---------------------------------------------------------------------- */

/* Diagnostic of the failure path shared by every bounded on-device wait:
 * launches one warp that waits on a barrier nothing will complete and gives
 * up after limit_ns (1 us .. 2 s), recording FP8_ERR_TIMEOUT in the status
 * block as a real wait whose peer never signals does.  The next
 * fp8_status_poll() returns FP8_ERR_TIMEOUT and clears it; the context stays
 * usable.  No fault, trap or hang is involved. */
fp8_status fp8_check_wait_expiry(int64_t limit_ns, fp8_stream_t stream);

/* Synchronizes `stream`, reads and clears the current device's status
 * block.  Returns FP8_OK, FP8_ERR_CHECKSUM, FP8_ERR_TIMEOUT or
 * FP8_ERR_INVALID_ARG (device-detected), or FP8_ERR_CUDA. */
fp8_status fp8_status_poll(fp8_stream_t stream);

/* Message describing the last non-OK status returned on this host thread. */
const char* fp8_last_error(void);

/* FP8BS_ABI_VERSION of the loaded library. */
int32_t fp8_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H */
