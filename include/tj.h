/*
 * tj.h - C ABI of the GB300 (sm_103a) TetraJet-v2 NVFP4 linear-layer library.
 *
 * The method: arXiv 2510.27527, "TetraJet-v2: Accurate NVFP4 Training for Large
 * Language Models with Oscillation Suppression and Outlier Control", as given
 * by its technical summary pages (gist.science, nl/es/ja; sections cited as
 * §2.A double-block quantization, §2.B OsciReset, §2.C OutControl).
 *
 * Conventions for every call
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates or frees device memory; scratch space is passed in as
 *     `workspace` with its size from tj_workspace_size().
 *   - Dense bf16/fp32 inputs (x, dy) need only their element alignment; rows that
 *     start on 64-byte boundaries (ld a multiple of 32) take a vectorised load path.
 *     Every other pointer (quantized tensors, outputs, workspace) must be 16-byte
 *     aligned (the workspace 256-byte); violations return TJ_ERR_ALIGN before any
 *     launch.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and never synchronize.  Argument/shape errors are detected on the
 *     host before any launch and leave outputs untouched; a failed launch maps to
 *     TJ_ERR_CUDA.  Device-side bounded waits that run out set a sticky device
 *     flag read by tj_get_device_status().
 *   - Inputs must be finite.  Padded regions of outputs are written (zeros).
 *   - Index arrays (sel, normal_idx, outlier_idx, col_map) are device data: the host
 *     checks their pointers and lengths, not their values.  Their values must lie in
 *     range (a channel index < the input's columns, a col_map entry < the output's
 *     columns) and be distinct, as tj_outlier_calibrate writes them; the kernels read
 *     and write through them unchecked.
 *   - Empty tensors: a tensor with no rows or no columns has no storage, and its
 *     pointers may be NULL.  A call whose outputs are all empty only checks its
 *     arguments.  A product over an empty contraction (K = 0 for a GEMM, no output
 *     features for dX, no tokens for dW) is zero and is written as zeros.  With every
 *     channel an outlier (k = K) normal_idx may be NULL and the NVFP4 parts are empty.
 *
 * Data layouts in HBM
 *   NVFP4 double-block tensor (tj_nvfp4), logical [rows, cols] quantized along
 *   cols (the contraction dimension of the GEMM that consumes it);
 *   rows_p = roundup(rows, 128), cols_p = roundup(cols, 128):
 *     codes  uint8 [rows_p][cols_p/2]   E2M1; element 2j in the LOW nibble of byte j;
 *                                        bit 3 of a code is the sign.
 *     sf     uint8 [rows_p*cols_p/16]   E4M3 inner scales (one per 1x16 group) in the
 *                                        MMA tile layout below.
 *     outer  float [cols_p/128][rows_p] FP32 outer scales (one per 1x128 block),
 *                                        block-major so one block's scales for 128
 *                                        consecutive rows are contiguous.
 *   MX outlier slice (tj_mxfp8), logical [rows, cols] along cols, element format fmt:
 *     codes  uint8 [rows_p][cols_p*bits/8]  packed element codes of `bits` bits each:
 *              E4M3 (8 bits): one byte per element;
 *              E2M3 / E3M2 (6 bits): each row is a little-endian bit stream, element c at
 *                bits 6c .. 6c+5 (16 elements in 12 bytes), sign in the code's bit 5;
 *              E2M1 (4 bits): element 2j in the low nibble of byte j, sign in bit 3.
 *     sf     uint8 [rows_p*cols_p/32]   UE8M0 scales (one per 1x32 group), tile layout.
 *   The packed FP6 / FP4 rows are the tensor core's operand order: the GEMM's TMA copies
 *   expand each 16-element run into the 16-byte shared-memory slot the MMA reads.
 *   Scale tile layout (both formats; B = 16 for NVFP4, 32 for MXFP8): the scales
 *   form tiles of 128 rows x 4 consecutive groups; tile (rt, kt) starts at byte
 *   (rt * (cols_p / (4*B)) + kt) * 512; inside it, the scale of row
 *   rt*128 + 32*i + j (i < 4, j < 32) and group 4*kt + q sits at byte 16*j + 4*i + q.
 *   This is the order in which the block-scaled tensor-core MMA reads its scale
 *   factors from tensor memory, so the GEMM copies tiles without rearranging.
 *
 * Number formats (§2.A): E2M1 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}; E4M3 inner
 * scales; FP32 outer scale s_o = amax_128 / 2688 (2688 = 6 * 448); inner scale =
 * the smallest normal E4M3 value s_i (2^-6 .. 448) whose dequantized top value
 * fl(fl(6 s_i) s_o) is >= amax_16, 448 if none is (decided on dequantized values, so
 * re-quantizing a dequantized tensor gives the same codes and scales, and an OsciReset
 * reset keeps the weight's quantized value); elements x * (1/(s_i s_o)) clamped to 6,
 * rounded to nearest-even (forward) or stochastically (backward).
 */
#ifndef TJ_H
#define TJ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TJ_OK = 0,
    TJ_ERR_INVALID_ARG = 1,   /* null pointer, bad enum, negative size */
    TJ_ERR_SHAPE = 2,         /* inconsistent or unsupported sizes */
    TJ_ERR_ALIGN = 3,         /* pointer or leading dimension misaligned */
    TJ_ERR_UNSUPPORTED = 4,   /* device is not sm_103a-class, or feature not built */
    TJ_ERR_CUDA = 5,          /* a CUDA runtime call or kernel launch failed */
    TJ_ERR_TIMEOUT = 6,       /* a device-side bounded wait ran out (sticky) */
    TJ_ERR_WORKSPACE = 7      /* workspace pointer null or smaller than required */
} tj_status;

typedef enum { TJ_RTN = 0, TJ_SR = 1 } tj_round;
typedef enum { TJ_BF16 = 0, TJ_FP32 = 1 } tj_dtype;

/* NVFP4 double-block tensor (caller-owned device buffers; layout above).  Every call
 * rejects with TJ_ERR_SHAPE an NVFP4 or MXFP8 descriptor whose padded size holds 2^31 or
 * more 128-element blocks (roundup(rows, 128) * roundup(cols, 128) / 128); such a tensor
 * would not fit in device memory together with its source. */
typedef struct {
    uint8_t *codes;
    uint8_t *sf;
    float *outer;
    int64_t rows;
    int64_t cols;
} tj_nvfp4;

/* Element formats of an MX outlier slice (the tensor core's own format numbers).  E4M3 is
 * the FP8 slice (§2.C); E2M3 / E3M2 (FP6) and E2M1 (FP4) serve the mixed FP6 x FP4
 * variant of the slice, which the pages name as a future direction (§5).  E2M3: bias 1,
 * max 7.5; E3M2: bias 3, max 28; E2M1: max 6; no infinities or NaN (OCP MX v1.0). */
typedef enum { TJ_MX_E4M3 = 0, TJ_MX_E2M3 = 3, TJ_MX_E3M2 = 4, TJ_MX_E2M1 = 5 } tj_mx_format;

/* MX outlier slice (caller-owned device buffers; layout above).  fmt is a tj_mx_format;
 * a zero-initialised descriptor is E4M3.  Slices in E2M3 / E3M2 / E2M1 need 32-byte aligned
 * codes (TJ_ERR_ALIGN otherwise); an unknown fmt is TJ_ERR_INVALID_ARG.  Every call that
 * writes a slice writes it in its descriptor's format; every call that reads one decodes
 * its descriptor's format. */
typedef struct {
    uint8_t *codes;
    uint8_t *sf;
    int64_t rows;
    int64_t cols;
    int32_t fmt;
} tj_mxfp8;

/* Philox tags used inside the backward calls (documented for reproducibility):
 * stochastic rounding of dY rows (dX operand), of dY^T rows (dW operand), of the
 * re-aligned W-hat^T and X-hat^T, and the RHT sign vectors of dX and dW. */
#define TJ_TAG_DY_ROW 1u
#define TJ_TAG_DY_COL 2u
#define TJ_TAG_WT 3u
#define TJ_TAG_XT 4u
#define TJ_TAG_RHT_DX 0x100u
#define TJ_TAG_RHT_DW 0x101u

/* ---------------------------------------------------------------------------
 * tj_quantize_nvfp4 - double-block NVFP4 quantization (§2.A), optionally after a
 * 128-point random Hadamard transform (§2.C).
 *
 *   x          device [rows_x, cols_x] bf16 or fp32 (dtype), row stride ld elements.
 *   along_cols 0: output row r = input row r, quantized along the input columns.
 *              1: transposed alignment (§2.A, 1x16 groups of the transposed
 *                 operand): output row c = input column c, quantized along the
 *                 input rows.
 *   sel, n_sel optional (sel may be NULL -> all columns, n_sel ignored): ascending
 *              int32 input-column indices to keep (OutControl's normal channels).
 *              A non-NULL sel with n_sel = 0 keeps no column (the output is empty and
 *              sel is not read).
 *              along_cols=0: they form the compacted contraction (out->cols = n_sel);
 *              along_cols=1: they are the output rows (out->rows = n_sel).
 *   mode       TJ_RTN or TJ_SR.  SR draws 16 bits per element from Philox4x32-10
 *              with key = seed, counter = (e >> 3, tag, 0), e = out_row*cols_p + col.
 *   rht        0/1: apply y = H128 * (d .* x) per 128-block of the quantized axis
 *              (zero-padded), d from Philox(key = seed, counter = (0, 0, rht_tag, 0)).
 *   out        caller-filled tj_nvfp4 whose rows/cols must equal the output shape.
 * Errors: TJ_ERR_INVALID_ARG, TJ_ERR_SHAPE, TJ_ERR_ALIGN, TJ_ERR_CUDA.
 * ------------------------------------------------------------------------- */
tj_status tj_quantize_nvfp4(const void *x, int dtype, int64_t rows_x, int64_t cols_x, int64_t ld,
                            int along_cols, const int32_t *sel, int64_t n_sel, int mode,
                            int rht, uint64_t seed, uint32_t tag, uint32_t rht_tag,
                            tj_nvfp4 *out, void *stream);

/* tj_quantize_mxfp8 - FP8 outlier slice (§2.C "kept in higher precision, e.g.
 * FP8"): E4M3 values with a UE8M0 scale 2^E per 1x32 group, E the smallest
 * integer with 448*2^E >= amax_32, values rounded to nearest-even and saturated.
 * With out->fmt = E2M3 / E3M2 / E2M1 the same rule with that format's maximum (7.5 / 28
 * / 6) in place of 448 (sign of a value that rounds to zero kept, as for E4M3).
 * Same x / along_cols / sel conventions as tj_quantize_nvfp4 (no RHT, no SR). */
tj_status tj_quantize_mxfp8(const void *x, int dtype, int64_t rows_x, int64_t cols_x, int64_t ld,
                            int along_cols, const int32_t *sel, int64_t n_sel,
                            tj_mxfp8 *out, void *stream);

/* tj_quantize_nvfp4_mxfp8 - tj_quantize_nvfp4 and tj_quantize_mxfp8 of the same input
 * from one read: `out` gets the NVFP4 quantization (mode / rht / seed / tags as in
 * tj_quantize_nvfp4) and `out8` the MXFP8 quantization of the same (selected) elements
 * without the transform, both in the same orientation and shape.  The results equal the
 * two separate calls byte for byte.  The backward of a linear layer with outlier channels
 * needs both of dY (§2.A SR operand, §2.C FP8 slice); this halves the reads of dY.
 * Errors as tj_quantize_nvfp4, also when out8's shape differs. */
tj_status tj_quantize_nvfp4_mxfp8(const void *x, int dtype, int64_t rows_x, int64_t cols_x, int64_t ld,
                                  int along_cols, const int32_t *sel, int64_t n_sel, int mode,
                                  int rht, uint64_t seed, uint32_t tag, uint32_t rht_tag,
                                  tj_nvfp4 *out, tj_mxfp8 *out8, void *stream);

/* tj_quantize_split - OutControl split of a forward operand (§2.C: a static set of outlier
 * channels kept in FP8, the others in NVFP4), row-wise, from one read of x:
 *   out  = tj_quantize_nvfp4(x, along_cols=0, sel=normal_idx, TJ_RTN, no RHT)  [rows, n_normal]
 *   out8 = tj_quantize_mxfp8(x, along_cols=0, sel=outlier_idx)                [rows, n_outlier]
 * byte for byte.  normal_idx / outlier_idx are the ascending complementary channel lists
 * of tj_outlier_calibrate (n_normal + n_outlier = cols); out8 may be NULL when
 * n_outlier = 0.  Rows longer than the kernel's shared-memory staging fall back to the two
 * gathering passes.  Errors as tj_quantize_nvfp4. */
tj_status tj_quantize_split(const void *x, int dtype, int64_t rows, int64_t cols, int64_t ld,
                            const int32_t *normal_idx, int64_t n_normal, const int32_t *outlier_idx,
                            int64_t n_outlier, tj_nvfp4 *out, tj_mxfp8 *out8, void *stream);

/* tj_requantize_nvfp4 - transposed re-alignment of a forward NVFP4 operand for the
 * backward (§2.A: the backward estimates with X-hat, the dequantized forward operand, and
 * the 1x16 groups of the transposed weight are re-formed along the new contraction axis):
 * out[c, r] = Q(RHT(X-hat[:, c])) along r, with X-hat[r, c] = (G s_i) s_o of `in`
 * [rows, cols].  out is [cols, rows]; mode / rht / seed / tags as in tj_quantize_nvfp4
 * (element index e = out_row * roundup(rows, 128) + r).  Used inside tj_linear_bwd_*. */
tj_status tj_requantize_nvfp4(const tj_nvfp4 *in, int mode, int rht, uint64_t seed, uint32_t tag, uint32_t rht_tag,
                              tj_nvfp4 *out, void *stream);

/* tj_requantize_mxfp8 - the same re-alignment for an FP8 outlier slice: out[c, r] =
 * Q8(X-hat_O[:, c]) along r (RTN, no RHT), in [rows, cols] -> out [cols, rows].  X-hat_O
 * is decoded in in->fmt and re-quantized in out->fmt. */
tj_status tj_requantize_mxfp8(const tj_mxfp8 *in, tj_mxfp8 *out, void *stream);

/* tj_requantize_nvfp4_mxfp8 - tj_requantize_nvfp4(in, mode, rht, seed, tag, rht_tag, out) and
 * tj_requantize_mxfp8(in8, out8) in one launch: the backward re-alignment of a forward
 * operand and of its outlier slice (§2.A, §2.C).  Alone the slice's few tiles leave the GPU
 * mostly idle; here they run beside the operand's.  Results equal the two calls byte for
 * byte (errors as theirs); used inside tj_linear_bwd_dx / _dw when there are outlier
 * channels. */
tj_status tj_requantize_nvfp4_mxfp8(const tj_nvfp4 *in, int mode, int rht, uint64_t seed, uint32_t tag,
                                    uint32_t rht_tag, tj_nvfp4 *out, const tj_mxfp8 *in8, tj_mxfp8 *out8,
                                    void *stream);

/* tj_rht - standalone random Hadamard transform (§2.C): for each row of x (fp32,
 * [rows, cols], cols a multiple of 128, contiguous) y = H128 * (d .* x) per
 * 128-block, unnormalised, fp32 butterflies in stage order 1, 2, ..., 64.
 * d from Philox(key = seed, counter = (0, 0, tag, 0)).  y may alias x. */
tj_status tj_rht(const float *x, float *y, int64_t rows, int64_t cols, uint64_t seed, uint32_t tag,
                 void *stream);

/* tj_dequantize_nvfp4 - fp32 X-hat = (G * s_i) * s_o of a tj_nvfp4 into y
 * [rows, cols] (row stride ldy).  The value the aligned backward re-quantizes. */
tj_status tj_dequantize_nvfp4(const tj_nvfp4 *q, float *y, int64_t ldy, void *stream);

/* tj_dequantize_mxfp8 - fp32 values (element value x 2^(e - 127), in q->fmt) of a
 * tj_mxfp8 into y [rows, cols] (row stride ldy); exact.  For inspecting the slices (§2.C). */
tj_status tj_dequantize_mxfp8(const tj_mxfp8 *q, float *y, int64_t ldy, void *stream);

/* tj_gemm_nvfp4 - block-scaled FP4 GEMM with FP32 outer-scale promotion:
 *   D[m, n] = alpha * sum_kb sA[m,kb] sB[n,kb] * (sum over the 128 elements of
 *             block kb of  (a s_iA)(b s_iB))  [+ sum over the FP8 slice a8 b8]
 * A [M, K] and B [N, K] are both quantized along K (tcgen05 kind::mxf4nvf4,
 * UE4M3 per 16; optional FP8 part kind::mxf8f6f4, UE8M0 per 32, accumulated into
 * the same tile).  The slice operands may have any two element formats (a8->fmt,
 * b8->fmt: e.g. E2M3 x E2M1, the FP6 x FP4 slice); this holds for every GEMM call.  a8/b8 may be NULL (no FP8 part).  D is row-major [M, N] with
 * row stride ldd, fp32 or bf16 (out_dtype); col_map (may be NULL) scatters
 * column n of the product to column col_map[n] of D.  The product of one 16-group
 * is exact; the FP32 accumulation is the only rounding (within 2e-3 sum|a||b|). */
tj_status tj_gemm_nvfp4(const tj_nvfp4 *a, const tj_nvfp4 *b, const tj_mxfp8 *a8, const tj_mxfp8 *b8,
                        float alpha, void *d, int out_dtype, int64_t ldd, const int32_t *col_map,
                        void *stream);

/* tj_gemm_mxfp8 - FP8 slice GEMM alone: D[m, col_map[n]] = sum a8 b8 (used for the
 * outlier columns of dX and dW, whose outputs are distinct columns). */
tj_status tj_gemm_mxfp8(const tj_mxfp8 *a8, const tj_mxfp8 *b8, void *d, int out_dtype, int64_t ldd,
                        const int32_t *col_map, void *stream);

/* tj_gemm_pair - tj_gemm_nvfp4(a, b, alpha, d, out_dtype, ldd, col_map) without an FP8
 * slice, and tj_gemm_mxfp8(a8, b8, d8, out8_dtype, ldd8, col_map8), in one launch: the
 * FP4 product of a backward pass and its FP8 outlier slice (§2.C) write disjoint column
 * sets (of the same or different outputs), and the FP8 slice alone is too small to fill
 * the GPU.  Same arguments, layouts and errors as the two calls; results are the same. */
tj_status tj_gemm_pair(const tj_nvfp4 *a, const tj_nvfp4 *b, float alpha, void *d, int out_dtype,
                       int64_t ldd, const int32_t *col_map, const tj_mxfp8 *a8, const tj_mxfp8 *b8,
                       void *d8, int out8_dtype, int64_t ldd8, const int32_t *col_map8, void *stream);

/* tj_gemm_pair_f32 - tj_gemm_pair for the case of a weight gradient: both products are fp32
 * and together fill one matrix out [rows][cols] (row pitch ld floats, 16-byte aligned), the
 * FP4 product through col_map (a->rows x b->rows) and the FP8 slice through col_map8
 * (a8->rows x b8->rows), with rows = a->rows = a8->rows and every column of out written by
 * exactly one product (col_map / col_map8 int32 device arrays, both required).
 * Because the call owns all of out, it may zero it and split a long K in two: each half of
 * a tile then adds its fp32 sum into out.  Two additions onto zero commute, so the result
 * is deterministic.  It equals tj_gemm_pair's up to the rounding of that one extra fp32
 * addition (the sum of the halves instead of one running sum).  The split is taken when K
 * has at least 8 stages (2 x 128 FP4 or 128 FP8 elements each) in both products and the
 * halves fill the GPU in fewer rounds.  Errors as tj_gemm_pair; TJ_ERR_SHAPE if the row
 * counts differ, cols < 1 or ld < cols. */
tj_status tj_gemm_pair_f32(const tj_nvfp4 *a, const tj_nvfp4 *b, float alpha, const int32_t *col_map,
                           const tj_mxfp8 *a8, const tj_mxfp8 *b8, const int32_t *col_map8, float *out,
                           int64_t cols, int64_t ld, void *stream);

/* ---------------------------------------------------------------------------
 * tj_linear_fwd - forward of the NVFP4 linear layer (§2: NVFP4 for activations,
 * weights and gradients of every linear layer; §2.A RTN double-block quantization;
 * §2.C static outlier channels kept in FP8):
 *   Y[M, N] = Q(X[:, NC]) Q(W[:, NC])^T + Q8(X[:, O]) Q8(W[:, O])^T
 * The slices take the formats of their descriptors: X's slice is quantized in x8->fmt, and
 * w8 holds W's in w8->fmt (E4M3 both for the FP8 slice; e.g. E2M3 and E2M1 for the
 * FP6 x FP4 variant).
 * x           bf16 [M, K], row stride ldx.
 * wq, w8      W's forward operands: NVFP4 [N, K_N] and FP8 slice [N, k] (w8 NULL iff
 *             k == 0), e.g. from tj_quantize_nvfp4/_mxfp8 with sel = normal_idx /
 *             outlier_idx, or wq from tj_osci_reset when k == 0.
 * normal_idx  int32 [K_N] ascending, outlier_idx int32 [k] ascending (device); both
 *             NULL with k == 0 means no OutControl (K_N = K).
 * xq, x8      caller buffers receiving the saved context X-hat: NVFP4 [M, K_N] and FP8
 *             [M, k] (x8 NULL iff k == 0); the backward reads them (alignment, §2.A).
 * y           [M, N] bf16 or fp32 (out_dtype), row stride ldy.
 * ------------------------------------------------------------------------- */
tj_status tj_linear_fwd(const void *x, int64_t M, int64_t K, int64_t ldx, const tj_nvfp4 *wq,
                        const tj_mxfp8 *w8, const int32_t *normal_idx, const int32_t *outlier_idx,
                        int64_t k, tj_nvfp4 *xq, tj_mxfp8 *x8, void *y, int out_dtype, int64_t ldy,
                        void *stream);

/* tj_linear_bwd_dx - input gradient (§2.A aligned backward with SR; §2.C RHT and
 * FP8 outlier columns):
 *   dX[:, NC] = 2^-7 SR(RHT(dY)) SR(RHT(W-hat_NC^T))^T   (RHT along N, tags above)
 *   dX[:, O]  = Q8(dY) Q8(W-hat_O^T)^T                   (RTN, no RHT)
 * Slice formats: W-hat_O^T keeps w8->fmt and dY's slice takes the partner format (E4M3 for
 * E4M3, E2M3 for E2M1, E2M1 for E2M3 or E3M2), so the slice product is FP8 x FP8 or
 * FP6 x FP4.  The workspace reserves each slice's FP8 size whatever its format.
 * W-hat is read from the forward operands wq / w8 (never the master weight).
 * dy bf16 [M, N] (lddy); dx [M, K] bf16 or fp32 (lddx); seed = per-step Philox key.
 * workspace: at least tj_workspace_size(TJ_OP_BWD_DX, M, N, K, k) bytes, 256-aligned.
 * On return the workspace holds the quantized operands, each buffer starting on a
 * 256-byte boundary in this order: S_dY (tj_nvfp4 [M, N]: codes, sf, outer),
 * S_W (tj_nvfp4 [K_N, N]), and when k > 0 Q8(dY) (tj_mxfp8 [M, N]: codes, sf) and
 * Q8(W-hat_O^T) (tj_mxfp8 [k, N]). */
tj_status tj_linear_bwd_dx(const void *dy, int64_t M, int64_t N, int64_t lddy, const tj_nvfp4 *wq,
                           const tj_mxfp8 *w8, const int32_t *normal_idx, const int32_t *outlier_idx,
                           int64_t k, uint64_t seed, void *dx, int out_dtype, int64_t lddx,
                           void *workspace, size_t ws_bytes, void *stream);

/* tj_linear_bwd_dw - weight gradient:
 *   dW[:, NC] = 2^-7 SR(RHT(dY^T)) SR(RHT(X-hat_NC^T))^T  (RHT along M)
 *   dW[:, O]  = Q8(dY^T) Q8(X-hat_O^T)^T
 * Slice formats: X-hat_O^T keeps x8->fmt and dY^T's slice takes the partner format (as
 * for dX).
 * xq / x8 are the saved forward context of tj_linear_fwd.  dw fp32 [N, K] (lddw).
 * The workspace then holds S_dY^T (tj_nvfp4 [N, M]), S_X (tj_nvfp4 [K_N, M]) and when
 * k > 0 Q8(dY^T) (tj_mxfp8 [N, M]) and Q8(X-hat_O^T) (tj_mxfp8 [k, M]), laid out as for dX.
 * The two products run as one tj_gemm_pair_f32 launch into dw, so a long M (the
 * contraction, tokens) with few output tiles may be split in two (see there). */
tj_status tj_linear_bwd_dw(const void *dy, int64_t M, int64_t N, int64_t lddy, const tj_nvfp4 *xq,
                           const tj_mxfp8 *x8, const int32_t *normal_idx, const int32_t *outlier_idx,
                           int64_t k, uint64_t seed, float *dw, int64_t lddw, void *workspace,
                           size_t ws_bytes, void *stream);

/* tj_linear_bwd_dx_noalloc - the same input gradient as tj_linear_bwd_dx, for callers
 * that cannot allocate device memory when the backward runs (code below the framework's
 * allocator, or deployments that only hand out buffers registered up front).  The paper
 * has no counterpart: this is an interface convenience of the library.
 *   - Takes the same arguments as tj_linear_bwd_dx minus the workspace: the scratch is a
 *     fixed array inside the library, tj_noalloc_scratch_bytes() = 16 MiB, kept resident
 *     on every GPU that loads the library until the process exits.
 *   - Problems whose tj_workspace_size(TJ_OP_BWD_DX, ...) exceeds it return
 *     TJ_ERR_WORKSPACE before any launch.
 *   - Allocates nothing (no cudaMalloc / cudaFree, no allocating library routine).
 *   - Each call looks up the scratch's device address in the current context
 *     (cudaGetSymbolAddress, a host call); nothing is cached, so the call stays valid
 *     after a cudaDeviceReset and under any context, and it may be captured into a
 *     CUDA graph.
 *   - All calls share the one scratch array, which keeps the last call's contents; calls
 *     whose executions overlap on the GPU (other streams, other threads) race on it, so
 *     serialise them.  Nothing needs clearing: each call writes all scratch it reads. */
tj_status tj_linear_bwd_dx_noalloc(const void *dy, int64_t M, int64_t N, int64_t lddy, const tj_nvfp4 *wq,
                                   const tj_mxfp8 *w8, const int32_t *normal_idx, const int32_t *outlier_idx,
                                   int64_t k, uint64_t seed, void *dx, int out_dtype, int64_t lddx, void *stream);
size_t tj_noalloc_scratch_bytes(void);

/* ---------------------------------------------------------------------------
 * The FP8 linear baseline (technical summary §4, efficiency: the pages measure
 * TetraJet-v2's training speed against FP8 training with TransformerEngine).  The
 * same linear layer with every GEMM operand in MXFP8 on the same GPU, so the NVFP4
 * path can be timed against it:
 *   - each operand is E4M3 with one UE8M0 scale per 1x32 block along the contraction
 *     axis of the GEMM that reads it (the format of tj_quantize_mxfp8), rounded to
 *     nearest, quantized from its bf16 source (X, W, dY), as an MXFP8 recipe does;
 *   - no RHT, no stochastic rounding, no outlier channels, no double-block scale;
 *   - the three GEMMs are FP8-only products of the library's GEMM (fp32 accumulation).
 * ------------------------------------------------------------------------- */
/* tj_fp8_linear_fwd:  Y[M, N] = Q8(X) Q8(W)^T.
 * x    bf16 [M, K] (ldx).  w8: MXFP8 [N, K], W along K (tj_quantize_mxfp8(W)).
 * x8   out: MXFP8 [M, K], X along K.  xt8: out, MXFP8 [K, M], X^T along M (the dW
 *      operand, saved for tj_fp8_linear_bwd_dw), or NULL to skip it.
 * y    [M, N] bf16 or fp32 (out_dtype), row stride ldy. */
tj_status tj_fp8_linear_fwd(const void *x, int64_t M, int64_t K, int64_t ldx, const tj_mxfp8 *w8, tj_mxfp8 *x8,
                            tj_mxfp8 *xt8, void *y, int out_dtype, int64_t ldy, void *stream);
/* tj_fp8_linear_bwd_dx:  dX[M, K] = Q8(dY) Q8(W^T)^T, both along N.
 * dy bf16 [M, N] (lddy); wt8 MXFP8 [K, N] = tj_quantize_mxfp8(W, along_cols = 1);
 * dx [M, K] bf16 or fp32 (lddx).  workspace: tj_workspace_size(TJ_OP_FP8_BWD_DX, M, N, K,
 * 0) bytes, 256-aligned; it then holds Q8(dY) (tj_mxfp8 [M, N]: codes, sf). */
tj_status tj_fp8_linear_bwd_dx(const void *dy, int64_t M, int64_t N, int64_t lddy, const tj_mxfp8 *wt8, void *dx,
                               int out_dtype, int64_t lddx, void *workspace, size_t ws_bytes, void *stream);
/* tj_fp8_linear_bwd_dw:  dW[N, K] = Q8(dY^T) Q8(X^T)^T, both along M (tokens).
 * xt8 from tj_fp8_linear_fwd; dw fp32 [N, K] (lddw), written whole (a long M may be
 * split in two, as in tj_gemm_pair_f32).  workspace: tj_workspace_size(TJ_OP_FP8_BWD_DW,
 * M, N, K, 0) bytes, 256-aligned; it then holds Q8(dY^T) (tj_mxfp8 [N, M]). */
tj_status tj_fp8_linear_bwd_dw(const void *dy, int64_t M, int64_t N, int64_t lddy, const tj_mxfp8 *xt8, float *dw,
                               int64_t lddw, void *workspace, size_t ws_bytes, void *stream);

#define TJ_OP_BWD_DX 1
#define TJ_OP_BWD_DW 2
#define TJ_OP_FP8_BWD_DX 3
#define TJ_OP_FP8_BWD_DW 4

/* Bytes of workspace the backward call `op` needs for these sizes (K = K_N + k). */
size_t tj_workspace_size(int op, int64_t M, int64_t N, int64_t K, int64_t k);

/* ---------------------------------------------------------------------------
 * tj_outlier_calibrate - OutControl's static outlier selection (§2.C: the top p%
 * channels by norm, found once in a short calibration window).
 * If x != NULL: sumsq[c] += sum over the batch of x[t, c]^2, fp64, in a fixed order
 * (each 128-token chunk summed in token order, then the chunks in order), so the
 * result is reproducible bit for bit.  x bf16/fp32 [M, K] (ld); M <= 2^20.
 * If finalize: the k channels with the largest sumsq (ties -> lower index) are
 * written ascending to outlier_idx [k], the rest ascending to normal_idx [K - k].
 * sumsq: device fp64 [K], zeroed by the caller before the first batch.
 * ------------------------------------------------------------------------- */
tj_status tj_outlier_calibrate(const void *x, int dtype, int64_t M, int64_t K, int64_t ld,
                               double *sumsq, int finalize, int64_t k, int32_t *outlier_idx,
                               int32_t *normal_idx, void *stream);

/* ---------------------------------------------------------------------------
 * tj_osci_reset - OsciReset (§2.B) over master weights w [rows, cols] (fp32,
 * contiguous), one pass after each optimizer step:
 *   dist_M += |w - w_prev|;  Q = RTN double-block quantization of w (rows along
 *   cols, written to q_out: the next forward's weight operand when k == 0);
 *   dist_Q += |Q-hat - Q-hat_prev| (Q-hat_prev decoded from q_prev);
 *   reset iff track && lr < lr_thr && dist_M > 0 && dist_Q > risk_thr * dist_M:
 *     w <- Q-hat (the centre of its bin), dist_Q = dist_M = 0, mask bit set;
 *   then w_prev <- w.  All in fp32.
 * reset_mask: uint32 [rows][ceil(cols/32)], bit c&31 of word c>>5 of row r; every
 * word is written.  q_out may equal q_prev.  Start tracking with w_prev = w,
 * dist = 0 and q_prev = tj_quantize_nvfp4(w, RTN).
 * ------------------------------------------------------------------------- */
tj_status tj_osci_reset(float *w, float *w_prev, float *dist_q, float *dist_m, const tj_nvfp4 *q_prev,
                        tj_nvfp4 *q_out, uint32_t *reset_mask, int64_t rows, int64_t cols, float lr,
                        float lr_thr, float risk_thr, int track, void *stream);

/* ---------------------------------------------------------------------------
 * tj_adamw_osci_reset - the training-step pass around OsciReset in one sweep over the
 * master weights: the AdamW update of w from its gradient, then tj_osci_reset of the
 * updated w (including its forward quantization into q_out).  The pages apply OsciReset
 * after the optimizer step (§2.B) and name no optimizer; this is AdamW with decoupled
 * weight decay, each step an fp32 round-to-nearest operation in this order:
 *   m <- beta1 m + (1 - beta1) g
 *   v <- beta2 v + (1 - beta2) (g g)
 *   w <- w (1 - lr wd) - (lr / (1 - beta1^t)) (m / (sqrt(v) / sqrt(1 - beta2^t) + eps))
 * The per-step constants (1 - beta1, 1 - beta2, 1 - lr wd, lr / (1 - beta1^t),
 * sqrt(1 - beta2^t)) are formed in double from the fp32 arguments and rounded once.
 * step = t >= 1.  g, m, v: fp32 [rows, cols] contiguous, 16-byte aligned (m, v updated in
 * place; g read only).  w is always written.  The other arguments, the reset and the
 * outputs are as for tj_osci_reset; the learning rate lr is also the one OsciReset
 * compares with lr_thr.  Same as tj_osci_reset applied to the result of the AdamW step,
 * bit for bit, in one pass (one read of w instead of two).
 * ------------------------------------------------------------------------- */
tj_status tj_adamw_osci_reset(float *w, const float *g, float *m, float *v, float *w_prev, float *dist_q,
                              float *dist_m, const tj_nvfp4 *q_prev, tj_nvfp4 *q_out, uint32_t *reset_mask,
                              int64_t rows, int64_t cols, float lr, float beta1, float beta2, float eps,
                              float weight_decay, int64_t step, float lr_thr, float risk_thr, int track,
                              void *stream);

/* Reads (synchronously) and clears the sticky device error flag: TJ_OK, or
 * TJ_ERR_TIMEOUT if a bounded device wait ran out since the last query. */
tj_status tj_get_device_status(void);

/* tj_debug_gemm_fault - test hook of the time-out path (not for production use).  Arms a
 * fault for the next GEMM launch that runs (tj_gemm_*, or one inside tj_linear_* /
 * tj_fp8_linear_*); the launch after it runs normally again:
 *   - skip_stage >= 0: in every CTA the producers never load the operands of that stage
 *     (its index among the CTA's stages, counted over its tiles), so the waits for it run
 *     out; -1: no fault;
 *   - wait_clk > 0: every mbarrier wait of the launch gives up after wait_clk SM clocks
 *     (the default is about 2 s); 0 keeps the default.
 * A launch whose wait runs out stops its work, keeps the protocol of its hardware
 * barriers, drains its copies and tensor-core work, frees its tensor memory and returns;
 * tj_get_device_status then reports TJ_ERR_TIMEOUT, the outputs of that launch are
 * undefined, and later launches are unaffected.  Not thread-safe: arm it and launch from
 * one host thread.  Returns TJ_ERR_INVALID_ARG for skip_stage < -1 or wait_clk < 0. */
tj_status tj_debug_gemm_fault(int skip_stage, int64_t wait_clk);

/* Static description of a status code. */
const char *tj_status_str(tj_status s);

#ifdef __cplusplus
}
#endif
#endif /* TJ_H */
