// api.cu - the C ABI of libtj (declared and documented in include/tj.h):
// argument validation, workspace carving and the composition of the linear
// layer's forward / backward out of the kernels (TetraJet-v2 technical summary
// §2.A aligned backward with SR, §2.C RHT and FP8 outlier channels).
#include <cstring>

#include "tj_common.cuh"
#include "tj_internal.h"

using namespace tj;

namespace {

inline bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
// Dense inputs need only their element alignment (the kernels take a vectorised
// path by themselves when rows are 64-byte aligned).
inline bool al_elem(const void *p, int dtype) {
    return (reinterpret_cast<uintptr_t>(p) & (dtype == TJ_FP32 ? 3 : 1)) == 0;
}

tj_status cuda_status(cudaError_t e) { return e == cudaSuccess ? TJ_OK : TJ_ERR_CUDA; }

#define TJ_TRY(expr)                          \
    do {                                      \
        const cudaError_t e_ = (expr);        \
        if (e_ != cudaSuccess) return TJ_ERR_CUDA; \
    } while (0)

// Fewer than 2^31 128-element blocks per tensor: the row quantizers (k_quant_rows)
// walk the (row, block) pairs of a tensor with 32-bit counters.  Every other index
// (element, byte, scale-tile and MXFP8 group offsets) is formed in 64 bits.
bool blocks_fit(int64_t rows, int64_t cols) {
    const int64_t lim = int64_t(1) << 31;
    if (rows > lim || cols > lim * 128) return false;
    return round_up(rows, 128) * (round_up(cols, 128) / 128) < lim;      // both factors <= 2^31
}

// The column (transposed) quantizers launch one grid row per 128 output columns, and
// a grid has at most 65535 rows: at most 8,388,480 output columns (input rows).
bool cols_grid_fits(int64_t out_cols) { return round_up(out_cols, 128) / 128 <= 65535; }

// An empty tensor (no rows or no columns) has no storage: its pointers may be null.
tj_status check_nv(const tj_nvfp4 *q, int64_t rows, int64_t cols) {
    if (q == nullptr) return TJ_ERR_INVALID_ARG;
    const bool empty = q->rows == 0 || q->cols == 0;
    if (!empty && (q->codes == nullptr || q->sf == nullptr || q->outer == nullptr)) return TJ_ERR_INVALID_ARG;
    if (q->rows != rows || q->cols != cols || rows < 0 || cols < 0) return TJ_ERR_SHAPE;
    if (empty) return TJ_OK;
    if (!blocks_fit(rows, cols)) return TJ_ERR_SHAPE;
    if (!al16(q->codes) || !al16(q->sf) || !al16(q->outer)) return TJ_ERR_ALIGN;
    return TJ_OK;
}

// An MX slice: a known element format; packed FP6 / FP4 codes start on 32 bytes (the
// tensor maps of the packed sub-byte types require it).
tj_status check_mx(const tj_mxfp8 *q, int64_t rows, int64_t cols) {
    if (q == nullptr) return TJ_ERR_INVALID_ARG;
    const bool empty = q->rows == 0 || q->cols == 0;
    if (!empty && (q->codes == nullptr || q->sf == nullptr)) return TJ_ERR_INVALID_ARG;
    if (!mx_fmt_valid(q->fmt)) return TJ_ERR_INVALID_ARG;
    if (q->rows != rows || q->cols != cols || rows < 0 || cols < 0) return TJ_ERR_SHAPE;
    if (empty) return TJ_OK;
    if (!blocks_fit(rows, cols)) return TJ_ERR_SHAPE;
    if (!al16(q->codes) || !al16(q->sf)) return TJ_ERR_ALIGN;
    if (q->fmt != kMxE4M3 && (reinterpret_cast<uintptr_t>(q->codes) & 31) != 0) return TJ_ERR_ALIGN;
    return TJ_OK;
}

// Format of dY's slice in a backward product whose other slice operand has format f: the
// FP8 slice stays FP8 x FP8, the FP6 / FP4 formats pair up as FP6 x FP4.
int slice_partner(int f) { return f == kMxE4M3 ? kMxE4M3 : (f == kMxE2M1 ? kMxE2M3 : kMxE2M1); }

int64_t nv_bytes(int64_t rows, int64_t cols) {
    const int64_t rp = round_up(rows, 128), cp = round_up(cols, 128);
    return round_up(rp * cp / 2, 256) + round_up(rp * cp / 16, 256) + round_up(rp * (cp / 128) * 4, 256);
}
int64_t mx_bytes(int64_t rows, int64_t cols) {
    const int64_t rp = round_up(rows, 128), cp = round_up(cols, 128);
    return round_up(rp * cp, 256) + round_up(rp * cp / 32, 256);
}

// Carve an NVFP4 / MXFP8 tensor out of a workspace cursor.
tj_nvfp4 carve_nv(uint8_t *&cur, int64_t rows, int64_t cols) {
    const int64_t rp = round_up(rows, 128), cp = round_up(cols, 128);
    tj_nvfp4 q;
    q.codes = cur;
    cur += round_up(rp * cp / 2, 256);
    q.sf = cur;
    cur += round_up(rp * cp / 16, 256);
    q.outer = reinterpret_cast<float *>(cur);
    cur += round_up(rp * (cp / 128) * 4, 256);
    q.rows = rows;
    q.cols = cols;
    return q;
}
// (the FP8 size is reserved whatever the format, so the workspace layout does not depend on it)
tj_mxfp8 carve_mx(uint8_t *&cur, int64_t rows, int64_t cols, int fmt = kMxE4M3) {
    const int64_t rp = round_up(rows, 128), cp = round_up(cols, 128);
    tj_mxfp8 q;
    q.codes = cur;
    cur += round_up(rp * cp, 256);
    q.sf = cur;
    cur += round_up(rp * cp / 32, 256);
    q.rows = rows;
    q.cols = cols;
    q.fmt = fmt;
    return q;
}

// A dense input: x may be null only when it has no elements.
bool dense_ok(const void *x, int dtype, int64_t ld, int64_t rows, int64_t cols) {
    return (x != nullptr || rows == 0 || cols == 0) && (dtype == TJ_BF16 || dtype == TJ_FP32) && ld >= cols;
}

}  // namespace

extern "C" {

const char *tj_status_str(tj_status s) {
    switch (s) {
        case TJ_OK: return "ok";
        case TJ_ERR_INVALID_ARG: return "invalid argument";
        case TJ_ERR_SHAPE: return "inconsistent or unsupported shape";
        case TJ_ERR_ALIGN: return "pointer or leading dimension misaligned";
        case TJ_ERR_UNSUPPORTED: return "unsupported device or feature";
        case TJ_ERR_CUDA: return "CUDA error";
        case TJ_ERR_TIMEOUT: return "device-side wait timed out";
        case TJ_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

tj_status tj_get_device_status(void) {
    const unsigned int v = read_and_clear_device_error();
    if (v == 0xFFFFFFFFu) return TJ_ERR_CUDA;
    return v ? TJ_ERR_TIMEOUT : TJ_OK;
}

tj_status tj_quantize_nvfp4(const void *x, int dtype, int64_t rows_x, int64_t cols_x, int64_t ld, int along_cols,
                            const int32_t *sel, int64_t n_sel, int mode, int rht, uint64_t seed, uint32_t tag,
                            uint32_t rht_tag, tj_nvfp4 *out, void *stream) {
    if (rows_x < 0 || cols_x < 0 || (mode != TJ_RTN && mode != TJ_SR) || out == nullptr) return TJ_ERR_INVALID_ARG;
    if (!dense_ok(x, dtype, ld, rows_x, cols_x)) return TJ_ERR_INVALID_ARG;
    if (!al_elem(x, dtype)) return TJ_ERR_ALIGN;
    const int64_t ncols = sel ? n_sel : cols_x;
    if (sel && (n_sel < 0 || n_sel > cols_x)) return TJ_ERR_SHAPE;
    const int64_t orows = along_cols ? ncols : rows_x, ocols = along_cols ? rows_x : ncols;
    if (along_cols && !cols_grid_fits(ocols)) return TJ_ERR_SHAPE;
    const tj_status st = check_nv(out, orows, ocols);
    if (st != TJ_OK) return st;
    if (orows == 0 || ocols == 0) return TJ_OK;
    return cuda_status(launch_quant_nv_dense(x, dtype, rows_x, ncols, ld, along_cols, sel, mode, rht, seed, tag,
                                             rht_tag, *out, static_cast<cudaStream_t>(stream)));
}

tj_status tj_quantize_mxfp8(const void *x, int dtype, int64_t rows_x, int64_t cols_x, int64_t ld, int along_cols,
                            const int32_t *sel, int64_t n_sel, tj_mxfp8 *out, void *stream) {
    if (rows_x < 0 || cols_x < 0 || out == nullptr) return TJ_ERR_INVALID_ARG;
    if (!dense_ok(x, dtype, ld, rows_x, cols_x)) return TJ_ERR_INVALID_ARG;
    if (!al_elem(x, dtype)) return TJ_ERR_ALIGN;
    const int64_t ncols = sel ? n_sel : cols_x;
    if (sel && (n_sel < 0 || n_sel > cols_x)) return TJ_ERR_SHAPE;
    const int64_t orows = along_cols ? ncols : rows_x, ocols = along_cols ? rows_x : ncols;
    if (along_cols && !cols_grid_fits(ocols)) return TJ_ERR_SHAPE;
    const tj_status st = check_mx(out, orows, ocols);
    if (st != TJ_OK) return st;
    if (orows == 0 || ocols == 0) return TJ_OK;
    return cuda_status(launch_quant_mx_dense(x, dtype, rows_x, ncols, ld, along_cols, sel, *out,
                                             static_cast<cudaStream_t>(stream)));
}

tj_status tj_quantize_nvfp4_mxfp8(const void *x, int dtype, int64_t rows_x, int64_t cols_x, int64_t ld,
                                  int along_cols, const int32_t *sel, int64_t n_sel, int mode, int rht,
                                  uint64_t seed, uint32_t tag, uint32_t rht_tag, tj_nvfp4 *out, tj_mxfp8 *out8,
                                  void *stream) {
    if (rows_x < 0 || cols_x < 0 || (mode != TJ_RTN && mode != TJ_SR) || out == nullptr || out8 == nullptr)
        return TJ_ERR_INVALID_ARG;
    if (!dense_ok(x, dtype, ld, rows_x, cols_x)) return TJ_ERR_INVALID_ARG;
    if (!al_elem(x, dtype)) return TJ_ERR_ALIGN;
    const int64_t ncols = sel ? n_sel : cols_x;
    if (sel && (n_sel < 0 || n_sel > cols_x)) return TJ_ERR_SHAPE;
    const int64_t orows = along_cols ? ncols : rows_x, ocols = along_cols ? rows_x : ncols;
    if (along_cols && !cols_grid_fits(ocols)) return TJ_ERR_SHAPE;
    tj_status st = check_nv(out, orows, ocols);
    if (st == TJ_OK) st = check_mx(out8, orows, ocols);
    if (st != TJ_OK) return st;
    if (orows == 0 || ocols == 0) return TJ_OK;
    return cuda_status(launch_quant_dual_dense(x, dtype, rows_x, ncols, ld, along_cols, sel, mode, rht, seed, tag,
                                               rht_tag, *out, *out8, static_cast<cudaStream_t>(stream)));
}

tj_status tj_quantize_split(const void *x, int dtype, int64_t rows, int64_t cols, int64_t ld,
                            const int32_t *normal_idx, int64_t n_normal, const int32_t *outlier_idx,
                            int64_t n_outlier, tj_nvfp4 *out, tj_mxfp8 *out8, void *stream) {
    if (rows < 0 || cols < 0 || n_normal < 0 || n_outlier < 0 || out == nullptr) return TJ_ERR_INVALID_ARG;
    if (n_normal + n_outlier != cols) return TJ_ERR_SHAPE;
    if ((n_normal > 0 && normal_idx == nullptr) || (n_outlier > 0 && (outlier_idx == nullptr || out8 == nullptr)))
        return TJ_ERR_INVALID_ARG;
    if (!dense_ok(x, dtype, ld, rows, cols)) return TJ_ERR_INVALID_ARG;
    if (!al_elem(x, dtype)) return TJ_ERR_ALIGN;
    tj_status st = check_nv(out, rows, n_normal);
    if (st == TJ_OK && n_outlier > 0) st = check_mx(out8, rows, n_outlier);
    if (st != TJ_OK) return st;
    if (rows == 0 || cols == 0) return TJ_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const tj_mxfp8 none{};
    const cudaError_t e = launch_quant_split(x, dtype, rows, cols, ld, normal_idx, n_normal, outlier_idx, n_outlier,
                                             *out, n_outlier > 0 ? *out8 : none, s);
    if (e != cudaErrorNotSupported) return cuda_status(e);
    // rows too long to stage: gather the two channel sets separately
    TJ_TRY(launch_quant_nv_dense(x, dtype, rows, n_normal, ld, 0, normal_idx, TJ_RTN, 0, 0, 0, 0, *out, s));
    if (n_outlier > 0) TJ_TRY(launch_quant_mx_dense(x, dtype, rows, n_outlier, ld, 0, outlier_idx, *out8, s));
    return TJ_OK;
}

tj_status tj_requantize_nvfp4(const tj_nvfp4 *in, int mode, int rht, uint64_t seed, uint32_t tag, uint32_t rht_tag,
                              tj_nvfp4 *out, void *stream) {
    if (in == nullptr || out == nullptr || (mode != TJ_RTN && mode != TJ_SR)) return TJ_ERR_INVALID_ARG;
    tj_status st = check_nv(in, in->rows, in->cols);
    if (st == TJ_OK) st = check_nv(out, in->cols, in->rows);
    if (st != TJ_OK) return st;
    if (!cols_grid_fits(in->rows)) return TJ_ERR_SHAPE;
    if (in->rows == 0 || in->cols == 0) return TJ_OK;
    return cuda_status(launch_realign_nv(*in, *out, mode, rht, seed, tag, rht_tag, static_cast<cudaStream_t>(stream)));
}

tj_status tj_requantize_mxfp8(const tj_mxfp8 *in, tj_mxfp8 *out, void *stream) {
    if (in == nullptr || out == nullptr) return TJ_ERR_INVALID_ARG;
    tj_status st = check_mx(in, in->rows, in->cols);
    if (st == TJ_OK) st = check_mx(out, in->cols, in->rows);
    if (st != TJ_OK) return st;
    if (!cols_grid_fits(in->rows)) return TJ_ERR_SHAPE;
    if (in->rows == 0 || in->cols == 0) return TJ_OK;
    return cuda_status(launch_realign_mx(*in, *out, static_cast<cudaStream_t>(stream)));
}

tj_status tj_requantize_nvfp4_mxfp8(const tj_nvfp4 *in, int mode, int rht, uint64_t seed, uint32_t tag,
                                    uint32_t rht_tag, tj_nvfp4 *out, const tj_mxfp8 *in8, tj_mxfp8 *out8,
                                    void *stream) {
    if (in == nullptr || out == nullptr || in8 == nullptr || out8 == nullptr || (mode != TJ_RTN && mode != TJ_SR))
        return TJ_ERR_INVALID_ARG;
    tj_status st = check_nv(in, in->rows, in->cols);
    if (st == TJ_OK) st = check_nv(out, in->cols, in->rows);
    if (st == TJ_OK) st = check_mx(in8, in8->rows, in8->cols);
    if (st == TJ_OK) st = check_mx(out8, in8->cols, in8->rows);
    if (st != TJ_OK) return st;
    if (!cols_grid_fits(in->rows) || !cols_grid_fits(in8->rows)) return TJ_ERR_SHAPE;
    // (an empty part leaves the other part alone in the launch)
    return cuda_status(launch_realign_pair(*in, *out, mode, rht, seed, tag, rht_tag, *in8, *out8,
                                           static_cast<cudaStream_t>(stream)));
}

tj_status tj_rht(const float *x, float *y, int64_t rows, int64_t cols, uint64_t seed, uint32_t tag, void *stream) {
    if (rows < 0 || cols < 0 || ((x == nullptr || y == nullptr) && rows > 0 && cols > 0)) return TJ_ERR_INVALID_ARG;
    if (cols % 128 != 0) return TJ_ERR_SHAPE;
    if (!al16(x) || !al16(y)) return TJ_ERR_ALIGN;
    if (rows == 0 || cols == 0) return TJ_OK;
    return cuda_status(launch_rht(x, y, rows, cols, seed, tag, static_cast<cudaStream_t>(stream)));
}

tj_status tj_dequantize_nvfp4(const tj_nvfp4 *q, float *y, int64_t ldy, void *stream) {
    if (q == nullptr || (y == nullptr && q->rows > 0 && q->cols > 0)) return TJ_ERR_INVALID_ARG;
    const tj_status st = check_nv(q, q->rows, q->cols);
    if (st != TJ_OK) return st;
    if (ldy < q->cols) return TJ_ERR_SHAPE;
    return cuda_status(launch_dequant_nv(*q, y, ldy, static_cast<cudaStream_t>(stream)));
}

tj_status tj_dequantize_mxfp8(const tj_mxfp8 *q, float *y, int64_t ldy, void *stream) {
    if (q == nullptr || (y == nullptr && q->rows > 0 && q->cols > 0)) return TJ_ERR_INVALID_ARG;
    const tj_status st = check_mx(q, q->rows, q->cols);
    if (st != TJ_OK) return st;
    if (ldy < q->cols) return TJ_ERR_SHAPE;
    return cuda_status(launch_dequant_mx(*q, y, ldy, static_cast<cudaStream_t>(stream)));
}

tj_status tj_gemm_nvfp4(const tj_nvfp4 *a, const tj_nvfp4 *b, const tj_mxfp8 *a8, const tj_mxfp8 *b8, float alpha,
                        void *d, int out_dtype, int64_t ldd, const int32_t *col_map, void *stream) {
    if (a == nullptr || b == nullptr || (d == nullptr && a->rows > 0 && b->rows > 0)) return TJ_ERR_INVALID_ARG;
    if (out_dtype != TJ_BF16 && out_dtype != TJ_FP32) return TJ_ERR_INVALID_ARG;
    tj_status st = check_nv(a, a->rows, a->cols);
    if (st == TJ_OK) st = check_nv(b, b->rows, a->cols);
    if (st != TJ_OK) return st;
    if ((a8 == nullptr) != (b8 == nullptr)) return TJ_ERR_INVALID_ARG;
    if (a8 != nullptr) {
        st = check_mx(a8, a->rows, a8->cols);
        if (st == TJ_OK) st = check_mx(b8, b->rows, a8->cols);
        if (st != TJ_OK) return st;
    }
    if (ldd < (col_map ? 1 : b->rows) || !al16(d)) return ldd < 1 ? TJ_ERR_SHAPE : TJ_ERR_ALIGN;
    return cuda_status(launch_gemm(a, b, a8, b8, alpha, d, out_dtype, ldd, a->rows, b->rows, col_map,
                                   static_cast<cudaStream_t>(stream)));
}

tj_status tj_gemm_mxfp8(const tj_mxfp8 *a8, const tj_mxfp8 *b8, void *d, int out_dtype, int64_t ldd,
                        const int32_t *col_map, void *stream) {
    if (a8 == nullptr || b8 == nullptr || (d == nullptr && a8->rows > 0 && b8->rows > 0)) return TJ_ERR_INVALID_ARG;
    if (out_dtype != TJ_BF16 && out_dtype != TJ_FP32) return TJ_ERR_INVALID_ARG;
    tj_status st = check_mx(a8, a8->rows, a8->cols);
    if (st == TJ_OK) st = check_mx(b8, b8->rows, a8->cols);
    if (st != TJ_OK) return st;
    if (!al16(d)) return TJ_ERR_ALIGN;
    return cuda_status(launch_gemm(nullptr, nullptr, a8, b8, 1.0f, d, out_dtype, ldd, a8->rows, b8->rows, col_map,
                                   static_cast<cudaStream_t>(stream)));
}

tj_status tj_gemm_pair(const tj_nvfp4 *a, const tj_nvfp4 *b, float alpha, void *d, int out_dtype, int64_t ldd,
                       const int32_t *col_map, const tj_mxfp8 *a8, const tj_mxfp8 *b8, void *d8, int out8_dtype,
                       int64_t ldd8, const int32_t *col_map8, void *stream) {
    if (a == nullptr || b == nullptr || a8 == nullptr || b8 == nullptr) return TJ_ERR_INVALID_ARG;
    if ((d == nullptr && a->rows > 0 && b->rows > 0) || (d8 == nullptr && a8->rows > 0 && b8->rows > 0))
        return TJ_ERR_INVALID_ARG;
    if ((out_dtype != TJ_BF16 && out_dtype != TJ_FP32) || (out8_dtype != TJ_BF16 && out8_dtype != TJ_FP32))
        return TJ_ERR_INVALID_ARG;
    tj_status st = check_nv(a, a->rows, a->cols);
    if (st == TJ_OK) st = check_nv(b, b->rows, a->cols);
    if (st == TJ_OK) st = check_mx(a8, a8->rows, a8->cols);
    if (st == TJ_OK) st = check_mx(b8, b8->rows, a8->cols);
    if (st != TJ_OK) return st;
    if (ldd < (col_map ? 1 : b->rows) || ldd8 < (col_map8 ? 1 : b8->rows)) return TJ_ERR_SHAPE;
    if (!al16(d) || !al16(d8)) return TJ_ERR_ALIGN;
    return cuda_status(launch_gemm_pair(a, b, alpha, d, out_dtype, ldd, a->rows, b->rows, col_map, a8, b8, d8,
                                        out8_dtype, ldd8, a8->rows, b8->rows, col_map8,
                                        static_cast<cudaStream_t>(stream)));
}

tj_status tj_gemm_pair_f32(const tj_nvfp4 *a, const tj_nvfp4 *b, float alpha, const int32_t *col_map,
                           const tj_mxfp8 *a8, const tj_mxfp8 *b8, const int32_t *col_map8, float *out,
                           int64_t cols, int64_t ld, void *stream) {
    if (a == nullptr || b == nullptr || a8 == nullptr || b8 == nullptr) return TJ_ERR_INVALID_ARG;
    if ((col_map == nullptr && b->rows > 0) || (col_map8 == nullptr && b8->rows > 0) ||
        (out == nullptr && a->rows > 0 && cols > 0))
        return TJ_ERR_INVALID_ARG;
    tj_status st = check_nv(a, a->rows, a->cols);
    if (st == TJ_OK) st = check_nv(b, b->rows, a->cols);
    if (st == TJ_OK) st = check_mx(a8, a8->rows, a8->cols);
    if (st == TJ_OK) st = check_mx(b8, b8->rows, a8->cols);
    if (st != TJ_OK) return st;
    if (a8->rows != a->rows || cols < 0 || ld < cols || b->rows + b8->rows > cols) return TJ_ERR_SHAPE;
    if (!al16(out)) return TJ_ERR_ALIGN;
    const SplitRegion whole{out, a->rows, cols, ld};
    return cuda_status(launch_gemm_pair(a, b, alpha, out, TJ_FP32, ld, a->rows, b->rows, col_map, a8, b8, out, TJ_FP32,
                                        ld, a8->rows, b8->rows, col_map8, static_cast<cudaStream_t>(stream), &whole));
}

size_t tj_workspace_size(int op, int64_t M, int64_t N, int64_t K, int64_t k) {
    if (M < 0 || N < 0 || K < 0 || k < 0 || k > K) return 0;
    const int64_t kn = K - k;
    int64_t b = 0;
    if (op == TJ_OP_BWD_DX) {
        b = nv_bytes(M, N) + nv_bytes(kn, N);
        if (k > 0) b += mx_bytes(M, N) + mx_bytes(k, N);
    } else if (op == TJ_OP_BWD_DW) {
        b = nv_bytes(N, M) + nv_bytes(kn, M);
        if (k > 0) b += mx_bytes(N, M) + mx_bytes(k, M);
    } else if (op == TJ_OP_FP8_BWD_DX) {
        b = mx_bytes(M, N);
    } else if (op == TJ_OP_FP8_BWD_DW) {
        b = mx_bytes(N, M);
    }
    return (size_t)b;
}

tj_status tj_linear_fwd(const void *x, int64_t M, int64_t K, int64_t ldx, const tj_nvfp4 *wq, const tj_mxfp8 *w8,
                        const int32_t *normal_idx, const int32_t *outlier_idx, int64_t k, tj_nvfp4 *xq,
                        tj_mxfp8 *x8, void *y, int out_dtype, int64_t ldy, void *stream) {
    if (wq == nullptr || xq == nullptr || M < 0 || K < 0 || k < 0 || k > K) return TJ_ERR_INVALID_ARG;
    if ((x == nullptr && M > 0 && K > 0) || (y == nullptr && M > 0 && wq->rows > 0)) return TJ_ERR_INVALID_ARG;
    if (out_dtype != TJ_BF16 && out_dtype != TJ_FP32) return TJ_ERR_INVALID_ARG;
    // (every channel an outlier: there is no normal channel to list)
    if (k > 0 && ((k < K && normal_idx == nullptr) || outlier_idx == nullptr || w8 == nullptr || x8 == nullptr))
        return TJ_ERR_INVALID_ARG;
    if (!al_elem(x, TJ_BF16) || !al16(y)) return TJ_ERR_ALIGN;
    if (ldx < K) return TJ_ERR_SHAPE;
    const int64_t kn = K - k, N = wq->rows;
    tj_status st = check_nv(wq, N, kn);
    if (st == TJ_OK) st = check_nv(xq, M, kn);
    if (st == TJ_OK && k > 0) st = check_mx(w8, N, k);
    if (st == TJ_OK && k > 0) st = check_mx(x8, M, k);
    if (st != TJ_OK) return st;
    if (ldy < N) return TJ_ERR_SHAPE;
    if (M == 0) return TJ_OK;                          // no tokens: nothing to quantize or write
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (k > 0) {
        // the OutControl split of X from one read (two gathering passes if a row is too long)
        const cudaError_t e = launch_quant_split(x, TJ_BF16, M, K, ldx, normal_idx, kn, outlier_idx, k, *xq, *x8, s);
        if (e != cudaErrorNotSupported) {
            TJ_TRY(e);
        } else {
            TJ_TRY(launch_quant_nv_dense(x, TJ_BF16, M, kn, ldx, 0, normal_idx, TJ_RTN, 0, 0, 0, 0, *xq, s));
            TJ_TRY(launch_quant_mx_dense(x, TJ_BF16, M, k, ldx, 0, outlier_idx, *x8, s));
        }
    } else {
        TJ_TRY(launch_quant_nv_dense(x, TJ_BF16, M, kn, ldx, 0, nullptr, TJ_RTN, 0, 0, 0, 0, *xq, s));
    }
    TJ_TRY(launch_gemm(xq, wq, k > 0 ? x8 : nullptr, k > 0 ? w8 : nullptr, 1.0f, y, out_dtype, ldy, M, N, nullptr, s));
    return TJ_OK;
}

tj_status tj_linear_bwd_dx(const void *dy, int64_t M, int64_t N, int64_t lddy, const tj_nvfp4 *wq,
                           const tj_mxfp8 *w8, const int32_t *normal_idx, const int32_t *outlier_idx, int64_t k,
                           uint64_t seed, void *dx, int out_dtype, int64_t lddx, void *workspace, size_t ws_bytes,
                           void *stream) {
    if (wq == nullptr || M < 0 || N < 0 || k < 0) return TJ_ERR_INVALID_ARG;
    const int64_t kn = wq->cols, K = kn + k;
    if ((dy == nullptr && M > 0 && N > 0) || (dx == nullptr && M > 0 && K > 0)) return TJ_ERR_INVALID_ARG;
    if (out_dtype != TJ_BF16 && out_dtype != TJ_FP32) return TJ_ERR_INVALID_ARG;
    if (k > 0 && ((kn > 0 && normal_idx == nullptr) || outlier_idx == nullptr || w8 == nullptr))
        return TJ_ERR_INVALID_ARG;
    if (!al_elem(dy, TJ_BF16) || !al16(dx)) return TJ_ERR_ALIGN;
    tj_status st = check_nv(wq, N, kn);
    if (st == TJ_OK && k > 0) st = check_mx(w8, N, k);
    if (st != TJ_OK) return st;
    if (lddy < N || lddx < K || !cols_grid_fits(N)) return TJ_ERR_SHAPE;
    const size_t need = tj_workspace_size(TJ_OP_BWD_DX, M, N, K, k);
    if ((workspace == nullptr && need > 0) || ws_bytes < need) return TJ_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return TJ_ERR_ALIGN;
    if (M == 0 || K == 0) return TJ_OK;                // dX is empty (N = 0: dX = 0, an empty contraction)
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *cur = static_cast<uint8_t *>(workspace);
    tj_nvfp4 s_dy = carve_nv(cur, M, N);
    tj_nvfp4 s_w = carve_nv(cur, kn, N);
    tj_mxfp8 q8_dy{}, q8_w{};
    if (k > 0) {
        // W-hat_O^T keeps the forward slice's format, dY takes its partner
        q8_dy = carve_mx(cur, M, N, slice_partner(w8->fmt));
        q8_w = carve_mx(cur, k, N, w8->fmt);
    }
    // dY rows: RHT along N + SR (the dX operand), and with an outlier slice also the
    // MXFP8 rows of dY, from one read; W-hat^T re-aligned with the same signs
    if (k > 0)
        TJ_TRY(launch_quant_dual_dense(dy, TJ_BF16, M, N, lddy, 0, nullptr, TJ_SR, 1, seed, TJ_TAG_DY_ROW,
                                       TJ_TAG_RHT_DX, s_dy, q8_dy, s));
    else
        TJ_TRY(launch_quant_nv_dense(dy, TJ_BF16, M, N, lddy, 0, nullptr, TJ_SR, 1, seed, TJ_TAG_DY_ROW,
                                     TJ_TAG_RHT_DX, s_dy, s));
    if (k > 0 && kn > 0) {
        // W-hat^T and its slice re-aligned in one launch
        TJ_TRY(launch_realign_pair(*wq, s_w, TJ_SR, 1, seed, TJ_TAG_WT, TJ_TAG_RHT_DX, *w8, q8_w, s));
    } else {
        TJ_TRY(launch_realign_nv(*wq, s_w, TJ_SR, 1, seed, TJ_TAG_WT, TJ_TAG_RHT_DX, s));
        if (k > 0) TJ_TRY(launch_realign_mx(*w8, q8_w, s));
    }
    if (k > 0) {
        // the FP4 product (normal columns of dX) and the slice (outlier columns) in one launch
        TJ_TRY(launch_gemm_pair(&s_dy, &s_w, 0.0078125f, dx, out_dtype, lddx, M, kn, normal_idx, &q8_dy, &q8_w, dx,
                                out_dtype, lddx, M, k, outlier_idx, s));
    } else {
        TJ_TRY(launch_gemm(&s_dy, &s_w, nullptr, nullptr, 0.0078125f, dx, out_dtype, lddx, M, kn, nullptr, s));
    }
    return TJ_OK;
}

tj_status tj_linear_bwd_dw(const void *dy, int64_t M, int64_t N, int64_t lddy, const tj_nvfp4 *xq,
                           const tj_mxfp8 *x8, const int32_t *normal_idx, const int32_t *outlier_idx, int64_t k,
                           uint64_t seed, float *dw, int64_t lddw, void *workspace, size_t ws_bytes, void *stream) {
    if (xq == nullptr || M < 0 || N < 0 || k < 0) return TJ_ERR_INVALID_ARG;
    const int64_t kn = xq->cols, K = kn + k;
    if ((dy == nullptr && M > 0 && N > 0) || (dw == nullptr && N > 0 && K > 0)) return TJ_ERR_INVALID_ARG;
    if (k > 0 && ((kn > 0 && normal_idx == nullptr) || outlier_idx == nullptr || x8 == nullptr))
        return TJ_ERR_INVALID_ARG;
    if (!al_elem(dy, TJ_BF16) || !al16(dw)) return TJ_ERR_ALIGN;
    tj_status st = check_nv(xq, M, kn);
    if (st == TJ_OK && k > 0) st = check_mx(x8, M, k);
    if (st != TJ_OK) return st;
    if (lddy < N || lddw < K || !cols_grid_fits(M)) return TJ_ERR_SHAPE;
    const size_t need = tj_workspace_size(TJ_OP_BWD_DW, M, N, K, k);
    if ((workspace == nullptr && need > 0) || ws_bytes < need) return TJ_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return TJ_ERR_ALIGN;
    if (N == 0 || K == 0) return TJ_OK;                // dW is empty (M = 0: dW = 0, an empty contraction)
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *cur = static_cast<uint8_t *>(workspace);
    tj_nvfp4 s_dy = carve_nv(cur, N, M);
    tj_nvfp4 s_x = carve_nv(cur, kn, M);
    tj_mxfp8 q8_dy{}, q8_x{};
    if (k > 0) {
        // X-hat_O^T keeps the forward slice's format, dY^T takes its partner
        q8_dy = carve_mx(cur, N, M, slice_partner(x8->fmt));
        q8_x = carve_mx(cur, k, M, x8->fmt);
    }
    // dY^T rows (RHT along M + SR), and with an outlier slice also the MXFP8 rows of
    // dY^T, from one read; X-hat^T re-aligned with the same signs
    if (k > 0)
        TJ_TRY(launch_quant_dual_dense(dy, TJ_BF16, M, N, lddy, 1, nullptr, TJ_SR, 1, seed, TJ_TAG_DY_COL,
                                       TJ_TAG_RHT_DW, s_dy, q8_dy, s));
    else
        TJ_TRY(launch_quant_nv_dense(dy, TJ_BF16, M, N, lddy, 1, nullptr, TJ_SR, 1, seed, TJ_TAG_DY_COL,
                                     TJ_TAG_RHT_DW, s_dy, s));
    if (k > 0 && kn > 0) {
        // X-hat^T and its slice re-aligned in one launch
        TJ_TRY(launch_realign_pair(*xq, s_x, TJ_SR, 1, seed, TJ_TAG_XT, TJ_TAG_RHT_DW, *x8, q8_x, s));
    } else {
        TJ_TRY(launch_realign_nv(*xq, s_x, TJ_SR, 1, seed, TJ_TAG_XT, TJ_TAG_RHT_DW, s));
        if (k > 0) TJ_TRY(launch_realign_mx(*x8, q8_x, s));
    }
    // dW [N][K] is fp32 and covered by the launch, so a long-K launch may split K in two
    const SplitRegion whole_dw{dw, N, K, lddw};
    if (k > 0) {
        // the FP4 product (normal columns of dW) and the slice (outlier columns) in one launch
        TJ_TRY(launch_gemm_pair(&s_dy, &s_x, 0.0078125f, dw, TJ_FP32, lddw, N, kn, normal_idx, &q8_dy, &q8_x, dw,
                                TJ_FP32, lddw, N, k, outlier_idx, s, &whole_dw));
    } else {
        TJ_TRY(launch_gemm(&s_dy, &s_x, nullptr, nullptr, 0.0078125f, dw, TJ_FP32, lddw, N, kn, nullptr, s, &whole_dw));
    }
    return TJ_OK;
}

// ---------------------------------------------------------------------------
// The FP8 linear baseline the pages compare against (technical summary §4: training
// speed vs FP8 TransformerEngine): every GEMM operand MXFP8 (E4M3, UE8M0 per 1x32
// along its contraction axis, round to nearest), quantized from its bf16 source; no
// RHT, no stochastic rounding, no outlier split.  The GEMMs are FP8-only products of
// the same kernel, whose power-of-two scales the tensor core applies itself.
// ---------------------------------------------------------------------------
tj_status tj_fp8_linear_fwd(const void *x, int64_t M, int64_t K, int64_t ldx, const tj_mxfp8 *w8, tj_mxfp8 *x8,
                            tj_mxfp8 *xt8, void *y, int out_dtype, int64_t ldy, void *stream) {
    if (w8 == nullptr || x8 == nullptr || M < 0 || K < 0) return TJ_ERR_INVALID_ARG;
    const int64_t N = w8->rows;
    if ((x == nullptr && M > 0 && K > 0) || (y == nullptr && M > 0 && N > 0)) return TJ_ERR_INVALID_ARG;
    if (out_dtype != TJ_BF16 && out_dtype != TJ_FP32) return TJ_ERR_INVALID_ARG;
    if (!al_elem(x, TJ_BF16) || !al16(y)) return TJ_ERR_ALIGN;
    if (ldx < K || ldy < N) return TJ_ERR_SHAPE;
    tj_status st = check_mx(w8, N, K);
    if (st == TJ_OK) st = check_mx(x8, M, K);
    if (st == TJ_OK && xt8 != nullptr) st = check_mx(xt8, K, M);
    if (st != TJ_OK) return st;
    if (xt8 != nullptr && !cols_grid_fits(M)) return TJ_ERR_SHAPE;
    if (M == 0) return TJ_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    TJ_TRY(launch_quant_mx_dense(x, TJ_BF16, M, K, ldx, 0, nullptr, *x8, s));
    if (xt8 != nullptr) TJ_TRY(launch_quant_mx_dense(x, TJ_BF16, M, K, ldx, 1, nullptr, *xt8, s));
    TJ_TRY(launch_gemm(nullptr, nullptr, x8, w8, 1.0f, y, out_dtype, ldy, M, N, nullptr, s));
    return TJ_OK;
}

tj_status tj_fp8_linear_bwd_dx(const void *dy, int64_t M, int64_t N, int64_t lddy, const tj_mxfp8 *wt8, void *dx,
                               int out_dtype, int64_t lddx, void *workspace, size_t ws_bytes, void *stream) {
    if (wt8 == nullptr || M < 0 || N < 0) return TJ_ERR_INVALID_ARG;
    const int64_t K = wt8->rows;
    if ((dy == nullptr && M > 0 && N > 0) || (dx == nullptr && M > 0 && K > 0)) return TJ_ERR_INVALID_ARG;
    if (out_dtype != TJ_BF16 && out_dtype != TJ_FP32) return TJ_ERR_INVALID_ARG;
    if (!al_elem(dy, TJ_BF16) || !al16(dx)) return TJ_ERR_ALIGN;
    tj_status st = check_mx(wt8, K, N);
    if (st != TJ_OK) return st;
    if (lddy < N || lddx < K) return TJ_ERR_SHAPE;
    const size_t need = tj_workspace_size(TJ_OP_FP8_BWD_DX, M, N, K, 0);
    if ((workspace == nullptr && need > 0) || ws_bytes < need) return TJ_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return TJ_ERR_ALIGN;
    if (M == 0 || K == 0) return TJ_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *cur = static_cast<uint8_t *>(workspace);
    tj_mxfp8 q8_dy = carve_mx(cur, M, N);
    TJ_TRY(launch_quant_mx_dense(dy, TJ_BF16, M, N, lddy, 0, nullptr, q8_dy, s));
    TJ_TRY(launch_gemm(nullptr, nullptr, &q8_dy, wt8, 1.0f, dx, out_dtype, lddx, M, K, nullptr, s));
    return TJ_OK;
}

tj_status tj_fp8_linear_bwd_dw(const void *dy, int64_t M, int64_t N, int64_t lddy, const tj_mxfp8 *xt8, float *dw,
                               int64_t lddw, void *workspace, size_t ws_bytes, void *stream) {
    if (xt8 == nullptr || M < 0 || N < 0) return TJ_ERR_INVALID_ARG;
    const int64_t K = xt8->rows;
    if ((dy == nullptr && M > 0 && N > 0) || (dw == nullptr && N > 0 && K > 0)) return TJ_ERR_INVALID_ARG;
    if (!al_elem(dy, TJ_BF16) || !al16(dw)) return TJ_ERR_ALIGN;
    tj_status st = check_mx(xt8, K, M);
    if (st != TJ_OK) return st;
    if (lddy < N || lddw < K || !cols_grid_fits(M)) return TJ_ERR_SHAPE;
    const size_t need = tj_workspace_size(TJ_OP_FP8_BWD_DW, M, N, K, 0);
    if ((workspace == nullptr && need > 0) || ws_bytes < need) return TJ_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return TJ_ERR_ALIGN;
    if (N == 0 || K == 0) return TJ_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *cur = static_cast<uint8_t *>(workspace);
    tj_mxfp8 q8_dyt = carve_mx(cur, N, M);
    TJ_TRY(launch_quant_mx_dense(dy, TJ_BF16, M, N, lddy, 1, nullptr, q8_dyt, s));
    // dW [N][K] is fp32 and covered by the launch, so a long-K launch may split K in two
    const SplitRegion whole_dw{dw, N, K, lddw};
    TJ_TRY(launch_gemm(nullptr, nullptr, &q8_dyt, xt8, 1.0f, dw, TJ_FP32, lddw, N, K, nullptr, s, &whole_dw));
    return TJ_OK;
}

tj_status tj_outlier_calibrate(const void *x, int dtype, int64_t M, int64_t K, int64_t ld, double *sumsq,
                               int finalize, int64_t k, int32_t *outlier_idx, int32_t *normal_idx, void *stream) {
    if (sumsq == nullptr || M < 0 || K <= 0 || K > (int64_t)1 << 24) return TJ_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (x != nullptr) {
        if (dtype != TJ_BF16 && dtype != TJ_FP32) return TJ_ERR_INVALID_ARG;
        if (ld < K || M > ((int64_t)1 << 20)) return TJ_ERR_SHAPE;
        if (!al_elem(x, dtype)) return TJ_ERR_ALIGN;
        TJ_TRY(launch_calib_accumulate(x, dtype, M, K, ld, sumsq, s));
    }
    if (finalize) {
        if (k < 0 || k > K) return TJ_ERR_SHAPE;
        if ((k > 0 && outlier_idx == nullptr) || (k < K && normal_idx == nullptr)) return TJ_ERR_INVALID_ARG;
        TJ_TRY(launch_calib_select(sumsq, K, k, outlier_idx, normal_idx, s));
    }
    return TJ_OK;
}

tj_status tj_osci_reset(float *w, float *w_prev, float *dist_q, float *dist_m, const tj_nvfp4 *q_prev,
                        tj_nvfp4 *q_out, uint32_t *reset_mask, int64_t rows, int64_t cols, float lr, float lr_thr,
                        float risk_thr, int track, void *stream) {
    if (rows < 0 || cols < 0) return TJ_ERR_INVALID_ARG;
    if ((w == nullptr || w_prev == nullptr || dist_q == nullptr || dist_m == nullptr || reset_mask == nullptr) &&
        rows > 0 && cols > 0)
        return TJ_ERR_INVALID_ARG;
    tj_status st = check_nv(q_prev, rows, cols);
    if (st == TJ_OK) st = check_nv(q_out, rows, cols);
    if (st != TJ_OK) return st;
    if (!al16(w) || !al16(w_prev) || !al16(dist_q) || !al16(dist_m) || !al16(reset_mask)) return TJ_ERR_ALIGN;
    if (rows == 0 || cols == 0) return TJ_OK;
    return cuda_status(launch_osci_reset(w, w_prev, dist_q, dist_m, *q_prev, *q_out, reset_mask, rows, cols, lr,
                                         lr_thr, risk_thr, track, static_cast<cudaStream_t>(stream)));
}

tj_status tj_adamw_osci_reset(float *w, const float *g, float *m, float *v, float *w_prev, float *dist_q,
                              float *dist_m, const tj_nvfp4 *q_prev, tj_nvfp4 *q_out, uint32_t *reset_mask,
                              int64_t rows, int64_t cols, float lr, float beta1, float beta2, float eps,
                              float weight_decay, int64_t step, float lr_thr, float risk_thr, int track,
                              void *stream) {
    if (rows < 0 || cols < 0 || step < 1) return TJ_ERR_INVALID_ARG;
    if ((w == nullptr || g == nullptr || m == nullptr || v == nullptr || w_prev == nullptr || dist_q == nullptr ||
         dist_m == nullptr || reset_mask == nullptr) &&
        rows > 0 && cols > 0)
        return TJ_ERR_INVALID_ARG;
    tj_status st = check_nv(q_prev, rows, cols);
    if (st == TJ_OK) st = check_nv(q_out, rows, cols);
    if (st != TJ_OK) return st;
    if (!al16(w) || !al16(g) || !al16(m) || !al16(v) || !al16(w_prev) || !al16(dist_q) || !al16(dist_m) ||
        !al16(reset_mask))
        return TJ_ERR_ALIGN;
    if (rows == 0 || cols == 0) return TJ_OK;
    return cuda_status(launch_adamw_osci_reset(w, g, m, v, w_prev, dist_q, dist_m, *q_prev, *q_out, reset_mask, rows,
                                               cols, lr, beta1, beta2, eps, weight_decay, step, lr_thr, risk_thr,
                                               track, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
