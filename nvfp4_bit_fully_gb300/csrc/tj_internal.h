// tj_internal.h - launchers shared between the kernel files and the C ABI layer.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "tj.h"

namespace tj {

cudaError_t launch_quant_nv_dense(const void *x, int dtype, int64_t rows_x, int64_t n_cols_sel, int64_t ld,
                                  int along_cols, const int32_t *sel, int mode, int rht, uint64_t seed,
                                  uint32_t tag, uint32_t rht_tag, const tj_nvfp4 &out, cudaStream_t s);
cudaError_t launch_quant_dual_dense(const void *x, int dtype, int64_t rows_x, int64_t n_cols_sel, int64_t ld,
                                    int along_cols, const int32_t *sel, int mode, int rht, uint64_t seed,
                                    uint32_t tag, uint32_t rht_tag, const tj_nvfp4 &out, const tj_mxfp8 &out8,
                                    cudaStream_t s);
cudaError_t launch_quant_split(const void *x, int dtype, int64_t rows, int64_t K, int64_t ld, const int32_t *sel_n,
                               int64_t kn, const int32_t *sel_o, int64_t k, const tj_nvfp4 &out,
                               const tj_mxfp8 &out8, cudaStream_t s);
cudaError_t launch_quant_mx_dense(const void *x, int dtype, int64_t rows_x, int64_t n_cols_sel, int64_t ld,
                                  int along_cols, const int32_t *sel, const tj_mxfp8 &out, cudaStream_t s);
cudaError_t launch_realign_nv(const tj_nvfp4 &in, const tj_nvfp4 &out, int mode, int rht, uint64_t seed,
                              uint32_t tag, uint32_t rht_tag, cudaStream_t s);
cudaError_t launch_realign_mx(const tj_mxfp8 &in, const tj_mxfp8 &out, cudaStream_t s);
cudaError_t launch_realign_pair(const tj_nvfp4 &in, const tj_nvfp4 &out, int mode, int rht, uint64_t seed,
                                uint32_t tag, uint32_t rht_tag, const tj_mxfp8 &in8, const tj_mxfp8 &out8,
                                cudaStream_t s);
cudaError_t launch_rht(const float *x, float *y, int64_t rows, int64_t cols, uint64_t seed, uint32_t tag,
                       cudaStream_t s);
cudaError_t launch_dequant_nv(const tj_nvfp4 &q, float *y, int64_t ldy, cudaStream_t s);
cudaError_t launch_dequant_mx(const tj_mxfp8 &q, float *y, int64_t ldy, cudaStream_t s);

// An fp32 output region [rows][cols] (row pitch ld floats) that holds every output of a GEMM
// launch.  Passing it allows the launch to split K in two when that shortens its schedule:
// the region is then zeroed on the stream and both halves add their sums into it (two fp32
// additions onto zero: the result does not depend on their order).
struct SplitRegion {
    float *base;
    int64_t rows, cols, ld;
};
// GEMM: D = alpha * A_fp4 B_fp4^T (+ A8 B8^T); a/b may be null for an FP8-only GEMM.
cudaError_t launch_gemm(const tj_nvfp4 *a, const tj_nvfp4 *b, const tj_mxfp8 *a8, const tj_mxfp8 *b8,
                        float alpha, void *d, int out_dtype, int64_t ldd, int64_t M, int64_t N,
                        const int32_t *col_map, cudaStream_t s, const SplitRegion *split = nullptr);
// An FP4 product and an FP8-only product (each with its own output) in one launch.
cudaError_t launch_gemm_pair(const tj_nvfp4 *a, const tj_nvfp4 *b, float alpha, void *d, int out_dtype, int64_t ldd,
                             int64_t M, int64_t N, const int32_t *col_map, const tj_mxfp8 *a8, const tj_mxfp8 *b8,
                             void *d8, int out8_dtype, int64_t ldd8, int64_t M8, int64_t N8, const int32_t *col_map8,
                             cudaStream_t s, const SplitRegion *split = nullptr);

cudaError_t launch_adamw_osci_reset(float *w, const float *grad, float *m, float *v, float *w_prev, float *dist_q,
                                    float *dist_m, const tj_nvfp4 &q_prev, const tj_nvfp4 &q_out, uint32_t *mask,
                                    int64_t rows, int64_t cols, float lr, float beta1, float beta2, float eps,
                                    float weight_decay, int64_t step, float lr_thr, float risk_thr, int track,
                                    cudaStream_t s);
cudaError_t launch_osci_reset(float *w, float *w_prev, float *dist_q, float *dist_m, const tj_nvfp4 &q_prev,
                              const tj_nvfp4 &q_out, uint32_t *mask, int64_t rows, int64_t cols, float lr,
                              float lr_thr, float risk_thr, int track, cudaStream_t s);

cudaError_t launch_calib_accumulate(const void *x, int dtype, int64_t M, int64_t K, int64_t ld, double *sumsq,
                                    cudaStream_t s);
cudaError_t launch_calib_select(const double *sumsq, int64_t K, int64_t k, int32_t *outlier_idx,
                                int32_t *normal_idx, cudaStream_t s);

// Sticky device error flag (set by bounded waits that run out).
unsigned int read_and_clear_device_error();

}  // namespace tj
