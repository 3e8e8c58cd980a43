// calib.cu - OutControl's static outlier calibration (TetraJet-v2 technical
// summary §2.C: the top p% channels, which consistently carry the largest norms,
// are found once during a short calibration window and kept in FP8).
//
// Accumulation: sumsq[c] += sum_t x[t, c]^2 in fp64 with a fixed order that any
// implementation reproduces bit for bit: each 128-token chunk is summed in token
// order, the chunk sums are added in chunk order, and the batch total is added to
// the running sum.  A CTA owns 32 channels (one per lane); its 32 warps sum 32
// chunks at a time into shared memory, and lane c of warp 0 folds them in order.
// Selection: rank(c) = #{c' : s[c'] > s[c] or (s[c'] == s[c] and c' < c)};
// channels with rank < k are outliers; both lists are written ascending.
#include <cuda_bf16.h>

#include "tj_common.cuh"
#include "tj_internal.h"

namespace tj {
namespace {

template <typename T>
__device__ __forceinline__ double to_d(T v);
template <>
__device__ __forceinline__ double to_d<__nv_bfloat16>(__nv_bfloat16 v) { return (double)__bfloat162float(v); }
template <>
__device__ __forceinline__ double to_d<float>(float v) { return (double)v; }

template <typename T>
__global__ void __launch_bounds__(1024) k_calib_accumulate(const T *x, int64_t M, int64_t K, int64_t ld,
                                                           double *sumsq) {
    __shared__ double part[32][33];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t c = (int64_t)blockIdx.x * 32 + lane;
    const int64_t nchunks = (M + 127) / 128;
    double total = 0.0;                          // used by warp 0 only
    for (int64_t g0 = 0; g0 < nchunks; g0 += 32) {
        const int64_t ch = g0 + warp;
        double s = 0.0;
        if (ch < nchunks && c < K) {
            const int64_t t1 = (ch + 1) * 128 < M ? (ch + 1) * 128 : M;
            for (int64_t t = ch * 128; t < t1; ++t) {
                const double v = to_d(x[t * ld + c]);
                s = __dadd_rn(s, __dmul_rn(v, v));
            }
        }
        part[warp][lane] = s;
        __syncthreads();
        if (warp == 0) {
            const int64_t n = nchunks - g0 < 32 ? nchunks - g0 : 32;
            for (int i = 0; i < n; ++i) total = __dadd_rn(total, part[i][lane]);
        }
        __syncthreads();
    }
    if (warp == 0 && c < K) sumsq[c] = __dadd_rn(sumsq[c], total);
}

__global__ void __launch_bounds__(1024) k_calib_select(const double *sumsq, int64_t K, int64_t k,
                                                       int32_t *outlier_idx, int32_t *normal_idx) {
    __shared__ int cnt_out[1024], cnt_norm[1024];
    const int tid = threadIdx.x;
    const int64_t per = (K + 1023) / 1024;
    const int64_t c_beg = tid * per, c_end = (c_beg + per < K) ? c_beg + per : K;
    // pass 1: count outliers among this thread's contiguous channels
    int n_out = 0, n_norm = 0;
    for (int64_t c = c_beg; c < c_end; ++c) {
        const double v = sumsq[c];
        int64_t rank = 0;
        for (int64_t j = 0; j < K && rank < k; ++j) {
            const double u = sumsq[j];
            rank += (u > v || (u == v && j < c)) ? 1 : 0;
        }
        if (rank < k) ++n_out; else ++n_norm;
    }
    cnt_out[tid] = n_out;
    cnt_norm[tid] = n_norm;
    __syncthreads();
    if (tid == 0) {                               // exclusive scan (1024 entries, cold path)
        int a = 0, b = 0;
        for (int i = 0; i < 1024; ++i) {
            const int ta = cnt_out[i], tb = cnt_norm[i];
            cnt_out[i] = a;
            cnt_norm[i] = b;
            a += ta;
            b += tb;
        }
    }
    __syncthreads();
    int po = cnt_out[tid], pn = cnt_norm[tid];
    for (int64_t c = c_beg; c < c_end; ++c) {
        const double v = sumsq[c];
        int64_t rank = 0;
        for (int64_t j = 0; j < K && rank < k; ++j) {
            const double u = sumsq[j];
            rank += (u > v || (u == v && j < c)) ? 1 : 0;
        }
        if (rank < k) outlier_idx[po++] = (int32_t)c;
        else normal_idx[pn++] = (int32_t)c;
    }
}

}  // namespace

cudaError_t launch_calib_accumulate(const void *x, int dtype, int64_t M, int64_t K, int64_t ld, double *sumsq,
                                    cudaStream_t s) {
    const unsigned grid = (unsigned)((K + 31) / 32);
    if (grid == 0 || M == 0) return cudaSuccess;
    if (dtype == TJ_BF16)
        k_calib_accumulate<__nv_bfloat16><<<grid, 1024, 0, s>>>(static_cast<const __nv_bfloat16 *>(x), M, K, ld, sumsq);
    else
        k_calib_accumulate<float><<<grid, 1024, 0, s>>>(static_cast<const float *>(x), M, K, ld, sumsq);
    return cudaGetLastError();
}

cudaError_t launch_calib_select(const double *sumsq, int64_t K, int64_t k, int32_t *outlier_idx,
                                int32_t *normal_idx, cudaStream_t s) {
    k_calib_select<<<1, 1024, 0, s>>>(sumsq, K, k, outlier_idx, normal_idx);
    return cudaGetLastError();
}

}  // namespace tj
