// osci.cu - OsciReset (TetraJet-v2 technical summary §2.B) fused with the
// forward quantization of the master weights.
//
// One pass over the master weights after each optimizer step.  Per element:
//   dist_M += |w - w_prev|
//   Q      = RTN double-block quantization of w (rows along cols, §2.A), written
//            out as the next forward's weight operand
//   dist_Q += |Q-hat - Q-hat_prev|          (Q-hat_prev decoded from the previous Q)
//   reset  <=> track && lr < lr_thr && dist_M > 0 && dist_Q > risk_thr * dist_M
//   on reset: w <- Q-hat (the centre of its quantization bin), distances <- 0
//   w_prev <- w
// The risk dist_Q / dist_M is compared without a division.  A quad of lanes
// owns one 128-element outer block (32 elements per lane), so each lane's
// reset bits form exactly one 32-bit mask word.  HBM-bound: ~29.3 bytes/element.
#include "quant_core.cuh"
#include "tj_internal.h"

namespace tj {
namespace {

__device__ __forceinline__ float e2m1_value(uint32_t code) {
    const uint32_t mag = code & 7u;
    const float g = mag < 4u ? __fmul_rn((float)mag, 0.5f)
                             : (mag == 4u ? 2.0f : (mag == 5u ? 3.0f : (mag == 6u ? 4.0f : 6.0f)));
    return (code & 8u) ? -g : g;
}

// fp32 dequantization (G * s_i) * s_o of element j of a lane's 32 codes.
__device__ __forceinline__ float deq(const uint32_t (&w)[4], int j, float s_i, float s_o) {
    const uint32_t code = (w[j >> 3] >> (4 * (j & 7))) & 15u;
    return __fmul_rn(__fmul_rn(e2m1_value(code), s_i), s_o);
}

__global__ void __launch_bounds__(256) k_osci_reset(float *w, float *w_prev, float *dist_q, float *dist_m,
                                                    const uint8_t *qp_codes, const uint8_t *qp_sf,
                                                    const float *qp_outer, OutNv qo, uint32_t *mask, int64_t rows,
                                                    int64_t cols, int lr_low, float risk_thr, int track) {
    const int lane = threadIdx.x & 31, t = lane & 3;
    const int64_t nseg = qo.cols_p / 128, total = qo.rows_p * nseg;
    const int64_t mask_words = (cols + 31) / 32;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const bool vec = (cols & 3) == 0;
    for (int64_t base = warp0 * 8; base < total; base += nwarps * 8) {
        const int64_t seg = base + (lane >> 2);
        const bool valid = seg < total;
        const int64_t row = valid ? seg / nseg : 0;
        const int64_t kb = valid ? seg % nseg : 0;
        const int64_t c0 = kb * 128 + 32 * t;
        const bool live = valid && row < rows;
        int n_live = 0;                                 // elements of this lane inside [0, cols)
        if (live) n_live = (int)(cols - c0 < 0 ? 0 : (cols - c0 > 32 ? 32 : cols - c0));
        const int64_t off = row * cols + c0;
        float x[32], xp[32], dq[32], dm[32];
        if (n_live == 32 && vec) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 a = __ldg(reinterpret_cast<const float4 *>(w + off) + i);
                const float4 b = __ldg(reinterpret_cast<const float4 *>(w_prev + off) + i);
                const float4 c = __ldg(reinterpret_cast<const float4 *>(dist_q + off) + i);
                const float4 d = __ldg(reinterpret_cast<const float4 *>(dist_m + off) + i);
                x[4 * i] = a.x; x[4 * i + 1] = a.y; x[4 * i + 2] = a.z; x[4 * i + 3] = a.w;
                xp[4 * i] = b.x; xp[4 * i + 1] = b.y; xp[4 * i + 2] = b.z; xp[4 * i + 3] = b.w;
                dq[4 * i] = c.x; dq[4 * i + 1] = c.y; dq[4 * i + 2] = c.z; dq[4 * i + 3] = c.w;
                dm[4 * i] = d.x; dm[4 * i + 1] = d.y; dm[4 * i + 2] = d.z; dm[4 * i + 3] = d.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const bool in = j < n_live;
                x[j] = in ? w[off + j] : 0.0f;
                xp[j] = in ? w_prev[off + j] : 0.0f;
                dq[j] = in ? dist_q[off + j] : 0.0f;
                dm[j] = in ? dist_m[off + j] : 0.0f;
            }
        }
        // previous Q: this lane's 16 code bytes, its two inner scales, the block's outer scale
        uint32_t pw[4] = {0u, 0u, 0u, 0u};
        float ps_i[2] = {0.0f, 0.0f}, ps_o = 0.0f;
        if (valid) {
            const uint4 pc = __ldg(reinterpret_cast<const uint4 *>(qp_codes + row * (qo.cols_p / 2) + kb * 64 + 16 * t));
            pw[0] = pc.x; pw[1] = pc.y; pw[2] = pc.z; pw[3] = pc.w;
            const uint32_t sw = __ldg(reinterpret_cast<const uint32_t *>(
                qp_sf + sf_word_offset(row, 2 * kb + (t >> 1), qo.cols_p / 64)));
            ps_i[0] = e4m3_to_float((sw >> (16 * (t & 1))) & 0xFFu);
            ps_i[1] = e4m3_to_float((sw >> (16 * (t & 1) + 8)) & 0xFFu);
            ps_o = __ldg(qp_outer + kb * qo.rows_p + row);
        }
        const NvSeg q = quant_nvfp4_seg<false>(x, 0, 0, 0);
        store_nv_seg(qo, row, kb, t, q, valid);
        const uint32_t nw[4] = {q.codes.x, q.codes.y, q.codes.z, q.codes.w};
        const float ns_i[2] = {e4m3_to_float(q.sf2 & 0xFFu), e4m3_to_float((q.sf2 >> 8) & 0xFFu)};
        uint32_t bits = 0u;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float qh = deq(nw, j, ns_i[j >> 4], q.s_o);
            const float qp = deq(pw, j, ps_i[j >> 4], ps_o);
            const float m = __fadd_rn(dm[j], fabsf(__fsub_rn(x[j], xp[j])));
            const float d = __fadd_rn(dq[j], fabsf(__fsub_rn(qh, qp)));
            const bool reset = track && lr_low && (m > 0.0f) && (d > __fmul_rn(risk_thr, m)) && j < n_live;
            if (reset) {
                bits |= 1u << j;
                x[j] = qh;
                dq[j] = 0.0f;
                dm[j] = 0.0f;
                w[off + j] = qh;
            } else {
                dq[j] = d;
                dm[j] = m;
            }
        }
        if (n_live == 32 && vec) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                reinterpret_cast<float4 *>(w_prev + off)[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
                reinterpret_cast<float4 *>(dist_q + off)[i] = make_float4(dq[4 * i], dq[4 * i + 1], dq[4 * i + 2], dq[4 * i + 3]);
                reinterpret_cast<float4 *>(dist_m + off)[i] = make_float4(dm[4 * i], dm[4 * i + 1], dm[4 * i + 2], dm[4 * i + 3]);
            }
        } else {
            for (int j = 0; j < n_live; ++j) {
                w_prev[off + j] = x[j];
                dist_q[off + j] = dq[j];
                dist_m[off + j] = dm[j];
            }
        }
        if (n_live > 0) mask[row * mask_words + (c0 >> 5)] = bits;
    }
}

}  // namespace

cudaError_t launch_osci_reset(float *w, float *w_prev, float *dist_q, float *dist_m, const tj_nvfp4 &q_prev,
                              const tj_nvfp4 &q_out, uint32_t *mask, int64_t rows, int64_t cols, float lr,
                              float lr_thr, float risk_thr, int track, cudaStream_t s) {
    const OutNv qo{q_out.codes, q_out.sf, q_out.outer, round_up(rows, 128), round_up(cols, 128)};
    const int64_t total = qo.rows_p * (qo.cols_p / 128);
    int64_t grid = (total + 63) / 64;
    if (grid > 152 * 16) grid = 152 * 16;
    if (grid < 1) grid = 1;
    k_osci_reset<<<(unsigned)grid, 256, 0, s>>>(w, w_prev, dist_q, dist_m, q_prev.codes, q_prev.sf, q_prev.outer, qo,
                                                 mask, rows, cols, (lr < lr_thr) ? 1 : 0, risk_thr, track);
    return cudaGetLastError();
}

}  // namespace tj
