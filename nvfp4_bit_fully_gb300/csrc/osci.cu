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
// The risk dist_Q / dist_M is compared without a division.  HBM-bound:
// ~29.3 bytes per element (read w, w_prev, dist_Q, dist_M and the previous Q;
// write w_prev, dist_Q, dist_M, the new Q and one mask bit; w only on reset).
#include <cmath>

#include "quant_core.cuh"
#include "tj_internal.h"

namespace tj {
namespace {

// Grid value of an E2M1 code's magnitude, built from its bits (exact).
__device__ __forceinline__ float e2m1_mag(uint32_t code) {
    const uint32_t m = code & 7u;
    return m < 2u ? __uint_as_float(m ? 0x3F000000u : 0u)                   // 0, 0.5
                  : __uint_as_float((((m >> 1) + 126u) << 23) | ((m & 1u) << 22));  // (1 + b/2) 2^(e-1)
}
__device__ __forceinline__ float e2m1_value(uint32_t code) {
    const float g = e2m1_mag(code);
    return (code & 8u) ? -g : g;
}

// 8 bits -> bit k at position 4k (interleave of the four per-element ballots).
__device__ __forceinline__ uint32_t spread4(uint32_t b) {
    b = (b | (b << 12)) & 0x000F000Fu;
    b = (b | (b << 6)) & 0x03030303u;
    b = (b | (b << 3)) & 0x11111111u;
    return b;
}

constexpr int kBlocksPerWarp = 1;   // 128-element blocks per warp iteration (one, with 5 CTAs per SM, measured fastest)

}  // namespace

// The fp32 constants of one AdamW step (formed in double on the host, rounded once).
struct AdamConsts {
    float b1, b2, om1, om2, decay, step_size, bc2, eps;
};

namespace {

// One AdamW update of an element, in the fixed fp32 order of the training-step pass:
//   m <- b1 m + (1 - b1) g;  v <- b2 v + (1 - b2) g g;
//   w <- w (1 - lr wd) - step_size * m / (sqrt(v) / bc2 + eps)
// (step_size = lr / (1 - b1^t), bc2 = sqrt(1 - b2^t)); every step is rounded separately.
__device__ __forceinline__ float adamw_elem(float w, float g, float &m, float &v, const AdamConsts &c) {
    m = __fadd_rn(__fmul_rn(c.b1, m), __fmul_rn(c.om1, g));
    v = __fadd_rn(__fmul_rn(c.b2, v), __fmul_rn(c.om2, __fmul_rn(g, g)));
    const float denom = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), c.bc2), c.eps);
    return __fsub_rn(__fmul_rn(w, c.decay), __fmul_rn(c.step_size, __fdiv_rn(m, denom)));
}

// One warp per 128-element block: lane l holds elements 4l .. 4l+3, so every
// load and store of the fp32 state is a fully coalesced 512-byte warp access.
// A 16-element inner group is 4 lanes; the outer block is the whole warp.
// ADAMW: the training-step pass, which first applies the AdamW update to w (reading the
// gradient and both moments, writing the moments and always writing w back).
template <bool ADAMW>
__global__ void __launch_bounds__(256, ADAMW ? 4 : 5) k_osci_reset(float *w, float *w_prev, float *dist_q,
                                                                float *dist_m, const uint8_t *qp_codes,
                                                                const uint8_t *qp_sf, const float *qp_outer, OutNv qo,
                                                                uint32_t *mask, int64_t rows, int64_t cols, int lr_low,
                                                                float risk_thr, int track, const float *grad,
                                                                float *adam_m, float *adam_v, AdamConsts ac) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;                                  // inner group within the block
    const int64_t nblk_row = qo.cols_p / 128, total = qo.rows_p * nblk_row;
    const int64_t mw = (cols + 31) / 32;                      // mask words per row
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const bool vec = (cols & 3) == 0;
    // (row, block) of the warp's block, stepped by nwarps blocks with a carry: a 64-bit
    // division per block cost more issue slots than the block's arithmetic.  32-bit counters:
    // the C ABI rejects tensors of 2^31 or more 128-element blocks
    static_assert(kBlocksPerWarp == 1, "one block per warp iteration");
    const uint32_t nbr = nblk_row > 0 ? (uint32_t)nblk_row : 1u;
    uint32_t row_i = (uint32_t)warp0 / nbr, kb_i = (uint32_t)warp0 - row_i * nbr;
    const uint32_t d_row = (uint32_t)nwarps / nbr, d_kb = (uint32_t)nwarps - d_row * nbr;
    for (int64_t base = warp0 * kBlocksPerWarp; base < total; base += nwarps * kBlocksPerWarp) {
        const int64_t row_w = row_i, kb_w = kb_i;
        row_i += d_row;
        kb_i += d_kb;
        if (kb_i >= nbr) { kb_i -= nbr; ++row_i; }
        float x[kBlocksPerWarp][4], xp[kBlocksPerWarp][4], dq[kBlocksPerWarp][4], dm[kBlocksPerWarp][4];
        float gr[kBlocksPerWarp][4], am[kBlocksPerWarp][4], av[kBlocksPerWarp][4];   // AdamW: g, m, v
        int n_live[kBlocksPerWarp];
        uint32_t pcode[kBlocksPerWarp], psb[kBlocksPerWarp];   // previous Q: this lane's 4 codes, its group's scale byte
        float pso[kBlocksPerWarp];                              // previous Q: the block's outer scale
        // ---- loads (all blocks first: many bytes in flight per warp)
#pragma unroll
        for (int b = 0; b < kBlocksPerWarp; ++b) {
            const int64_t blk = base + b;
            const int64_t row = row_w, kb = kb_w, c = kb * 128 + 4 * lane;
            int nl = 0;
            if (blk < total && row < rows) nl = (int)(cols - c <= 0 ? 0 : (cols - c >= 4 ? 4 : cols - c));
            n_live[b] = nl;
            // the previous Q of these elements, in the same batch of loads as the state
            pcode[b] = 0u;
            psb[b] = 0u;
            pso[b] = 0.0f;
            if (blk < total) {
                const int64_t gg = kb * 8 + g;
                pcode[b] = (uint32_t)__ldg(reinterpret_cast<const uint16_t *>(qp_codes + row * (qo.cols_p / 2) + kb * 64 + 2 * lane));
                psb[b] = __ldg(qp_sf + sf_word_offset(row, gg >> 2, qo.cols_p / 64) + (gg & 3));
                pso[b] = __ldg(qp_outer + kb * qo.rows_p + row);
            }
            const int64_t off = row * cols + c;
            if (nl == 4 && vec) {
                const float4 a = __ldg(reinterpret_cast<const float4 *>(w + off));
                const float4 p = __ldg(reinterpret_cast<const float4 *>(w_prev + off));
                const float4 q = __ldg(reinterpret_cast<const float4 *>(dist_q + off));
                const float4 m = __ldg(reinterpret_cast<const float4 *>(dist_m + off));
                x[b][0] = a.x; x[b][1] = a.y; x[b][2] = a.z; x[b][3] = a.w;
                xp[b][0] = p.x; xp[b][1] = p.y; xp[b][2] = p.z; xp[b][3] = p.w;
                dq[b][0] = q.x; dq[b][1] = q.y; dq[b][2] = q.z; dq[b][3] = q.w;
                dm[b][0] = m.x; dm[b][1] = m.y; dm[b][2] = m.z; dm[b][3] = m.w;
                if (ADAMW) {
                    const float4 gg = __ldg(reinterpret_cast<const float4 *>(grad + off));
                    const float4 mm = *reinterpret_cast<const float4 *>(adam_m + off);
                    const float4 vv = *reinterpret_cast<const float4 *>(adam_v + off);
                    gr[b][0] = gg.x; gr[b][1] = gg.y; gr[b][2] = gg.z; gr[b][3] = gg.w;
                    am[b][0] = mm.x; am[b][1] = mm.y; am[b][2] = mm.z; am[b][3] = mm.w;
                    av[b][0] = vv.x; av[b][1] = vv.y; av[b][2] = vv.z; av[b][3] = vv.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const bool in = i < nl;
                    x[b][i] = in ? w[off + i] : 0.0f;
                    xp[b][i] = in ? w_prev[off + i] : 0.0f;
                    dq[b][i] = in ? dist_q[off + i] : 0.0f;
                    dm[b][i] = in ? dist_m[off + i] : 0.0f;
                    if (ADAMW) {
                        gr[b][i] = in ? grad[off + i] : 0.0f;
                        am[b][i] = in ? adam_m[off + i] : 0.0f;
                        av[b][i] = in ? adam_v[off + i] : 0.0f;
                    }
                }
            }
        }
        // ---- per block: quantize, compare with the previous Q, update, store
#pragma unroll
        for (int b = 0; b < kBlocksPerWarp; ++b) {
            const int64_t blk = base + b;
            const bool valid = blk < total;                  // warp-uniform
            if (!valid) break;
            const int64_t row = row_w, kb = kb_w;
            const int64_t c = kb * 128 + 4 * lane;
            if (ADAMW) {
                // the optimizer step first; padding elements stay 0
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (i < n_live[b]) x[b][i] = adamw_elem(x[b][i], gr[b][i], am[b][i], av[b][i], ac);
            }
            // double-block RTN quantization (TetraJet-v2 §2.A) of the master weights
            float a = fmaxf(fmaxf(fabsf(x[b][0]), fabsf(x[b][1])), fmaxf(fabsf(x[b][2]), fabsf(x[b][3])));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
            const float a_i = a;
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
            const float a_o = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 16));
            float s_o = __fdiv_rn(a_o, 2688.0f);
            if (a_o > 0.0f && s_o == 0.0f) s_o = __uint_as_float(1u);
            uint32_t sb = 0u;
            if (a_i > 0.0f) sb = inner_scale_byte(a_i, s_o, rcp_approx(__fmul_rn(s_o, 6.0f)));
            const float s_i = e4m3_to_float(sb);
            const float s = __fmul_rn(s_i, s_o);
            uint32_t code16 = 0u;
            if (s > 0.0f) {
                const float r = __fdiv_rn(1.0f, s);
                uint32_t b0 = e2m1x2_rn(__fmul_rn(x[b][0], r), __fmul_rn(x[b][1], r));
                uint32_t b1 = e2m1x2_rn(__fmul_rn(x[b][2], r), __fmul_rn(x[b][3], r));
                if (x[b][0] == 0.0f) b0 &= 0xF0u;
                if (x[b][1] == 0.0f) b0 &= 0x0Fu;
                if (x[b][2] == 0.0f) b1 &= 0xF0u;
                if (x[b][3] == 0.0f) b1 &= 0x0Fu;
                code16 = b0 | (b1 << 8);
            }
            // previous Q of these elements
            const uint32_t pc = pcode[b];
            const float ps_i = e4m3_to_float(psb[b]);
            const float ps_o = pso[b];
            // OsciReset (TetraJet-v2 §2.B)
            bool rs[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float qh = __fmul_rn(__fmul_rn(e2m1_value((code16 >> (4 * i)) & 15u), s_i), s_o);
                const float qp = __fmul_rn(__fmul_rn(e2m1_value((pc >> (4 * i)) & 15u), ps_i), ps_o);
                const float m = __fadd_rn(dm[b][i], fabsf(__fsub_rn(x[b][i], xp[b][i])));
                const float d = __fadd_rn(dq[b][i], fabsf(__fsub_rn(qh, qp)));
                rs[i] = track && lr_low && (m > 0.0f) && (d > __fmul_rn(risk_thr, m)) && i < n_live[b];
                if (rs[i]) {
                    x[b][i] = qh;
                    dq[b][i] = 0.0f;
                    dm[b][i] = 0.0f;
                } else {
                    dq[b][i] = d;
                    dm[b][i] = m;
                }
            }
            // stores: Q codes / scales, state, reset mask
            *reinterpret_cast<uint16_t *>(qo.codes + row * (qo.cols_p / 2) + kb * 64 + 2 * lane) = (uint16_t)code16;
            const uint32_t s1 = __shfl_down_sync(0xffffffffu, sb, 4);
            const uint32_t s2 = __shfl_down_sync(0xffffffffu, sb, 8);
            const uint32_t s3 = __shfl_down_sync(0xffffffffu, sb, 12);
            if ((lane & 15) == 0)
                *reinterpret_cast<uint32_t *>(qo.sf + sf_word_offset(row, 2 * kb + (lane >> 4), qo.cols_p / 64)) =
                    sb | (s1 << 8) | (s2 << 16) | (s3 << 24);
            if (lane == 0) qo.outer[kb * qo.rows_p + row] = s_o;
            const uint32_t bal[4] = {__ballot_sync(0xffffffffu, rs[0]), __ballot_sync(0xffffffffu, rs[1]),
                                     __ballot_sync(0xffffffffu, rs[2]), __ballot_sync(0xffffffffu, rs[3])};
            if (row < rows) {
                const int64_t off = row * cols + c;
                const int nl = n_live[b];
                if (ADAMW && nl == 4 && vec) {
                    *reinterpret_cast<float4 *>(w + off) = make_float4(x[b][0], x[b][1], x[b][2], x[b][3]);
                    *reinterpret_cast<float4 *>(adam_m + off) = make_float4(am[b][0], am[b][1], am[b][2], am[b][3]);
                    *reinterpret_cast<float4 *>(adam_v + off) = make_float4(av[b][0], av[b][1], av[b][2], av[b][3]);
                } else if (ADAMW) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (i < nl) {
                            w[off + i] = x[b][i];
                            adam_m[off + i] = am[b][i];
                            adam_v[off + i] = av[b][i];
                        }
                    }
                }
                if (nl == 4 && vec) {
                    *reinterpret_cast<float4 *>(w_prev + off) = make_float4(x[b][0], x[b][1], x[b][2], x[b][3]);
                    *reinterpret_cast<float4 *>(dist_q + off) = make_float4(dq[b][0], dq[b][1], dq[b][2], dq[b][3]);
                    *reinterpret_cast<float4 *>(dist_m + off) = make_float4(dm[b][0], dm[b][1], dm[b][2], dm[b][3]);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (i < nl) {
                            w_prev[off + i] = x[b][i];
                            dist_q[off + i] = dq[b][i];
                            dist_m[off + i] = dm[b][i];
                        }
                    }
                }
                if (!ADAMW) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (rs[i]) w[off + i] = x[b][i];      // master weight moves only on a reset
                }
                if (lane < 4) {
                    const int64_t word = kb * 4 + lane;        // bits of elements 32*lane .. +31 of the block
                    if (word < mw) {
                        uint32_t v = 0u;
#pragma unroll
                        for (int i = 0; i < 4; ++i) v |= spread4((bal[i] >> (8 * lane)) & 0xFFu) << i;
                        mask[row * mw + word] = v;
                    }
                }
            }
        }
    }
}

}  // namespace

namespace {
template <bool ADAMW>
cudaError_t launch_osci(float *w, float *w_prev, float *dist_q, float *dist_m, const tj_nvfp4 &q_prev,
                        const tj_nvfp4 &q_out, uint32_t *mask, int64_t rows, int64_t cols, float lr, float lr_thr,
                        float risk_thr, int track, const float *grad, float *m, float *v, const AdamConsts &ac,
                        cudaStream_t s) {
    const OutNv qo{q_out.codes, q_out.sf, q_out.outer, round_up(rows, 128), round_up(cols, 128)};
    const int64_t total = qo.rows_p * (qo.cols_p / 128);
    int64_t grid = (total + 8 * kBlocksPerWarp - 1) / (8 * kBlocksPerWarp);
    if (grid > 152 * 12) grid = 152 * 12;
    if (grid < 1) grid = 1;
    k_osci_reset<ADAMW><<<(unsigned)grid, 256, 0, s>>>(w, w_prev, dist_q, dist_m, q_prev.codes, q_prev.sf,
                                                        q_prev.outer, qo, mask, rows, cols, (lr < lr_thr) ? 1 : 0,
                                                        risk_thr, track, grad, m, v, ac);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_osci_reset(float *w, float *w_prev, float *dist_q, float *dist_m, const tj_nvfp4 &q_prev,
                              const tj_nvfp4 &q_out, uint32_t *mask, int64_t rows, int64_t cols, float lr,
                              float lr_thr, float risk_thr, int track, cudaStream_t s) {
    return launch_osci<false>(w, w_prev, dist_q, dist_m, q_prev, q_out, mask, rows, cols, lr, lr_thr, risk_thr, track,
                              nullptr, nullptr, nullptr, AdamConsts{}, s);
}

cudaError_t launch_adamw_osci_reset(float *w, const float *grad, float *m, float *v, float *w_prev, float *dist_q,
                                    float *dist_m, const tj_nvfp4 &q_prev, const tj_nvfp4 &q_out, uint32_t *mask,
                                    int64_t rows, int64_t cols, float lr, float beta1, float beta2, float eps,
                                    float weight_decay, int64_t step, float lr_thr, float risk_thr, int track,
                                    cudaStream_t s) {
    const double t = (double)step;
    AdamConsts ac;
    ac.b1 = beta1;
    ac.b2 = beta2;
    ac.om1 = (float)(1.0 - (double)beta1);
    ac.om2 = (float)(1.0 - (double)beta2);
    ac.decay = (float)(1.0 - (double)lr * (double)weight_decay);
    ac.step_size = (float)((double)lr / (1.0 - std::pow((double)beta1, t)));
    ac.bc2 = (float)std::sqrt(1.0 - std::pow((double)beta2, t));
    ac.eps = eps;
    return launch_osci<true>(w, w_prev, dist_q, dist_m, q_prev, q_out, mask, rows, cols, lr, lr_thr, risk_thr, track,
                             grad, m, v, ac, s);
}

}  // namespace tj
