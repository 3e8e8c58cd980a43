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

// One warp per 128-element block: lane l holds elements 4l .. 4l+3, so every
// load and store of the fp32 state is a fully coalesced 512-byte warp access.
// A 16-element inner group is 4 lanes; the outer block is the whole warp.
__global__ void __launch_bounds__(256, 5) k_osci_reset(float *w, float *w_prev, float *dist_q, float *dist_m,
                                                    const uint8_t *qp_codes, const uint8_t *qp_sf,
                                                    const float *qp_outer, OutNv qo, uint32_t *mask, int64_t rows,
                                                    int64_t cols, int lr_low, float risk_thr, int track) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;                                  // inner group within the block
    const int64_t nblk_row = qo.cols_p / 128, total = qo.rows_p * nblk_row;
    const int64_t mw = (cols + 31) / 32;                      // mask words per row
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const bool vec = (cols & 3) == 0;
    for (int64_t base = warp0 * kBlocksPerWarp; base < total; base += nwarps * kBlocksPerWarp) {
        float x[kBlocksPerWarp][4], xp[kBlocksPerWarp][4], dq[kBlocksPerWarp][4], dm[kBlocksPerWarp][4];
        int n_live[kBlocksPerWarp];
        uint32_t pcode[kBlocksPerWarp], psb[kBlocksPerWarp];   // previous Q: this lane's 4 codes, its group's scale byte
        float pso[kBlocksPerWarp];                              // previous Q: the block's outer scale
        // ---- loads (all blocks first: many bytes in flight per warp)
#pragma unroll
        for (int b = 0; b < kBlocksPerWarp; ++b) {
            const int64_t blk = base + b;
            const int64_t row = blk / nblk_row, kb = blk % nblk_row, c = kb * 128 + 4 * lane;
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
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const bool in = i < nl;
                    x[b][i] = in ? w[off + i] : 0.0f;
                    xp[b][i] = in ? w_prev[off + i] : 0.0f;
                    dq[b][i] = in ? dist_q[off + i] : 0.0f;
                    dm[b][i] = in ? dist_m[off + i] : 0.0f;
                }
            }
        }
        // ---- per block: quantize, compare with the previous Q, update, store
#pragma unroll
        for (int b = 0; b < kBlocksPerWarp; ++b) {
            const int64_t blk = base + b;
            const bool valid = blk < total;                  // warp-uniform
            if (!valid) break;
            const int64_t row = blk / nblk_row, kb = blk % nblk_row;
            const int64_t c = kb * 128 + 4 * lane;
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
            if (a_i > 0.0f) sb = e4m3_ceil_byte(__fdiv_rn(a_i, __fmul_rn(s_o, 6.0f)));
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
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (rs[i]) w[off + i] = x[b][i];          // master weight moves only on a reset
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

cudaError_t launch_osci_reset(float *w, float *w_prev, float *dist_q, float *dist_m, const tj_nvfp4 &q_prev,
                              const tj_nvfp4 &q_out, uint32_t *mask, int64_t rows, int64_t cols, float lr,
                              float lr_thr, float risk_thr, int track, cudaStream_t s) {
    const OutNv qo{q_out.codes, q_out.sf, q_out.outer, round_up(rows, 128), round_up(cols, 128)};
    const int64_t total = qo.rows_p * (qo.cols_p / 128);
    int64_t grid = (total + 8 * kBlocksPerWarp - 1) / (8 * kBlocksPerWarp);
    if (grid > 152 * 12) grid = 152 * 12;
    if (grid < 1) grid = 1;
    k_osci_reset<<<(unsigned)grid, 256, 0, s>>>(w, w_prev, dist_q, dist_m, q_prev.codes, q_prev.sf, q_prev.outer, qo,
                                                 mask, rows, cols, (lr < lr_thr) ? 1 : 0, risk_thr, track);
    return cudaGetLastError();
}

}  // namespace tj
