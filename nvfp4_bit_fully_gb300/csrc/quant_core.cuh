// quant_core.cuh - the per-segment quantizers used by every quantize kernel.
//
// Work split: one 128-element segment of the quantized axis (one outer block of
// TetraJet-v2 §2.A) is held by a quad of 4 adjacent lanes, 32 consecutive elements
// per lane (lane t of the quad holds elements 32t .. 32t+31).  So each lane owns
// two whole 16-element inner groups, one whole 32-element FP8 group, four whole
// Philox calls (8 elements each), and the 128-point Hadamard butterfly needs only
// two cross-lane stages.
#pragma once
#include "tj_common.cuh"

namespace tj {

// 128-point unnormalised Walsh-Hadamard transform of a quad's segment, after
// multiplying by the random +-1 diagonal (bit j of `sign_word` set -> negate
// element j of this lane).  Stages h = 1, 2, 4, 8, 16 run inside the lane, h = 32
// and h = 64 pair lanes t^1 and t^2; every stage maps (a, b) -> (a + b, a - b) in
// fp32, in the fixed order h = 1, 2, ..., 64 (TetraJet-v2 §2.C RHT).  The
// cross-lane stages use one FMA with a +-1 factor: s*x + p is exact before its
// single rounding, so it rounds exactly like x + p or p - x.
// kFlip = false: the caller has applied the diagonal already (while loading).
template <bool kFlip = true>
__device__ __forceinline__ void rht128_quad(float (&x)[32], uint32_t sign_word, int t) {
    if (kFlip) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            x[j] = __uint_as_float(__float_as_uint(x[j]) ^ ((sign_word << (31 - j)) & 0x80000000u));
    }
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const float a = x[j], b = x[j + 1];
        x[j] = __fadd_rn(a, b);
        x[j + 1] = __fsub_rn(a, b);
    }
    // h = 2 .. 16 on packed pairs: (x[j], x[j+1]) with (x[j+h], x[j+h+1])
#pragma unroll
    for (int h = 2; h < 32; h <<= 1) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            if ((j & h) == 0) {
                const uint64_t a = f2_pack(x[j], x[j + 1]), b = f2_pack(x[j + h], x[j + h + 1]);
                f2_unpack(f2_add(a, b), x[j], x[j + 1]);
                f2_unpack(f2_sub(a, b), x[j + h], x[j + h + 1]);
            }
        }
    }
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
        const float sgn = (t & m) ? -1.0f : 1.0f;
        const uint64_t sgn2 = f2_pack(sgn, sgn);
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            const float p0 = __shfl_xor_sync(0xffffffffu, x[j], m);
            const float p1 = __shfl_xor_sync(0xffffffffu, x[j + 1], m);
            f2_unpack(f2_fma(sgn2, f2_pack(x[j], x[j + 1]), f2_pack(p0, p1)), x[j], x[j + 1]);
        }
    }
}

// max |x[j0 .. j0+15]| by three-input maxima
__device__ __forceinline__ float amax16(const float (&x)[32], int j0) {
    float m = amax3(x[j0], x[j0 + 1], x[j0 + 2]);
#pragma unroll
    for (int j = 3; j < 15; j += 2) m = amax3(m, x[j0 + j], x[j0 + j + 1]);
    return fmaxf(m, fabsf(x[j0 + 15]));
}

struct NvSeg {
    uint4 codes;    // 32 E2M1 codes, element 2j in the low nibble of byte j
    uint32_t sf2;   // inner scale bytes of this lane's groups (low byte = first group)
    float s_o;      // the segment's FP32 outer scale (same in all 4 lanes)
};

// Double-block NVFP4 quantization of one 128-segment (§2.A), readings as in tj.h:
// s_o = amax/2688 (2^-149 if that underflows), s_i = inner_scale_byte (the
// smallest normal E4M3 scale whose dequantized top value covers amax_16),
// v = x * (1/(s_i s_o)); RTN = nearest E2M1 value, ties even,
// saturated at 6 (hardware conversion); SR = exact integer test on min(|v|, 6)
// with the 16-bit uniforms of Philox call (elem0 + 8q) >> 3.  A zero element,
// or any element of a group whose scale is zero, gets code 0.  elem0 = index of
// x[0] in the operand's quantized layout (row * cols_p + col), a multiple of 8.
template <bool SR>
__device__ __forceinline__ NvSeg quant_nvfp4_seg(const float (&x)[32], uint64_t elem0, const PhiloxKeys &pk,
                                                 uint32_t tag) {
    float a_i[2];
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        a_i[g] = amax16(x, 16 * g);
    }
    float a_o = fmaxf(a_i[0], a_i[1]);
    a_o = fmaxf(a_o, __shfl_xor_sync(0xffffffffu, a_o, 1));
    a_o = fmaxf(a_o, __shfl_xor_sync(0xffffffffu, a_o, 2));

    float s_o = __fdiv_rn(a_o, 2688.0f);
    if (a_o > 0.0f && s_o == 0.0f) s_o = __uint_as_float(1u);     // 2^-149
    const float inv_m6 = rcp_approx(__fmul_rn(s_o, 6.0f));    // first guess of the inner scales

    NvSeg out;
    out.s_o = s_o;
    out.sf2 = 0u;
    uint32_t words[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        uint32_t sb = 0u;
        if (a_i[g] > 0.0f) sb = inner_scale_byte(a_i[g], s_o, inv_m6);
        out.sf2 |= sb << (8 * g);
        const float s = __fmul_rn(e4m3_to_float(sb), s_o);
        const float r = s > 0.0f ? __fdiv_rn(1.0f, s) : 0.0f;
        if (!(s > 0.0f)) continue;                         // zero group: codes stay 0
        if (SR && r <= 3.4028235e38f) {
            // two elements at a time: y = x * r + 0 (so x = -0 gives +0 and its code 0,
            // while a negative x whose product underflows keeps its sign), then the
            // packed stochastic rounding; uniforms drawn just in time, 8 elements a call
            const uint64_t r2 = f2_pack(r, r), z2 = f2_pack(0.0f, 0.0f);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint4 w4 = sr_bits8((elem0 >> 3) + (uint64_t)(2 * g + h), pk, tag);
                const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
                // byte 3 of pb[i] = the code byte of elements 2i, 2i+1 (first in the low
                // nibble): the top nibble of t1, and t0's top nibble shifted down by 4
                uint32_t pb[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int e = 16 * g + 8 * h + 2 * i;
                    uint32_t t0, t1;
                    e2m1x2_sr_nib(f2_fma(f2_pack(x[e], x[e + 1]), r2, z2), (ws[i] << 12) & 0x0FFFF000u,
                                  (ws[i] >> 4) & 0x0FFFF000u, t0, t1);
                    pb[i] = (t1 & 0xF0000000u) | ((t0 >> 4) & 0x0FFFFFFFu);
                }
                const uint32_t lo = __byte_perm(pb[0], pb[1], 0x0073u), hi = __byte_perm(pb[2], pb[3], 0x0073u);
                words[2 * g + h] = __byte_perm(lo, hi, 0x5410u);
            }
        } else if (SR) {
            // a group whose 1 / s overflows (denormal inputs): element by element
            uint4 w4;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int e = 16 * g + j;
                if ((e & 7) == 0) w4 = sr_bits8((elem0 >> 3) + (uint64_t)(e >> 3), pk, tag);
                const float xv = x[e];
                const float a = fminf(fabsf(__fmul_rn(xv, r)), 6.0f);
                const int wi = (e & 7) >> 1;
                const uint32_t w = wi == 0 ? w4.x : (wi == 1 ? w4.y : (wi == 2 ? w4.z : w4.w));
                uint32_t code = e2m1_sr(a, (w >> (16 * (e & 1))) & 0xFFFFu) | (xv < 0.0f ? 8u : 0u);
                if (xv == 0.0f) code = 0u;
                words[e >> 3] |= code << (4 * (e & 7));
            }
        } else if (r <= 3.4028235e38f) {
            // RTN by the hardware conversion on y = x * r + 0: as above, x = -0 gives +0
            // and code 0, a negative x whose product rounds to zero keeps its sign
            const uint64_t r2 = f2_pack(r, r), z2 = f2_pack(0.0f, 0.0f);
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                const int e = 16 * g + j;
                float v0, v1;
                f2_unpack(f2_fma(f2_pack(x[e], x[e + 1]), r2, z2), v0, v1);
                words[e >> 3] |= e2m1x2_rn(v0, v1) << (4 * (e & 7));
            }
        } else {
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                const int e = 16 * g + j;
                const float x0 = x[e], x1 = x[e + 1];
                uint32_t byte = e2m1x2_rn(__fmul_rn(x0, r), __fmul_rn(x1, r));
                if (x0 == 0.0f) byte &= 0xF0u;                 // -0 or 0 input -> code 0
                if (x1 == 0.0f) byte &= 0x0Fu;
                words[e >> 3] |= byte << (4 * (e & 7));
            }
        }
    }
    out.codes = make_uint4(words[0], words[1], words[2], words[3]);
    return out;
}

struct MxSeg {
    uint4 codes[2];  // the group's packed codes: 32 bytes (E4M3), 24 (E2M3 / E3M2) or 16 (E2M1)
    uint32_t e8;     // UE8M0 scale byte
};

// Block exponent of an MX group: the smallest integer E with max * 2^E >= amax, for a
// format maximum max = (1 + f) 2^emax whose fraction bits are `manlim` (448: 8 and
// 0x600000; 7.5: 2 and 0x700000; 28: 4 and 0x600000; 6: 2 and 0x400000), clamped to
// [-127, 127]; 0 for an all-zero group.
__device__ __forceinline__ int mx_block_exponent(float amax, int emax, uint32_t manlim) {
    if (!(amax > 0.0f)) return 0;
    uint32_t b = __float_as_uint(amax);
    int ex = (int)(b >> 23) - 127;
    if (ex == -127) {                                   // fp32 subnormal: renormalise
        b = __float_as_uint(__fmul_rn(amax, 4294967296.0f));
        ex = (int)(b >> 23) - 127 - 32;
    }
    const int E = ((b & 0x7FFFFFu) <= manlim) ? ex - emax : ex - emax + 1;
    return E < -127 ? -127 : (E > 127 ? 127 : E);
}

// 2^-E as an exact fp32 (E in [-127, 127])
__device__ __forceinline__ float mx_inv_scale(int E) {
    const int e2 = -E;
    return e2 >= -126 ? __uint_as_float((uint32_t)(e2 + 127) << 23) : __uint_as_float(0x400000u);
}

// MXFP8 quantization of one 32-element group (this lane's elements), §2.C FP8
// slice: E = smallest integer with 448 * 2^E >= amax (clamped to [-127, 127],
// 0 for an all-zero group), values x * 2^-E rounded to nearest-even E4M3 with
// saturation at +-448.
__device__ __forceinline__ MxSeg quant_mxfp8_group(const float (&x)[32]) {
    const float amax = fmaxf(amax16(x, 0), amax16(x, 16));
    const int E = mx_block_exponent(amax, 8, 0x600000u);          // 448 = 1.75 * 2^8
    const float inv = mx_inv_scale(E);
    MxSeg out;
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t word = 0u;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float2 f;
            f2_unpack(f2_mul(f2_pack(x[4 * i + 2 * h], x[4 * i + 2 * h + 1]), f2_pack(inv, inv)), f.x, f.y);
            const __nv_fp8x2_storage_t p = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
            word |= (uint32_t)p << (16 * h);
        }
        w[i] = word;
    }
    out.codes[0] = make_uint4(w[0], w[1], w[2], w[3]);
    out.codes[1] = make_uint4(w[4], w[5], w[6], w[7]);
    out.e8 = (uint32_t)(E + 127);
    return out;
}

// The MXFP8 codes of a lane's 32 elements computed on sign-flipped inputs, turned
// into the codes of the unflipped inputs: the E4M3 conversion is symmetric in the
// sign (zeros included), so each flipped element's code byte has its sign bit
// toggled.  Bit j of `sign_word` set = element j was negated.
__device__ __forceinline__ void mx_unflip(MxSeg &m, uint32_t sign_word) {
    uint32_t w[8] = {m.codes[0].x, m.codes[0].y, m.codes[0].z, m.codes[0].w,
                     m.codes[1].x, m.codes[1].y, m.codes[1].z, m.codes[1].w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        // bits 4i .. 4i+3 -> bit 7 of bytes 0 .. 3 (the multiply spreads the four bits 7 apart)
        w[i] ^= (((sign_word >> (4 * i)) & 0xFu) * 0x00204081u & 0x01010101u) << 7;
    }
    m.codes[0] = make_uint4(w[0], w[1], w[2], w[3]);
    m.codes[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// FP6 (E2M3 / E3M2) quantization of one 32-element group with the FP8 slice's rule and the
// format's maximum (7.5 = 1.875 * 2^2, 28 = 1.75 * 2^4).  Element j is negated first when
// bit j of `flip` is set.  The 32 6-bit codes are packed as a little-endian bit stream
// (element j at bits 6j .. 6j+5): 24 bytes, the tensor core's FP6 operand order.
__device__ __forceinline__ MxSeg quant_mx6_group(const float (&x)[32], bool e3m2, uint32_t flip) {
    const float amax = fmaxf(amax16(x, 0), amax16(x, 16));
    const int E = e3m2 ? mx_block_exponent(amax, 4, 0x600000u) : mx_block_exponent(amax, 2, 0x700000u);
    const float inv = mx_inv_scale(E);
    uint32_t p[8];                                      // 4 codes = 24 bits each
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float v[4];
#pragma unroll
        for (int h = 0; h < 4; ++h)
            v[h] = __uint_as_float(__float_as_uint(__fmul_rn(x[4 * i + h], inv)) ^ (((flip >> (4 * i + h)) & 1u) << 31));
        const uint32_t w = e3m2 ? (e3m2x2_rn(v[0], v[1]) | (e3m2x2_rn(v[2], v[3]) << 16))
                                : (e2m3x2_rn(v[0], v[1]) | (e2m3x2_rn(v[2], v[3]) << 16));
        p[i] = (w & 0x3Fu) | ((w >> 2) & 0xFC0u) | ((w >> 4) & 0x3F000u) | ((w >> 6) & 0xFC0000u);
    }
    MxSeg out;
    out.codes[0] = make_uint4(p[0] | (p[1] << 24), (p[1] >> 8) | (p[2] << 16), (p[2] >> 16) | (p[3] << 8),
                              p[4] | (p[5] << 24));
    out.codes[1] = make_uint4((p[5] >> 8) | (p[6] << 16), (p[6] >> 16) | (p[7] << 8), 0u, 0u);
    out.e8 = (uint32_t)(E + 127);
    return out;
}

// FP4 (E2M1) quantization of one 32-element group with the same rule (6 = 1.5 * 2^2):
// codes packed two per byte, element 2j in the low nibble (16 bytes).  `flip` as above.
__device__ __forceinline__ MxSeg quant_mx4_group(const float (&x)[32], uint32_t flip) {
    const float amax = fmaxf(amax16(x, 0), amax16(x, 16));
    const int E = mx_block_exponent(amax, 2, 0x400000u);
    const float inv = mx_inv_scale(E);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t word = 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = 8 * i + 2 * j;
            const float a = __uint_as_float(__float_as_uint(__fmul_rn(x[e], inv)) ^ (((flip >> e) & 1u) << 31));
            const float b = __uint_as_float(__float_as_uint(__fmul_rn(x[e + 1], inv)) ^ (((flip >> (e + 1)) & 1u) << 31));
            word |= e2m1x2_rn(a, b) << (8 * j);
        }
        w[i] = word;
    }
    MxSeg out;
    out.codes[0] = make_uint4(w[0], w[1], w[2], w[3]);
    out.codes[1] = make_uint4(0u, 0u, 0u, 0u);
    out.e8 = (uint32_t)(E + 127);
    return out;
}

// MX quantization of one group in the slice format fmt (uniform across the warp).  With
// kFlip, element j is taken negated when bit j of `flip` is set (the sign-flipped rows of
// the transposed RHT quantizer); the E4M3 path turns its codes' sign bits instead.
template <bool kFlip = false>
__device__ __forceinline__ MxSeg quant_mx_group(const float (&x)[32], int fmt, uint32_t flip = 0u) {
    if (fmt == kMxE2M1) return quant_mx4_group(x, kFlip ? flip : 0u);
    if (fmt != kMxE4M3) return quant_mx6_group(x, fmt == kMxE3M2, kFlip ? flip : 0u);
    MxSeg m = quant_mxfp8_group(x);
    if (kFlip) mx_unflip(m, flip);
    return m;
}

// Output descriptors (device pointers and padded sizes).
struct OutNv {
    uint8_t *codes;
    uint8_t *sf;
    float *outer;
    int64_t rows_p, cols_p;
};
struct OutMx {
    uint8_t *codes;
    uint8_t *sf;
    int64_t rows_p, cols_p;
    int fmt;                  // slice element format (kMxE4M3 / kMxE2M3 / kMxE3M2 / kMxE2M1)
};

// Store one quad's NVFP4 segment (row, block kb).  Lane t writes its 16 code
// bytes; lanes 0 and 2 write the two 4-byte scale words (groups 8kb..8kb+3 and
// 8kb+4..8kb+7); lane 0 writes the outer scale.  All 4 lanes must call.
__device__ __forceinline__ void store_nv_seg(const OutNv &o, int64_t row, int64_t kb, int t, const NvSeg &s,
                                             bool valid) {
    const uint32_t other = __shfl_xor_sync(0xffffffffu, s.sf2, 1);
    if (!valid) return;
    *reinterpret_cast<uint4 *>(o.codes + row * (o.cols_p / 2) + kb * 64 + 16 * t) = s.codes;
    if ((t & 1) == 0) {
        const uint32_t word = (s.sf2 & 0xFFFFu) | (other << 16);
        *reinterpret_cast<uint32_t *>(o.sf + sf_word_offset(row, 2 * kb + (t >> 1), o.cols_p / 64)) = word;
    }
    if (t == 0) o.outer[kb * o.rows_p + row] = s.s_o;
}

// Store one quad's MX segment (row, 128-block kb) in the slice format: lane t owns group 4kb+t.
__device__ __forceinline__ void store_mx_seg(const OutMx &o, int64_t row, int64_t kb, int t, const MxSeg &s,
                                             bool valid) {
    const uint32_t b1 = __shfl_xor_sync(0xffffffffu, s.e8, 1);
    const uint32_t b2 = __shfl_xor_sync(0xffffffffu, s.e8, 2);
    const uint32_t b3 = __shfl_xor_sync(0xffffffffu, s.e8, 3);
    if (!valid) return;
    if (o.fmt == kMxE4M3) {
        uint4 *dst = reinterpret_cast<uint4 *>(o.codes + row * o.cols_p + kb * 128 + 32 * t);
        dst[0] = s.codes[0];
        dst[1] = s.codes[1];
    } else if (o.fmt == kMxE2M1) {
        *reinterpret_cast<uint4 *>(o.codes + row * (o.cols_p / 2) + kb * 64 + 16 * t) = s.codes[0];
    } else {                                          // 24 bytes, 8-byte aligned
        uint2 *dst = reinterpret_cast<uint2 *>(o.codes + row * (o.cols_p / 4 * 3) + kb * 96 + 24 * t);
        dst[0] = make_uint2(s.codes[0].x, s.codes[0].y);
        dst[1] = make_uint2(s.codes[0].z, s.codes[0].w);
        dst[2] = make_uint2(s.codes[1].x, s.codes[1].y);
    }
    if (t == 0) {
        const uint32_t word = s.e8 | (b1 << 8) | (b2 << 16) | (b3 << 24);
        *reinterpret_cast<uint32_t *>(o.sf + sf_word_offset(row, kb, o.cols_p / 128)) = word;
    }
}

}  // namespace tj
