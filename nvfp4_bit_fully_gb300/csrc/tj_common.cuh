// tj_common.cuh - device helpers shared by the sm_103a kernels of libtj.
//
// Number formats and rounding follow the TetraJet-v2 technical summary §2.A
// (NVFP4: E2M1 values, 16-element groups with an 8-bit E4M3 scale, a 128-element
// outer block with an FP32 scale; RTN forward, stochastic rounding backward) and
// §2.C (128-point random Hadamard transform in the backward; FP8 outlier slice).
// Every arithmetic step that decides a code is an explicit IEEE fp32 operation
// (__fmul_rn / __fdiv_rn / __fadd_rn) so that no FMA contraction or reordering
// can change a rounding.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "tj.h"

namespace tj {

constexpr int kOuter = 128;  // outer block (FP32 scale)
constexpr int kInner = 16;   // inner group (E4M3 scale)
constexpr int kMx = 32;      // FP8 slice group (UE8M0 scale)

__host__ __device__ inline int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): 10 rounds of two 32x32->64
// multiplications with the constants 0xD2511F53 / 0xCD9E8D57, the high halves
// xored with the other counter words and the round key, the key advanced by the
// Weyl increments 0x9E3779B9 / 0xBB67AE85 after every round.
// ---------------------------------------------------------------------------
// The ten round keys of Philox4x32-10 for one 64-bit seed (key = (lo, hi), each
// round adds the Weyl constants 0x9E3779B9 / 0xBB67AE85).  They are the same for
// every call of a launch, so the host computes them once and the kernels read them
// as launch parameters instead of re-deriving them in every call.
struct PhiloxKeys {
    uint32_t k[20];     // k[2r], k[2r+1]: the key words of round r
};
inline PhiloxKeys philox_keys(uint64_t seed) {
    PhiloxKeys pk;
    uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
    for (int r = 0; r < 10; ++r) {
        pk.k[2 * r] = k0;
        pk.k[2 * r + 1] = k1;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return pk;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxKeys &pk) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        uint32_t lo0, hi0, lo1, hi1;        // both halves of each 32 x 32 -> 64-bit product at once
        asm("{\n\t.reg .b64 p;\n\tmul.wide.u32 p, %2, 0xD2511F53;\n\tmov.b64 {%0, %1}, p;\n\t}"
            : "=r"(lo0), "=r"(hi0) : "r"(c.x));
        asm("{\n\t.reg .b64 p;\n\tmul.wide.u32 p, %2, 0xCD9E8D57;\n\tmov.b64 {%0, %1}, p;\n\t}"
            : "=r"(lo1), "=r"(hi1) : "r"(c.z));
        c = make_uint4(hi1 ^ c.y ^ pk.k[2 * r], lo1, hi0 ^ c.w ^ pk.k[2 * r + 1], lo0);
    }
    return c;
}

// Random bits for stochastic rounding: element e (row * cols_p + col of the
// quantized operand) takes 16 bits of Philox(counter = (e>>3, tag, 0), key = seed);
// elements 8g .. 8g+7 share call g: word (e&7)>>1, low half for even e.
__device__ __forceinline__ uint4 sr_bits8(uint64_t g, const PhiloxKeys &pk, uint32_t tag) {
    return philox4x32_10(make_uint4((uint32_t)g, (uint32_t)(g >> 32), tag, 0u), pk);
}

// The +-1 diagonal of the RHT as 128 sign bits (bit i set -> d[i] = -1):
// one Philox call with counter (0, 0, tag, 0) and key = seed.
__device__ __forceinline__ uint4 rht_sign_bits(const PhiloxKeys &pk, uint32_t tag) {
    return philox4x32_10(make_uint4(0u, 0u, tag, 0u), pk);
}

// ---------------------------------------------------------------------------
// E4M3 (bias 7, max 448, subnormal step 2^-9) helpers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float e4m3_to_float(uint32_t b) {
    const uint32_t e = (b >> 3) & 15u, m = b & 7u;
    float v = (e == 0) ? __fmul_rn((float)m, 0.001953125f)                   // m * 2^-9
                       : __uint_as_float(((e + 120u) << 23) | (m << 20));    // (1+m/8) 2^(e-7)
    return (b & 0x80u) ? -v : v;
}

// Smallest E4M3 value >= t (t >= 0), clamped to 448; returns its byte.
__device__ __forceinline__ uint32_t e4m3_ceil_byte(float t) {
    if (!(t > 0.0f)) return 0u;
    if (t >= 448.0f) return 0x7Eu;
    const uint32_t bits = __float_as_uint(t);
    const int ex = (int)((bits >> 23) & 0xFFu) - 127;
    if (ex < -6) {                                   // below the smallest normal 2^-6
        const float s = __fmul_rn(t, 512.0f);        // t / 2^-9, exact
        const uint32_t k = (uint32_t)ceilf(s);       // 1 .. 8
        return k >= 8u ? 0x08u : (k == 0u ? 1u : k);
    }
    uint32_t m3 = (bits >> 20) & 7u;
    uint32_t eb = (uint32_t)(ex + 7);
    if (bits & 0xFFFFFu) {                           // not exactly representable: round up
        if (++m3 == 8u) { m3 = 0u; ++eb; }
    }
    const uint32_t byte = (eb << 3) | m3;
    return byte > 0x7Eu ? 0x7Eu : byte;
}

// Value of a normal E4M3 byte (0x08 .. 0x7E): exponent and mantissa bits moved into
// place and the exponent rebiased (7 -> 127) by one add.
__device__ __forceinline__ float e4m3_normal_to_float(uint32_t b) { return __uint_as_float((b << 20) + 0x3C000000u); }

// Approximate reciprocal (one special-function instruction); only used for a first
// guess that inner_scale_byte corrects exactly.
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Inner-scale byte of a 16-element group with amax a_i > 0 in an outer block of
// scale s_o.  Reading of §2.A's group scale: the smallest normal E4M3 value sigma
// (2^-6 .. 448) whose top value fl(fl(6 sigma) s_o), dequantized the way every
// consumer dequantizes, is >= a_i; 448 if none is.  Rounding up keeps |x / s| <= 6,
// so no element clips and stochastic rounding stays unbiased; deciding on the
// dequantized value makes the quantizer idempotent, so an OsciReset reset (§2.B: the
// weight moved onto its own Q-hat) re-quantizes to the same code and scales.
// The search starts from c, the E4M3 ceiling of a_i * inv_m6 (inv_m6 ~ 1 / fl(6 s_o),
// an approximate reciprocal), clamped to the normal bytes.  From a start within an ulp
// or two of the quotient the answer is c - 1, c or c + 1 whenever the products are
// normal fp32 numbers (s_o >= 2^-110), and the top values of c - 1 and c decide it.
// Below that the top values of c - 2 .. c + 1, computed side by side, take one step,
// and where that is not enough (fp32-subnormal products) two walks reach the exact
// answer, since the top value grows with sigma.
__device__ __forceinline__ float inner_top(uint32_t b, float s_o) {
    return __fmul_rn(__fmul_rn(6.0f, e4m3_normal_to_float(b)), s_o);   // 6 sigma is exact
}
__device__ __forceinline__ uint32_t inner_scale_byte(float a_i, float s_o, float inv_m6) {
    // c: the E4M3 ceiling of the first guess from its fp32 bits (rounded up to 3 mantissa
    // bits, exponent rebiased 127 -> 7), clamped to the normal bytes 0x08 .. 0x7E
    const int cb = (int)((__float_as_uint(__fmul_rn(a_i, inv_m6)) + 0xFFFFFu) >> 20) - 960;
    const uint32_t c = (uint32_t)min(max(cb, 0x08), 0x7E);
    if (s_o >= 0x1p-110f) {
        // every top value is a normal fp32 number, and the first guess is a few ulps off at
        // most: the answer is c - 1, c or c + 1, told apart by the top values of c - 1 and c
        const uint32_t cm = c > 0x08u ? c - 1u : c;
        const float t0 = inner_top(c, s_o), tm = inner_top(cm, s_o);
        return t0 < a_i ? (c < 0x7Eu ? c + 1u : c) : ((cm < c && tm >= a_i) ? cm : c);
    }
    // the top values of c - 2 .. c + 1 as independent products (clamped to the normal range)
    const uint32_t cp = c < 0x7Eu ? c + 1u : c, cm = c > 0x08u ? c - 1u : c, cmm = cm > 0x08u ? cm - 1u : cm;
    const float tp = inner_top(cp, s_o), t0 = inner_top(c, s_o), tm = inner_top(cm, s_o), tmm = inner_top(cmm, s_o);
    uint32_t sb;
    bool more;
    if (t0 < a_i) {
        sb = cp;
        more = cp < 0x7Eu && tp < a_i;               // still below: walk further up
    } else if (cm < c && tm >= a_i) {
        sb = cm;
        more = cmm < cm && tmm >= a_i;               // the next lower scale fits too: walk down
    } else {
        sb = c;
        more = false;
    }
    if (more) {                                      // only where the products are fp32 subnormals
        while (sb < 0x7Eu && inner_top(sb, s_o) < a_i) ++sb;
        while (sb > 0x08u && inner_top(sb - 1u, s_o) >= a_i) --sb;
    }
    return sb;
}

// ---------------------------------------------------------------------------
// E2M1 grid {0, .5, 1, 1.5, 2, 3, 4, 6}: rounding of a magnitude a in [0, 6].
// ---------------------------------------------------------------------------
// Nearest grid point, ties to the even code (the midpoints .25, .75, 1.25, 1.75,
// 2.5, 3.5, 5 go to codes 0, 2, 2, 4, 4, 6, 6).  Reference form, used by the
// scalar paths; the vector paths use the hardware E2M1 conversion, which rounds
// to nearest-even on the same grid and saturates at 6.
__device__ __forceinline__ uint32_t e2m1_rtn(float a) {
    return (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
           (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) +
           (uint32_t)(a > 5.0f);
}

// Two signed values -> one byte of E2M1 codes (lo in the low nibble), rounded
// to nearest-even and saturated to +-6 by cvt.rn.satfinite.e2m1x2.f32.
__device__ __forceinline__ uint32_t e2m1x2_rn(float lo, float hi) {
    uint16_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
        : "=h"(r)
        : "f"(hi), "f"(lo));
    return (uint32_t)r & 0xFFu;
}

// ---------------------------------------------------------------------------
// Element formats of an MX outlier slice (tj.h tj_mx_format: the tensor core's format
// numbers).  E2M3 (bias 1, max 7.5) and E3M2 (bias 3, max 28) are the FP6 formats, E2M1
// the FP4 one, of the mixed FP6 x FP4 slice; E4M3 is the FP8 slice.
// ---------------------------------------------------------------------------
constexpr int kMxE4M3 = 0, kMxE2M3 = 3, kMxE3M2 = 4, kMxE2M1 = 5;
__host__ __device__ constexpr int mx_bits(int fmt) { return fmt == kMxE4M3 ? 8 : (fmt == kMxE2M1 ? 4 : 6); }
__host__ __device__ constexpr bool mx_fmt_valid(int fmt) {
    return fmt == kMxE4M3 || fmt == kMxE2M3 || fmt == kMxE3M2 || fmt == kMxE2M1;
}

// Two signed values -> two 6-bit codes, one per byte (lo in the low byte), rounded to
// nearest-even and saturated by cvt.rn.satfinite.{e2m3x2,e3m2x2}.f32 (which puts its
// first operand in the high byte).
__device__ __forceinline__ uint32_t e2m3x2_rn(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e2m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return (uint32_t)r;
}
__device__ __forceinline__ uint32_t e3m2x2_rn(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e3m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return (uint32_t)r;
}

// Exact fp32 value of a 6-bit E2M3 / E3M2 code (sign in bit 5): the normal values are
// built from their exponent and mantissa bits, the subnormals as m / 8 or m / 16.
__device__ __forceinline__ float e2m3_to_float(uint32_t c) {
    const uint32_t e = (c >> 3) & 3u, m = c & 7u;
    const float v = e ? __uint_as_float(((e + 126u) << 23) | (m << 20)) : __fmul_rn((float)m, 0.125f);
    return (c & 0x20u) ? -v : v;
}
__device__ __forceinline__ float e3m2_to_float(uint32_t c) {
    const uint32_t e = (c >> 2) & 7u, m = c & 3u;
    const float v = e ? __uint_as_float(((e + 124u) << 23) | (m << 21)) : __fmul_rn((float)m, 0.0625f);
    return (c & 0x20u) ? -v : v;
}
__device__ __forceinline__ float e2m1_to_float(uint32_t c) {
    const uint32_t mag = c & 7u;
    const float v = mag < 4u ? __fmul_rn((float)mag, 0.5f)
                             : (mag == 4u ? 2.0f : (mag == 5u ? 3.0f : (mag == 6u ? 4.0f : 6.0f)));
    return (c & 8u) ? -v : v;
}

// Stochastic rounding of a in [0, 6] between its grid neighbours lo <= a <= hi:
// up with probability p = (a - lo) / (hi - lo), decided as float(u16) < p * 65536.
// Integer form of that same test: for a >= 1 in the binade [2^e, 2^(e+1)) the grid
// keeps 1 mantissa bit, so p = r / 2^22 with r the 22 lower mantissa bits and the
// test is 128 * u16 < 2 r; on [0.5, 1) p = m / 2^23 (test 128 * u16 < m); below 0.5
// lo = 0 and p * 65536 = a * 2^17 exactly, compared with u16 converted exactly
// (2^23 + u16 as fp32, minus 2^23).  Every case is evaluated and selected, without
// branches.  Returns the grid index (0..7).
__device__ __forceinline__ uint32_t e2m1_sr(float a, uint32_t u16) {
    const uint32_t A = __float_as_uint(a);
    const uint32_t big = A >= 0x3F800000u ? 1u : 0u;              // a >= 1
    const bool mid = A >= 0x3F000000u;                            // a >= 0.5
    const bool up_hi = (u16 << 7) < ((A << big) & 0x7FFFFFu);
    const float uf = __fsub_rn(__uint_as_float(0x4B000000u | u16), 8388608.0f);
    const bool up_lo = uf < __fmul_rn(a, 131072.0f);
    const uint32_t lo = big ? (A >> 22) - 252u : (mid ? 1u : 0u);
    return lo + ((mid ? up_hi : up_lo) ? 1u : 0u);
}

// ---------------------------------------------------------------------------
// Scale tile layout of the block-scaled MMA (see tj.h): byte offset of the scale
// of (row, group) for a tensor with `ntile_k` = cols_p / (4 * group) tiles per row
// tile.  Groups 4kt..4kt+3 of one row are 4 consecutive bytes.
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ int64_t sf_word_offset(int64_t row, int64_t kt, int64_t ntile_k) {
    const int64_t rt = row >> 7, rr = row & 127;
    return (rt * ntile_k + kt) * 512 + 16 * (rr & 31) + 4 * (rr >> 5);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) { return __uint_as_float(h << 16); }

// max(|a|, |b|, |c|) (one three-input maximum; NaN inputs are not propagated)
__device__ __forceinline__ float amax3(float a, float b, float c) {
    float d;
    asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// ---------------------------------------------------------------------------
// Packed fp32 pairs (one 64-bit register, low word = first element): the sm_100+
// f32x2 instructions round each half exactly like the scalar instruction.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// a * b + c rounded toward +infinity
__device__ __forceinline__ uint64_t f2_fma_rp(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rp.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Stochastic rounding of two scaled values y0, y1 (fp32, |y| may exceed 6 slightly)
// to signed E2M1 codes, returned in bits 28..31 of the two results (bits 0..27 are
// not part of the code).  u_lo4096 / u_hi4096 hold each element's 16-bit uniform U
// at bits 12..27 (U << 12, other bits zero).  Same decision as e2m1_sr on
// a = min(|y|, 6), with the sign of y:
//   a >= 1: the float bits A of a carry the grid index in bits 22.. (index
//           (A >> 22) - 252) and the fraction p * 2^22 in bits 0..21;
//   a < 1:  the grid {0, .5, 1} is uniform, and 0.5 + a / 2 rounded up to a
//           multiple of 2^-24 has the bits 0x3F000000 + ceil(a * 2^23), index *
//           2^22 plus the fraction rounded up (exact for the test below, whose
//           left side is a multiple of 64);
// the larger of the two floats is the right one in each range.  Adding
// 2^22 - 1 - 64 U to that bit pattern carries into the index exactly when the
// fraction exceeds 64 U, which is the exact test U < p * 2^16.  The sum minus
// 0x3F000000, times 64, puts the index in bits 28..30 (the index is <= 7, so bit
// 31 is clear); the sign of y fills bit 31.  y = -0 gives the code of -0.
__device__ __forceinline__ void e2m1x2_sr_nib(uint64_t y2, uint32_t u_lo4096, uint32_t u_hi4096, uint32_t &t0,
                                              uint32_t &t1) {
    float y0, y1;
    f2_unpack(y2, y0, y1);
    const float a0 = fminf(fabsf(y0), 6.0f), a1 = fminf(fabsf(y1), 6.0f);
    float f0, f1;
    f2_unpack(f2_fma_rp(f2_pack(a0, a1), f2_pack(0.5f, 0.5f), f2_pack(0.5f, 0.5f)), f0, f1);
    const uint32_t s0 = __float_as_uint(fmaxf(f0, a0)), s1 = __float_as_uint(fmaxf(f1, a1));
    // (2^22 - 1 - 64 U) * 64 - 0x3F000000 * 64 (mod 2^32) = 0x4FFFFFC0 - 4096 U, and
    // 4096 U only has bits that 0x4FFFFFC0 has, so the subtraction is an xor
    t0 = (s0 * 64u + (u_lo4096 ^ 0x4FFFFFC0u)) | (__float_as_uint(y0) & 0x80000000u);
    t1 = (s1 * 64u + (u_hi4096 ^ 0x4FFFFFC0u)) | (__float_as_uint(y1) & 0x80000000u);
}

}  // namespace tj
