// quant.cu - quantize kernels (sm_103a): row-wise and transposed-alignment
// double-block NVFP4 (RTN / SR, optional RHT), the MXFP8 outlier slice, the
// standalone RHT and fp32 dequantization.  TetraJet-v2 technical summary §2.A
// (double-block quantization, SR, 1x16 groups re-aligned for the transposed
// operand) and §2.C (RHT, FP8 outlier channels).
//
// HBM-bound kernels: every input byte is read once with coalesced loads, every
// output written once; no intermediate fp32/bf16 tensor is materialised.
#include "quant_core.cuh"
#include "tj_internal.h"

namespace tj {

// ---------------------------------------------------------------------------
// Sources.  elem(r, c) is the fp32 value at input row r and (selected) column c;
// rows beyond `rows` or columns beyond the selection read as 0 (zero padding).
// ---------------------------------------------------------------------------
template <typename T>
struct SrcDense {
    const T *p;
    int64_t ld, rows, cols;   // cols = number of (selected) columns
    const int32_t *sel;       // nullptr: identity
    __device__ __forceinline__ float load(int64_t r, int64_t c) const {
        if (r >= rows || c >= cols) return 0.0f;
        const int64_t ci = sel ? (int64_t)sel[c] : c;
        return to_f(p[r * ld + ci]);
    }
    __device__ static __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ static __forceinline__ float to_f(float v) { return v; }
    // elem(r, c .. c+7), c a multiple of 8: one or two 16-byte loads when the octet is
    // inside the tensor, unselected and 16-byte aligned.  flip = ~0u negates all eight
    // (the RHT diagonal entry of input row r), 0 leaves them.
    __device__ __forceinline__ void load8(int64_t r, int64_t c, float (&v)[8], uint32_t flip = 0u) const {
        const T *q = p + r * ld + c;
        if (sel == nullptr && r < rows && c + 8 <= cols && (reinterpret_cast<uintptr_t>(q) & 15) == 0) {
            vec8(q, v, flip);
            return;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(__float_as_uint(load(r, c + j)) ^ (flip & 0x80000000u));
    }
    __device__ static __forceinline__ void vec8(const __nv_bfloat16 *q, float (&v)[8], uint32_t flip) {
        const uint4 w = __ldg(reinterpret_cast<const uint4 *>(q));
        const uint32_t f = flip & 0x80008000u;
        const uint32_t ws[4] = {w.x ^ f, w.y ^ f, w.z ^ f, w.w ^ f};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[2 * k] = __uint_as_float(ws[k] << 16);
            v[2 * k + 1] = __uint_as_float(ws[k] & 0xFFFF0000u);
        }
    }
    __device__ static __forceinline__ void vec8(const float *q, float (&v)[8], uint32_t flip) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(q)), b = __ldg(reinterpret_cast<const float4 *>(q) + 1);
        const float av[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        const uint32_t f = flip & 0x80000000u;
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = __uint_as_float(__float_as_uint(av[k]) ^ f);
    }
};

// NVFP4 tensor [rows, cols] read back as its fp32 dequantization (G * s_i) * s_o.
struct SrcNv {
    const uint8_t *codes, *sf;
    const float *outer;
    int64_t rows, cols, rows_p, cols_p;
    __device__ __forceinline__ float load(int64_t r, int64_t c) const {
        if (r >= rows || c >= cols) return 0.0f;
        const uint32_t byte = codes[r * (cols_p / 2) + (c >> 1)];
        const uint32_t code = (c & 1) ? (byte >> 4) : (byte & 15u);
        const int64_t g = c >> 4;
        const uint32_t sb = sf[sf_word_offset(r, g >> 2, cols_p / 64) + (g & 3)];
        const uint32_t mag = code & 7u;
        const float gv = mag < 4u ? __fmul_rn((float)mag, 0.5f)
                                  : (mag == 4u ? 2.0f : (mag == 5u ? 3.0f : (mag == 6u ? 4.0f : 6.0f)));
        const float v = __fmul_rn(__fmul_rn(gv, e4m3_to_float(sb)), outer[(c >> 7) * rows_p + r]);
        return (code & 8u) ? -v : v;
    }
    // elem(r, c .. c+7), c a multiple of 8, inside the padded tensor (whose padding holds
    // zero codes and scales): one 4-byte code load, one scale byte, one outer scale.
    // Two codes' magnitudes at a time are looked up as 2G in {0,1,2,3,4,6,8,12} with a
    // byte permute, turned into fp32 exactly, and scaled as (G * s_i) * s_o.
    __device__ __forceinline__ void load8(int64_t r, int64_t c, float (&v)[8], uint32_t flip = 0u) const {
        // flipping the eight code sign bits negates the eight values (zeros included)
        const uint32_t w = *reinterpret_cast<const uint32_t *>(codes + r * (cols_p / 2) + (c >> 1)) ^ (flip & 0x88888888u);
        const int64_t g = c >> 4;
        const uint32_t sb = sf[sf_word_offset(r, g >> 2, cols_p / 64) + (g & 3)];
        const float half_si = __fmul_rn(e4m3_to_float(sb), 0.5f);        // exact
        const float so = outer[(c >> 7) * rows_p + r];
        const uint32_t mag = w & 0x77777777u;
        const uint32_t two_g[2] = {__byte_perm(0x03020100u, 0x0C080604u, mag & 0xFFFFu),
                                   __byte_perm(0x03020100u, 0x0C080604u, mag >> 16)};
        const uint64_t m2 = f2_pack(-8388608.0f, -8388608.0f), hs2 = f2_pack(half_si, half_si), so2 = f2_pack(so, so);
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            // 0x4B0000nn = 2^23 + nn as fp32; subtracting 2^23 leaves nn = 2G exactly.  Two
            // elements at a time on packed f32x2 instructions, which round each half like
            // the scalar ones: (2G * s_i / 2) * s_o
            const uint64_t gg = f2_add(f2_pack(__uint_as_float(__byte_perm(two_g[k >> 2], 0x4B000000u, (k & 3) | 0x7440)),
                                               __uint_as_float(__byte_perm(two_g[k >> 2], 0x4B000000u, ((k + 1) & 3) | 0x7440))),
                                       m2);
            float a0, a1;
            f2_unpack(f2_mul(f2_mul(gg, hs2), so2), a0, a1);
            v[k] = __uint_as_float(__float_as_uint(a0) ^ ((w << (28 - 4 * k)) & 0x80000000u));
            v[k + 1] = __uint_as_float(__float_as_uint(a1) ^ ((w << (24 - 4 * k)) & 0x80000000u));
        }
    }
};

// MX slice [rows, cols] read back as fp32 (element value times 2^(byte-127)), in the
// slice's element format (E4M3 bytes, packed 6-bit E2M3 / E3M2 or packed 4-bit E2M1).
struct SrcMx {
    const uint8_t *codes, *sf;
    int64_t rows, cols, rows_p, cols_p;
    int fmt;
    __device__ __forceinline__ float scale(int64_t r, int64_t c) const {
        const int64_t g = c >> 5;
        const int e = (int)sf[sf_word_offset(r, g >> 2, cols_p / 128) + (g & 3)] - 127;
        return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x400000u);
    }
    __device__ __forceinline__ float value(uint32_t code) const {
        return fmt == kMxE4M3 ? e4m3_to_float(code)
                              : (fmt == kMxE2M1 ? e2m1_to_float(code)
                                                : (fmt == kMxE2M3 ? e2m3_to_float(code) : e3m2_to_float(code)));
    }
    __device__ __forceinline__ float load(int64_t r, int64_t c) const {
        if (r >= rows || c >= cols) return 0.0f;
        const uint8_t *row = codes + r * (cols_p * mx_bits(fmt) / 8);
        uint32_t code;
        if (fmt == kMxE4M3) {
            code = row[c];
        } else if (fmt == kMxE2M1) {
            code = (row[c >> 1] >> (4 * (c & 1))) & 15u;
        } else {                                       // bits 6c .. 6c+5 of the row
            const int64_t b = (6 * c) >> 3;
            const int sh = (int)((6 * c) & 7);
            uint32_t w = row[b];
            if (sh > 2) w |= (uint32_t)row[b + 1] << 8;   // the code spills into the next byte
            code = (w >> sh) & 63u;
        }
        return __fmul_rn(value(code), scale(r, c));
    }
    // elem(r, c .. c+7), c a multiple of 8, inside the padded tensor: one 8-, 6- or 4-byte
    // read of the eight codes (never used with the RHT: flip must be 0)
    __device__ __forceinline__ void load8(int64_t r, int64_t c, float (&v)[8], uint32_t flip = 0u) const {
        const float s = scale(r, c);
        if (fmt == kMxE4M3) {
            const uint2 w = *reinterpret_cast<const uint2 *>(codes + r * cols_p + c);
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = __fmul_rn(e4m3_to_float(((k < 4 ? w.x : w.y) >> (8 * (k & 3))) & 0xFFu), s);
        } else if (fmt == kMxE2M1) {
            const uint32_t w = *reinterpret_cast<const uint32_t *>(codes + r * (cols_p / 2) + (c >> 1));
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = __fmul_rn(e2m1_to_float((w >> (4 * k)) & 15u), s);
        } else {                                       // 6 bytes at a 2-byte boundary
            const uint16_t *p = reinterpret_cast<const uint16_t *>(codes + r * (cols_p / 4 * 3) + (c / 4) * 3);
            const uint64_t w = (uint64_t)p[0] | ((uint64_t)p[1] << 16) | ((uint64_t)p[2] << 32);
            const bool e3 = fmt == kMxE3M2;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t code = (uint32_t)(w >> (6 * k)) & 63u;
                v[k] = __fmul_rn(e3 ? e3m2_to_float(code) : e2m3_to_float(code), s);
            }
        }
    }
};

// Fast path of the row kernel: 32 consecutive bf16 of one row, 64-byte aligned.
__device__ __forceinline__ void load32_bf16_vec(const __nv_bfloat16 *p, float (&x)[32]) {
    const uint4 *q = reinterpret_cast<const uint4 *>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = __ldg(q + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[8 * i + 2 * k] = bf16_bits_to_float(w[k] & 0xFFFFu);
            x[8 * i + 2 * k + 1] = bf16_bits_to_float(w[k] >> 16);
        }
    }
}

template <typename Src>
__device__ __forceinline__ void load_row32(const Src &src, int64_t r, int64_t c0, float (&x)[32]) {
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = src.load(r, c0 + j);
}

__device__ __forceinline__ void load_row32(const SrcDense<__nv_bfloat16> &src, int64_t r, int64_t c0,
                                           float (&x)[32]) {
    if (src.sel == nullptr && r < src.rows && c0 + 32 <= src.cols && (src.ld & 31) == 0 &&
        ((reinterpret_cast<uintptr_t>(src.p) & 63) == 0)) {
        load32_bf16_vec(src.p + r * src.ld + c0, x);
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = src.load(r, c0 + j);
    }
}

// ---------------------------------------------------------------------------
// Row-wise kernel: output row r = input row r, quantized along the columns.
// One quad per (row, 128-block); a warp covers 8 consecutive segments.
// FMT 0 = NVFP4, 1 = MXFP8, 2 = both from one read (MXFP8 of the input, NVFP4 of
// its optional RHT), into outputs of the same shape.
// ---------------------------------------------------------------------------
template <typename Src, int FMT, bool SR, bool RHT>
__global__ void __launch_bounds__(256, 4) k_quant_rows(Src src, OutNv onv, OutMx omx, int64_t nseg, const PhiloxKeys pk,
                                                    uint32_t tag, uint32_t rht_tag) {
    const int lane = threadIdx.x & 31;
    const int t = lane & 3;
    const int64_t rows_p = FMT != 1 ? onv.rows_p : omx.rows_p;
    const int64_t cols_p = FMT != 1 ? onv.cols_p : omx.cols_p;
    const int64_t total = rows_p * nseg;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    uint32_t sign_word = 0u;
    if (RHT) {
        const uint4 sb = rht_sign_bits(pk, rht_tag);
        sign_word = t == 0 ? sb.x : (t == 1 ? sb.y : (t == 2 ? sb.z : sb.w));
    }
    // segment seg = row * nseg + kb of this quad; the (row, kb) pair advances by the loop
    // stride without a division per iteration.  Segment counts fit in 32 bits: the C ABI
    // rejects tensors of 2^31 or more 128-element blocks.
    const uint32_t nseg32 = (uint32_t)nseg;
    const uint32_t stride = (uint32_t)(nwarps * 8);
    const uint32_t seg0 = (uint32_t)(warp0 * 8) + (uint32_t)(lane >> 2);
    const uint32_t d_row = stride / nseg32, d_kb = stride % nseg32;
    uint32_t row_i = seg0 / nseg32, kb_i = seg0 % nseg32;
    for (int64_t base = warp0 * 8; base < total; base += stride) {   // warp-uniform loop
        const bool valid = (int64_t)row_i < rows_p;
        const int64_t row = valid ? (int64_t)row_i : 0;
        const int64_t kb = valid ? (int64_t)kb_i : 0;
        row_i += d_row;
        kb_i += d_kb;
        if (kb_i >= nseg32) {
            kb_i -= nseg32;
            ++row_i;
        }
        float x[32];
        if (valid) load_row32(src, row, kb * 128 + 32 * t, x);
        else {
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = 0.0f;
        }
        if (FMT != 1) {
            if (FMT == 2) {
                const MxSeg m = quant_mx_group(x, omx.fmt);
                store_mx_seg(omx, row, kb, t, m, valid);
            }
            if (RHT) {
                // an opaque copy per segment: otherwise the compiler hoists the 32 sign masks
                // (sign_word << (31 - j)) out of the loop, where they spill (6% of the kernel)
                uint32_t sw;
                asm volatile("mov.b32 %0, %1;" : "=r"(sw) : "r"(sign_word));
                rht128_quad(x, sw, t);
            }
            const NvSeg s = quant_nvfp4_seg<SR>(x, (uint64_t)(row * cols_p + kb * 128 + 32 * t), pk, tag);
            store_nv_seg(onv, row, kb, t, s, valid);
        } else {
            const MxSeg s = quant_mx_group(x, omx.fmt);
            store_mx_seg(omx, row, kb, t, s, valid);
        }
    }
}

// ---------------------------------------------------------------------------
// Transposed-alignment kernel: output row c = input column c, quantized along
// the input rows.  A CTA stages a 128 (input rows = one output block) x 64
// (output rows) fp32 tile in shared memory, then each quad quantizes one output
// row's 128-segment.  The tile is XOR-swizzled so that both the row-major fill
// and the column reads (lanes = 8 columns x 4 quad lanes) are conflict-free:
// element (r, c) sits at r*64 + (c ^ (((r >> 5) & 3) << 3)).
// ---------------------------------------------------------------------------
// One tile (output rows 64 bx .., input-row block by), with the CTA's staging tile.
template <typename Src, int FMT, bool SR, bool RHT>
__device__ __forceinline__ void quant_cols_tile(const Src &src, const OutNv &onv, const OutMx &omx, const PhiloxKeys &pk,
                                                uint32_t tag, uint32_t rht_tag, int64_t bx, int64_t by, float *tile) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t c0 = bx * 64;                       // first output row of the tile
    const int64_t kb = by;                            // 128-block along the input rows
    const int64_t r0 = kb * 128;
    // with the RHT, input row rr (element rr of every output segment) is negated while
    // loading when its diagonal entry is -1
    const uint4 sbits = RHT && FMT != 1 ? rht_sign_bits(pk, rht_tag) : make_uint4(0u, 0u, 0u, 0u);
    // fill: 128 rows x 8 column octets, one octet (8 consecutive columns of a row) per
    // thread and pass, stored as two 16-byte words (the swizzle keeps an octet contiguous)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = i * 256 + (int)threadIdx.x;
        const int rr = idx >> 3, o = idx & 7;                   // rr = 32 i + threadIdx.x / 8
        const uint32_t sw = i == 0 ? sbits.x : (i == 1 ? sbits.y : (i == 2 ? sbits.z : sbits.w));
        const uint32_t flip = 0u - ((sw >> (threadIdx.x >> 3)) & 1u);
        float v[8];
        src.load8(r0 + rr, c0 + 8 * o, v, flip);
        float4 *dst = reinterpret_cast<float4 *>(&tile[rr * 64 + ((8 * o) ^ (((rr >> 5) & 3) << 3))]);
        dst[0] = make_float4(v[0], v[1], v[2], v[3]);
        dst[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
    __syncthreads();
    const int t = lane & 3;
    const int cl = warp * 8 + (lane >> 2);            // output row within the tile
    float x[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = tile[(32 * t + j) * 64 + (cl ^ (t << 3))];
    const int64_t row = c0 + cl;
    const int64_t rows_p = FMT != 1 ? onv.rows_p : omx.rows_p;
    const int64_t cols_p = FMT != 1 ? onv.cols_p : omx.cols_p;
    const bool valid = row < rows_p;
    if (FMT != 1) {
        const uint32_t sign_word = t == 0 ? sbits.x : (t == 1 ? sbits.y : (t == 2 ? sbits.z : sbits.w));
        if (FMT == 2) {
            const MxSeg m = quant_mx_group<RHT>(x, omx.fmt, sign_word);
            store_mx_seg(omx, row, kb, t, m, valid);
        }
        if (RHT) rht128_quad<false>(x, sign_word, t);
        const NvSeg s = quant_nvfp4_seg<SR>(x, (uint64_t)(row * cols_p + r0 + 32 * t), pk, tag);
        store_nv_seg(onv, row, kb, t, s, valid);
    } else {
        const MxSeg s = quant_mx_group(x, omx.fmt);
        store_mx_seg(omx, row, kb, t, s, valid);
    }
}

template <typename Src, int FMT, bool SR, bool RHT>
__global__ void __launch_bounds__(256, (FMT == 2 || (FMT == 0 && !SR && !RHT)) ? 5 : 4) k_quant_cols(Src src, OutNv onv, OutMx omx, const PhiloxKeys pk, uint32_t tag,
                                                    uint32_t rht_tag) {
    __shared__ __align__(16) float tile[128 * 64];
    quant_cols_tile<Src, FMT, SR, RHT>(src, onv, omx, pk, tag, rht_tag, blockIdx.x, blockIdx.y, tile);
}

// The backward re-alignment of a forward NVFP4 operand and of its outlier slice in one
// launch: blocks [0, nb) take the slice's tiles (nxb per input-row block), the others the
// NVFP4 operand's (nxa per input-row block).  Alone the slice's few tiles leave the GPU
// mostly idle; here they run beside the operand's.
template <bool SR, bool RHT>
__global__ void __launch_bounds__(256, 4) k_realign_pair(SrcNv sa, OutNv oa, SrcMx sb, OutMx ob, const PhiloxKeys pk,
                                                         uint32_t tag, uint32_t rht_tag, int nxa, int nxb, int nb) {
    __shared__ __align__(16) float tile[128 * 64];
    const int b = (int)blockIdx.x;
    if (b < nb) quant_cols_tile<SrcMx, 1, false, false>(sb, OutNv{}, ob, pk, 0u, 0u, b % nxb, b / nxb, tile);
    else quant_cols_tile<SrcNv, 0, SR, RHT>(sa, oa, OutMx{}, pk, tag, rht_tag, (b - nb) % nxa, (b - nb) / nxa, tile);
}

// ---------------------------------------------------------------------------
// OutControl split of a forward operand, row-wise, one read (§2.C): the normal
// channels (ascending `sel_n`, compacted) -> NVFP4 RTN, the outlier channels
// (`sel_o`) -> MXFP8.  Same results as the two gathering calls
// (tj_quantize_nvfp4 RTN with sel = normal, tj_quantize_mxfp8 with sel = outliers).
//
// A CTA stages tiles of `tr` whole input rows in shared memory as 32-bit words,
// two pad words after every 32, and gathers the selected columns from there
// through two tables of byte offsets built once per CTA.  Two staging buffers: the
// rows of the next tile arrive by asynchronous copies (cp.async, 8 bytes each, which
// the two-word pad keeps aligned) while the current tile is gathered and quantized.
// The tables list the channels in output order, padded by 4 entries after every 32,
// so a lane reads its 32 offsets with eight 16-byte loads; entries past the end of a
// list point at a zero word of the row.  The quads of all warps take (row, segment)
// tasks of the whole tile: first every NVFP4 task, then every MXFP8 task.
// ---------------------------------------------------------------------------
constexpr int kSplitThreads = 256;

// words of one staged row: the data words, two pads after every 32, one zero word, 16-byte rows
__host__ __device__ inline int split_row_words(int K, int esz) {
    const int nw = esz == 2 ? (K + 1) / 2 : K;
    return (int)round_up(nw + 2 * ((nw + 31) / 32) + 1, 4);
}
__host__ __device__ inline int split_tab_words(int len) { return len + len / 8; }    // len: a multiple of 128
__device__ __forceinline__ int split_pad_row(int w) { return w + 2 * (w >> 5); }

// 8-byte asynchronous copy global -> shared; src_bytes 0 writes zeros and reads nothing
__device__ __forceinline__ void cp_async8(void *smem_dst, const void *gsrc, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
                 "l"(gsrc), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ int split_pad_tab(int i) { return i + 4 * (i >> 5); }

template <typename T>
__device__ __forceinline__ uint32_t split_byte_off(int c) {
    return sizeof(T) == 2 ? 4u * (uint32_t)split_pad_row(c >> 1) + 2u * (uint32_t)(c & 1)
                          : 4u * (uint32_t)split_pad_row(c);
}

// input word w (elements 2w, 2w+1 for bf16; element w for fp32) of row `row`, zero past the end
template <typename T>
__device__ __forceinline__ uint32_t split_word(const T *x, int64_t ld, int64_t row, int64_t rows, int K, int w) {
    if (row >= rows) return 0u;
    const T *p = x + row * ld;
    if (sizeof(T) == 2) {
        const uint32_t lo = 2 * w < K ? (uint32_t)__bfloat16_as_ushort(reinterpret_cast<const __nv_bfloat16 *>(p)[2 * w]) : 0u;
        const uint32_t hi = 2 * w + 1 < K ? (uint32_t)__bfloat16_as_ushort(reinterpret_cast<const __nv_bfloat16 *>(p)[2 * w + 1]) : 0u;
        return lo | (hi << 16);
    }
    return w < K ? __float_as_uint(reinterpret_cast<const float *>(p)[w]) : 0u;
}

template <typename T>
__device__ __forceinline__ float split_elem(const uint8_t *p) {
    if (sizeof(T) == 2) return __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t *>(p) << 16);
    return *reinterpret_cast<const float *>(p);
}

// 32 elements of one staged row through 32 table entries (8 x 16-byte reads)
template <typename T>
__device__ __forceinline__ void split_gather32(const uint8_t *rowp, const uint32_t *tab, float (&v)[32]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint4 o = *reinterpret_cast<const uint4 *>(tab + 4 * i);
        v[4 * i] = split_elem<T>(rowp + o.x);
        v[4 * i + 1] = split_elem<T>(rowp + o.y);
        v[4 * i + 2] = split_elem<T>(rowp + o.z);
        v[4 * i + 3] = split_elem<T>(rowp + o.w);
    }
}

template <typename T>
__global__ void __launch_bounds__(kSplitThreads) k_quant_split(const T *x, int64_t ld, int64_t rows, int K,
                                                              const int32_t *sel_n, int kn, const int32_t *sel_o,
                                                              int k, OutNv onv, OutMx omx, int tr) {
    extern __shared__ __align__(16) uint8_t smem_split[];
    const int nseg_n = (int)(onv.cols_p / 128), nseg_o = k > 0 ? (int)(omx.cols_p / 128) : 0;
    const int rw = split_row_words(K, (int)sizeof(T));
    uint32_t *tab_n = reinterpret_cast<uint32_t *>(smem_split);
    uint32_t *tab_o = tab_n + split_tab_words(128 * nseg_n);
    uint32_t *tiles[2];
    tiles[0] = tab_o + split_tab_words(128 * nseg_o);
    tiles[1] = tiles[0] + tr * rw;
    const uint32_t zero_off = 4u * (uint32_t)(rw - 1);
    for (int i = threadIdx.x; i < 128 * nseg_n; i += blockDim.x)
        tab_n[split_pad_tab(i)] = i < kn ? split_byte_off<T>(sel_n[i]) : zero_off;
    for (int i = threadIdx.x; i < 128 * nseg_o; i += blockDim.x)
        tab_o[split_pad_tab(i)] = i < k ? split_byte_off<T>(sel_o[i]) : zero_off;
    for (int r = threadIdx.x; r < 2 * tr; r += blockDim.x) tiles[0][r * rw + rw - 1] = 0u;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = lane & 3, qd = lane >> 2;
    const int nwarp = blockDim.x >> 5;
    const int64_t rows_p = onv.rows_p;
    const int64_t ntile = (rows_p + tr - 1) / tr;
    const bool vec = ((reinterpret_cast<uintptr_t>(x) & 15) == 0) && ((ld * (int64_t)sizeof(T)) % 16 == 0);
    constexpr int kv = 16 / (int)sizeof(T);              // elements per 16-byte chunk
    const int nch = vec ? K / kv : 0;                    // full chunks per row, copied asynchronously
    const int nw = sizeof(T) == 2 ? (K + 1) / 2 : K;     // data words per row
    const int wtail = 4 * nch, ntail = nw - wtail;       // words loaded one at a time
    const int fill_dr = nch > 0 ? (int)blockDim.x / nch : 0, fill_dc = (int)blockDim.x - fill_dr * nch;
    // the (row, segment) of a quad's task, stepped by nwarp * 8 tasks per pass
    const int step_t = nwarp * 8;
    const int dr_n = nseg_n > 0 ? step_t / nseg_n : 0, dk_n = step_t - dr_n * nseg_n;
    const int dr_o = nseg_o > 0 ? step_t / nseg_o : 0, dk_o = step_t - dr_o * nseg_o;

    // Start the copies of tile tl's rows into buf: chunk i of the tile is (row i / nch, chunk
    // i % nch), stepped by blockDim.x chunks with a carry instead of dividing; rows past the end
    // are filled with zeros.  The words past a row's last full chunk are loaded and stored here.
    auto stage = [&](int64_t tl, uint32_t *buf) {
        const int64_t r0 = tl * tr;
        int fr = (int)threadIdx.x / (nch > 0 ? nch : 1), fc = (int)threadIdx.x - fr * nch;   // chunk threadIdx.x
        for (int i = threadIdx.x; i < tr * nch; i += blockDim.x) {
            const int rr = fr, cc = fc;
            fr += fill_dr;
            fc += fill_dc;
            if (fc >= nch) { fc -= nch; ++fr; }
            const bool in = r0 + rr < rows;
            const uint8_t *src = reinterpret_cast<const uint8_t *>(in ? x + (r0 + rr) * ld + (int64_t)cc * kv : x);
            uint32_t *d = buf + rr * rw + split_pad_row(4 * cc);       // 4 words inside one 32-word run
            cp_async8(d, src, in ? 8u : 0u);
            cp_async8(d + 2, src + (in ? 8 : 0), in ? 8u : 0u);
        }
        for (int i = threadIdx.x; i < tr * ntail; i += blockDim.x) {
            const int r = i / ntail, w = wtail + (i - r * ntail);
            buf[r * rw + split_pad_row(w)] = split_word(x, ld, r0 + r, rows, K, w);
        }
    };
    int64_t tl = blockIdx.x;
    if (tl < ntile) stage(tl, tiles[0]);
    cp_async_commit();
    for (int b = 0; tl < ntile; tl += gridDim.x, b ^= 1) {
        const int64_t r0 = tl * tr;
        const uint32_t *tile = tiles[b];
        if (tl + gridDim.x < ntile) stage(tl + gridDim.x, tiles[b ^ 1]);   // lands during this tile
        cp_async_commit();
        cp_async_wait_one();                             // this thread's copies of tile tl have landed
        __syncthreads();                                 // ... and every thread's
        const int nt_n = tr * nseg_n;
        int tr_n = nseg_n > 0 ? (warp * 8 + qd) / nseg_n : 0, tk_n = (warp * 8 + qd) - tr_n * nseg_n;   // task warp*8 + qd
        for (int q0 = warp * 8; q0 < nt_n; q0 += nwarp * 8) {          // warp-uniform
            const int task = q0 + qd;
            const bool ok = task < nt_n;
            const int r = ok ? tr_n : 0, kb = ok ? tk_n : 0;
            tr_n += dr_n;
            tk_n += dk_n;
            if (tk_n >= nseg_n) { tk_n -= nseg_n; ++tr_n; }
            float v[32];
            split_gather32<T>(reinterpret_cast<const uint8_t *>(tile + r * rw), tab_n + split_pad_tab(kb * 128 + 32 * t), v);
            const NvSeg sg = quant_nvfp4_seg<false>(v, 0, PhiloxKeys{}, 0u);
            store_nv_seg(onv, r0 + r, kb, t, sg, ok && r0 + r < rows_p);
        }
        const int nt_o = tr * nseg_o;
        int tr_o = nseg_o > 0 ? (warp * 8 + qd) / nseg_o : 0, tk_o = (warp * 8 + qd) - tr_o * nseg_o;
        for (int q0 = warp * 8; q0 < nt_o; q0 += nwarp * 8) {
            const int task = q0 + qd;
            const bool ok = task < nt_o;
            const int r = ok ? tr_o : 0, kb = ok ? tk_o : 0;
            tr_o += dr_o;
            tk_o += dk_o;
            if (tk_o >= nseg_o) { tk_o -= nseg_o; ++tr_o; }
            float v[32];
            split_gather32<T>(reinterpret_cast<const uint8_t *>(tile + r * rw), tab_o + split_pad_tab(kb * 128 + 32 * t), v);
            const MxSeg m = quant_mx_group(v, omx.fmt);
            store_mx_seg(omx, r0 + r, kb, t, m, ok && r0 + r < omx.rows_p);
        }
        __syncthreads();                                 // the gathers are done before the buffer is refilled
    }
}

// ---------------------------------------------------------------------------
// Standalone RHT (fp32 -> fp32), one quad per 128-block, same butterfly as the
// fused quantizers.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_rht(const float *x, float *y, int64_t rows, int64_t cols, const PhiloxKeys pk,
                                             uint32_t tag) {
    const int lane = threadIdx.x & 31, t = lane & 3;
    const int64_t nseg = cols / 128, total = rows * nseg;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const uint4 sb = rht_sign_bits(pk, tag);
    const uint32_t sign_word = t == 0 ? sb.x : (t == 1 ? sb.y : (t == 2 ? sb.z : sb.w));
    for (int64_t base = warp0 * 8; base < total; base += nwarps * 8) {
        const int64_t seg = base + (lane >> 2);
        const bool valid = seg < total;
        const int64_t off = valid ? (seg / nseg) * cols + (seg % nseg) * 128 + 32 * t : 0;
        float v[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 f = valid ? reinterpret_cast<const float4 *>(x + off)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
            v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
        }
        rht128_quad(v, sign_word, t);
        if (valid) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                reinterpret_cast<float4 *>(y + off)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
    }
}

// fp32 dequantization of an NVFP4 tensor, one thread per element.
__global__ void k_dequant_nv(SrcNv src, float *y, int64_t ldy) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= src.rows * src.cols) return;
    const int64_t r = i / src.cols, c = i % src.cols;
    y[r * ldy + c] = src.load(r, c);
}

// fp32 values of an MXFP8 tensor, one thread per element.
__global__ void k_dequant_mx(SrcMx src, float *y, int64_t ldy) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= src.rows * src.cols) return;
    const int64_t r = i / src.cols, c = i % src.cols;
    y[r * ldy + c] = src.load(r, c);
}

// ---------------------------------------------------------------------------
// Host launchers.
// ---------------------------------------------------------------------------
namespace {
constexpr int kThreads = 256;

int64_t row_grid(int64_t total_segments) {
    const int64_t ctas = (total_segments + 63) / 64;          // 64 segments per CTA pass
    return ctas < 152 * 32 ? (ctas > 0 ? ctas : 1) : 152 * 32;
}

OutNv out_nv(const tj_nvfp4 &q) {
    return OutNv{q.codes, q.sf, q.outer, round_up(q.rows, 128), round_up(q.cols, 128)};
}
OutMx out_mx(const tj_mxfp8 &q) {
    return OutMx{q.codes, q.sf, round_up(q.rows, 128), round_up(q.cols, 128), (int)q.fmt};
}

template <typename Src, int FMT = 0>
cudaError_t rows_nv(const Src &src, const OutNv &o, int mode, int rht, uint64_t seed, uint32_t tag,
                    uint32_t rht_tag, cudaStream_t s, const OutMx none = OutMx{}) {
    const int64_t nseg = o.cols_p / 128, grid = row_grid(o.rows_p * nseg);
    const PhiloxKeys pk = philox_keys(seed);
    if (mode == TJ_SR && rht)  k_quant_rows<Src, FMT, true, true><<<grid, kThreads, 0, s>>>(src, o, none, nseg, pk, tag, rht_tag);
    else if (mode == TJ_SR)    k_quant_rows<Src, FMT, true, false><<<grid, kThreads, 0, s>>>(src, o, none, nseg, pk, tag, rht_tag);
    else if (rht)              k_quant_rows<Src, FMT, false, true><<<grid, kThreads, 0, s>>>(src, o, none, nseg, pk, tag, rht_tag);
    else                       k_quant_rows<Src, FMT, false, false><<<grid, kThreads, 0, s>>>(src, o, none, nseg, pk, tag, rht_tag);
    return cudaGetLastError();
}

template <typename Src, int FMT = 0>
cudaError_t cols_nv(const Src &src, const OutNv &o, int mode, int rht, uint64_t seed, uint32_t tag,
                    uint32_t rht_tag, cudaStream_t s, const OutMx none = OutMx{}) {
    if (o.rows_p == 0 || o.cols_p == 0) return cudaSuccess;          // an empty output
    const dim3 grid((unsigned)(o.rows_p / 64), (unsigned)(o.cols_p / 128));
    const PhiloxKeys pk = philox_keys(seed);
    if (mode == TJ_SR && rht)  k_quant_cols<Src, FMT, true, true><<<grid, kThreads, 0, s>>>(src, o, none, pk, tag, rht_tag);
    else if (mode == TJ_SR)    k_quant_cols<Src, FMT, true, false><<<grid, kThreads, 0, s>>>(src, o, none, pk, tag, rht_tag);
    else if (rht)              k_quant_cols<Src, FMT, false, true><<<grid, kThreads, 0, s>>>(src, o, none, pk, tag, rht_tag);
    else                       k_quant_cols<Src, FMT, false, false><<<grid, kThreads, 0, s>>>(src, o, none, pk, tag, rht_tag);
    return cudaGetLastError();
}

template <typename Src>
cudaError_t rows_mx(const Src &src, const OutMx &o, cudaStream_t s) {
    const int64_t nseg = o.cols_p / 128, grid = row_grid(o.rows_p * nseg);
    k_quant_rows<Src, 1, false, false><<<grid, kThreads, 0, s>>>(src, OutNv{}, o, nseg, PhiloxKeys{}, 0, 0);
    return cudaGetLastError();
}

template <typename Src>
cudaError_t cols_mx(const Src &src, const OutMx &o, cudaStream_t s) {
    if (o.rows_p == 0 || o.cols_p == 0) return cudaSuccess;          // an empty output
    const dim3 grid((unsigned)(o.rows_p / 64), (unsigned)(o.cols_p / 128));
    k_quant_cols<Src, 1, false, false><<<grid, kThreads, 0, s>>>(src, OutNv{}, o, PhiloxKeys{}, 0, 0);
    return cudaGetLastError();
}
}  // namespace

SrcNv src_nv(const tj_nvfp4 &q) {
    return SrcNv{q.codes, q.sf, q.outer, q.rows, q.cols, round_up(q.rows, 128), round_up(q.cols, 128)};
}
SrcMx src_mx(const tj_mxfp8 &q) {
    return SrcMx{q.codes, q.sf, q.rows, q.cols, round_up(q.rows, 128), round_up(q.cols, 128), (int)q.fmt};
}

// Dense input (bf16 / fp32) -> NVFP4, either orientation.  n_cols_sel = number of
// selected input columns (cols_x when sel == nullptr).
cudaError_t launch_quant_nv_dense(const void *x, int dtype, int64_t rows_x, int64_t n_cols_sel, int64_t ld,
                                  int along_cols, const int32_t *sel, int mode, int rht, uint64_t seed,
                                  uint32_t tag, uint32_t rht_tag, const tj_nvfp4 &out, cudaStream_t s) {
    const OutNv o = out_nv(out);
    if (dtype == TJ_BF16) {
        const SrcDense<__nv_bfloat16> src{static_cast<const __nv_bfloat16 *>(x), ld, rows_x, n_cols_sel, sel};
        return along_cols ? cols_nv(src, o, mode, rht, seed, tag, rht_tag, s)
                          : rows_nv(src, o, mode, rht, seed, tag, rht_tag, s);
    }
    const SrcDense<float> src{static_cast<const float *>(x), ld, rows_x, n_cols_sel, sel};
    return along_cols ? cols_nv(src, o, mode, rht, seed, tag, rht_tag, s)
                      : rows_nv(src, o, mode, rht, seed, tag, rht_tag, s);
}

// Dense input -> NVFP4 (mode / rht) and MXFP8 of the same elements, one read.
cudaError_t launch_quant_dual_dense(const void *x, int dtype, int64_t rows_x, int64_t n_cols_sel, int64_t ld,
                                    int along_cols, const int32_t *sel, int mode, int rht, uint64_t seed,
                                    uint32_t tag, uint32_t rht_tag, const tj_nvfp4 &out, const tj_mxfp8 &out8,
                                    cudaStream_t s) {
    const OutNv o = out_nv(out);
    const OutMx m = out_mx(out8);
    if (dtype == TJ_BF16) {
        const SrcDense<__nv_bfloat16> src{static_cast<const __nv_bfloat16 *>(x), ld, rows_x, n_cols_sel, sel};
        return along_cols ? cols_nv<decltype(src), 2>(src, o, mode, rht, seed, tag, rht_tag, s, m)
                          : rows_nv<decltype(src), 2>(src, o, mode, rht, seed, tag, rht_tag, s, m);
    }
    const SrcDense<float> src{static_cast<const float *>(x), ld, rows_x, n_cols_sel, sel};
    return along_cols ? cols_nv<decltype(src), 2>(src, o, mode, rht, seed, tag, rht_tag, s, m)
                      : rows_nv<decltype(src), 2>(src, o, mode, rht, seed, tag, rht_tag, s, m);
}

cudaError_t launch_quant_mx_dense(const void *x, int dtype, int64_t rows_x, int64_t n_cols_sel, int64_t ld,
                                  int along_cols, const int32_t *sel, const tj_mxfp8 &out, cudaStream_t s) {
    const OutMx o = out_mx(out);
    if (dtype == TJ_BF16) {
        const SrcDense<__nv_bfloat16> src{static_cast<const __nv_bfloat16 *>(x), ld, rows_x, n_cols_sel, sel};
        return along_cols ? cols_mx(src, o, s) : rows_mx(src, o, s);
    }
    const SrcDense<float> src{static_cast<const float *>(x), ld, rows_x, n_cols_sel, sel};
    return along_cols ? cols_mx(src, o, s) : rows_mx(src, o, s);
}

// OutControl split of a forward operand (row-wise): NVFP4 RTN of the normal channels
// and MXFP8 of the outlier channels from one read of x.  Returns cudaErrorNotSupported
// when a row does not fit the shared-memory staging (the caller then gathers twice).
cudaError_t launch_quant_split(const void *x, int dtype, int64_t rows, int64_t K, int64_t ld, const int32_t *sel_n,
                               int64_t kn, const int32_t *sel_o, int64_t k, const tj_nvfp4 &out,
                               const tj_mxfp8 &out8, cudaStream_t s) {
    if (K > (1 << 24)) return cudaErrorNotSupported;
    if (rows == 0 || K == 0) return cudaSuccess;                      // empty outputs
    const int esz = dtype == TJ_BF16 ? 2 : 4;
    const OutNv o = out_nv(out);
    const OutMx m = k > 0 ? out_mx(out8) : OutMx{};
    const int64_t tabs = 4 * (int64_t)(split_tab_words((int)o.cols_p) + (k > 0 ? split_tab_words((int)m.cols_p) : 0));
    const int64_t row_bytes = 4 * (int64_t)split_row_words((int)K, esz);
    // two staging buffers of about 24 KB of rows each, so that three or four CTAs share an SM
    int64_t tr = (24 * 1024) / row_bytes;
    tr = tr < 1 ? 1 : (tr > 64 ? 64 : tr);
    if (tr >= 8) tr -= tr % 8;     // whole passes of the 64 quads when a row has 8 segments
    const size_t smem = (size_t)(tabs + 2 * tr * row_bytes);
    if (smem > 200 * 1024) return cudaErrorNotSupported;
    const int64_t ntile = (o.rows_p + tr - 1) / tr;
    const int per_sm = smem <= 56 * 1024 ? 4 : (smem <= 75 * 1024 ? 3 : (smem <= 113 * 1024 ? 2 : 1));
    const int64_t grid = ntile < 152 * per_sm ? ntile : 152 * per_sm;
    if (dtype == TJ_BF16) {
        cudaFuncSetAttribute(k_quant_split<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        k_quant_split<__nv_bfloat16><<<(unsigned)grid, kSplitThreads, smem, s>>>(
            static_cast<const __nv_bfloat16 *>(x), ld, rows, (int)K, sel_n, (int)kn, sel_o, (int)k, o, m, (int)tr);
    } else {
        cudaFuncSetAttribute(k_quant_split<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        k_quant_split<float><<<(unsigned)grid, kSplitThreads, smem, s>>>(static_cast<const float *>(x), ld, rows,
                                                                        (int)K, sel_n, (int)kn, sel_o, (int)k, o,
                                                                        m, (int)tr);
    }
    return cudaGetLastError();
}

// Re-alignment of a forward NVFP4 operand for the backward (§2.A "estimate
// X-hat instead of X", 1x16 groups of the transposed weight): dequantize, read
// transposed, optional RHT along the new contraction axis, SR re-quantize.
cudaError_t launch_realign_nv(const tj_nvfp4 &in, const tj_nvfp4 &out, int mode, int rht, uint64_t seed,
                              uint32_t tag, uint32_t rht_tag, cudaStream_t s) {
    return cols_nv(src_nv(in), out_nv(out), mode, rht, seed, tag, rht_tag, s);
}

// The FP8 outlier slice of a forward operand, transposed and re-quantized (RTN).
cudaError_t launch_realign_mx(const tj_mxfp8 &in, const tj_mxfp8 &out, cudaStream_t s) {
    return cols_mx(src_mx(in), out_mx(out), s);
}

// Both re-alignments of a forward operand with an outlier slice, in one launch.
cudaError_t launch_realign_pair(const tj_nvfp4 &in, const tj_nvfp4 &out, int mode, int rht, uint64_t seed,
                                uint32_t tag, uint32_t rht_tag, const tj_mxfp8 &in8, const tj_mxfp8 &out8,
                                cudaStream_t s) {
    const OutNv oa = out_nv(out);
    const OutMx ob = out_mx(out8);
    const int64_t nxa = oa.rows_p / 64, nya = oa.cols_p / 128, nxb = ob.rows_p / 64, nyb = ob.cols_p / 128;
    if (nxa * nya == 0 || nxb * nyb == 0) {          // an empty part: the other one alone
        if (nxa * nya > 0) return launch_realign_nv(in, out, mode, rht, seed, tag, rht_tag, s);
        if (nxb * nyb > 0) return launch_realign_mx(in8, out8, s);
        return cudaSuccess;
    }
    const int64_t nb = nxb * nyb, n = nb + nxa * nya;
    if (n > 0x7fffffff) return cudaErrorInvalidValue;
    const PhiloxKeys pk = philox_keys(seed);
    const SrcNv sa = src_nv(in);
    const SrcMx sb = src_mx(in8);
    const unsigned grid = (unsigned)n;
    if (mode == TJ_SR && rht)  k_realign_pair<true, true><<<grid, kThreads, 0, s>>>(sa, oa, sb, ob, pk, tag, rht_tag, (int)nxa, (int)nxb, (int)nb);
    else if (mode == TJ_SR)    k_realign_pair<true, false><<<grid, kThreads, 0, s>>>(sa, oa, sb, ob, pk, tag, rht_tag, (int)nxa, (int)nxb, (int)nb);
    else if (rht)              k_realign_pair<false, true><<<grid, kThreads, 0, s>>>(sa, oa, sb, ob, pk, tag, rht_tag, (int)nxa, (int)nxb, (int)nb);
    else                       k_realign_pair<false, false><<<grid, kThreads, 0, s>>>(sa, oa, sb, ob, pk, tag, rht_tag, (int)nxa, (int)nxb, (int)nb);
    return cudaGetLastError();
}

cudaError_t launch_rht(const float *x, float *y, int64_t rows, int64_t cols, uint64_t seed, uint32_t tag,
                       cudaStream_t s) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    const int64_t grid = row_grid(rows * (cols / 128));
    k_rht<<<grid, kThreads, 0, s>>>(x, y, rows, cols, philox_keys(seed), tag);
    return cudaGetLastError();
}

cudaError_t launch_dequant_nv(const tj_nvfp4 &q, float *y, int64_t ldy, cudaStream_t s) {
    const int64_t n = q.rows * q.cols;
    if (n == 0) return cudaSuccess;
    k_dequant_nv<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(src_nv(q), y, ldy);
    return cudaGetLastError();
}

cudaError_t launch_dequant_mx(const tj_mxfp8 &q, float *y, int64_t ldy, cudaStream_t s) {
    const int64_t n = q.rows * q.cols;
    if (n == 0) return cudaSuccess;
    k_dequant_mx<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(src_mx(q), y, ldy);
    return cudaGetLastError();
}

}  // namespace tj
