// gemm.cu - block-scaled NVFP4 GEMM with FP32 outer-scale promotion, plus the
// MXFP8 outlier slice accumulated into the same tile (sm_103a, tcgen05 + TMA).
//
// TetraJet-v2 technical summary §2 / §2.A: all three GEMMs of a linear layer take
// NVFP4 operands whose 16-element groups carry an E4M3 scale and whose
// 128-element blocks carry an FP32 scale; §2.C: outlier channels are kept in FP8.
// The tensor core applies the per-16 scales natively (kind::mxf4nvf4, UE4M3,
// 4 scale factors per K = 64 MMA); the per-128 FP32 scales differ per row and per
// block, so every 128-K block is accumulated into its own tensor-memory partial P
// and promoted by CUDA cores:  acc[m, n] += sA[m, kb] * sB[n, kb] * P[m, n].
// The FP8 slice (kind::mxf8f6f4, UE8M0 per 32) has only power-of-two scales and
// accumulates over its whole K into one tensor-memory buffer added at the end.
//
// Persistent CTAs (one per SM) walk the 128 x 128 output tiles; 18 warps:
//   warp 0     TMA producer (one lane): operand tiles (128 B rows, 128-byte swizzle)
//              and scale-factor tiles into a 5-stage ring, and the FP32 outer
//              scales of every 128-K block into a 12-slot ring (bulk copies);
//   warp 1     tensor-memory owner and MMA issuer (one lane): tcgen05.cp of the
//              scale tiles into a 3-slot tensor-memory ring, tcgen05.mma into the
//              double-buffered partials;
//   warps 2-17 promotion + epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 (its
//              rows) and columns 32*((w-2)/4) .. +31, accumulates in registers with
//              packed f32x2 FMAs and writes its row segment with 16-byte stores.
// Tensor memory (512 columns): P0 [0,128), P1 [128,256), FP8 accumulator
// [256,384), scale factors 32 columns per slot [384,480).
// Every mbarrier wait is bounded; a wait that runs out sets the sticky device
// error flag and an abort flag that makes every role leave its loop, after which
// in-flight copies and MMAs are drained (bounded) and tensor memory is freed.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>

#include "sm100_ptx.cuh"
#include "tj_common.cuh"
#include "tj_internal.h"

namespace tj {

__device__ unsigned int g_tj_dev_error = 0u;

namespace {

constexpr int kStages = 5;                     // operand ring (2 x 128-K blocks per stage)
constexpr int kSfSlots = 3;                    // tensor-memory scale-factor slots (stages in flight)
constexpr int kScaleSlots = 12;                // FP32 outer-scale ring (one 128-K block per slot)
constexpr int kPromoWarps = 16;                // 4 per TMEM lane quadrant, 32 columns each
constexpr int kTileBytes = 128 * 128;          // one operand tile: 128 rows x 128 bytes
constexpr int kSfStageBytes = 2048;            // 4 scale tiles of 512 bytes
constexpr int kSmemA = 0;
constexpr int kSmemB = kSmemA + kStages * kTileBytes;
constexpr int kSmemSfa = kSmemB + kStages * kTileBytes;
constexpr int kSmemSfb = kSmemSfa + kStages * kSfStageBytes;
constexpr int kSmemOuter = kSmemSfb + kStages * kSfStageBytes;      // [slot][A 128 | B 128] floats
constexpr int kSmemBar = kSmemOuter + kScaleSlots * 1024;
constexpr int kSmemBytes = kSmemBar + 512;
constexpr int kThreadsGemm = 32 * (2 + kPromoWarps);
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s per wait
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColP = 0, kColAcc8 = 256, kColSf = 384;

struct GemmArgs {
    int64_t M, N;                 // logical output size
    int tiles_m, tiles_n;         // 128 x 128 output tiles
    int nkb4;                     // 128-K blocks of the FP4 part (0: none)
    int nk8;                      // 128-K stages of the FP8 part (0: none)
    const uint8_t *sfa4, *sfb4;   // scale tiles, FP4 operands
    int64_t ntk_a4, ntk_b4;       // scale tiles per 128-row tile (cols_p / 64)
    const float *outa, *outb;     // FP32 outer scales [cols_p/128][rows_p]
    int64_t rpa, rpb;             // rows_p of A and B
    const uint8_t *sfa8, *sfb8;   // scale tiles, FP8 operands
    int64_t ntk_a8, ntk_b8;       // cols_p / 128
    float alpha;
    void *d;
    int out_bf16;
    int64_t ldd;
    const int32_t *col_map;
};

struct Bars {
    uint64_t full[kStages], empty[kStages];
    uint64_t pfull[2], pempty[2];
    uint64_t sfull[kScaleSlots], sempty[kScaleSlots];
    uint64_t a8full, a8empty, drain;
    uint32_t tmem_base;
    volatile int abort_flag;
};

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on an mbarrier phase: gives up after kWaitNs of wall time (or as
// soon as another role has aborted), setting the sticky device error flag and
// the CTA's abort flag.  No wait in this kernel can spin forever.
__device__ __forceinline__ bool wait_bounded(uint64_t *bar, uint32_t parity, Bars *bars) {
    if (ptx::mbar_try_wait(bar, parity)) return true;         // fast path: no clock read
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0;; ++i) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 63u) {
            if (bars->abort_flag) return false;
            if (global_ns() - t0 > kWaitNs) break;
        }
    }
    atomicOr(&g_tj_dev_error, 1u);
    bars->abort_flag = 1;
    return false;
}

// Warp-uniform bounded wait: every lane waits (lane 0 first), the verdict is
// agreed by vote, so warp-collective operations that follow see one decision.
__device__ __forceinline__ bool warp_wait_bounded(uint64_t *bar, uint32_t parity, Bars *bars, int lane) {
    int ok = 0;
    if (lane == 0) ok = wait_bounded(bar, parity, bars) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok && lane != 0) ok = wait_bounded(bar, parity, bars) ? 1 : 0;
    return __all_sync(0xffffffffu, ok) != 0;
}

// Instruction descriptors (bits: 4-5 B scale id, 7-9 A format, 10-12 B format,
// 15/16 A/B major (0 = K), 17-22 N>>3, 23 scale format (0 UE4M3, 1 UE8M0),
// 24-28 M>>4, 29-30 A scale id).
__host__ __device__ constexpr uint32_t idesc_nvf4() {
    return (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | (0u << 23) | ((128u >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_mxf8(uint32_t sf_id) {
    return (sf_id << 4) | (0u << 7) | (0u << 10) | ((128u >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24) |
           (sf_id << 29);
}

// Packed fp32 pair helpers (two accumulator columns per instruction).
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    return ((uint64_t)__float_as_uint(hi) << 32) | (uint64_t)__float_as_uint(lo);
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__global__ void __launch_bounds__(kThreadsGemm, 1)
    k_gemm_nvfp4(const __grid_constant__ CUtensorMap tm_a4, const __grid_constant__ CUtensorMap tm_b4,
                 const __grid_constant__ CUtensorMap tm_a8, const __grid_constant__ CUtensorMap tm_b8,
                 const GemmArgs args) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars *bars = reinterpret_cast<Bars *>(smem + kSmemBar);
    float *outer_s = reinterpret_cast<float *>(smem + kSmemOuter);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntiles = args.tiles_m * args.tiles_n;
    const int nst4 = (args.nkb4 + 1) / 2;
    const int nstages = nst4 + args.nk8;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(&bars->full[s], 1);
            ptx::mbar_init(&bars->empty[s], 1);
        }
        for (int p = 0; p < 2; ++p) {
            ptx::mbar_init(&bars->pfull[p], 1);
            ptx::mbar_init(&bars->pempty[p], kPromoWarps);
        }
        for (int s = 0; s < kScaleSlots; ++s) {
            ptx::mbar_init(&bars->sfull[s], 1);
            ptx::mbar_init(&bars->sempty[s], kPromoWarps);
        }
        ptx::mbar_init(&bars->a8full, 1);
        ptx::mbar_init(&bars->a8empty, kPromoWarps);
        ptx::mbar_init(&bars->drain, 1);
        bars->abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) ptx::tmem_alloc(&bars->tmem_base, kTmemCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tbase = bars->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            if (args.nkb4 > 0) { ptx::prefetch_tmap(&tm_a4); ptx::prefetch_tmap(&tm_b4); }
            if (args.nk8 > 0) { ptx::prefetch_tmap(&tm_a8); ptx::prefetch_tmap(&tm_b8); }
            int it = 0, sk = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                const int64_t m0 = (int64_t)(tile / args.tiles_n) * 128, n0 = (int64_t)(tile % args.tiles_n) * 128;
                const int64_t rta = m0 / 128, rtb = n0 / 128;
                for (int st = 0; st < nstages; ++st, ++it) {
                    const int slot = it % kStages;
                    if (it >= kStages && !wait_bounded(&bars->empty[slot], ((it / kStages) - 1) & 1, bars)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sa = smem + kSmemA + slot * kTileBytes;
                    uint8_t *sb = smem + kSmemB + slot * kTileBytes;
                    uint8_t *sfa = smem + kSmemSfa + slot * kSfStageBytes;
                    uint8_t *sfb = smem + kSmemSfb + slot * kSfStageBytes;
                    if (st < nst4) {
                        const int nkbs = min(2, args.nkb4 - 2 * st);
                        const uint32_t sfbytes = (uint32_t)nkbs * 1024u;
                        ptx::mbar_arrive_expect_tx(&bars->full[slot], 2u * kTileBytes + 2u * sfbytes);
                        ptx::tma_load_2d(sa, &tm_a4, st * 128, (int32_t)m0, &bars->full[slot]);
                        ptx::tma_load_2d(sb, &tm_b4, st * 128, (int32_t)n0, &bars->full[slot]);
                        ptx::bulk_load(sfa, args.sfa4 + (rta * args.ntk_a4 + 4 * st) * 512, sfbytes, &bars->full[slot]);
                        ptx::bulk_load(sfb, args.sfb4 + (rtb * args.ntk_b4 + 4 * st) * 512, sfbytes, &bars->full[slot]);
                        // the FP32 outer scales of these blocks, for the promotion warps
                        for (int j = 0; j < nkbs && ok; ++j, ++sk) {
                            const int ss = sk % kScaleSlots;
                            if (sk >= kScaleSlots &&
                                !wait_bounded(&bars->sempty[ss], ((sk / kScaleSlots) - 1) & 1, bars)) {
                                ok = false;
                                break;
                            }
                            const int64_t kb = 2 * st + j;
                            ptx::mbar_arrive_expect_tx(&bars->sfull[ss], 1024u);
                            ptx::bulk_load(outer_s + ss * 256, args.outa + kb * args.rpa + m0, 512u, &bars->sfull[ss]);
                            ptx::bulk_load(outer_s + ss * 256 + 128, args.outb + kb * args.rpb + n0, 512u,
                                           &bars->sfull[ss]);
                        }
                        if (!ok) { ++it; break; }
                    } else {
                        const int s8 = st - nst4;
                        ptx::mbar_arrive_expect_tx(&bars->full[slot], 2u * kTileBytes + 1024u);
                        ptx::tma_load_2d(sa, &tm_a8, s8 * 128, (int32_t)m0, &bars->full[slot]);
                        ptx::tma_load_2d(sb, &tm_b8, s8 * 128, (int32_t)n0, &bars->full[slot]);
                        ptx::bulk_load(sfa, args.sfa8 + (rta * args.ntk_a8 + s8) * 512, 512u, &bars->full[slot]);
                        ptx::bulk_load(sfb, args.sfb8 + (rtb * args.ntk_b8 + s8) * 512, 512u, &bars->full[slot]);
                    }
                }
            }
            // drain: every copy issued must have landed before the CTA exits
            for (int j = (it > kStages ? it - kStages : 0); j < it; ++j)
                wait_bounded(&bars->full[j % kStages], (j / kStages) & 1, bars);
            for (int j = (sk > kScaleSlots ? sk - kScaleSlots : 0); j < sk; ++j)
                wait_bounded(&bars->sfull[j % kScaleSlots], (j / kScaleSlots) & 1, bars);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc4 = idesc_nvf4();
            int it = 0, pcount = 0, a8count = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                for (int st = 0; st < nstages; ++st, ++it) {
                    const int slot = it % kStages;
                    if (!wait_bounded(&bars->full[slot], (it / kStages) & 1, bars)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_u32(smem + kSmemA + slot * kTileBytes);
                    const uint32_t sb = ptx::smem_u32(smem + kSmemB + slot * kTileBytes);
                    const uint32_t sfa = ptx::smem_u32(smem + kSmemSfa + slot * kSfStageBytes);
                    const uint32_t sfb = ptx::smem_u32(smem + kSmemSfb + slot * kSfStageBytes);
                    // scale-factor slot it % kSfSlots was last read by the MMAs of stage
                    // it - kSfSlots; those have completed once that stage's ring slot was
                    // released (its empty barrier phase)
                    if (it >= kSfSlots) {
                        const int prev = it - kSfSlots;
                        if (!wait_bounded(&bars->empty[prev % kStages], (prev / kStages) & 1, bars)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                    }
                    const uint32_t sfcol = tbase + kColSf + 32u * (uint32_t)(it % kSfSlots);
                    if (st < nst4) {
                        const int nkbs = min(2, args.nkb4 - 2 * st);
                        for (int j = 0; j < 2 * nkbs; ++j) {   // one 512-byte scale tile per K = 64 MMA
                            ptx::tc_cp_32x128b_warpx4(sfcol + 4 * j, ptx::smem_desc(sfa + 512 * j, 0, 128, 0));
                            ptx::tc_cp_32x128b_warpx4(sfcol + 16 + 4 * j, ptx::smem_desc(sfb + 512 * j, 0, 128, 0));
                        }
                        for (int kbl = 0; kbl < nkbs; ++kbl) {
                            const int pb = pcount & 1;
                            if (pcount >= 2 && !wait_bounded(&bars->pempty[pb], ((pcount >> 1) - 1) & 1, bars)) {
                                ok = false;
                                break;
                            }
                            ptx::tc_fence_after();
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                const uint32_t koff = 64u * kbl + 32u * j;
                                ptx::mma_nvf4(tbase + kColP + 128u * pb, ptx::smem_desc(sa + koff, 16, 1024, 2),
                                              ptx::smem_desc(sb + koff, 16, 1024, 2), idesc4,
                                              sfcol + 4 * (2 * kbl + j), sfcol + 16 + 4 * (2 * kbl + j), (uint32_t)j);
                            }
                            ptx::tc_commit(&bars->pfull[pb]);
                            ++pcount;
                        }
                        if (!ok) break;
                    } else {
                        const int s8 = st - nst4;
                        if (s8 == 0 && a8count >= 1 &&
                            !wait_bounded(&bars->a8empty, (a8count - 1) & 1, bars)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        ptx::tc_cp_32x128b_warpx4(sfcol, ptx::smem_desc(sfa, 0, 128, 0));
                        ptx::tc_cp_32x128b_warpx4(sfcol + 16, ptx::smem_desc(sfb, 0, 128, 0));
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            ptx::mma_mxf8(tbase + kColAcc8, ptx::smem_desc(sa + 32u * j, 16, 1024, 2),
                                          ptx::smem_desc(sb + 32u * j, 16, 1024, 2), idesc_mxf8((uint32_t)j), sfcol,
                                          sfcol + 16, (uint32_t)(s8 > 0 || j > 0));
                        }
                        if (s8 == args.nk8 - 1) {
                            ptx::tc_commit(&bars->a8full);
                            ++a8count;
                        }
                    }
                    ptx::tc_commit(&bars->empty[slot]);
                }
            }
            // drain: all MMAs / copies issued by this thread complete before TMEM is freed
            ptx::tc_commit(&bars->drain);
            wait_bounded(&bars->drain, 0, bars);
        }
    } else {
        // ------------------------------------------------------------ promotion + epilogue
        const int pw = warp - 2;
        const int q = warp & 3;                 // TMEM lane quadrant of this warp
        const int cq = pw >> 2;                 // column quarter: columns 32*cq .. +31
        const int row_l = 32 * q + lane;
        const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
        int kbc = 0, a8c = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
            uint64_t acc[16];                  // 32 fp32 accumulators as packed pairs
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j] = 0ull;
            for (int kb = 0; kb < args.nkb4; ++kb, ++kbc) {
                const int pb = kbc & 1;
                const int ss = kbc % kScaleSlots;
                if (!warp_wait_bounded(&bars->pfull[pb], (kbc >> 1) & 1, bars, lane)) { ok = false; break; }
                ptx::tc_fence_after();
                uint32_t pv[32];
                ptx::tmem_ld_32x32b_x32(tbase + lane_addr + kColP + 128u * pb + 32u * cq, pv);
                ptx::tmem_wait_ld();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&bars->pempty[pb]);
                if (!warp_wait_bounded(&bars->sfull[ss], (kbc / kScaleSlots) & 1, bars, lane)) { ok = false; break; }
                const float sa = outer_s[ss * 256 + row_l] * args.alpha;
                const uint64_t sa2 = pack2(sa, sa);
                const float4 *sbp = reinterpret_cast<const float4 *>(outer_s + ss * 256 + 128 + 32 * cq);
                float4 sbv[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) sbv[i] = sbp[i];    // broadcast reads: all lanes, same address
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&bars->sempty[ss]);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint64_t c01 = mul2(sa2, pack2(sbv[i].x, sbv[i].y));
                    const uint64_t c23 = mul2(sa2, pack2(sbv[i].z, sbv[i].w));
                    acc[2 * i] = fma2(pack2(__uint_as_float(pv[4 * i]), __uint_as_float(pv[4 * i + 1])), c01, acc[2 * i]);
                    acc[2 * i + 1] =
                        fma2(pack2(__uint_as_float(pv[4 * i + 2]), __uint_as_float(pv[4 * i + 3])), c23, acc[2 * i + 1]);
                }
            }
            if (!ok) break;
            if (args.nk8 > 0) {
                if (!warp_wait_bounded(&bars->a8full, a8c & 1, bars, lane)) { ok = false; break; }
                ptx::tc_fence_after();
                uint32_t pv[32];
                ptx::tmem_ld_32x32b_x32(tbase + lane_addr + kColAcc8 + 32u * cq, pv);
                ptx::tmem_wait_ld();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&bars->a8empty);
                ++a8c;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    acc[i] = add2(acc[i], pack2(__uint_as_float(pv[2 * i]), __uint_as_float(pv[2 * i + 1])));
            }
            // epilogue: this thread's row segment of 32 columns, written with 16-byte stores
            const int64_t m0 = (int64_t)(tile / args.tiles_n) * 128, n0 = (int64_t)(tile % args.tiles_n) * 128;
            const int64_t row = m0 + row_l;
            const int64_t nb = n0 + 32 * cq;
            if (row < args.M) {
                float v[32];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    v[2 * i] = __uint_as_float((uint32_t)acc[i]);
                    v[2 * i + 1] = __uint_as_float((uint32_t)(acc[i] >> 32));
                }
                const bool fast = args.col_map == nullptr && nb + 32 <= args.N && (args.ldd & 7) == 0;
                if (fast && args.out_bf16) {
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(args.d) + row * args.ldd + nb);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t w4[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            __nv_bfloat162 b2 = __floats2bfloat162_rn(v[8 * i + 2 * k], v[8 * i + 2 * k + 1]);
                            w4[k] = *reinterpret_cast<uint32_t *>(&b2);
                        }
                        dst[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                } else if (fast) {
                    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(args.d) + row * args.ldd + nb);
#pragma unroll
                    for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int64_t n = nb + j;
                        if (n < args.N) {
                            const int64_t col = args.col_map ? (int64_t)args.col_map[n] : n;
                            if (args.out_bf16)
                                static_cast<__nv_bfloat16 *>(args.d)[row * args.ldd + col] = __float2bfloat16_rn(v[j]);
                            else
                                static_cast<float *>(args.d)[row * args.ldd + col] = v[j];
                        }
                    }
                }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tbase, kTmemCols);
    }
}

}  // namespace

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D byte tensor [rows_p][row_bytes] -> tiles of 128 rows x 128 bytes, 128-byte swizzle.
bool make_tile_map(CUtensorMap *m, const void *base, int64_t rows_p, int64_t row_bytes) {
    EncodeTiledFn enc = get_encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows_p};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {128u, 128u};
    const cuuint32_t estr[2] = {1u, 1u};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_gemm(const tj_nvfp4 *a, const tj_nvfp4 *b, const tj_mxfp8 *a8, const tj_mxfp8 *b8, float alpha,
                        void *d, int out_dtype, int64_t ldd, int64_t M, int64_t N, const int32_t *col_map,
                        cudaStream_t s) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm_nvfp4, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes + 1024);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    CUtensorMap tm[4];
    memset(tm, 0, sizeof(tm));
    GemmArgs g{};
    g.M = M;
    g.N = N;
    g.alpha = alpha;
    g.d = d;
    g.out_bf16 = out_dtype == TJ_BF16;
    g.ldd = ldd;
    g.col_map = col_map;
    int64_t rows_pa = 0, rows_pb = 0;
    if (a != nullptr && b != nullptr) {
        const int64_t kp = round_up(a->cols, 128);
        rows_pa = round_up(a->rows, 128);
        rows_pb = round_up(b->rows, 128);
        g.nkb4 = (int)(kp / 128);
        g.sfa4 = a->sf;
        g.sfb4 = b->sf;
        g.ntk_a4 = kp / 64;
        g.ntk_b4 = kp / 64;
        g.outa = a->outer;
        g.outb = b->outer;
        g.rpa = rows_pa;
        g.rpb = rows_pb;
        if (!make_tile_map(&tm[0], a->codes, rows_pa, kp / 2) || !make_tile_map(&tm[1], b->codes, rows_pb, kp / 2))
            return cudaErrorInvalidValue;
    }
    if (a8 != nullptr && b8 != nullptr && a8->cols > 0) {
        const int64_t kp8 = round_up(a8->cols, 128);
        rows_pa = round_up(a8->rows, 128);
        rows_pb = round_up(b8->rows, 128);
        g.nk8 = (int)(kp8 / 128);
        g.sfa8 = a8->sf;
        g.sfb8 = b8->sf;
        g.ntk_a8 = kp8 / 128;
        g.ntk_b8 = kp8 / 128;
        if (!make_tile_map(&tm[2], a8->codes, rows_pa, kp8) || !make_tile_map(&tm[3], b8->codes, rows_pb, kp8))
            return cudaErrorInvalidValue;
    }
    g.tiles_m = (int)(round_up(M, 128) / 128);
    g.tiles_n = (int)(round_up(N, 128) / 128);
    const int ntiles = g.tiles_m * g.tiles_n;
    if (ntiles == 0) return cudaSuccess;
    static int num_sms = 0;
    if (num_sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (num_sms <= 0) num_sms = 148;
    }
    const int grid = ntiles < num_sms ? ntiles : num_sms;     // persistent CTAs, one per SM
    k_gemm_nvfp4<<<grid, kThreadsGemm, kSmemBytes + 1024, s>>>(tm[0], tm[1], tm[2], tm[3], g);
    return cudaGetLastError();
}

unsigned int read_and_clear_device_error() {
    unsigned int v = 0u, z = 0u;
    if (cudaMemcpyFromSymbol(&v, g_tj_dev_error, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
    cudaMemcpyToSymbol(g_tj_dev_error, &z, sizeof(z));
    return v;
}

}  // namespace tj
