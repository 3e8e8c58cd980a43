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
// Persistent CTAs (one per SM) walk the 128 x 128 output tiles; 10 warps:
//   warp 0     TMA producer (one lane): operand tiles (128 B rows, 128-byte swizzle)
//              and scale-factor tiles into a 5-stage ring, and the FP32 outer
//              scales of every 128-K block into a 16-slot ring (bulk copies);
//   warp 1     tensor-memory owner and MMA issuer (one lane): tcgen05.cp of the
//              scale tiles into a 3-slot tensor-memory ring, tcgen05.mma into the
//              double-buffered partials;
//   warps 2-9  promotion + epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 (its
//              rows) and columns 64*((w-2)/4) .. +63, accumulates in registers
//              (one multiply and one FMA per element and block) and writes its row
//              segment with 16-byte stores.
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
constexpr int kScaleSlots = 16;                // FP32 outer-scale ring (one 128-K block per slot; power of 2)
constexpr int kPromoWarps = 8;                 // 2 per TMEM lane quadrant, 64 columns each
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
        // sleep in hardware until the phase completes (or 20 us pass): a waiting
        // thread takes no issue slots from the warps doing the work
        if (ptx::mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (bars->abort_flag) return false;
        if ((i & 15u) == 15u && global_ns() - t0 > kWaitNs) break;
    }
    atomicOr(&g_tj_dev_error, 1u);
    bars->abort_flag = 1;
    return false;
}

// Warp-uniform bounded wait: lane 0 waits, the verdict is broadcast, and
// __syncwarp orders the other lanes' following accesses after lane 0's
// observation of the completed phase.
__device__ __forceinline__ bool warp_wait_bounded(uint64_t *bar, uint32_t parity, Bars *bars, int lane) {
    int ok = 1;
    if (lane == 0) ok = wait_bounded(bar, parity, bars) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
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

template <int CM, int CN>
__global__ void __launch_bounds__(kThreadsGemm, 1)
    k_gemm_nvfp4(const __grid_constant__ CUtensorMap tm_a4, const __grid_constant__ CUtensorMap tm_b4,
                 const __grid_constant__ CUtensorMap tm_a8, const __grid_constant__ CUtensorMap tm_b8,
                 const GemmArgs args) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars *bars = reinterpret_cast<Bars *>(smem + kSmemBar);
    float *outer_s = reinterpret_cast<float *>(smem + kSmemOuter);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // cluster of CM x CN CTAs computing a (CM*128) x (CN*128) block of tiles; the CTAs
    // with the same m share the A tile, those with the same n the B tile
    constexpr int CS = CM * CN;
    const uint32_t crank = CS > 1 ? ptx::cluster_ctarank() : 0u;
    const int cm = (int)(crank % CM), cn = (int)(crank / CM);
    const int cid = (int)blockIdx.x / CS, ncl = (int)gridDim.x / CS;
    const int ctn = args.tiles_n / CN;
    const int ntiles = (args.tiles_m / CM) * ctn;          // cluster tiles
    auto tile_m0 = [&](int ct) { return (int64_t)((ct / ctn) * CM + cm) * 128; };
    auto tile_n0 = [&](int ct) { return (int64_t)((ct % ctn) * CN + cn) * 128; };
    const int nst4 = (args.nkb4 + 1) / 2;
    const int nstages = nst4 + args.nk8;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(&bars->full[s], 1);
            ptx::mbar_init(&bars->empty[s], CS);            // every CTA of the cluster releases each stage
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
    if (CS > 1) ptx::cluster_sync();                        // partners' barriers exist before any multicast
    const uint32_t tbase = bars->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            if (args.nkb4 > 0) { ptx::prefetch_tmap(&tm_a4); ptx::prefetch_tmap(&tm_b4); }
            if (args.nk8 > 0) { ptx::prefetch_tmap(&tm_a8); ptx::prefetch_tmap(&tm_b8); }
            int it = 0, sk = 0;
            bool ok = true;
            // multicast masks: the CTAs sharing this CTA's A tile (same cm) and B tile (same cn)
            uint16_t mask_a = 0, mask_b = 0;
            for (int j = 0; j < CN; ++j) mask_a |= (uint16_t)(1u << (cm + CM * j));
            for (int i = 0; i < CM; ++i) mask_b |= (uint16_t)(1u << (i + CM * cn));
            constexpr int ra = 128 / CN, rb = 128 / CM;      // rows of A / B this CTA loads
            for (int tile = cid; tile < ntiles && ok; tile += ncl) {
                const int64_t m0 = tile_m0(tile), n0 = tile_n0(tile);
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
                        if (CN > 1)
                            ptx::tma_load_2d_multicast(sa + cn * ra * 128, &tm_a4, st * 128, (int32_t)(m0 + cn * ra),
                                                       &bars->full[slot], mask_a);
                        else
                            ptx::tma_load_2d(sa, &tm_a4, st * 128, (int32_t)m0, &bars->full[slot]);
                        if (CM > 1)
                            ptx::tma_load_2d_multicast(sb + cm * rb * 128, &tm_b4, st * 128, (int32_t)(n0 + cm * rb),
                                                       &bars->full[slot], mask_b);
                        else
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
                        if (CN > 1)
                            ptx::tma_load_2d_multicast(sa + cn * ra * 128, &tm_a8, s8 * 128, (int32_t)(m0 + cn * ra),
                                                       &bars->full[slot], mask_a);
                        else
                            ptx::tma_load_2d(sa, &tm_a8, s8 * 128, (int32_t)m0, &bars->full[slot]);
                        if (CM > 1)
                            ptx::tma_load_2d_multicast(sb + cm * rb * 128, &tm_b8, s8 * 128, (int32_t)(n0 + cm * rb),
                                                       &bars->full[slot], mask_b);
                        else
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
            for (int tile = cid; tile < ntiles && ok; tile += ncl) {
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
                    // release the stage in every CTA whose shared memory this cluster's loads fill
                    if (CS > 1)
                        ptx::tc_commit_multicast(&bars->empty[slot], (uint16_t)((1u << CS) - 1u));
                    else
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
        const int h = pw >> 2;                  // column half: columns 64*h .. +63
        const int row_l = 32 * q + lane;
        const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
        int kbc = 0, a8c = 0;
        bool ok = true;
        for (int tile = cid; tile < ntiles && ok; tile += ncl) {
            float acc[64];
#pragma unroll
            for (int j = 0; j < 64; ++j) acc[j] = 0.0f;
            for (int kb = 0; kb < args.nkb4; ++kb, ++kbc) {
                const int pb = kbc & 1;
                const int ss = kbc & (kScaleSlots - 1);
                if (!warp_wait_bounded(&bars->pfull[pb], (kbc >> 1) & 1, bars, lane)) { ok = false; break; }
                ptx::tc_fence_after();
                uint32_t p0[32], p1[32];
                ptx::tmem_ld_32x32b_x32(tbase + lane_addr + kColP + 128u * pb + 64u * h, p0);
                ptx::tmem_ld_32x32b_x32(tbase + lane_addr + kColP + 128u * pb + 64u * h + 32u, p1);
                ptx::tmem_wait_ld();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&bars->pempty[pb]);
                if (!warp_wait_bounded(&bars->sfull[ss], (kbc / kScaleSlots) & 1, bars, lane)) { ok = false; break; }
                const float sa = outer_s[ss * 256 + row_l] * args.alpha;
                const float4 *sbp = reinterpret_cast<const float4 *>(outer_s + ss * 256 + 128 + 64 * h);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float4 sb = sbp[i];                     // broadcast read: all lanes, same address
                    const uint32_t *pp = i < 8 ? p0 : p1;
                    const int jj = (4 * i) & 31;
                    acc[4 * i] = fmaf(__uint_as_float(pp[jj]), sa * sb.x, acc[4 * i]);
                    acc[4 * i + 1] = fmaf(__uint_as_float(pp[jj + 1]), sa * sb.y, acc[4 * i + 1]);
                    acc[4 * i + 2] = fmaf(__uint_as_float(pp[jj + 2]), sa * sb.z, acc[4 * i + 2]);
                    acc[4 * i + 3] = fmaf(__uint_as_float(pp[jj + 3]), sa * sb.w, acc[4 * i + 3]);
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&bars->sempty[ss]);
            }
            if (!ok) break;
            if (args.nk8 > 0) {
                if (!warp_wait_bounded(&bars->a8full, a8c & 1, bars, lane)) { ok = false; break; }
                ptx::tc_fence_after();
                uint32_t p0[32], p1[32];
                ptx::tmem_ld_32x32b_x32(tbase + lane_addr + kColAcc8 + 64u * h, p0);
                ptx::tmem_ld_32x32b_x32(tbase + lane_addr + kColAcc8 + 64u * h + 32u, p1);
                ptx::tmem_wait_ld();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&bars->a8empty);
                ++a8c;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    acc[j] += __uint_as_float(p0[j]);
                    acc[32 + j] += __uint_as_float(p1[j]);
                }
            }
            // epilogue: this thread's row segment of 64 columns, written with 16-byte stores
            const int64_t m0 = tile_m0(tile), n0 = tile_n0(tile);
            const int64_t row = m0 + row_l;
            const int64_t nb = n0 + 64 * h;
            if (row < args.M) {
                const bool fast = args.col_map == nullptr && nb + 64 <= args.N && (args.ldd & 7) == 0;
                if (fast && args.out_bf16) {
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(args.d) + row * args.ldd + nb);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        uint32_t w4[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[8 * i + 2 * k], acc[8 * i + 2 * k + 1]);
                            w4[k] = *reinterpret_cast<uint32_t *>(&b2);
                        }
                        dst[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                } else if (fast) {
                    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(args.d) + row * args.ldd + nb);
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        dst[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        const int64_t n = nb + j;
                        if (n < args.N) {
                            const int64_t col = args.col_map ? (int64_t)args.col_map[n] : n;
                            if (args.out_bf16)
                                static_cast<__nv_bfloat16 *>(args.d)[row * args.ldd + col] = __float2bfloat16_rn(acc[j]);
                            else
                                static_cast<float *>(args.d)[row * args.ldd + col] = acc[j];
                        }
                    }
                }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (CS > 1) ptx::cluster_sync();                        // no partner still writes into this CTA
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

// 2-D byte tensor [rows_p][row_bytes] -> boxes of box_rows rows x 128 bytes, 128-byte swizzle.
bool make_tile_map(CUtensorMap *m, const void *base, int64_t rows_p, int64_t row_bytes, uint32_t box_rows) {
    EncodeTiledFn enc = get_encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows_p};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {128u, box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms_of_current_device() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
}

// Launch one cluster shape: persistent grid of as many clusters as fit at once.
template <int CM, int CN>
cudaError_t launch_cluster(const CUtensorMap (&tm)[4], const GemmArgs &g, cudaStream_t s) {
    constexpr int CS = CM * CN;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm_nvfp4<CM, CN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes + 1024);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int nctiles = (g.tiles_m / CM) * (g.tiles_n / CN);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreadsGemm);
    cfg.dynamicSmemBytes = kSmemBytes + 1024;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static int max_clusters = 0;
    if (max_clusters == 0) {
        cfg.gridDim = dim3(CS * 64);
        int n = 0;
        if (CS > 1 && cudaOccupancyMaxActiveClusters(&n, k_gemm_nvfp4<CM, CN>, &cfg) == cudaSuccess && n > 0)
            max_clusters = n;
        else
            max_clusters = num_sms_of_current_device() / CS;
    }
    const int nclusters = nctiles < max_clusters ? nctiles : max_clusters;
    cfg.gridDim = dim3((unsigned)(nclusters * CS));
    return cudaLaunchKernelEx(&cfg, k_gemm_nvfp4<CM, CN>, tm[0], tm[1], tm[2], tm[3], g);
}

}  // namespace

cudaError_t launch_gemm(const tj_nvfp4 *a, const tj_nvfp4 *b, const tj_mxfp8 *a8, const tj_mxfp8 *b8, float alpha,
                        void *d, int out_dtype, int64_t ldd, int64_t M, int64_t N, const int32_t *col_map,
                        cudaStream_t s) {
    GemmArgs g{};
    g.M = M;
    g.N = N;
    g.alpha = alpha;
    g.d = d;
    g.out_bf16 = out_dtype == TJ_BF16;
    g.ldd = ldd;
    g.col_map = col_map;
    g.tiles_m = (int)(round_up(M, 128) / 128);
    g.tiles_n = (int)(round_up(N, 128) / 128);
    if (g.tiles_m == 0 || g.tiles_n == 0) return cudaSuccess;
    // cluster shape: pair tiles along M (sharing B) and along N (sharing A) when the
    // tile counts allow; each CTA then loads half of each shared operand tile
    const int cm = (g.tiles_m % 2 == 0) ? 2 : 1;
    const int cn = (g.tiles_n % 2 == 0) ? 2 : 1;
    CUtensorMap tm[4];
    memset(tm, 0, sizeof(tm));
    if (a != nullptr && b != nullptr) {
        const int64_t kp = round_up(a->cols, 128);
        g.nkb4 = (int)(kp / 128);
        g.sfa4 = a->sf;
        g.sfb4 = b->sf;
        g.ntk_a4 = kp / 64;
        g.ntk_b4 = kp / 64;
        g.outa = a->outer;
        g.outb = b->outer;
        g.rpa = round_up(a->rows, 128);
        g.rpb = round_up(b->rows, 128);
        if (!make_tile_map(&tm[0], a->codes, g.rpa, kp / 2, 128u / cn) ||
            !make_tile_map(&tm[1], b->codes, g.rpb, kp / 2, 128u / cm))
            return cudaErrorInvalidValue;
    }
    if (a8 != nullptr && b8 != nullptr && a8->cols > 0) {
        const int64_t kp8 = round_up(a8->cols, 128);
        g.nk8 = (int)(kp8 / 128);
        g.sfa8 = a8->sf;
        g.sfb8 = b8->sf;
        g.ntk_a8 = kp8 / 128;
        g.ntk_b8 = kp8 / 128;
        if (!make_tile_map(&tm[2], a8->codes, round_up(a8->rows, 128), kp8, 128u / cn) ||
            !make_tile_map(&tm[3], b8->codes, round_up(b8->rows, 128), kp8, 128u / cm))
            return cudaErrorInvalidValue;
    }
    if (cm == 2 && cn == 2) return launch_cluster<2, 2>(tm, g, s);
    if (cm == 2) return launch_cluster<2, 1>(tm, g, s);
    if (cn == 2) return launch_cluster<1, 2>(tm, g, s);
    return launch_cluster<1, 1>(tm, g, s);
}

unsigned int read_and_clear_device_error() {
    unsigned int v = 0u, z = 0u;
    if (cudaMemcpyFromSymbol(&v, g_tj_dev_error, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
    cudaMemcpyToSymbol(g_tj_dev_error, &z, sizeof(z));
    return v;
}

}  // namespace tj
