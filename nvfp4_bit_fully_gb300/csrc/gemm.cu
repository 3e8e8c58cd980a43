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
// The outlier slice (kind::mxf8f6f4, UE8M0 per 32; E4M3 operands, or the FP6 / FP4
// formats of the FP6 x FP4 variant in any pairing) has only power-of-two scales and
// accumulates over its whole K into one tensor-memory buffer added at the end.
//
// Persistent CTAs (one per SM) walk the 128 x 128 output tiles; every CTA loads its
// own operand tiles.  12 warps:
//   warps 0-2   TMA producers (one lane each; stage it is issued by warp it % 3): the
//               operand tiles (128-byte rows, 128-byte swizzle) and their scale-factor
//               tiles into a 5-stage ring, and the FP32 outer scales of the stage's
//               128-K blocks into an 8-slot ring, all on the stage's barrier;
//   warp 3      tensor-memory owner and MMA issuer (lane 0 issues): per block,
//               tcgen05.cp of its scale-factor tiles and two tcgen05.mma into a
//               3-slot ring of partials, so the MMAs run up to two blocks ahead of
//               the promotion;
//   warps 4-11  promotion + epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 (its
//               rows) and columns 64*((w-4)/4) .. +63, accumulates in registers with
//               packed f32x2 multiplies and FMAs, and writes its slice (a TMA store
//               or row-at-a-time stores).  (Sixteen warps of 32 columns measured slower.)
// A thread can observe only one barrier handoff every few hundred cycles, so the
// design keeps handoffs few: the partial slots are released through hardware named
// barriers, the scale factors of a block share its partial slot's lifetime, and the
// outer scales travel with the operands and are handed back by the promotion warps once
// their math is done with them.
// The FP8 slice accumulates over its whole K into the next partial slot, which the
// promotion adds with weight 1.
// Tensor memory (512 columns): partials [0,384) (128 per slot), FP4 scale factors
// [384,432) (16 per partial slot), FP8 scale factors [432,472) (8 per operand ring slot).
// Every mbarrier wait is bounded; a wait that runs out sets the sticky device
// error flag and an abort flag.  The roles then stop working but keep the named-
// barrier protocol (whose counts depend only on the problem size), in-flight copies
// and MMAs are drained (bounded) and tensor memory is freed.
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
constexpr int kPSlots = 3;                     // tensor-memory partial slots (128-K blocks in flight)
constexpr int kProdWarps = 3;                  // TMA producers; stage it is issued by warp it % kProdWarps
constexpr int kMmaWarp = kProdWarps;           // tensor-memory owner and MMA issuer
constexpr int kPromo0 = kProdWarps + 1;        // first promotion warp
constexpr int kPromoWarps = 8;                 // 2 per TMEM lane quadrant
constexpr int kColsW = 512 / kPromoWarps;      // accumulator columns per promotion warp
constexpr int kLdCols = kColsW < 64 ? kColsW : 64;   // partial columns held in registers at a time
constexpr int kTileBytes = 128 * 128;          // one operand tile: 128 rows x 128 bytes
constexpr int kSfStageBytes = 2048;            // 4 scale tiles of 512 bytes
constexpr int kSmemA = 0;
constexpr int kSmemB = kSmemA + kStages * kTileBytes;
constexpr int kSmemSfa = kSmemB + kStages * kTileBytes;
constexpr int kSmemSfb = kSmemSfa + kStages * kSfStageBytes;
constexpr int kScaleSlots = 8;                 // FP32 outer-scale ring: one FP4 block per slot, [A 128 | B 128]
constexpr int kSmemScale = kSmemSfb + kStages * kSfStageBytes;
constexpr int kSmemBar = kSmemScale + kScaleSlots * 1024;
// Epilogue staging, per promotion warp: a 32-row box of kColsW bf16 for TMA stores
// (stride kEpiTma, 1024-aligned) or 32 rows of kColsW / 2 words plus a pad word for the
// row-at-a-time writes (stride kEpiRow).  A launch uses only one of the two layouts (TMA
// stores only in single-product launches).
constexpr int kSmemEpi = (kSmemBar + 512 + 1023) & ~1023;
constexpr int kEpiTma = 32 * 2 * kColsW;
constexpr int kEpiRow = 32 * (kColsW / 2 + 1) * 4;
constexpr int kSmemBytes = kSmemEpi + kPromoWarps * (kEpiTma > kEpiRow ? kEpiTma : kEpiRow);
static_assert(kSmemBytes + 1024 <= 227 * 1024, "shared memory budget");
constexpr int kThreadsGemm = 32 * (kPromo0 + kPromoWarps);
constexpr int kNamedP = 1;                     // named barriers kNamedP .. +kPSlots-1: partial slot released
constexpr int kNamedCount = 32 * (1 + kPromoWarps);   // the MMA warp and every promotion warp
constexpr long long kWaitClk = 4000000000ll;  // per wait: about 2 s at the maximum SM clock, longer below it
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColP = 0;                                   // partials: 128 columns per slot
constexpr uint32_t kColSf = 128 * kPSlots;                      // FP4 scale factors: 16 columns per partial slot
constexpr uint32_t kColSf8 = kColSf + 16 * kPSlots;             // FP8 scale factors: 8 columns per operand slot
static_assert(kColSf8 + 8 * kStages <= kTmemCols, "tensor memory budget");
static_assert(kColsW == 32 || kColsW == 64, "epilogue: 64- or 128-byte bf16 rows per warp slice");
static_assert(kEpiTma % 1024 == 0, "TMA staging boxes stay 1024-aligned");
static_assert(kNamedP + kPSlots <= 16, "named barriers");

// One product D = alpha * A B^T of the launch.  A launch computes one or two of them:
// pr[0] with FP4 blocks (and optionally an FP8 K-slice into the same tiles), and
// optionally pr[1], an FP8-only product with its own output (the outlier slice of a
// backward GEMM).  When both cover the same output rows, the works are taken row block by
// row block (FP8 works first), so writes to the same rows meet in L2.
struct GemmProblem {
    int64_t M, N;                 // logical output size
    int tiles_m, tiles_n;         // 128 x 128 output tiles (0 x 0: absent)
    int nkb4;                     // 128-K blocks of the FP4 part (0: none)
    int nk8;                      // 128-K stages of the FP8 part (0: none)
    float alpha;                  // applied to the FP4 part
    void *d;
    int out_bf16;
    int64_t ldd;
    const int32_t *col_map;       // output column n goes to column col_map[n] (nullptr: n)
    int tma_store;                // bf16, no col_map, ldd % 8 == 0: tiles leave by TMA stores (map tm_d)
    int splits;                   // 1, or 2: each tile's K schedule is halved over two tile works whose
                                  // fp32 sums are added into the (zeroed) output
};
__host__ __device__ __forceinline__ int problem_works(const GemmProblem &p) { return p.tiles_m * p.tiles_n * p.splits; }

struct GemmArgs {
    GemmProblem pr[2];
    const uint8_t *sfa4, *sfb4;   // scale tiles, FP4 operands
    int64_t ntk_a4, ntk_b4;       // scale tiles per 128-row tile (cols_p / 64)
    const float *outa, *outb;     // FP32 outer scales [cols_p/128][rows_p]
    int64_t rpa, rpb;             // rows_p of A and B
    const uint8_t *sfa8, *sfb8;   // scale tiles, FP8 operands (of whichever product has FP8 stages)
    int64_t ntk_a8, ntk_b8;       // cols_p / 128
    uint32_t tx8;                 // bytes one slice stage brings in: both operand tiles (128 rows x 128
                                  // elements of 8, 6 or 4 bits, as stored in HBM) and two scale tiles
    uint32_t idesc8;              // the slice's element formats in the instruction descriptor (bits 7-12)
    long long wait_clk;           // bound of every mbarrier wait, in SM clocks
    int skip_stage;               // test hook: the producers never load this stage of each CTA (-1: none)
};

// The work of one output tile (or, with a split, of one half of its K): its product,
// origin and K schedule (FP4 stages of two 128-K blocks first, then the FP8 stages, which
// accumulate into one partial).  st0 / k80: the first FP4 stage and the first FP8 stage
// of the tile's K that this work covers.
struct TileWork {
    int p;
    int64_t m0, n0;
    int nkb4, nk8, nst4, nstages, nblk, st0, k80;
};
__device__ __forceinline__ TileWork tile_work(const GemmArgs &a, int t) {
    const int t1 = problem_works(a.pr[1]);
    TileWork w;
    int i;
    if (t1 > 0 && a.pr[0].tiles_m == a.pr[1].tiles_m) {
        // both products cover the same output rows: take them row block by row block (the
        // FP8 works of a row block, then its FP4 works), so that the two products' writes to
        // the same output rows follow each other while those rows are still in L2
        const int w1 = a.pr[1].tiles_n * a.pr[1].splits, w0 = a.pr[0].tiles_n * a.pr[0].splits;
        const int mb = t / (w0 + w1), r = t - mb * (w0 + w1);
        w.p = r < w1 ? 1 : 0;
        i = w.p ? mb * w1 + r : mb * w0 + (r - w1);
    } else {
        w.p = t < t1 ? 1 : 0;
        i = w.p ? t : t - t1;
    }
    const int split = w.p ? a.pr[1].splits : a.pr[0].splits;
    const int tn = w.p ? a.pr[1].tiles_n : a.pr[0].tiles_n;
    const int nkb4 = w.p ? a.pr[1].nkb4 : a.pr[0].nkb4, nk8 = w.p ? a.pr[1].nk8 : a.pr[0].nk8;
    const int sp = split == 2 ? (i & 1) : 0, ti = split == 2 ? (i >> 1) : i;
    w.m0 = (int64_t)(ti / tn) * 128;
    w.n0 = (int64_t)(ti % tn) * 128;
    w.st0 = 0;
    w.k80 = 0;
    w.nkb4 = nkb4;
    w.nk8 = nk8;
    if (split == 2) {
        const int s4a = ((nkb4 + 1) / 2 + 1) / 2, k8a = (nk8 + 1) / 2;
        const int kb4a = nkb4 < 2 * s4a ? nkb4 : 2 * s4a;
        w.st0 = sp ? s4a : 0;
        w.k80 = sp ? k8a : 0;
        w.nkb4 = sp ? nkb4 - kb4a : kb4a;
        w.nk8 = sp ? nk8 - k8a : k8a;
    }
    w.nst4 = (w.nkb4 + 1) / 2;
    w.nstages = w.nst4 + w.nk8;
    w.nblk = w.nkb4 + (w.nk8 > 0 ? 1 : 0);
    return w;
}

struct Bars {
    uint64_t full[kStages], empty[kStages];
    uint64_t pfull[kPSlots];
    uint64_t sempty[kScaleSlots];
    uint64_t drain;
    uint32_t tmem_base;
    volatile int abort_flag;
    volatile int met[kPSlots];    // generations of each slot's named barrier the MMA warp has met
                                  // (written by the MMA warp alone, as plain stores)
};
static_assert(sizeof(Bars) <= 512, "barrier block");

// Bounded wait on an mbarrier phase: gives up after kWaitClk SM clocks (or as
// soon as another role has aborted), setting the sticky device error flag and
// the CTA's abort flag.  No wait in this kernel can spin forever.  The bound is
// kept in SM clocks because the clock register is read in a few cycles.
__device__ __forceinline__ bool wait_bounded(uint64_t *bar, uint32_t parity, Bars *bars, long long wait_clk) {
    if (ptx::mbar_try_wait(bar, parity)) return true;         // fast path
    const long long t0 = clock64();
    for (;;) {
        if (bars->abort_flag) return false;
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > wait_clk) break;
    }
    atomicOr(&g_tj_dev_error, 1u);
    bars->abort_flag = 1;
    return false;
}

// Bounded wait that ignores the abort flag: used only to drain asynchronous work
// (copies, MMAs) that is already in flight before the CTA frees its memory.
__device__ __forceinline__ void wait_drain(uint64_t *bar, uint32_t parity, long long wait_clk) {
    const long long t0 = clock64();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > wait_clk) {
            atomicOr(&g_tj_dev_error, 1u);
            return;
        }
    }
}

// Hardware named barriers (ids 1..15; 0 is __syncthreads).  `count` threads, a
// multiple of 32, take part; every warp executes them warp-uniformly.
__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("barrier.cta.sync.aligned %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_arrive(int id, int count) {
    asm volatile("barrier.cta.arrive.aligned %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Warp-uniform bounded wait.  Every lane polls the barrier: a completed phase is
// seen several hundred cycles sooner by a warp whose lanes all wait than by one
// that waits on lane 0 and broadcasts (measured on GB300 in the partial-slot
// handshake: 802 against 858 cycles per block).  The result is the lanes'
// conjunction; a phase, once complete, stays complete, so the lanes agree unless
// the wait ran out.
__device__ __forceinline__ bool warp_wait_bounded(uint64_t *bar, uint32_t parity, Bars *bars, long long wait_clk) {
    const bool ok = wait_bounded(bar, parity, bars, wait_clk);
    return __all_sync(0xffffffffu, ok);
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

// Packed pairs of fp32 (element 0 in the low half): one instruction for two lanes of work.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ float lo2(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi2(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
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

// A 16-byte shared-memory load issued where it stands in the program: each of the
// promotion's column-scale loads then sits right before the math that uses it.  Left to
// the compiler, the same loads were scheduled otherwise and the layer set's GEMMs took 5%
// longer (1.88 against 1.78 ms per step).
__device__ __forceinline__ float4 lds128_in_order(const float4 *p) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(ptx::smem_u32(p)));
    return v;
}

// The barrier protocol of a promotion warp that has stopped waiting for partials (a
// wait ran out, or another role aborted), from block kb of `tile` on: it takes part in
// every remaining generation of the partial slots' named barriers with a sync.  A live
// warp arrives on them without waiting, which is safe because it reached each block only
// after the MMA warp had met the slot's previous generation; a warp that stops being live
// may have arrived on that generation already, and a second participation in one
// generation would derail every later one.  So before each sync it waits until the MMA
// warp has published (met[]) that it met the slot's previous generation.  The MMA warp
// meets the generations in order and waits on nothing else once the launch has aborted,
// so this takes microseconds; the wait is bounded by the default limit.  Not inlined: it
// keeps the code of the working loop as it was.
__device__ __noinline__ void promo_drain(const GemmArgs &args, Bars *bars, int tile, int kb, int ps, uint32_t pph,
                                         int ncta, int ntiles) {
    for (; tile < ntiles; tile += ncta, kb = 0) {
        const TileWork w = tile_work(args, tile);
        for (; kb < w.nblk; ++kb) {
            // this is use u of slot ps, and met[ps] is u - 1 or u here (this warp took part in
            // generation u - 1 already), so its parity, that of the slot's phase bit
            // pph = u & 1, tells the two apart
            const long long t0 = clock64();
            while (((uint32_t)bars->met[ps] & 1u) != pph && clock64() - t0 <= kWaitClk) {
            }
            named_sync(kNamedP + ps, kNamedCount);
            if (++ps == kPSlots) { ps = 0; pph ^= 1u; }
        }
    }
}

// kTestHook: the launch honours the test hook of tj_debug_gemm_fault (a stage the
// producers never load, a shorter bound for every wait); production launches use the
// instantiation without it, whose bound is the constant kWaitClk.
template <bool kTestHook>
__global__ void __launch_bounds__(kThreadsGemm, 1)
    k_gemm_nvfp4(const __grid_constant__ CUtensorMap tm_a4, const __grid_constant__ CUtensorMap tm_b4,
                 const __grid_constant__ CUtensorMap tm_a8, const __grid_constant__ CUtensorMap tm_b8,
                 const __grid_constant__ CUtensorMap tm_d, const GemmArgs args) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars *bars = reinterpret_cast<Bars *>(smem + kSmemBar);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long wclk = kTestHook ? args.wait_clk : kWaitClk;    // bound of every mbarrier wait
    const int ntiles = problem_works(args.pr[0]) + problem_works(args.pr[1]);
    const int cta = (int)blockIdx.x, ncta = (int)gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(&bars->full[s], 1);
            ptx::mbar_init(&bars->empty[s], 1);
        }
        for (int p = 0; p < kPSlots; ++p) ptx::mbar_init(&bars->pfull[p], 1);
        for (int q = 0; q < kScaleSlots; ++q) ptx::mbar_init(&bars->sempty[q], kPromoWarps);
        ptx::mbar_init(&bars->drain, 1);
        bars->abort_flag = 0;
        for (int p = 0; p < kPSlots; ++p) bars->met[p] = 0;
        ptx::fence_mbar_init();
    }
    if (warp == kMmaWarp) ptx::tmem_alloc(&bars->tmem_base, kTmemCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tbase = bars->tmem_base;

    if (warp < kProdWarps) {
        // ------------------------------------------------------------ producers: one thread can
        // issue a stage only every few hundred cycles, so stages alternate between warps
        if (lane == 0) {
            if (args.pr[0].nkb4 > 0) { ptx::prefetch_tmap(&tm_a4); ptx::prefetch_tmap(&tm_b4); }
            if (args.pr[0].nk8 > 0 || args.pr[1].nk8 > 0) { ptx::prefetch_tmap(&tm_a8); ptx::prefetch_tmap(&tm_b8); }
            int it = 0, fbase = 0;                            // stages / FP4 blocks of earlier tiles
            bool ok = true;
            for (int tile = cta; tile < ntiles && ok; tile += ncta) {
                const TileWork w = tile_work(args, tile);
                const int64_t rta = w.m0 / 128, rtb = w.n0 / 128;
                for (int st = 0; st < w.nstages; ++st, ++it) {
                    if (it % kProdWarps != warp) continue;
                    const int slot = it % kStages;
                    if (it >= kStages && !wait_bounded(&bars->empty[slot], ((it / kStages) - 1) & 1, bars, wclk)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sa = smem + kSmemA + slot * kTileBytes;
                    uint8_t *sb = smem + kSmemB + slot * kTileBytes;
                    uint8_t *sfa = smem + kSmemSfa + slot * kSfStageBytes;
                    uint8_t *sfb = smem + kSmemSfb + slot * kSfStageBytes;
                    const bool fp4 = st < w.nst4;
                    const int k0 = fp4 ? w.st0 + st : w.k80 + st - w.nst4;   // 128-byte column of the operand rows
                    const int nkbs = fp4 ? min(2, w.nkb4 - 2 * st) : 0;
                    const uint32_t sfbytes = fp4 ? (uint32_t)nkbs * 1024u : 512u;
                    // the outer-scale slots of the stage's blocks: FP4 block f (counted over this
                    // CTA's tiles) uses slot f % kScaleSlots, freed when the promotion of block
                    // f - kScaleSlots has finished with it
                    const int f0 = fbase + 2 * st;
                    for (int j = 0; j < nkbs && ok; ++j) {
                        const int f = f0 + j;
                        if (f >= kScaleSlots &&
                            !wait_bounded(&bars->sempty[f % kScaleSlots], ((f / kScaleSlots) - 1) & 1, bars, wclk))
                            ok = false;
                    }
                    if (!ok) break;
                    // test hook: this stage is never loaded, so the waits for it run out
                    if (kTestHook && it == args.skip_stage) continue;
                    // operands, their scale-factor tiles and, for FP4 stages, the FP32 outer
                    // scales of the stage's blocks all land on one barrier
                    ptx::mbar_arrive_expect_tx(&bars->full[slot], fp4 ? 2u * kTileBytes + 2u * sfbytes + (uint32_t)nkbs * 1024u
                                                                   : args.tx8);
                    ptx::tma_load_2d(sa, fp4 ? &tm_a4 : &tm_a8, k0 * 128, (int32_t)w.m0, &bars->full[slot]);
                    ptx::tma_load_2d(sb, fp4 ? &tm_b4 : &tm_b8, k0 * 128, (int32_t)w.n0, &bars->full[slot]);
                    if (fp4) {
                        ptx::bulk_load(sfa, args.sfa4 + (rta * args.ntk_a4 + 4 * k0) * 512, sfbytes, &bars->full[slot]);
                        ptx::bulk_load(sfb, args.sfb4 + (rtb * args.ntk_b4 + 4 * k0) * 512, sfbytes, &bars->full[slot]);
                        for (int j = 0; j < nkbs; ++j) {
                            const int64_t kb = 2 * k0 + j;
                            uint8_t *so = smem + kSmemScale + ((f0 + j) % kScaleSlots) * 1024;
                            ptx::bulk_load(so, args.outa + kb * args.rpa + w.m0, 512u, &bars->full[slot]);
                            ptx::bulk_load(so + 512, args.outb + kb * args.rpb + w.n0, 512u, &bars->full[slot]);
                        }
                    } else {
                        ptx::bulk_load(sfa, args.sfa8 + (rta * args.ntk_a8 + k0) * 512, 512u, &bars->full[slot]);
                        ptx::bulk_load(sfb, args.sfb8 + (rtb * args.ntk_b8 + k0) * 512, 512u, &bars->full[slot]);
                    }
                }
                fbase += w.nkb4;
            }
            // drain: every copy this warp issued must have landed before the CTA exits
            for (int j = (it > kStages ? it - kStages : 0); j < it; ++j)
                if (j % kProdWarps == warp && (!kTestHook || j != args.skip_stage))
                    wait_drain(&bars->full[j % kStages], (j / kStages) & 1, wclk);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer (warp-uniform loop;
        // lane 0 issues).  Before a partial slot is rewritten, the named barrier of that slot
        // meets every promotion warp's release of the block that used it three blocks earlier;
        // that also frees the slot's scale-factor columns, which only that block's MMAs read.
        const uint32_t idesc4 = idesc_nvf4();
        int it = 0, pc = 0;
        bool live = true;
        for (int tile = cta; tile < ntiles; tile += ncta) {
            const TileWork w = tile_work(args, tile);
            for (int st = 0; st < w.nstages; ++st, ++it) {
                const int slot = it % kStages;
                if (live) live = warp_wait_bounded(&bars->full[slot], (it / kStages) & 1, bars, wclk);
                ptx::tc_fence_after();
                const uint32_t sa = ptx::smem_u32(smem + kSmemA + slot * kTileBytes);
                const uint32_t sb = ptx::smem_u32(smem + kSmemB + slot * kTileBytes);
                const uint32_t sfa = ptx::smem_u32(smem + kSmemSfa + slot * kSfStageBytes);
                const uint32_t sfb = ptx::smem_u32(smem + kSmemSfb + slot * kSfStageBytes);
                if (st < w.nst4) {
                    const int nkbs = min(2, w.nkb4 - 2 * st);
                    for (int kbl = 0; kbl < nkbs; ++kbl, ++pc) {
                        const int ps = pc % kPSlots;
                        if (pc >= kPSlots) named_sync(kNamedP + ps, kNamedCount);
                        ptx::tc_fence_after();
                        if (live && lane == 0) {
                            const uint32_t sfcol = tbase + kColSf + 16u * (uint32_t)ps;
#pragma unroll
                            for (int j = 0; j < 2; ++j) {   // one 512-byte scale tile per K = 64 MMA
                                ptx::tc_cp_32x128b_warpx4(sfcol + 4 * j,
                                                          ptx::smem_desc(sfa + 512 * (2 * kbl + j), 0, 128, 0));
                                ptx::tc_cp_32x128b_warpx4(sfcol + 8 + 4 * j,
                                                          ptx::smem_desc(sfb + 512 * (2 * kbl + j), 0, 128, 0));
                            }
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                const uint32_t koff = 64u * kbl + 32u * j;
                                ptx::mma_nvf4(tbase + kColP + 128u * ps, ptx::smem_desc(sa + koff, 16, 1024, 2),
                                              ptx::smem_desc(sb + koff, 16, 1024, 2), idesc4, sfcol + 4 * j,
                                              sfcol + 8 + 4 * j, (uint32_t)j);
                            }
                            ptx::tc_commit(&bars->pfull[ps]);
                        }
                        __syncwarp();
                        // the generation just met, published for the promotion warps' abort path
                        // (a plain store, after the issue so that it stays off the meet-to-issue path)
                        if (pc >= kPSlots && lane == 0) bars->met[ps] = pc / kPSlots;
                    }
                } else {
                    // the FP8 slice: all its stages accumulate into one partial slot.  A stage's
                    // scale factors use the tensor-memory slot of its operand ring slot: the
                    // previous user of that slot, stage it - kStages, has completed its MMAs,
                    // because the producers refilled the ring slot only after its release
                    const int s8 = st - w.nst4;
                    const int ps = pc % kPSlots;
                    if (s8 == 0 && pc >= kPSlots) named_sync(kNamedP + ps, kNamedCount);
                    ptx::tc_fence_after();
                    if (live && lane == 0) {
                        const uint32_t sfcol = tbase + kColSf8 + 8u * (uint32_t)slot;
                        ptx::tc_cp_32x128b_warpx4(sfcol, ptx::smem_desc(sfa, 0, 128, 0));
                        ptx::tc_cp_32x128b_warpx4(sfcol + 4, ptx::smem_desc(sfb, 0, 128, 0));
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            ptx::mma_mxf8(tbase + kColP + 128u * ps, ptx::smem_desc(sa + 32u * j, 16, 1024, 2),
                                          ptx::smem_desc(sb + 32u * j, 16, 1024, 2), idesc_mxf8((uint32_t)j) | args.idesc8, sfcol,
                                          sfcol + 4, (uint32_t)(s8 > 0 || j > 0));
                        }
                        if (s8 == w.nk8 - 1) ptx::tc_commit(&bars->pfull[ps]);
                    }
                    __syncwarp();
                    if (s8 == 0 && pc >= kPSlots && lane == 0) bars->met[ps] = pc / kPSlots;
                    if (s8 == w.nk8 - 1) ++pc;
                }
                // the stage's buffers are free once its MMAs complete
                if (live && lane == 0) ptx::tc_commit(&bars->empty[slot]);
                __syncwarp();
            }
        }
        // meet the promotion warps' releases of the last blocks
        for (int j = (pc > kPSlots ? pc - kPSlots : 0); j < pc; ++j) {
            named_sync(kNamedP + j % kPSlots, kNamedCount);
            if (lane == 0) bars->met[j % kPSlots] = j / kPSlots + 1;
        }
        // all MMAs / copies issued by this thread complete before TMEM is freed
        if (lane == 0) {
            ptx::tc_commit(&bars->drain);
            wait_drain(&bars->drain, 0, wclk);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ promotion + epilogue
        const int pw = warp - kPromo0;
        const int q = warp & 3;                 // TMEM lane quadrant of this warp
        const int cq = pw >> 2;                 // columns kColsW*cq .. +kColsW-1
        const uint32_t taddr0 = tbase + ((uint32_t)(32 * q) << 16) + kColP + (uint32_t)(kColsW * cq);
        int f4c = 0;                            // FP4 blocks promoted so far (outer-scale ring position)
        int ps = 0;
        uint32_t pph = 0;                       // partial ring slot and phase
        bool aborted = false;                   // a wait ran out: promo_drain keeps the barrier protocol
        for (int tile = cta; tile < ntiles && !aborted; tile += ncta) {
            const TileWork w = tile_work(args, tile);
            const GemmProblem &g = w.p ? args.pr[1] : args.pr[0];
            const int64_t m0 = w.m0, n0 = w.n0;
            const float alpha = g.alpha;
            uint64_t acc[kColsW / 2];
#pragma unroll
            for (int j = 0; j < kColsW / 2; ++j) acc[j] = 0ull;
            for (int kb = 0; kb < w.nblk; ++kb) {
                if (!warp_wait_bounded(&bars->pfull[ps], pph, bars, wclk)) {
                    promo_drain(args, bars, tile, kb, ps, pph, ncta, ntiles);
                    aborted = true;
                    break;
                }
                const float *so = reinterpret_cast<const float *>(smem + kSmemScale + (f4c % kScaleSlots) * 1024);
#pragma unroll
                for (int ch = 0; ch < kColsW / kLdCols; ++ch) {
                    uint32_t p[kLdCols];
                    ptx::tc_fence_after();
#pragma unroll
                    for (int c = 0; c < kLdCols / 32; ++c)
                        ptx::tmem_ld_32x32b_x32(taddr0 + 128u * (uint32_t)ps + (uint32_t)(kLdCols * ch + 32 * c),
                                                *reinterpret_cast<uint32_t(*)[32]>(p + 32 * c));
                    ptx::tmem_wait_ld();
                    if (ch == kColsW / kLdCols - 1) {
                        ptx::tc_fence_before();
                        __syncwarp();
                        // release the partial slot.  The warp arrives without waiting: it reached this
                        // block only after the MMA warp had met the previous use of the slot.
                        named_arrive(kNamedP + ps, kNamedCount);
                    }
                    uint64_t *ac = acc + (kLdCols / 2) * ch;
                    if (kb < w.nkb4) {
                        {
                            // the block's outer scales: their slot goes back to the producers once
                            // every promotion warp has done this math (the arrivals below)
                            const float sa = so[32 * q + lane] * alpha;
                            const uint64_t sa2 = pack2(sa, sa);
                            const float4 *sbp = reinterpret_cast<const float4 *>(
                                so + 128 + kColsW * cq + kLdCols * ch);
#pragma unroll
                            for (int i = 0; i < kLdCols / 4; ++i) {
                                const float4 sb = lds128_in_order(sbp + i);   // broadcast: all lanes, one address
                                const uint64_t w0 = mul2(sa2, pack2(sb.x, sb.y));
                                const uint64_t w1 = mul2(sa2, pack2(sb.z, sb.w));
                                ac[2 * i] = fma2((uint64_t)p[4 * i] | ((uint64_t)p[4 * i + 1] << 32), w0, ac[2 * i]);
                                ac[2 * i + 1] =
                                    fma2((uint64_t)p[4 * i + 2] | ((uint64_t)p[4 * i + 3] << 32), w1, ac[2 * i + 1]);
                            }
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < kLdCols / 2; ++i)
                            ac[i] = add2(ac[i], (uint64_t)p[2 * i] | ((uint64_t)p[2 * i + 1] << 32));
                    }
                }
                if (kb < w.nkb4) {
                    // this warp is done with the block's outer scales: its share of handing their
                    // slot back to the producers (the slot's barrier counts the promotion warps)
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&bars->sempty[f4c % kScaleSlots]);
                    ++f4c;
                }
                if (++ps == kPSlots) { ps = 0; pph ^= 1u; }
            }
            if (aborted) break;
            // epilogue: the warp's 32 x kColsW slice of the tile (rows 32q.., columns kColsW*cq..)
            const int64_t rbase = m0 + 32 * q;
            const int64_t nb = n0 + kColsW * cq;
            if (g.tma_store) {
                uint32_t *stg = reinterpret_cast<uint32_t *>(smem + kSmemEpi + pw * kEpiTma);
                if (lane == 0) ptx::bulk_wait_read_all();     // this warp's previous TMA store has read it
                __syncwarp();
                // bf16 without scatter: each lane's row segment (2 kColsW bytes) goes to the staging
                // buffer in the swizzle of the output tensor map (128-byte rows: 16-byte chunk c of
                // row r at c ^ (r & 7); 64-byte rows: c ^ ((r >> 1) & 3)), and one TMA store writes
                // the slice (clipping rows >= M and columns >= N) while the warp moves on
                uint8_t *rowp = reinterpret_cast<uint8_t *>(stg) + lane * (2 * kColsW);
                const int sw = kColsW == 64 ? (lane & 7) : ((lane >> 1) & 3);
#pragma unroll
                for (int i = 0; i < kColsW / 8; ++i) {
                    uint32_t w4[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        __nv_bfloat162 b2 = __floats2bfloat162_rn(lo2(acc[4 * i + k]), hi2(acc[4 * i + k]));
                        w4[k] = *reinterpret_cast<uint32_t *>(&b2);
                    }
                    *reinterpret_cast<uint4 *>(rowp + ((i ^ sw) << 4)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ptx::tma_store_2d(&tm_d, (int32_t)nb, (int32_t)rbase, stg);
                    ptx::bulk_commit_group();
                }
                continue;
            }
            // fp32 outputs, scattered columns (col_map), ragged edges or unaligned row pitches: the
            // warp stages its slice in shared memory, kColsW / 2 words per row plus a pad word (so
            // row writes and column reads are both free of bank conflicts), and writes it a few
            // rows per store instruction, a lane per word, so each instruction covers contiguous
            // row segments.  bf16: one pass of kColsW / 2 column pairs; fp32: two passes of
            // kColsW / 2 columns.
            constexpr int kW = kColsW / 2, kRp = 32 / kW;      // words per staged row, rows per store
            uint32_t *stg = reinterpret_cast<uint32_t *>(smem + kSmemEpi + pw * kEpiRow);
            const int wl = lane % kW, rsub = lane / kW;
            if (g.out_bf16) {
#pragma unroll
                for (int j = 0; j < kW; ++j) {
                    __nv_bfloat162 b2 = __floats2bfloat162_rn(lo2(acc[j]), hi2(acc[j]));
                    stg[lane * (kW + 1) + j] = *reinterpret_cast<uint32_t *>(&b2);
                }
                __syncwarp();
                const int64_t na = nb + 2 * wl, nz = na + 1;     // this lane's column pair
                const bool va = na < g.N, vz = nz < g.N;
                const int64_t ca = va ? (g.col_map ? (int64_t)g.col_map[na] : na) : 0;
                const int64_t cz = vz ? (g.col_map ? (int64_t)g.col_map[nz] : nz) : 0;
                // two 2-byte stores per lane and row, the same for every lane: choosing a 4-byte
                // store where a lane's pair happens to be adjacent and aligned splits the warp
                // into divergent store instructions, which measured slower
                for (int r = rsub; r < 32 && rbase + r < g.M; r += kRp) {
                    const uint32_t w = stg[r * (kW + 1) + wl];
                    __nv_bfloat16 *drow = static_cast<__nv_bfloat16 *>(g.d) + (rbase + r) * g.ldd;
                    if (va) drow[ca] = __ushort_as_bfloat16((unsigned short)(w & 0xffffu));
                    if (vz) drow[cz] = __ushort_as_bfloat16((unsigned short)(w >> 16));
                }
                __syncwarp();
            } else {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
#pragma unroll
                    for (int j = 0; j < kW; ++j) {
                        const int e = kW * h + j;
                        stg[lane * (kW + 1) + j] = __float_as_uint((e & 1) ? hi2(acc[e >> 1]) : lo2(acc[e >> 1]));
                    }
                    __syncwarp();
                    const int64_t n = nb + kW * h + wl;
                    const bool v = n < g.N;
                    const int64_t c = v ? (g.col_map ? (int64_t)g.col_map[n] : n) : 0;
                    float *dcol = static_cast<float *>(g.d) + c;
                    if (g.splits > 1) {                                  // half of a split K: add
                        for (int r = rsub; r < 32 && rbase + r < g.M; r += kRp)
                            if (v) atomicAdd(dcol + (rbase + r) * g.ldd, __uint_as_float(stg[r * (kW + 1) + wl]));
                    } else {
                        for (int r = rsub; r < 32 && rbase + r < g.M; r += kRp)
                            if (v) dcol[(rbase + r) * g.ldd] = __uint_as_float(stg[r * (kW + 1) + wl]);
                    }
                    __syncwarp();
                }
            }
        }
        // every TMA store of this warp has completed before the CTA exits
        if (lane == 0) ptx::bulk_wait_all();
        __syncwarp();
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
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

// An MX slice operand [rows_p][cols_p] of element format fmt -> boxes of 128 rows x 128
// elements.  E4M3 rows are plain bytes.  Packed E2M3 / E3M2 / E2M1 rows use the packed
// sub-byte tensor-map types, whose copies expand each run of 16 codes (12 or 8 bytes in
// HBM) into the 16-byte shared-memory slot the f8f6f4 MMA reads, so the shared tile has the
// E4M3 tile's shape; coordinates count elements, and a box moves 128 x 96 or 128 x 64
// bytes of HBM (the transaction count its barrier sees).
bool make_mx_map(CUtensorMap *m, const void *base, int64_t rows_p, int64_t cols_p, int fmt) {
    if (fmt == kMxE4M3) return make_tile_map(m, base, rows_p, cols_p, 128u);
    EncodeTiledFn enc = get_encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols_p, (cuuint64_t)rows_p};
    const cuuint64_t strides[1] = {(cuuint64_t)(cols_p * mx_bits(fmt) / 8)};
    const cuuint32_t box[2] = {128u, 128u};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUtensorMapDataType t =
        fmt == kMxE2M1 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_16U6_ALIGN16B;
    return enc(m, t, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 output [M][ldd] -> boxes of 32 rows x kColsW columns (one promotion warp's slice),
// swizzled to the row width (128 or 64 bytes), for the epilogue's TMA stores.
bool make_out_map(CUtensorMap *m, void *d, int64_t M, int64_t N, int64_t ldd) {
    EncodeTiledFn enc = get_encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)ldd * 2u};
    const cuuint32_t box[2] = {(cuuint32_t)kColsW, 32u};
    const cuuint32_t estr[2] = {1u, 1u};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               kColsW == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms_of_current_device() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
}

// The test hook of tj_debug_gemm_fault, armed for the next launch that runs.
int g_fault_skip_stage = -1;
long long g_fault_wait_clk = 0;        // 0: the default bound kWaitClk

// Persistent launch: one CTA per SM (or per tile, if fewer).
cudaError_t launch_persistent(const CUtensorMap (&tm)[5], const GemmArgs &g_in, cudaStream_t s) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e =
            cudaFuncSetAttribute(k_gemm_nvfp4<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes + 1024);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_gemm_nvfp4<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes + 1024);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int ntiles = problem_works(g_in.pr[0]) + problem_works(g_in.pr[1]);
    if (ntiles == 0) return cudaSuccess;
    GemmArgs g = g_in;
    const bool armed = g_fault_skip_stage >= 0 || g_fault_wait_clk > 0;
    g.wait_clk = g_fault_wait_clk > 0 ? g_fault_wait_clk : kWaitClk;
    g.skip_stage = g_fault_skip_stage;
    g_fault_skip_stage = -1;
    g_fault_wait_clk = 0;
    const int nsm = num_sms_of_current_device();
    const unsigned grid = (unsigned)(ntiles < nsm ? ntiles : nsm);
    if (armed)
        k_gemm_nvfp4<true><<<grid, kThreadsGemm, kSmemBytes + 1024, s>>>(tm[0], tm[1], tm[2], tm[3], tm[4], g);
    else
        k_gemm_nvfp4<false><<<grid, kThreadsGemm, kSmemBytes + 1024, s>>>(tm[0], tm[1], tm[2], tm[3], tm[4], g);
    return cudaGetLastError();
}

GemmProblem problem(int64_t M, int64_t N, float alpha, void *d, int out_dtype, int64_t ldd, const int32_t *col_map) {
    GemmProblem p{};
    p.M = M;
    p.N = N;
    p.alpha = alpha;
    p.d = d;
    p.out_bf16 = out_dtype == TJ_BF16;
    p.ldd = ldd;
    p.col_map = col_map;
    p.tiles_m = (int)(round_up(M, 128) / 128);
    p.tiles_n = (int)(round_up(N, 128) / 128);
    p.splits = 1;
    return p;
}

// Split K in two when the caller allows it (an fp32 output region), every product of the
// launch has at least 8 stages of K (so each half keeps 4), and the halves fill the SMs in
// fewer rounds of half-length works than whole tiles would (e.g. 72 tiles on 152 SMs: one
// round of halves instead of one of wholes; 216 tiles: three rounds of halves instead of two
// of wholes).  The output region is zeroed on the stream first.
cudaError_t maybe_split(GemmArgs &g, const SplitRegion *split, cudaStream_t s) {
    if (split == nullptr) return cudaSuccess;
    for (const GemmProblem &p : g.pr)
        if (p.tiles_m * p.tiles_n > 0 && (p.out_bf16 || p.tma_store || (p.nkb4 + 1) / 2 + p.nk8 < 8)) return cudaSuccess;
    const int nsm = num_sms_of_current_device();
    const int t = g.pr[0].tiles_m * g.pr[0].tiles_n + g.pr[1].tiles_m * g.pr[1].tiles_n;
    const int whole = (t + nsm - 1) / nsm, halves = (2 * t + nsm - 1) / nsm;
    if (t == 0 || halves >= 2 * whole) return cudaSuccess;
    const cudaError_t e = cudaMemset2DAsync(split->base, (size_t)split->ld * sizeof(float), 0,
                                            (size_t)split->cols * sizeof(float), (size_t)split->rows, s);
    if (e != cudaSuccess) return e;
    g.pr[0].splits = g.pr[1].splits = 2;
    return cudaSuccess;
}

// FP4 operands -> tensor maps 0/1 and the scale pointers; returns the 128-K block count.
bool set_fp4(const tj_nvfp4 &a, const tj_nvfp4 &b, GemmArgs &g, CUtensorMap (&tm)[5], int &nkb4) {
    const int64_t kp = round_up(a.cols, 128);
    nkb4 = (int)(kp / 128);
    if (nkb4 == 0 || a.rows == 0 || b.rows == 0) { nkb4 = 0; return true; }   // no FP4 blocks: no loads
    g.sfa4 = a.sf;
    g.sfb4 = b.sf;
    g.ntk_a4 = kp / 64;
    g.ntk_b4 = kp / 64;
    g.outa = a.outer;
    g.outb = b.outer;
    g.rpa = round_up(a.rows, 128);
    g.rpb = round_up(b.rows, 128);
    return make_tile_map(&tm[0], a.codes, g.rpa, kp / 2, 128u) && make_tile_map(&tm[1], b.codes, g.rpb, kp / 2, 128u);
}

// Slice operands (FP8, or FP6 / FP4 in any pairing) -> tensor maps 2/3, the scale pointers,
// the stage's transaction bytes and the formats of the instruction descriptor; returns the
// 128-K stage count.
bool set_fp8(const tj_mxfp8 &a8, const tj_mxfp8 &b8, GemmArgs &g, CUtensorMap (&tm)[5], int &nk8) {
    const int64_t kp8 = round_up(a8.cols, 128);
    nk8 = (int)(kp8 / 128);
    if (nk8 == 0 || a8.rows == 0 || b8.rows == 0) { nk8 = 0; return true; }   // no slice stages: no loads
    g.sfa8 = a8.sf;
    g.sfb8 = b8.sf;
    g.ntk_a8 = kp8 / 128;
    g.ntk_b8 = kp8 / 128;
    g.tx8 = (uint32_t)(128 * 128 * (mx_bits(a8.fmt) + mx_bits(b8.fmt)) / 8 + 2 * 512);
    g.idesc8 = ((uint32_t)a8.fmt << 7) | ((uint32_t)b8.fmt << 10);
    return make_mx_map(&tm[2], a8.codes, round_up(a8.rows, 128), kp8, a8.fmt) &&
           make_mx_map(&tm[3], b8.codes, round_up(b8.rows, 128), kp8, b8.fmt);
}

// Plain bf16 outputs (no column map, 16-byte row pitch) of a single-product launch leave the
// kernel by TMA stores.
void set_tma_store(GemmProblem &p, CUtensorMap &tm) {
    p.tma_store = p.out_bf16 && p.col_map == nullptr && (p.ldd & 7) == 0 &&
                  (reinterpret_cast<uintptr_t>(p.d) & 15) == 0 && p.M > 0 && p.N > 0 &&
                  make_out_map(&tm, p.d, p.M, p.N, p.ldd);
}

}  // namespace

cudaError_t launch_gemm(const tj_nvfp4 *a, const tj_nvfp4 *b, const tj_mxfp8 *a8, const tj_mxfp8 *b8, float alpha,
                        void *d, int out_dtype, int64_t ldd, int64_t M, int64_t N, const int32_t *col_map,
                        cudaStream_t s, const SplitRegion *split) {
    GemmArgs g{};
    g.pr[0] = problem(M, N, alpha, d, out_dtype, ldd, col_map);
    if (g.pr[0].tiles_m == 0 || g.pr[0].tiles_n == 0) return cudaSuccess;
    CUtensorMap tm[5];
    memset(tm, 0, sizeof(tm));
    if (a != nullptr && b != nullptr && !set_fp4(*a, *b, g, tm, g.pr[0].nkb4)) return cudaErrorInvalidValue;
    if (a8 != nullptr && b8 != nullptr && a8->cols > 0 && !set_fp8(*a8, *b8, g, tm, g.pr[0].nk8))
        return cudaErrorInvalidValue;
    set_tma_store(g.pr[0], tm[4]);
    const cudaError_t e = maybe_split(g, split, s);
    if (e != cudaSuccess) return e;
    return launch_persistent(tm, g, s);
}

cudaError_t launch_gemm_pair(const tj_nvfp4 *a, const tj_nvfp4 *b, float alpha, void *d, int out_dtype, int64_t ldd,
                             int64_t M, int64_t N, const int32_t *col_map, const tj_mxfp8 *a8, const tj_mxfp8 *b8,
                             void *d8, int out8_dtype, int64_t ldd8, int64_t M8, int64_t N8, const int32_t *col_map8,
                             cudaStream_t s, const SplitRegion *split) {
    GemmArgs g{};
    g.pr[0] = problem(M, N, alpha, d, out_dtype, ldd, col_map);
    g.pr[1] = problem(M8, N8, 1.0f, d8, out8_dtype, ldd8, col_map8);
    CUtensorMap tm[5];
    memset(tm, 0, sizeof(tm));
    if (!set_fp4(*a, *b, g, tm, g.pr[0].nkb4) || !set_fp8(*a8, *b8, g, tm, g.pr[1].nk8)) return cudaErrorInvalidValue;
    if (g.pr[0].tiles_m * g.pr[0].tiles_n == 0) g.pr[0].tiles_m = g.pr[0].tiles_n = 0;
    // a product over an empty contraction is zero: its tiles run with no blocks and write zeros
    if (g.pr[1].tiles_m * g.pr[1].tiles_n == 0) g.pr[1].tiles_m = g.pr[1].tiles_n = 0;
    const cudaError_t e = maybe_split(g, split, s);
    if (e != cudaSuccess) return e;
    return launch_persistent(tm, g, s);
}

unsigned int read_and_clear_device_error() {
    unsigned int v = 0u, z = 0u;
    if (cudaMemcpyFromSymbol(&v, g_tj_dev_error, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
    cudaMemcpyToSymbol(g_tj_dev_error, &z, sizeof(z));
    return v;
}

}  // namespace tj

// Test hook: arm a fault for the next GEMM launch (see tj.h).
extern "C" tj_status tj_debug_gemm_fault(int skip_stage, int64_t wait_clk) {
    if (skip_stage < -1 || wait_clk < 0) return TJ_ERR_INVALID_ARG;
    tj::g_fault_skip_stage = skip_stage;
    tj::g_fault_wait_clk = (long long)wait_clk;
    return TJ_OK;
}
