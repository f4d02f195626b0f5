// Tensor-core GEMM of libtern for M > 16 tokens (batched decode, prefill):
//   Y[M,N] = X[M,K] . (s (.) T)^T
//
// Method ("Ternary embedding model in vLLM", 2kiu.com/news/5082861, §4.2):
// the packed weights are dequantised tile by tile on chip and fed to the
// tensor cores (the page's "dequantise, then a dense GEMM" route, with the
// dequantisation fused into the GEMM instead of materialising W).
//
// Exactness: the dequantised weight t * s is exactly representable in fp16
// (t in {-1,0,+1}, s an FP16 scale).  The activations are converted once by
// `xprep_kernel` to fp16 after scaling each token row by a power of two
// 2^c_m chosen so that its largest magnitude lies in [2^14, 2^15): every
// bf16 value at most 2^-32 of the row's maximum converts exactly.  The
// products are then exact in fp32 and each item's K range accumulates in
// fp32 in tensor memory; the epilogue multiplies by 2^-c_m (exact).
//
// Work item = 256 weight rows (two 128-row tiles) x NT tokens x a range of
// 128-wide groups along K.  Both row tiles share every activation tile,
// halving the activation traffic per flop.  One launch may serve up to
// kMaxGroup independent linears with the same M (their items concatenated).
// Warp roles of the persistent CTA (one per SM):
//   * weight producer warp: bulk copies of 4 groups per row tile per stage;
//     two activation producer warps, alternate stages: one 3-D TMA copy of
//     a group (2 chunks of 64 along K, 128-byte swizzle) per stage -- a
//     CTA's copy engine completes only a few copies per microsecond per
//     issuing warp, so copies are few and large;
//   * two decode warpgroups, one per row tile (one thread per weight row =
//     one tensor-memory lane): code word -> exact fp16 t (LOP3 + FMA), times
//     the row's scale (one multiply) -> tcgen05.st into the row tile's A
//     ring (2 units, 3 when NT <= 64);
//   * MMA warp (warp-uniform loop, one elected lane issues): per group and
//     row tile eight tcgen05.mma (M = 128, N = NT, K = 16, f16 -> fp32);
//   * epilogue warpgroup: tcgen05.ld of both accumulators, times 2^-c_m,
//     stores (or, when K is split across items, the item's fp32 partial,
//     which split_reduce_kernel sums in split order after the GEMM).
// Every wait is bounded; a timeout raises the workspace error word.

#include <cuda.h>

#include <mutex>
#include <type_traits>
#include <vector>

#include "tern_common.cuh"
#include "tern_internal.h"
#include "tern_sm100.cuh"

namespace tern {
namespace {

// The MMA warp and the producers come first: a scheduler choosing among
// ready warps favours the older ones, and the decode warps are always
// ready with long runs of integer and FMA work.  Warp w reaches
// tensor-memory lanes 32 (w mod 4) .. +31, so the decode and epilogue
// warpgroups start at multiples of 4.
constexpr int kMmaWarp = 0;
constexpr int kProducerWarp = 1;                // weights
constexpr int kXWarp0 = 2;                      // 2 warps: activation stages, alternately
constexpr int kDecWarp0 = 4;
constexpr int kDecWarps = 8;                    // warpgroup r decodes row tile r of the pair
constexpr int kEpiWarp0 = kDecWarp0 + kDecWarps;   // 4 warps
constexpr int kThreads = (kEpiWarp0 + 4) * 32;
constexpr int kMaxNT = 128;                     // tokens per tile (UMMA N)
constexpr int kTmemCols = 512;
constexpr int kACols = 64;                      // one unit of fp16 A (128 per row)
// A ring per row tile: AU slots of kACols columns for each of the two row
// tiles, then the two accumulators of NT columns.  Three slots fit beside
// accumulators of up to 64 tokens, two beside 128 (see au_for).
constexpr int kAUMax = 3;
constexpr int kMaxNTForAU3 = (kTmemCols - 2 * 3 * kACols) / 2;
static_assert(2 * 2 * kACols + 2 * kMaxNT <= kTmemCols, "tensor-memory budget");
constexpr int kWG = 4;                          // groups per weight stage
constexpr int kWS = 2;                          // weight stages
constexpr int kXG = 1;                          // groups per activation stage (one TMA copy)
constexpr int kXS = 4;                          // activation stages; producer warp = stage mod 2
constexpr int kXStageMax = kXG * 2 * kMaxNT * 128;          // 2 chunks of 64 per group
constexpr int kWStage = 2 * kWG * kUnitBytes;              // both row tiles
constexpr int kCtrlBytes = 1024;
constexpr int kYTok = 16;                       // tokens per output staging buffer
constexpr int kYStage = kYTok * kTileRows * 4;  // one buffer: 16 tokens x 128 rows, up to 4 bytes each
constexpr int kSmemBytes = 1024 + kXS * kXStageMax + kWS * kWStage + 2 * kYStage + kCtrlBytes;
static_assert(kSmemBytes <= 232448, "shared-memory budget");
static_assert(kXS % 2 == 0, "each activation stage has one producer warp");

// control block offsets
constexpr int kBarXFull = 0;                                 // [kXS]
constexpr int kBarXEmpty = kBarXFull + 8 * kXS;              // [kXS]
constexpr int kBarWFull = kBarXEmpty + 8 * kXS;              // [kWS]
constexpr int kBarWEmpty = kBarWFull + 8 * kWS;              // [kWS]
constexpr int kBarAFull = kBarWEmpty + 8 * kWS;              // [AU], both row tiles
constexpr int kBarAEmpty = kBarAFull + 8 * kAUMax;           // [AU]
constexpr int kBarDFull = kBarAEmpty + 8 * kAUMax;
constexpr int kBarDEmpty = kBarDFull + 8;
constexpr int kBarDrain = kBarDEmpty + 8;
constexpr int kTmemPtr = kBarDrain + 8;
constexpr int kAbort = kTmemPtr + 4;
static_assert(kAbort + 4 <= kCtrlBytes, "control block");

// One linear of the launch (a launch serves up to kMaxGroup independent
// linears with the same M; their items are concatenated).
struct GemmProb {
    const uint8_t* codes;
    const uint8_t* scales;     // per unit: 128 FP16 scales, or (s8) 128 int8 scales
    const float* inv_scale;    // [T * NT + 32]: 2^-c_m of the problem's tokens
    float* partial;            // K split: [RP * T][KS][2][NT / 4][128][4]
    OutputSplit out;
    int64_t N;
    int64_t item_begin;        // items of the problems before this one
    int G;                     // groups along K
    int R;                     // 128-row tiles
    int RP;                    // pairs of row tiles
    int KS;                    // splits of K
    int tma_store;             // outputs written through ymaps.map[ymap0 + j] (see launch_gemm)
    int ymap0;
};

// Parameters of a grouped launch: up to kMaxGroup problems.
struct GemmArgsG {
    const float* row_factor;   // unused (int8 scales need a single problem)
    int s8;
    int scale_unit;            // 256
    const uint8_t* zflags;     // unused
    int M;
    int NT;                    // tokens per tile
    int T;                     // token tiles
    int P;                     // problems
    int64_t items;             // sum over problems of RP * T * KS
    int* err;
    GemmProb prob[kMaxGroup];
};

// Parameters of a single-problem launch: the problem's fields at the top
// level (one shared parameter layout with the grouped launch measured 6 %
// slower at 4096 tokens).
struct GemmArgs1 {
    const uint8_t* codes;
    const uint8_t* scales;     // per unit: 128 FP16 scales, or (s8) 128 int8 scales
    const float* row_factor;   // s8: per row, the factor of its int8 scales
    int s8;
    int scale_unit;            // 256 or 128 (s8)
    const uint8_t* zflags;     // optional, per unit: 1 = every weight of the unit is 0 (skipped)
    const float* inv_scale;    // [T * NT + 32]: 2^-c_m
    int M;
    int NT;                    // tokens per tile
    int G;                     // groups along K
    int R;                     // 128-row tiles
    int RP;                    // pairs of row tiles
    int T;                     // token tiles
    int KS;                    // splits of K
    int64_t N;
    int64_t items;             // RP * T * KS
    OutputSplit out;
    int* err;
    float* partial;            // [RP * T][KS][2][NT / 4][128][4]
    int tma_store;             // outputs written through ymaps (see launch_gemm)
    int ymap0;                 // 0
};
template <bool GROUPED>
using GemmArgsT = std::conditional_t<GROUPED, GemmArgsG, GemmArgs1>;

// Tensor maps of the activations (fp16, one per problem) and of the outputs
// (inner dimension: the output's rows n, outer: tokens m; box 128 x kYTok)
// for stores by TMA: one per output of a single problem, or one per problem.
template <int NP>
struct XMaps {
    CUtensorMap map[NP];
};
template <int NP>
struct YMaps {
    CUtensorMap map[NP > kMaxOutputs ? NP : kMaxOutputs];
};
template <bool GROUPED>
constexpr int kProbs = GROUPED ? kMaxGroup : 1;

// The fields of problem p: a grouped launch's entry, or the single
// problem's parameter block itself.
template <bool GROUPED, typename A>
__device__ __forceinline__ const auto& prob_ref(const A& a, int p) {
    if constexpr (GROUPED)
        return a.prob[p];
    else
        return a;
}
__device__ __forceinline__ int nprob(const GemmArgs1&) { return 1; }
__device__ __forceinline__ int nprob(const GemmArgsG& a) { return a.P; }

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
    const bool got = mbar_wait(bar, parity, abort);
    return __all_sync(0xffffffffu, got);
}

// Each lane with `active` set waits for its own barrier; the warp goes on when
// all have completed.  The common case (all complete) costs one test and one
// vote: a wait in the MMA warp is time the tensor pipe stands idle, since the
// issue of a group's MMAs returns only once the pipe has taken all but the last.
__device__ __forceinline__ bool vote_wait(uint32_t bar, uint32_t parity, bool active, volatile int* abort) {
    if (__all_sync(0xffffffffu, !active || mbar_test_wait(bar, parity))) return true;
    const bool got = !active || mbar_wait(bar, parity, abort);
    return __all_sync(0xffffffffu, got);
}

// 3-D TMA load (coordinates c0 innermost).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1, int32_t c2,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// 2^-c_m of C consecutive tokens (the workspace holds at least 32 entries
// past the last token tile).  Every lane reads the same addresses.
template <int C>
__device__ __forceinline__ void load_inv(const float* p, float (&inv)[C]) {
    const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
    for (int i = 0; i < C / 4; ++i) {
        const float4 v = __ldg(q + i);
        inv[4 * i] = v.x;
        inv[4 * i + 1] = v.y;
        inv[4 * i + 2] = v.z;
        inv[4 * i + 3] = v.w;
    }
}

__device__ __forceinline__ bool unit_zero(const uint8_t* zflags, int G, int64_t tile, int g) {
    return zflags != nullptr && zflags[tile * G + g] != 0;
}

// Whether row tile `tile` has a non-zero unit among groups [g0, g1).
__device__ __forceinline__ bool tile_has_data(const uint8_t* zflags, int G, int64_t tile, int g0, int g1) {
    if (zflags == nullptr) return true;
    for (int g = g0; g < g1; ++g)
        if (zflags[tile * G + g] == 0) return true;
    return false;
}

// Item i -> (problem, row-tile pair, token tile, K split); within a problem
// the token tile is slowest, so that the CTAs working at the same time
// share activation tiles in L2.
struct Item {
    int p, bp, n, ks;
};
template <bool GROUPED, typename A>
__device__ __forceinline__ Item item_of(const A& a, int64_t i) {
    Item it;
    int p = 0;
    int64_t local = i;
    if constexpr (GROUPED) {
        while (p + 1 < a.P && i >= a.prob[p + 1].item_begin) ++p;
        local = i - a.prob[p].item_begin;
    }
    const auto& q = prob_ref<GROUPED>(a, p);
    it.p = p;
    it.ks = static_cast<int>(local % q.KS);
    const int64_t t = local / q.KS;
    it.bp = static_cast<int>(t % q.RP);
    it.n = static_cast<int>(t / q.RP);
    return it;
}
template <typename Q>
__device__ __forceinline__ void group_range(const Q& q, int ks, int& g0, int& g1) {
    g0 = static_cast<int>((int64_t)q.G * ks / q.KS);
    g1 = static_cast<int>((int64_t)q.G * (ks + 1) / q.KS);
}

// EXT: the weights may carry int8 scales (a.s8) or zero-unit flags
// (a.zflags); the plain instantiation has neither check on its hot paths.
// AU: A-ring slots per row tile (3 needs a.NT <= kMaxNTForAU3).
// GROUPED: a.P problems (else one, whose fields the compiler then reads at
// fixed offsets).
// The current item's problem.
#define GQ (prob_ref<GROUPED>(a, it.p))

template <bool EXT, int AU, bool GROUPED>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ XMaps<kProbs<GROUPED>> xmaps, const __grid_constant__ YMaps<kProbs<GROUPED>> ymaps,
            const GemmArgsT<GROUPED> a) {
    static_assert(AU == 2 || AU == kAUMax, "A-ring depth");
    constexpr int kAU = AU;
    constexpr int kDCol0 = 2 * kAU * kACols;   // two accumulators of NT columns follow the A rings
    const bool s8 = EXT && a.s8 != 0;
    const uint8_t* const zflags = EXT ? a.zflags : nullptr;
    const int scale_unit = EXT ? a.scale_unit : kUnitScaleBytes;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const int NT = a.NT;
    const int x_stage = kXG * 2 * NT * 128;       // bytes of one activation stage
    const uint32_t xring = sbase;
    const uint32_t wring = sbase + kXS * kXStageMax;
    uint8_t* wring_ptr = smem + kXS * kXStageMax;
    uint8_t* ystage = smem + kXS * kXStageMax + kWS * kWStage;   // 2 output staging buffers
    uint8_t* ctrl = ystage + 2 * kYStage;
    const uint32_t cb = smem_u32(ctrl);
    uint32_t* tmem_base_ptr = reinterpret_cast<uint32_t*>(ctrl + kTmemPtr);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + kAbort);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kXS; ++i) {
            mbar_init(cb + kBarXFull + 8 * i, 1);
            mbar_init(cb + kBarXEmpty + 8 * i, 1);   // MMA commit
        }
        for (int i = 0; i < kWS; ++i) {
            mbar_init(cb + kBarWFull + 8 * i, 1);
            mbar_init(cb + kBarWEmpty + 8 * i, kDecWarps);
        }
        for (int i = 0; i < kAU; ++i) {
            mbar_init(cb + kBarAFull + 8 * i, kDecWarps);   // both row tiles
            mbar_init(cb + kBarAEmpty + 8 * i, 1);          // MMA commit
        }
        mbar_init(cb + kBarDFull, 1);
        mbar_init(cb + kBarDEmpty, 4);
        mbar_init(cb + kBarDrain, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_base_ptr), kTmemCols);
        tmem_relinquish();
    }
    if (warp == kXWarp0 && lane < nprob(a)) prefetch_tensormap(&xmaps.map[lane]);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_base_ptr;
    grid_launch_dependents();

    if (warp == kProducerWarp) {
        // -------------------------------------------------- weight producer
        // a CTA's copies complete at a rate per issuing warp, so weights and
        // activations have their own producer warps
        int ws = 0;
        uint32_t w_round = 0;
        int64_t wcount = 0;
        bool ok = true;
        for (int64_t i = blockIdx.x; i < a.items && ok; i += gridDim.x) {
            const Item it = item_of<GROUPED>(a, i);
            int g0, g1;
            group_range(GQ, it.ks, g0, g1);
            const bool two = 2 * it.bp + 1 < GQ.R;
            for (int g = g0; g < g1; g += kWG) {   // weights of up to kWG groups, both row tiles
                if (wcount >= kWS && !(ok = warp_wait(cb + kBarWEmpty + 8 * ws, (w_round - 1) & 1u, abort_flag))) break;
                const int cnt = g1 - g < kWG ? g1 - g : kWG;
                const uint32_t st = wring + ws * kWStage;
                if (elect_one()) {
                    mbar_arrive_expect_tx(cb + kBarWFull + 8 * ws, (two ? 2 : 1) * cnt * (kUnitCodeBytes + scale_unit));
#pragma unroll
                    for (int rt = 0; rt < 2; ++rt) {
                        if (rt == 1 && !two) break;
                        const int64_t u = (int64_t)(2 * it.bp + rt) * GQ.G + g;
                        bulk_load(st + rt * kWG * kUnitCodeBytes, GQ.codes + u * kUnitCodeBytes, cnt * kUnitCodeBytes,
                                  cb + kBarWFull + 8 * ws);
                        bulk_load(st + 2 * kWG * kUnitCodeBytes + rt * kWG * kUnitScaleBytes,
                                  GQ.scales + u * scale_unit, cnt * scale_unit, cb + kBarWFull + 8 * ws);
                    }
                }
                __syncwarp();
                ++wcount;
                if (++ws == kWS) {
                    ws = 0;
                    ++w_round;
                }
            }
        }
        if (*abort_flag) {
            volatile int no_abort = 0;
            for (int t = 0; t < kWS; ++t) {
                (void)mbar_wait(cb + kBarWFull + 8 * t, 0, &no_abort);
                (void)mbar_wait(cb + kBarWFull + 8 * t, 1, &no_abort);
            }
        }
    } else if (warp == kXWarp0 || warp == kXWarp0 + 1) {
        // ---------------------------------------------- activation producers
        // activation stage j (over all items' groups, in order) belongs to
        // producer warp j mod 2; it is stage j mod kXS of the ring
        const int q = warp - kXWarp0;
        grid_dependency_wait();   // the converted activations come from the kernel before
        int64_t j = 0;            // activation stages so far (all producers)
        bool ok = true;
        for (int64_t i = blockIdx.x; i < a.items && ok; i += gridDim.x) {
            const Item it = item_of<GROUPED>(a, i);
            int g0, g1;
            group_range(GQ, it.ks, g0, g1);
            for (int g = g0; g < g1; g += kXG, ++j) {
                if ((j & 1) != q) continue;
                const int xs = static_cast<int>(j % kXS);
                const uint32_t round = static_cast<uint32_t>(j / kXS);
                if (round > 0 && !(ok = warp_wait(cb + kBarXEmpty + 8 * xs, (round - 1) & 1u, abort_flag))) break;
                if (elect_one()) {
                    mbar_arrive_expect_tx(cb + kBarXFull + 8 * xs, x_stage);
                    tma_load_3d(xring + xs * kXStageMax, &xmaps.map[it.p], 0, it.n * NT, 2 * g, cb + kBarXFull + 8 * xs);
                }
                __syncwarp();
            }
        }
        if (*abort_flag) {
            volatile int no_abort = 0;
            for (int t = q; t < kXS; t += 2) {
                (void)mbar_wait(cb + kBarXFull + 8 * t, 0, &no_abort);
                (void)mbar_wait(cb + kBarXFull + 8 * t, 1, &no_abort);
            }
        }
    } else if (warp == kMmaWarp) {
        // --------------------------------------------------------------- MMA
        // per group one vote over: activation stage full (lane 1), A slot of
        // both row tiles full (lane 2), accumulators drained (lane 3, first
        // group of an item).  Lane 0 issues the MMAs and commits and tests
        // no barrier: a thread's barrier operations wait behind its own
        // commits, that is, until its last MMAs have completed.
        const uint32_t idesc = idesc_fp16_f32(128, static_cast<uint32_t>(NT));
        const uint64_t bdesc0 = smem_desc_kmajor_sw128(xring);
        int xs = 0, al = 0;
        uint32_t x_ph = 0, a_ph = 0;
        uint32_t d_round = 0;
        bool ok = true;
        for (int64_t i = blockIdx.x; i < a.items && ok; i += gridDim.x) {
            const Item it = item_of<GROUPED>(a, i);
            int g0, g1;
            group_range(GQ, it.ks, g0, g1);
            const bool two = 2 * it.bp + 1 < GQ.R;
            bool started0 = false, started1 = false;   // accumulators written this item
            for (int g = g0; g < g1; ++g) {
                const int xg = (g - g0) % kXG;
                const bool z0 = unit_zero(zflags, GQ.G, 2 * it.bp, g), z1 = !two || unit_zero(zflags, GQ.G, 2 * it.bp + 1, g);
                uint32_t bar = 0, par = 0;
                bool act = false;
                if (lane == 1) {
                    act = xg == 0;
                    bar = cb + kBarXFull + 8 * xs;
                    par = x_ph;
                } else if (lane == 2) {
                    act = true;
                    bar = cb + kBarAFull + 8 * al;
                    par = a_ph;
                } else if (lane == 3) {
                    act = g == g0 && d_round > 0;
                    bar = cb + kBarDEmpty;
                    par = (d_round - 1) & 1u;
                }
                if (!(ok = vote_wait(bar, par, act, abort_flag))) break;
                tc_fence_after_sync();
                // chunk 2*xg (+1) of the stage; +32 bytes per K-step inside a chunk
                const uint64_t b0 = bdesc0 + ((uint32_t)(xs * kXStageMax + 2 * xg * NT * 128) >> 4);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t bdesc = b0 + (uint32_t)((kk >> 2) * (NT * 128 / 16)) + 2 * (kk & 3);
                        if (!z0)
                            umma_bf16_tmem_a(tmem + kDCol0, tmem + al * kACols + 8 * kk, bdesc, idesc,
                                             (started0 || kk > 0) ? 1u : 0u);
                        if (!z1)
                            umma_bf16_tmem_a(tmem + kDCol0 + NT, tmem + (kAU + al) * kACols + 8 * kk, bdesc, idesc,
                                             (started1 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(cb + kBarAEmpty + 8 * al);
                    if (xg == kXG - 1 || g == g1 - 1) umma_commit(cb + kBarXEmpty + 8 * xs);
                    if (g == g1 - 1) umma_commit(cb + kBarDFull);
                }
                __syncwarp();
                started0 |= !z0;
                started1 |= !z1;
                if (++al == kAU) {
                    al = 0;
                    a_ph ^= 1u;
                }
                if (xg == kXG - 1 || g == g1 - 1) {
                    if (++xs == kXS) {
                        xs = 0;
                        x_ph ^= 1u;
                    }
                }
            }
            ++d_round;
        }
        if (elect_one()) umma_commit(cb + kBarDrain);
        __syncwarp();
        volatile int no_abort = 0;
        (void)mbar_wait(cb + kBarDrain, 0, &no_abort);
    } else if (warp >= kDecWarp0 && warp < kDecWarp0 + kDecWarps) {
        // ------------------------------------------------------------ decode
        // both warpgroups keep the A ring's phases even when an item has no
        // second row tile (they then arrive without decoding)
        const int rt = (warp - kDecWarp0) >> 2;         // row tile of the pair
        const int r = threadIdx.x & 127;                // weight row in the tile = tensor-memory lane
        const uint32_t tm = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + rt * kAU * kACols;
        const uint32_t bar_afull = cb + kBarAFull;
        const uint32_t bar_aempty = cb + kBarAEmpty;
        const DecodeConsts dk = decode_consts_fp16();
        int ws = 0, al = 0;
        uint32_t w_ph = 0, a_ph = 0;
        int64_t acount = 0;
        bool ok = true;
        for (int64_t i = blockIdx.x; i < a.items && ok; i += gridDim.x) {
            const Item it = item_of<GROUPED>(a, i);
            int g0, g1;
            group_range(GQ, it.ks, g0, g1);
            const bool tile_exists = rt == 0 || 2 * it.bp + 1 < GQ.R;
            for (int g = g0; g < g1; ++g) {
                const int wg = (g - g0) % kWG;
                if (wg == 0 && !(ok = warp_wait(cb + kBarWFull + 8 * ws, w_ph, abort_flag))) break;
                const bool mine = tile_exists && !unit_zero(zflags, GQ.G, 2 * it.bp + rt, g);   // a zero unit needs no A
                uint4 c0 = make_uint4(0, 0, 0, 0), c1 = c0;
                uint32_t s2 = 0;
                if (mine) {
                    const uint8_t* st = wring_ptr + ws * kWStage;
                    c0 = lds_v4(st + rt * kWG * kUnitCodeBytes + wg * kUnitCodeBytes + 16 * r);
                    c1 = lds_v4(st + rt * kWG * kUnitCodeBytes + wg * kUnitCodeBytes + 2048 + 16 * r);
                    const uint8_t* sp = st + 2 * kWG * kUnitCodeBytes + rt * kWG * kUnitScaleBytes + wg * scale_unit;
                    // int8 scale q: t * q is exact in fp16 (|q| <= 127); the row's factor comes at the end
                    const uint32_t sb = s8 ? __half_as_ushort(__int2half_rn(*reinterpret_cast<const int8_t*>(sp + r)))
                                             : *reinterpret_cast<const uint16_t*>(sp + 2 * r);
                    s2 = sb | (sb << 16);
                }
                if (acount >= kAU) {
                    if (!(ok = warp_wait(bar_aempty + 8 * al, a_ph ^ 1u, abort_flag))) break;
                    tc_fence_after_sync();
                }
                if (mine) {
                    // two stores of 32 columns: the first runs while the
                    // second half decodes (the empty asm keeps that decode
                    // after the first store)
                    uint32_t p[64];
                    decode_word_fp16_scaled(c0.x, s2, dk, p);
                    decode_word_fp16_scaled(c0.y, s2, dk, p + 8);
                    decode_word_fp16_scaled(c0.z, s2, dk, p + 16);
                    decode_word_fp16_scaled(c0.w, s2, dk, p + 24);
                    tmem_st_32x32b_x32(tm + al * kACols, p);
                    asm volatile("" : "+r"(c1.x), "+r"(c1.y), "+r"(c1.z), "+r"(c1.w));
                    decode_word_fp16_scaled(c1.x, s2, dk, p + 32);
                    decode_word_fp16_scaled(c1.y, s2, dk, p + 40);
                    decode_word_fp16_scaled(c1.z, s2, dk, p + 48);
                    decode_word_fp16_scaled(c1.w, s2, dk, p + 56);
                    tmem_st_32x32b_x32(tm + al * kACols + 32, p + 32);
                    tmem_st_wait();
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_afull + 8 * al);
                ++acount;
                if (++al == kAU) {
                    al = 0;
                    a_ph ^= 1u;
                }
                if (wg == kWG - 1 || g == g1 - 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(cb + kBarWEmpty + 8 * ws);
                    if (++ws == kWS) {
                        ws = 0;
                        w_ph ^= 1u;
                    }
                }
            }
        }
    } else if (warp >= kEpiWarp0) {
        // ---------------------------------------------------------- epilogue
        const int r = threadIdx.x & 127;
        const uint32_t tm = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + kDCol0;
        grid_dependency_wait();   // outputs and workspace belong to earlier kernels until now
        uint32_t d_ph = 0;
        uint32_t ybuf = 0;        // output staging buffers used so far
        for (int64_t i = blockIdx.x; i < a.items; i += gridDim.x) {
            const Item it = item_of<GROUPED>(a, i);
            // the four warps decide together (they meet at barrier 1 below)
            const bool got = warp_wait(cb + kBarDFull, d_ph, abort_flag);
            if (named_barrier_or(1, 128, !got)) break;
            d_ph ^= 1u;
            tc_fence_after_sync();
            const int m0 = it.n * NT;
            const int mvalid = a.M - m0 < NT ? a.M - m0 : NT;
            const bool two = 2 * it.bp + 1 < GQ.R;
            const int64_t tile = (int64_t)it.n * GQ.RP + it.bp;
            if (GQ.KS == 1 && GQ.tma_store) {
                // Through shared memory and TMA: the stores of the plain load
                // and store path hold back the whole kernel.  16 tokens at a
                // time into one of two staging buffers ([token][row]), one TMA
                // store per buffer by thread 0 of the warpgroup.
                const int nchunk = (mvalid + kYTok - 1) / kYTok;
                const int ebytes = GQ.out.bf16 ? 2 : 4;
                for (int rt = 0; rt < 2; ++rt) {
                    if (rt == 1 && !two) break;
                    const int64_t row0 = (int64_t)(2 * it.bp + rt) * kTileRows;
                    const int j = output_of(GQ.out, row0);
                    const int32_t n0 = static_cast<int32_t>(row0 - GQ.out.offset[j]);
                    const float f = s8 ? a.row_factor[row0 + r] : 1.0f;
                    const bool data = tile_has_data(zflags, GQ.G, 2 * it.bp + rt, 0, GQ.G);
                    for (int qc = 0; qc < nchunk; ++qc) {
                        const int c = qc * kYTok;
                        uint32_t d[16];
                        tmem_ld16_sync(tm + rt * NT + c, d);
                        float inv[16];
                        load_inv(GQ.inv_scale + m0 + c, inv);
                        // the buffer written two chunks ago has been read by its store
                        if (r == 0) bulk_wait_group_read<1>();
                        asm volatile("bar.sync 2, 128;" ::: "memory");
                        uint8_t* buf = ystage + (ybuf & 1) * kYStage;
#pragma unroll
                        for (int m = 0; m < 16; ++m) {
                            const float v = data ? __uint_as_float(d[m]) * (inv[m] * f) : 0.f;
                            if (ebytes == 4)
                                reinterpret_cast<float*>(buf)[m * kTileRows + r] = v;
                            else if (GQ.out.bf16 == 1)
                                reinterpret_cast<__nv_bfloat16*>(buf)[m * kTileRows + r] = __float2bfloat16_rn(v);
                            else
                                reinterpret_cast<__half*>(buf)[m * kTileRows + r] = __float2half_rn(v);
                        }
                        fence_proxy_async_smem();
                        asm volatile("bar.sync 2, 128;" ::: "memory");
                        if (r == 0) {
                            tma_store_2d(&ymaps.map[GROUPED ? GQ.ymap0 + j : j], n0, m0 + c, smem_u32(buf));
                            bulk_commit_group();
                        }
                        ++ybuf;
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(cb + kBarDEmpty);
            } else if (GQ.KS == 1) {
                // final values straight from tensor memory, 32 tokens per load
                for (int rt = 0; rt < 2; ++rt) {
                    if (rt == 1 && !two) break;
                    const int64_t row = (int64_t)(2 * it.bp + rt) * kTileRows + r;
                    const bool live = row < GQ.N;
                    const RowOut o = row_out(GQ.out, live ? row : 0);
                    const float f = s8 ? a.row_factor[row] : 1.0f;
                    const bool data = tile_has_data(zflags, GQ.G, 2 * it.bp + rt, 0, GQ.G);   // else the accumulators are stale
                    for (int c = 0; c < NT; c += 32) {
                        float inv[32];
                        load_inv(GQ.inv_scale + m0 + c, inv);
#pragma unroll
                        for (int m = 0; m < 32; ++m) inv[m] *= data ? f : 0.f;
                        uint32_t d[32];
                        if (c + 32 <= NT)
                            tmem_ld32_sync(tm + rt * NT + c, d);
                        else
                            tmem_ld16_sync(tm + rt * NT + c, d);
                        if (!data)
#pragma unroll
                            for (int m = 0; m < 32; ++m) d[m] = 0u;
                        float v[32];
#pragma unroll
                        for (int m = 0; m < 32; ++m) v[m] = __uint_as_float(d[m]) * inv[m];
                        store_run(GQ.out, o, m0 + c, m0 + mvalid, row, v, live);
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(cb + kBarDEmpty);
            } else {
                // this split's partial, laid out [rt][token / 4][row][4]: a
                // thread's four tokens are one 16-byte store, a warp's 512
                // contiguous bytes; split_reduce_kernel sums the splits
                float4* base = reinterpret_cast<float4*>(GQ.partial) + (tile * GQ.KS + it.ks) * (2 * (int64_t)NT * kTileRows / 4);
                int g0, g1;
                group_range(GQ, it.ks, g0, g1);
                for (int rt = 0; rt < 2; ++rt) {
                    if (rt == 1 && !two) break;
                    const bool data = tile_has_data(zflags, GQ.G, 2 * it.bp + rt, g0, g1);
                    for (int c = 0; c < NT; c += 32) {
                        uint32_t d[32];
                        if (c + 32 <= NT)
                            tmem_ld32_sync(tm + rt * NT + c, d);
                        else
                            tmem_ld16_sync(tm + rt * NT + c, d);
                        if (!data)
#pragma unroll
                            for (int m = 0; m < 32; ++m) d[m] = 0u;
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            if (c + 4 * u < NT)
                                base[((int64_t)(rt * NT + c) / 4 + u) * kTileRows + r] =
                                    make_float4(__uint_as_float(d[4 * u]), __uint_as_float(d[4 * u + 1]),
                                                __uint_as_float(d[4 * u + 2]), __uint_as_float(d[4 * u + 3]));
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(cb + kBarDEmpty);
            }
        }
    }

    // ------------------------------------------------------------ teardown
    if (threadIdx.x == kEpiWarp0 * 32) bulk_wait_group_all();   // output stores complete
    tc_fence_before_sync();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) atomicOr(a.err, 1);
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

#undef GQ

// Activation rows -> fp16 scaled by 2^c_m (largest magnitude in [2^14,
// 2^15)), and 2^-c_m per row.  One CTA per row.
__device__ __forceinline__ float x_lo(uint32_t w, int x_f16) {
    return x_f16 ? __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu))) : __uint_as_float(w << 16);
}
__device__ __forceinline__ float x_hi(uint32_t w, int x_f16) {
    return x_f16 ? __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16))) : __uint_as_float(w & 0xFFFF0000u);
}

struct XPrepProb {
    const uint16_t* X;
    int64_t ldx;
    int K;
    __half* X16;
    float* inv_scale;
};
struct XPrepArgs {
    XPrepProb prob[kMaxGroup];
    int x_f16;
};

__global__ void __launch_bounds__(256) xprep_kernel(const XPrepArgs args) {
    const int m = blockIdx.x;
    const XPrepProb& pr = args.prob[blockIdx.y];
    const int x_f16 = args.x_f16;
    const int K = pr.K;
    const uint16_t* xr = pr.X + (int64_t)m * pr.ldx;
    __half* yr = pr.X16 + (int64_t)m * K;
    float* inv_scale = pr.inv_scale;
    grid_dependency_wait();
    float mx = 0.f;
    for (int k = threadIdx.x * 8; k < K; k += 256 * 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(xr + k);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            mx = fmaxf(mx, fabsf(x_lo(w[i], x_f16)));
            mx = fmaxf(mx, fabsf(x_hi(w[i], x_f16)));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    __shared__ float wmax[8];
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = wmax[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) mx = fmaxf(mx, wmax[i]);
    // exponent of the largest magnitude; c brings it to 2^14
    int c = 0;
    if (mx > 0.f && mx < INFINITY) {
        const int e = static_cast<int>((__float_as_uint(mx) >> 23) & 0xFF) - 127;   // floor(log2), normal mx
        c = 14 - e;
        if (c > 120) c = 120;
        if (c < -120) c = -120;
    }
    const float scale = __uint_as_float(static_cast<uint32_t>(127 + c) << 23);
    if (threadIdx.x == 0) inv_scale[m] = __uint_as_float(static_cast<uint32_t>(127 - c) << 23);
    for (int k = threadIdx.x * 8; k < K; k += 256 * 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(xr + k);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half lo = __float2half_rn(x_lo(w[i], x_f16) * scale);
            const __half hi = __float2half_rn(x_hi(w[i], x_f16) * scale);
            o[i] = static_cast<uint32_t>(__half_as_ushort(lo)) | (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
        }
        *reinterpret_cast<uint4*>(yr + k) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    grid_launch_dependents();
}

// K split across items: the sum of a tile's partials in split order, times
// 2^-c_m (and, with int8 scales, the row's factor), to the outputs.  One
// thread per weight row, 16 tokens per CTA; the loads of kSumSplits splits
// are in flight together.  The CTAs of the split problems of a launch are
// concatenated.  Launched after gemm_kernel, whose completion it waits for.
struct ReduceProb {
    const float4* partial;     // [RP * T][KS][2][NT / 4][128] float4
    const float* inv_scale;
    OutputSplit out;
    int64_t N;
    int64_t block_begin;       // CTAs of the split problems before this one
    int R, RP, KS;
};
struct ReduceArgs {
    const float* row_factor;   // null unless int8 scales (one problem)
    int M, NT, P;
    ReduceProb prob[kMaxGroup];
};

__global__ void __launch_bounds__(kTileRows) split_reduce_kernel(const ReduceArgs a) {
    grid_dependency_wait();   // every split's partial is written
    grid_launch_dependents();
    constexpr int kSumSplits = 4;
    int p = 0;
    while (p + 1 < a.P && static_cast<int64_t>(blockIdx.x) >= a.prob[p + 1].block_begin) ++p;
    const ReduceProb& q = a.prob[p];
    const int64_t b = blockIdx.x - q.block_begin;
    const int nb = a.NT / 16;                      // 16-token blocks per tile
    const int cb = static_cast<int>(b % nb);
    const int rt = static_cast<int>((b / nb) & 1);
    const int64_t tile = b / (2 * nb);             // token tile * RP + row pair
    const int bp = static_cast<int>(tile % q.RP);
    const int m0 = static_cast<int>(tile / q.RP) * a.NT;
    const int mvalid = a.M - m0 < a.NT ? a.M - m0 : a.NT;
    const int c = 16 * cb;
    if (c >= mvalid || 2 * bp + rt >= q.R) return;
    const int r = threadIdx.x;
    const int64_t split_stride = 2 * (int64_t)a.NT * kTileRows / 4;
    const float4* src = q.partial + tile * q.KS * split_stride + ((int64_t)(rt * a.NT + c) / 4) * kTileRows + r;
    float v[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) v[m] = 0.f;
    for (int k0 = 0; k0 < q.KS; k0 += kSumSplits) {
        float4 t[kSumSplits][4];
#pragma unroll
        for (int kk = 0; kk < kSumSplits; ++kk)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                t[kk][j] = k0 + kk < q.KS ? __ldcg(src + (k0 + kk) * split_stride + j * kTileRows)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int kk = 0; kk < kSumSplits; ++kk) {
            if (k0 + kk >= q.KS) break;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[4 * j] += t[kk][j].x;
                v[4 * j + 1] += t[kk][j].y;
                v[4 * j + 2] += t[kk][j].z;
                v[4 * j + 3] += t[kk][j].w;
            }
        }
    }
    const int64_t row = (int64_t)(2 * bp + rt) * kTileRows + r;
    const bool live = row < q.N;
    const RowOut o = row_out(q.out, live ? row : 0);
    const float f = a.row_factor != nullptr && live ? a.row_factor[row] : 1.0f;
    float inv[16];
    load_inv(q.inv_scale + m0 + c, inv);
#pragma unroll
    for (int m = 0; m < 16; ++m) v[m] *= inv[m] * f;
    store_run(q.out, o, m0 + c, m0 + mvalid, row, v, live);
}

// ---------------------------------------------------------------- host

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

template <bool EXT, int AU, bool GROUPED>
cudaError_t set_smem_limit() {
    static cudaError_t status = cudaErrorUnknown;
    static std::once_flag once;
    std::call_once(once, [] {
        status = cudaFuncSetAttribute(gemm_kernel<EXT, AU, GROUPED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      kSmemBytes);
    });
    return status;
}

// The launch with the parameter block of its problem count (prepared for
// kMaxGroup problems).
template <bool EXT, int AU, bool GROUPED>
cudaError_t launch_kernel(const cudaLaunchConfig_t& cfg, const XMaps<kMaxGroup>& xm, const YMaps<kMaxGroup>& ym,
                          const GemmArgsG& a) {
    constexpr int NP = kProbs<GROUPED>;
    XMaps<NP> x;
    YMaps<NP> y;
    memcpy(&x, &xm, sizeof(x));   // the first NP maps
    memcpy(&y, &ym, sizeof(y));
    if constexpr (GROUPED) {
        return cudaLaunchKernelEx(&cfg, gemm_kernel<EXT, AU, GROUPED>, x, y, a);
    } else {
        const GemmProb& q = a.prob[0];
        GemmArgs1 b = {};
        b.codes = q.codes;
        b.scales = q.scales;
        b.row_factor = a.row_factor;
        b.s8 = a.s8;
        b.scale_unit = a.scale_unit;
        b.zflags = a.zflags;
        b.inv_scale = q.inv_scale;
        b.M = a.M;
        b.NT = a.NT;
        b.G = q.G;
        b.R = q.R;
        b.RP = q.RP;
        b.T = a.T;
        b.KS = q.KS;
        b.N = q.N;
        b.items = a.items;
        b.out = q.out;
        b.err = a.err;
        b.partial = q.partial;
        b.tma_store = q.tma_store;
        b.ymap0 = 0;
        return cudaLaunchKernelEx(&cfg, gemm_kernel<EXT, AU, GROUPED>, x, y, b);
    }
}

// A-ring depth for a token tile of NT: the deeper ring wherever tensor
// memory holds it beside the accumulators (the decode -> MMA hand-off of
// a slot is latency-bound at small NT).
int au_for(int NT) { return NT <= kMaxNTForAU3 ? kAUMax : 2; }

}  // namespace

namespace {

// Splits of one linear's K: as many as one wave holds when its row-pair x
// token tiles fill less than one wave.  With more tiles than SMs, the fewest
// splits (up to 4) that cut the waves of whole-item time by a tenth (216 row
// pairs on 152 SMs: 2 waves -> 3 waves of half items), if the fp32 partials
// stay within 64 MB (about half of L2) or the split items are still long
// (64 groups or more), so that writing and summing the partials costs less
// than the waves save.
int64_t splits_one(int64_t tiles, int64_t G, int NT, int sm_count) {
    int64_t ks = tiles < sm_count ? sm_count / tiles : 1;
    if (tiles >= sm_count) {
        const int64_t w1 = ceil_div(tiles, (int64_t)sm_count);
        for (int64_t k = 2; k <= 4; ++k) {
            const int64_t partial_bytes = tiles * k * 2 * NT * kTileRows * 4;
            if (ceil_div(tiles * k, (int64_t)sm_count) * 10 <= w1 * k * 9 &&
                (partial_bytes <= (int64_t(64) << 20) || G / k >= 64)) {
                ks = k;
                break;
            }
        }
    }
    if (ks > G / 4) ks = G / 4;
    return ks < 1 ? 1 : ks;
}

// Splits of a group of linears served by one launch.  The CTAs take items in
// turn (item i -> CTA i mod grid), so the launch lasts as long as its most
// loaded CTA.  For each target item length L (in groups) every problem's K is
// cut into about G / L splits; the CTA loads are tallied in groups, plus a
// fixed cost per item (pipeline fill, accumulator drain), plus per split item
// its partial's write and read (NT / 32 groups), plus the reduction launch;
// the lowest maximum wins (the longer items on a tie).  Targets that make
// more than 16 items per SM are not considered.
void splits_group(int P, const int64_t* tiles, const int64_t* G, int NT, int sm_count, int64_t* KS) {
    int64_t whole = 0;
    for (int q = 0; q < P; ++q) {
        KS[q] = 1;
        whole += tiles[q];
    }
    if (whole > 16 * int64_t(sm_count)) return;   // no split can help: already more items than any target allows
    // longest items first: the unsplit plan is always tallied
    static const int64_t kTargets[] = {int64_t(1) << 40, 216, 108, 64, 54, 40, 32, 27, 20, 16, 12, 8};
    constexpr int64_t kItemCost = 2, kReduceCost = 4;
    int64_t best = -1;
    for (const int64_t L : kTargets) {
        int64_t ks[kMaxGroup], items = 0;
        bool split = false;
        for (int q = 0; q < P; ++q) {
            int64_t k = (G[q] + L / 2) / L;
            if (k > G[q] / 4) k = G[q] / 4;
            if (k < 1) k = 1;
            ks[q] = k;
            split |= k > 1;
            items += tiles[q] * k;
        }
        if (items > 16 * int64_t(sm_count) && best >= 0) continue;
        const int64_t grid = items < sm_count ? items : sm_count;
        std::vector<int64_t> load(static_cast<size_t>(grid), 0);
        int64_t i = 0;
        for (int q = 0; q < P; ++q)
            for (int64_t t = 0; t < tiles[q]; ++t)
                for (int64_t k = 0; k < ks[q]; ++k, ++i) {
                    const int64_t len = G[q] * (k + 1) / ks[q] - G[q] * k / ks[q];
                    load[static_cast<size_t>(i % grid)] += len + kItemCost + (ks[q] > 1 ? NT / 32 : 0);
                }
        int64_t span = 0;
        for (const int64_t l : load) span = l > span ? l : span;
        if (split) span += kReduceCost;
        if (best < 0 || span < best) {
            best = span;
            for (int q = 0; q < P; ++q) KS[q] = ks[q];
        }
    }
}

}  // namespace

GemmPlan plan_gemm(int64_t M, const int64_t* N, const int64_t* K, int P, int sm_count) {
    GemmPlan p = {};
    if (sm_count <= 0) sm_count = 152;
    p.P = P;
    p.T = ceil_div(M, kMaxNT);
    p.NT = static_cast<int>(round_up(ceil_div(M, p.T), 16));
    int64_t tiles[kMaxGroup];
    for (int q = 0; q < P; ++q) {
        p.R[q] = ceil_div(N[q], kTileRows);
        p.RP[q] = ceil_div(p.R[q], 2);
        p.G[q] = K[q] / kGroup;
        tiles[q] = p.RP[q] * p.T;
    }
    if (P == 1)
        p.KS[0] = splits_one(tiles[0], p.G[0], p.NT, sm_count);
    else
        splits_group(P, tiles, p.G, p.NT, sm_count, p.KS);
    p.items = 0;
    for (int q = 0; q < P; ++q) {
        p.item_begin[q] = p.items;
        p.items += tiles[q] * p.KS[q];
    }
    p.grid = p.items < sm_count ? p.items : sm_count;
    // workspace: error word, then per problem: X16 [M][K] fp16 | 2^-c per
    // token | split partials
    size_t off = kWorkspaceErrBytes;
    for (int q = 0; q < P; ++q) {
        p.off_x16[q] = off;
        off += round_up(M * K[q] * 2, 1024);
        p.off_inv[q] = off;
        off += round_up((p.T * p.NT + 32) * 4, 256);   // read 32 at a time from any token tile
        p.off_partial[q] = off;
        if (p.KS[q] > 1) off += static_cast<size_t>(tiles[q] * p.KS[q] * 2 * p.NT * kTileRows) * sizeof(float);
    }
    p.ws_bytes = off;
    return p;
}

cudaError_t launch_gemm(const StreamProblem* probs, int P, bool x_f16, bool s8, const uint8_t* zflags, int64_t M,
                        void* ws, const GemmPlan& plan, cudaStream_t stream) {
    uint8_t* w = static_cast<uint8_t*>(ws);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // activations -> fp16, one CTA per (token, problem) (programmatic
    // dependent launch: waits for the kernel before)
    {
        XPrepArgs xa = {};
        xa.x_f16 = x_f16 ? 1 : 0;
        for (int q = 0; q < P; ++q)
            xa.prob[q] = {probs[q].x, probs[q].ldx, static_cast<int>(probs[q].K),
                          reinterpret_cast<__half*>(w + plan.off_x16[q]), reinterpret_cast<float*>(w + plan.off_inv[q])};
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(M), static_cast<unsigned>(P));
        cfg.blockDim = dim3(256);
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, xprep_kernel, xa);
        if (e != cudaSuccess) return e;
    }
    EncodeTiledFn enc = encode_tiled_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    const bool ext = s8 || zflags != nullptr;
    if (ext && P != 1) return cudaErrorInvalidValue;
    const int au = au_for(plan.NT);
    const bool grouped = P > 1;
    cudaError_t e = ext       ? (au == 3 ? set_smem_limit<true, 3, false>() : set_smem_limit<true, 2, false>())
                    : grouped ? (au == 3 ? set_smem_limit<false, 3, true>() : set_smem_limit<false, 2, true>())
                              : (au == 3 ? set_smem_limit<false, 3, false>() : set_smem_limit<false, 2, false>());
    if (e != cudaSuccess) return e;
    GemmArgsG a = {};
    a.s8 = s8 ? 1 : 0;
    a.zflags = zflags;
    a.scale_unit = s8 ? kUnitScaleBytesS8 : kUnitScaleBytes;
    a.row_factor = s8 ? reinterpret_cast<const float*>(probs[0].tiled + plan.R[0] * plan.G[0] *
                                                                            (kUnitCodeBytes + kUnitScaleBytesS8))
                      : nullptr;
    a.M = static_cast<int>(M);
    a.NT = plan.NT;
    a.T = static_cast<int>(plan.T);
    a.P = P;
    a.items = plan.items;
    a.err = reinterpret_cast<int*>(w);
    XMaps<kMaxGroup> xmaps;
    YMaps<kMaxGroup> ymaps;
    memset(&xmaps, 0, sizeof(xmaps));
    memset(&ymaps, 0, sizeof(ymaps));
    for (int q = 0; q < P; ++q) {
        const StreamProblem& pr = probs[q];
        const OutputSplit& out = pr.out;
        GemmProb& g = a.prob[q];
        g.codes = pr.tiled;
        g.scales = pr.tiled + plan.R[q] * plan.G[q] * kUnitCodeBytes;
        g.inv_scale = reinterpret_cast<float*>(w + plan.off_inv[q]);
        g.partial = reinterpret_cast<float*>(w + plan.off_partial[q]);
        g.out = out;
        g.N = pr.N;
        g.item_begin = plan.item_begin[q];
        g.G = static_cast<int>(plan.G[q]);
        g.R = static_cast<int>(plan.R[q]);
        g.RP = static_cast<int>(plan.RP[q]);
        g.KS = static_cast<int>(plan.KS[q]);
        // X16 viewed as [K/64 chunks][M rows][64]: one box = 64 x NT x 2 chunks
        const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(pr.K / 64)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(pr.K) * 2, 128};
        const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(plan.NT), 2 * kXG};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (enc(&xmaps.map[q], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, w + plan.off_x16[q], dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        // outputs by TMA when every row tile falls in one output and the
        // outputs meet TMA's alignment (else the plain stores); one map per
        // output of a single problem, one per problem in a group (one output
        // each)
        g.ymap0 = P == 1 ? 0 : q;
        const int eb = out.bf16 ? 2 : 4;
        bool ok = g.KS == 1 && !out.glu && (P == 1 || out.n_out == 1);
        for (int j = 0; j < out.n_out && ok; ++j) {
            const int64_t nj = out.offset[j + 1] - out.offset[j];
            if (nj == 0) continue;
            ok = out.offset[j] % kTileRows == 0 && (reinterpret_cast<uintptr_t>(out.y[j]) & 15) == 0 &&
                 (out.ldy[j] * eb) % 16 == 0;
            if (!ok) break;
            const cuuint64_t ydims[2] = {static_cast<cuuint64_t>(nj), static_cast<cuuint64_t>(M)};
            const cuuint64_t ystrides[1] = {static_cast<cuuint64_t>(out.ldy[j]) * eb};
            const cuuint32_t ybox[2] = {static_cast<cuuint32_t>(kTileRows), static_cast<cuuint32_t>(kYTok)};
            const cuuint32_t yestr[2] = {1, 1};
            const CUtensorMapDataType dt = out.bf16 == 1   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                           : out.bf16 == 2 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
            ok = enc(&ymaps.map[g.ymap0 + j], dt, 2, out.y[j], ydims, ystrides, ybox, yestr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        }
        g.tma_store = ok ? 1 : 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (ext)
        e = au == 3 ? launch_kernel<true, 3, false>(cfg, xmaps, ymaps, a)
                    : launch_kernel<true, 2, false>(cfg, xmaps, ymaps, a);
    else if (grouped)
        e = au == 3 ? launch_kernel<false, 3, true>(cfg, xmaps, ymaps, a)
                    : launch_kernel<false, 2, true>(cfg, xmaps, ymaps, a);
    else
        e = au == 3 ? launch_kernel<false, 3, false>(cfg, xmaps, ymaps, a)
                    : launch_kernel<false, 2, false>(cfg, xmaps, ymaps, a);
    if (e != cudaSuccess) return e;
    // the split problems' reduction, one launch
    ReduceArgs ra = {};
    ra.row_factor = a.row_factor;
    ra.M = a.M;
    ra.NT = a.NT;
    int64_t blocks = 0;
    for (int q = 0; q < P; ++q) {
        if (plan.KS[q] == 1) continue;
        ReduceProb& r = ra.prob[ra.P++];
        r.partial = reinterpret_cast<const float4*>(a.prob[q].partial);
        r.inv_scale = a.prob[q].inv_scale;
        r.out = probs[q].out;
        r.N = probs[q].N;
        r.block_begin = blocks;
        r.R = a.prob[q].R;
        r.RP = a.prob[q].RP;
        r.KS = a.prob[q].KS;
        blocks += plan.RP[q] * plan.T * 2 * (plan.NT / 16);
    }
    if (ra.P == 0) return cudaSuccess;
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kTileRows);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, split_reduce_kernel, ra);
}

}  // namespace tern
