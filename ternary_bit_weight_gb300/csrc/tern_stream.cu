// Streaming kernel of libtern for M <= 16 tokens:
//   Y[M,N] = X[M,K] . (s (.) T)^T
// with the 2-bit weights read once from HBM and decoded on chip.
//
// Method ("Ternary embedding model in vLLM", 2kiu.com/news/5082861, §4.2,
// §4.3): the weights stay packed in memory; signs are summed inside each
// 128-wide scale group and the FP16 scale is applied once per group.  The
// page's CUDA-core kernel is replaced by tensor cores fed from tensor
// memory:
//
//   * work unit = one 128-row x 128-weight block of the tiled layout (4 KB
//     of codes + 256 B of scales);
//   * one persistent CTA per SM; a producer warp fills a ring of shared-
//     memory stages with bulk copies (one unit per worker per stage);
//   * two decode workers (warpgroups; one thread per weight row = one
//     tensor-memory lane) turn each 16-weight code word into eight exact
//     bf16 pairs t in {-1,0,+1} (one LOP3 + one bf16x2 FMA per pair) and
//     store the unit's 64 columns of A with tcgen05.st into a 3-deep ring;
//   * an MMA warp issues eight tcgen05.mma (M = 128, N = 16, K = 16, bf16
//     -> fp32) per unit, A from tensor memory, B = X from shared memory,
//     into a per-unit accumulator ("D");
//   * promotion: the workers read the units' fp32 group partials with
//     tcgen05.ld one batch behind the decode and add s * partial to register
//     accumulators -- the FP16 scale is converted exactly to fp32 and never
//     rounded to bf16.
//
// M == 1 ("one"): the activation row (2K bytes) is copied once into shared
// memory and used as B in the no-swizzle layout: row 0 of every core matrix
// is the real row, rows 1..15 are whatever bytes follow it (they only feed
// accumulator columns 1..15, which nobody reads), and only column 0 of each
// unit's accumulator is promoted.
//
// M in 2..16: each stage also carries the unit's 16-row X tile, copied by
// TMA (128-byte swizzle, rows >= M zero-filled); accumulators are 16
// columns per unit, two units per promotion batch.
//
// Work split: worker v owns the contiguous unit range [U*v/V, U*(v+1)/V)
// in (row tile, group) order.  A tile whose groups span two or more
// workers is finished by the last of them to arrive (per 32-row quarter),
// which sums the partials in worker order (deterministic; no waiting on
// other CTAs).  Every mbarrier wait is bounded; on a timeout the kernel
// raises the workspace error word, drains its own copies and MMAs, frees
// its tensor memory and returns.

#include <cuda.h>

#include <mutex>

#include "tern_common.cuh"
#include "tern_internal.h"
#include "tern_sm100.cuh"

namespace tern {
namespace {

constexpr int kNW = 2;                          // decode workers per CTA
constexpr int kDecWarps = 4 * kNW;
constexpr int kProducerWarp = kDecWarps;
constexpr int kMmaWarp = kDecWarps + 1;
constexpr int kThreads = (kDecWarps + 2) * 32;
constexpr int kTmemCols = 512;
constexpr int kWorkerCols = kTmemCols / kNW;    // 256 columns per worker
constexpr int kAU = 3;                          // decoded-A ring depth (units)
constexpr int kACols = 64;                      // 128 bf16 per row = 64 columns
constexpr int kDCol0 = kAU * kACols;            // accumulators after the A ring
constexpr int kNtok = 16;                       // UMMA N
constexpr int kSmemLimit = 232448;              // 227 KB opt-in per CTA
constexpr int kCtrlBytes = 1024;
constexpr int kMaxStages = 48;

template <bool ONE>
struct SCfg {
    static constexpr int PB = 2;                        // units per promotion batch
    static constexpr int DS = 2 * PB;                   // 16-column accumulator slots in the ring
    static constexpr int LAGB = 2;                      // batches between reuses of a slot
    static constexpr int NCOL = ONE ? 1 : kNtok;        // token columns promoted per unit
    static constexpr int XUnit = ONE ? 0 : kNtok * kGroup * 2;   // one unit's X tile
    static constexpr int StageBytes =
        ONE ? kNW * kUnitBytes : static_cast<int>(round_up(kNW * (XUnit + kUnitBytes), 1024));
    static constexpr int OffCodes = kNW * XUnit;
    static constexpr int OffScales = OffCodes + kNW * kUnitCodeBytes;
};
static_assert(kNW == 2, "stage release count assumes two workers");
static_assert(kDCol0 + SCfg<true>::DS * kNtok <= kWorkerCols, "tensor-memory budget");

// control block offsets
constexpr int kBarAFull = 0;                                 // [kNW][kAU]
constexpr int kBarAEmpty = kBarAFull + 8 * kNW * kAU;        // [kNW][kAU]
constexpr int kBarDFull = kBarAEmpty + 8 * kNW * kAU;        // [kNW][4]
constexpr int kBarDEmpty = kBarDFull + 8 * kNW * 4;          // [kNW][4]
constexpr int kBarX = kBarDEmpty + 8 * kNW * 4;
constexpr int kBarDrain = kBarX + 8;
constexpr int kTmemPtr = kBarDrain + 8;
constexpr int kAbort = kTmemPtr + 4;
constexpr int kBarStages = 256;                              // full[S], empty[S]
static_assert(kAbort + 4 <= kBarStages, "control block");
static_assert(kBarStages + 16 * kMaxStages <= kCtrlBytes, "control block");

struct StreamArgs {
    const uint8_t* codes;
    const uint8_t* scales;
    const uint16_t* x;         // M == 1: the activation row
    int M;
    int G;                     // groups per row
    int stages;
    uint32_t x_bytes;          // M == 1: 2K
    uint32_t x_smem;           // shared memory reserved for X (multiple of 1024)
    int64_t N;
    int64_t R;
    int64_t U;
    int64_t V;
    OutputSplit out;
    int* err;                  // workspace error word
    int* counters;             // [R][4 row quarters]
    float* slots;              // [2V][NCOL][128]
};

__device__ __forceinline__ int64_t owner_worker(int64_t u, int64_t U, int64_t V) {
    return ((u + 1) * V - 1) / U;
}

// Finish tile b whose group partials this worker holds in acc (thread = row
// r of the tile, acc[m] = token m).  `whole`: this worker covered every
// group of the tile and owns the result.  Otherwise each warp publishes its
// 32 rows' partials in the worker's slot, and the last contributing worker
// to arrive for that row quarter sums all partials in worker order.
template <int NCOL>
__device__ __forceinline__ void flush_tile(const StreamArgs& a, int64_t v, int64_t b, int64_t first_tile,
                                           bool whole, float (&acc)[NCOL], int r) {
    const int lane = r & 31, quad = r >> 5;
    const int64_t row = b * kTileRows + r;
    const int mvalid = a.M < NCOL ? a.M : NCOL;
    if (whole) {
        if (row < a.N)
#pragma unroll
            for (int m = 0; m < NCOL; ++m)
                if (m < mvalid) store_y(a.out, m, row, acc[m]);
        return;
    }
    const int64_t slot = 2 * v + (b == first_tile ? 0 : 1);
    float* sp = a.slots + slot * (kTileRows * NCOL) + r;
#pragma unroll
    for (int m = 0; m < NCOL; ++m)
        if (m < mvalid) sp[m * kTileRows] = acc[m];
    __syncwarp();
    const int64_t t0 = b * a.G;
    const int64_t w_first = owner_worker(t0, a.U, a.V);
    const int64_t w_last = owner_worker(t0 + a.G - 1, a.U, a.V);
    int* counter = a.counters + b * 4 + quad;
    int last = 0;
    if (lane == 0) {
        __threadfence();   // publish the warp's slot writes (ordered by the warp barrier)
        last = atomicAdd(counter, 1) == static_cast<int>(w_last - w_first);
        if (last) __threadfence();
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __syncwarp();   // order the lanes' loads after lane 0's acquire
    // the first contributor's range starts before this tile (its partial is
    // its "last tile" slot) unless it starts exactly at the tile start
    const int first_side = (a.U * w_first < t0 * a.V) ? 1 : 0;
    float sum[NCOL];
#pragma unroll
    for (int m = 0; m < NCOL; ++m) sum[m] = 0.f;
    for (int64_t ww = w_first; ww <= w_last; ++ww) {
        const int64_t sl = 2 * ww + (ww == w_first ? first_side : 0);
        const float* src = a.slots + sl * (kTileRows * NCOL) + r;
#pragma unroll
        for (int m = 0; m < NCOL; ++m)
            if (m < mvalid) sum[m] += __ldcg(src + m * kTileRows);
    }
    if (row < a.N)
#pragma unroll
        for (int m = 0; m < NCOL; ++m)
            if (m < mvalid) store_y(a.out, m, row, sum[m]);
    if (lane == 0) *counter = 0;   // leave the workspace zeroed
}

// Warp-uniform bounded wait (every lane observes the barrier itself).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
    const bool got = mbar_wait(bar, parity, abort);
    return __all_sync(0xffffffffu, got);
}

template <bool ONE>
__global__ void __launch_bounds__(kThreads, 1)
stream_kernel(const __grid_constant__ CUtensorMap xmap, const StreamArgs a) {
    using C = SCfg<ONE>;
    constexpr int PB = C::PB;
    constexpr int NCOL = C::NCOL;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base (swizzle atoms)
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    uint8_t* ring_ptr = smem + a.x_smem;
    const uint32_t ring = sbase + a.x_smem;
    const int S = a.stages;
    uint8_t* ctrl = ring_ptr + S * C::StageBytes;
    const uint32_t cb = smem_u32(ctrl);
    const uint32_t bar_full = cb + kBarStages;
    const uint32_t bar_empty = bar_full + 8 * S;
    uint32_t* tmem_base_ptr = reinterpret_cast<uint32_t*>(ctrl + kTmemPtr);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + kAbort);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.G;

    // the workers of this CTA: contiguous unit ranges
    int64_t w_u0[kNW];
    int32_t w_n[kNW];
    int32_t max_n = 0;
#pragma unroll
    for (int w = 0; w < kNW; ++w) {
        const int64_t v = (int64_t)blockIdx.x * kNW + w;
        w_u0[w] = v < a.V ? a.U * v / a.V : 0;
        w_n[w] = v < a.V ? static_cast<int32_t>(a.U * (v + 1) / a.V - w_u0[w]) : 0;
        max_n = w_n[w] > max_n ? w_n[w] : max_n;
    }

    if (threadIdx.x == 0) {
        // a stage is released by the four warps of every worker with units
        // (plus the MMA commit when X travels in the stage)
        const int active = (w_n[0] > 0) + (w_n[1] > 0);
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 4 * active + (ONE ? 0 : 1));
        }
        for (int i = 0; i < kNW * kAU; ++i) {
            mbar_init(cb + kBarAFull + 8 * i, 4);
            mbar_init(cb + kBarAEmpty + 8 * i, 1);
        }
        for (int i = 0; i < kNW * 4; ++i) {
            mbar_init(cb + kBarDFull + 8 * i, 1);
            mbar_init(cb + kBarDEmpty + 8 * i, 4);
        }
        mbar_init(cb + kBarX, 1);
        mbar_init(cb + kBarDrain, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_base_ptr), kTmemCols);
        tmem_relinquish();
    }
    if (!ONE && warp == kProducerWarp && lane == 0) prefetch_tensormap(&xmap);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_base_ptr;
    grid_launch_dependents();

    if (warp == kProducerWarp) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            constexpr uint32_t kPerUnit = kUnitBytes + C::XUnit;
            int64_t uw[kNW];   // next unit whose weights are loaded
            int32_t gx[kNW];   // group of the next X tile
#pragma unroll
            for (int w = 0; w < kNW; ++w) {
                uw[w] = w_u0[w];
                gx[w] = static_cast<int32_t>(w_u0[w] % G);
            }
            auto load_weights = [&](int f, uint32_t st, uint32_t bar) {
                uint32_t bytes = 0;
#pragma unroll
                for (int w = 0; w < kNW; ++w) bytes += f < w_n[w] ? kPerUnit : 0u;
                mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
                for (int w = 0; w < kNW; ++w) {
                    if (f >= w_n[w]) continue;
                    bulk_load(st + C::OffCodes + w * kUnitCodeBytes, a.codes + uw[w] * kUnitCodeBytes,
                              kUnitCodeBytes, bar);
                    bulk_load(st + C::OffScales + w * kUnitScaleBytes, a.scales + uw[w] * kUnitScaleBytes,
                              kUnitScaleBytes, bar);
                    ++uw[w];
                }
            };
            // the weights of the first stages do not depend on earlier kernels
            const int32_t pre = max_n < S ? max_n : S;
            for (int32_t f = 0; f < pre; ++f) load_weights(f, ring + f * C::StageBytes, bar_full + 8 * f);
            grid_dependency_wait();
            if (ONE) {
                mbar_arrive_expect_tx(cb + kBarX, a.x_bytes);
                bulk_load(sbase, a.x, a.x_bytes, cb + kBarX);
            }
            int s = 0;
            uint32_t round = 0;   // completed passes over the ring
            for (int32_t f = 0; f < max_n; ++f) {
                const uint32_t st = ring + s * C::StageBytes;
                if (f >= pre) {
                    if (!mbar_wait(bar_empty + 8 * s, (round - 1) & 1u, abort_flag)) break;
                    load_weights(f, st, bar_full + 8 * s);
                }
                if (!ONE) {
#pragma unroll
                    for (int w = 0; w < kNW; ++w) {
                        if (f >= w_n[w]) continue;
                        const int32_t k0 = gx[w] * kGroup;
                        tma_load_2d(st + w * C::XUnit, &xmap, k0, 0, bar_full + 8 * s);
                        tma_load_2d(st + w * C::XUnit + kNtok * 128, &xmap, k0 + 64, 0, bar_full + 8 * s);
                        if (++gx[w] == G) gx[w] = 0;
                    }
                }
                if (++s == S) {
                    s = 0;
                    ++round;
                }
            }
            if (*abort_flag) {
                // drain the copies this CTA may still have in flight (bounded)
                volatile int no_abort = 0;
                for (int t = 0; t < S; ++t) {
                    (void)mbar_wait(bar_full + 8 * t, 0, &no_abort);
                    (void)mbar_wait(bar_full + 8 * t, 1, &no_abort);
                }
                (void)mbar_wait(cb + kBarX, 0, &no_abort);
            }
        }
    } else if (warp == kMmaWarp) {
        // --------------------------------------------------------------- MMA
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, kNtok);
            bool ok = true;
            if (ONE) ok = mbar_wait(cb + kBarX, 0, abort_flag);
            int32_t gm[kNW];   // group of the next unit (B address when M == 1)
#pragma unroll
            for (int w = 0; w < kNW; ++w) gm[w] = static_cast<int32_t>(w_u0[w] % G);
            int s = 0, aslot = 0;
            uint32_t full_ph = 0, around = 0;
            for (int32_t f = 0; f < max_n && ok; ++f) {
                const uint32_t st = ring + s * C::StageBytes;
                if (!ONE && !mbar_wait(bar_full + 8 * s, full_ph, abort_flag)) {
                    ok = false;
                    break;
                }
                const int i = f % PB, beta = f / PB;
#pragma unroll
                for (int w = 0; w < kNW; ++w) {
                    if (!ok || f >= w_n[w]) continue;
                    if (i == 0 && beta >= C::LAGB) {
                        const int bb = beta - C::LAGB;
                        if (!mbar_wait(cb + kBarDEmpty + 8 * (w * 4 + (bb & 3)), (bb >> 2) & 1, abort_flag)) {
                            ok = false;
                            continue;
                        }
                    }
                    if (!mbar_wait(cb + kBarAFull + 8 * (w * kAU + aslot), around, abort_flag)) {
                        ok = false;
                        continue;
                    }
                    tc_fence_after_sync();
                    const uint32_t a_tm = tmem + w * kWorkerCols + aslot * kACols;
                    const uint32_t d_tm = tmem + w * kWorkerCols + kDCol0 + kNtok * (f & (C::DS - 1));
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        uint64_t bdesc;
                        if (ONE)
                            bdesc = smem_desc_kmajor_noswz(sbase + 2u * (uint32_t)(kGroup * gm[w] + 16 * kk), 16, 16);
                        else   // +32 bytes per K-step = +2 in the address field
                            bdesc = smem_desc_kmajor_sw128(st + w * C::XUnit + (kk >> 2) * (kNtok * 128)) + 2 * (kk & 3);
                        umma_bf16_tmem_a(d_tm, a_tm + 8 * kk, bdesc, idesc, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(cb + kBarAEmpty + 8 * (w * kAU + aslot));
                    if (i == PB - 1 || f == w_n[w] - 1) umma_commit(cb + kBarDFull + 8 * (w * 4 + (beta & 3)));
                    if (++gm[w] == G) gm[w] = 0;
                }
                if (!ONE && ok) umma_commit(bar_empty + 8 * s);
                if (++aslot == kAU) {
                    aslot = 0;
                    around ^= 1u;
                }
                if (++s == S) {
                    s = 0;
                    full_ph ^= 1u;
                }
            }
            // every MMA issued has completed before tensor memory is freed
            umma_commit(cb + kBarDrain);
            volatile int no_abort = 0;
            (void)mbar_wait(cb + kBarDrain, 0, &no_abort);
        }
    } else {
        // ---------------------------------------------------- decode workers
        const int wg = warp >> 2;
        const int r = threadIdx.x & 127;   // weight row in the tile = tensor-memory lane
        const int64_t v = (int64_t)blockIdx.x * kNW + wg;
        const int32_t n = w_n[wg == 0 ? 0 : 1];
        const int64_t u0 = w_u0[wg == 0 ? 0 : 1];
        const uint32_t tm = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + wg * kWorkerCols;
        const uint32_t bar_afull = cb + kBarAFull + 8 * kAU * wg;
        const uint32_t bar_aempty = cb + kBarAEmpty + 8 * kAU * wg;
        const uint32_t bar_dfull = cb + kBarDFull + 8 * 4 * wg;
        const uint32_t bar_dempty = cb + kBarDEmpty + 8 * 4 * wg;
        if (n > 0) {
            const int codes_off = C::OffCodes + wg * kUnitCodeBytes + 16 * r;
            const int scale_off = C::OffScales + wg * kUnitScaleBytes + 2 * r;
            // promotion cursor (tile, group) of the next unit to promote
            const int64_t first_tile = u0 / G;
            const int32_t first_g = static_cast<int32_t>(u0 - first_tile * G);
            int64_t pb = first_tile;
            int32_t pg = first_g;
            float acc[NCOL];
#pragma unroll
            for (int m = 0; m < NCOL; ++m) acc[m] = 0.f;
            float s_cur[PB], s_prev[PB];
#pragma unroll
            for (int i = 0; i < PB; ++i) s_cur[i] = s_prev[i] = 0.f;
            bool ok = true, waited = false;
            int s = 0, aslot = 0;
            uint32_t full_ph = 0, around = 0;

            // acc += s * partial for the units of batch b, finishing tiles
            auto promote = [&](int32_t b) {
                if (!waited) {
                    grid_dependency_wait();   // outputs and workspace belong to earlier kernels until now
                    waited = true;
                }
                if (!warp_wait(bar_dfull + 8 * (b & 3), (b >> 2) & 1, abort_flag)) {
                    ok = false;
                    return;
                }
                tc_fence_after_sync();
                const int32_t cnt = (n - b * PB) < PB ? (n - b * PB) : PB;
                uint32_t d[PB * NCOL];
#pragma unroll
                for (int i = 0; i < PB; ++i) {
                    const uint32_t col = tm + kDCol0 + kNtok * ((b * PB + i) & (C::DS - 1));
                    // straight into d: the registers are valid only after the wait
                    if (ONE)
                        tmem_ld_32x32b_x1(col, d[i]);
                    else
                        tmem_ld_32x32b_x16(col, *reinterpret_cast<uint32_t(*)[16]>(d + i * NCOL));
                }
                tmem_ld_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_dempty + 8 * (b & 3));
#pragma unroll
                for (int i = 0; i < PB; ++i) {
                    if (i >= cnt) continue;
#pragma unroll
                    for (int m = 0; m < NCOL; ++m) acc[m] = fmaf(s_prev[i], __uint_as_float(d[i * NCOL + m]), acc[m]);
                    const int32_t u = b * PB + i;
                    if (pg == G - 1 || u == n - 1) {
                        const bool whole = (pb != first_tile || first_g == 0) && pg == G - 1;
                        flush_tile<NCOL>(a, v, pb, first_tile, whole, acc, r);
#pragma unroll
                        for (int m = 0; m < NCOL; ++m) acc[m] = 0.f;
                    }
                    if (++pg == G) {
                        pg = 0;
                        ++pb;
                    }
                }
            };

            int32_t beta = 0;
            for (; beta * PB < n && ok; ++beta) {
#pragma unroll
                for (int i = 0; i < PB; ++i) {
                    const int32_t j = beta * PB + i;
                    if (j >= n || !ok) continue;
                    // ---- unit j: codes and scale from the stage, then release it
                    if (!warp_wait(bar_full + 8 * s, full_ph, abort_flag)) {
                        ok = false;
                        continue;
                    }
                    const uint8_t* stp = ring_ptr + s * C::StageBytes;
                    const uint4 c0 = lds_v4(stp + codes_off);
                    const uint4 c1 = lds_v4(stp + codes_off + 2048);
                    const uint32_t sc = *reinterpret_cast<const uint16_t*>(stp + scale_off);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_empty + 8 * s);
                    if (++s == S) {
                        s = 0;
                        full_ph ^= 1u;
                    }
                    // ---- decode into the A ring slot
                    if (j >= kAU) {
                        if (!warp_wait(bar_aempty + 8 * aslot, around ^ 1u, abort_flag)) {
                            ok = false;
                            continue;
                        }
                        tc_fence_after_sync();
                    }
                    const uint32_t a_tm = tm + aslot * kACols;
                    {
                        uint32_t p[32];
                        decode_word_bf16(c0.x, p);
                        decode_word_bf16(c0.y, p + 8);
                        decode_word_bf16(c0.z, p + 16);
                        decode_word_bf16(c0.w, p + 24);
                        tmem_st_32x32b_x32(a_tm, p);
                    }
                    {
                        uint32_t p[32];
                        decode_word_bf16(c1.x, p);
                        decode_word_bf16(c1.y, p + 8);
                        decode_word_bf16(c1.z, p + 16);
                        decode_word_bf16(c1.w, p + 24);
                        tmem_st_32x32b_x32(a_tm + 32, p);
                    }
                    tmem_st_wait();
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_afull + 8 * aslot);
                    if (++aslot == kAU) {
                        aslot = 0;
                        around ^= 1u;
                    }
                    s_cur[i] = fp16_bits_to_float(sc);
                }
                if (ok && beta >= 1) promote(beta - 1);
#pragma unroll
                for (int i = 0; i < PB; ++i) s_prev[i] = s_cur[i];
            }
            if (ok && beta >= 1) promote(beta - 1);
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before_sync();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) atomicOr(a.err, 1);
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
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

template <bool ONE>
cudaError_t set_smem_limit() {
    static cudaError_t status = cudaErrorUnknown;
    static std::once_flag once;
    std::call_once(once, [] {
        status = cudaFuncSetAttribute(stream_kernel<ONE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    });
    return status;
}

template <bool ONE>
cudaError_t launch_one(const uint16_t* X, int64_t ldx, const StreamArgs& a, const StreamPlan& plan,
                       cudaStream_t stream) {
    CUtensorMap map;
    memset(&map, 0, sizeof(map));
    if (!ONE) {
        EncodeTiledFn enc = encode_tiled_fn();
        if (enc == nullptr) return cudaErrorNotSupported;
        const int64_t K = (int64_t)a.G * kGroup;
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(a.M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldx) * 2};
        const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kNtok)};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(X), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    cudaError_t e = set_smem_limit<ONE>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, stream_kernel<ONE>, map, a);
}

}  // namespace

StreamPlan plan_stream(int64_t M, int64_t N, int64_t K, int sm_count) {
    StreamPlan p = {};
    if (sm_count <= 0) sm_count = 152;
    p.R = ceil_div(N, kTileRows);
    p.G = K / kGroup;
    p.U = p.R * p.G;
    int64_t workers = (int64_t)sm_count * kNW;
    if (workers > p.U) workers = p.U;
    p.V = workers;
    p.grid = ceil_div(workers, kNW);
    // M == 1 keeps the activation row in shared memory when at least four
    // stages still fit beside it
    const int64_t x_smem = round_up(2 * K + 256, 1024);
    const int64_t avail_one = kSmemLimit - 1024 - kCtrlBytes - x_smem;
    p.one = (M == 1) && avail_one >= 4 * SCfg<true>::StageBytes;
    const int64_t stage_bytes = p.one ? SCfg<true>::StageBytes : SCfg<false>::StageBytes;
    const int64_t avail = p.one ? avail_one : kSmemLimit - 1024 - kCtrlBytes;
    int64_t stages = avail / stage_bytes;
    if (stages > kMaxStages) stages = kMaxStages;
    p.stages = static_cast<int>(stages);
    p.smem = static_cast<size_t>(1024 + (p.one ? x_smem : 0) + stages * stage_bytes + kCtrlBytes);
    const int64_t ncol = p.one ? SCfg<true>::NCOL : SCfg<false>::NCOL;
    const size_t counters = static_cast<size_t>(round_up(p.R * 4 * 4, 256));
    p.ws_bytes = kWorkspaceErrBytes + counters + static_cast<size_t>(2 * p.V * kTileRows * ncol) * sizeof(float);
    return p;
}

cudaError_t launch_stream(const uint16_t* X, int64_t ldx, const uint8_t* tiled, int64_t M, int64_t N,
                          int64_t K, const OutputSplit& out, void* ws, const StreamPlan& plan,
                          cudaStream_t stream) {
    StreamArgs a = {};
    a.codes = tiled;
    a.scales = tiled + plan.U * kUnitCodeBytes;
    a.x = X;
    a.M = static_cast<int>(M);
    a.G = static_cast<int>(plan.G);
    a.stages = plan.stages;
    a.x_bytes = static_cast<uint32_t>(2 * K);
    a.x_smem = plan.one ? static_cast<uint32_t>(round_up(2 * K + 256, 1024)) : 0u;
    a.N = N;
    a.R = plan.R;
    a.U = plan.U;
    a.V = plan.V;
    a.out = out;
    uint8_t* w = static_cast<uint8_t*>(ws);
    a.err = reinterpret_cast<int*>(w);
    a.counters = reinterpret_cast<int*>(w + kWorkspaceErrBytes);
    a.slots = reinterpret_cast<float*>(w + kWorkspaceErrBytes + static_cast<size_t>(round_up(plan.R * 4 * 4, 256)));
    return plan.one ? launch_one<true>(X, ldx, a, plan, stream) : launch_one<false>(X, ldx, a, plan, stream);
}

}  // namespace tern
