// Streaming kernel of libtern for M <= 16 tokens:
//   Y[M,N] = X[M,K] . (s (.) T)^T
// with the 2-bit weights read once from HBM and decoded on chip.
//
// Method ("Ternary embedding model in vLLM", 2kiu.com/news/5082861, §4.2,
// §4.3): the weights stay packed in memory; signs are summed inside each
// 128-wide scale group and the FP16 scale is applied once per group.  The
// page's CUDA-core kernel is replaced by tensor cores fed from tensor
// memory.  One persistent CTA per SM owns a contiguous range of work units
// (one unit = one 128-row x 128-weight block of the tiled layout: 4 KB of
// codes + 256 B of scales) and runs a pipeline of warp roles:
//
//   * producer warp: a ring of shared-memory stages of 8 consecutive units,
//     filled with two bulk copies per stage (codes, scales) -- few large
//     copies, since a CTA's copy ring completes only a few copies per
//     microsecond whatever their size;
//   * two decode streams (even units / odd units), one warpgroup each (one
//     thread per weight row = one tensor-memory lane): each 16-weight code
//     word becomes eight exact bf16 pairs t in {-1,0,+1} (one LOP3 + one
//     bf16x2 FMA per pair, balanced between the integer and FMA pipes)
//     stored with tcgen05.st (two stores of 32 columns, the first running
//     while the second half decodes) into the stream's 3-unit ring of A
//     operands;
//   * three MMA warps taking units in turn: eight tcgen05.mma (M = 128,
//     N = 16, K = 16, bf16 -> fp32) per unit, A from tensor memory, B = X
//     from shared memory, into one of 8 accumulator slots; the whole warp runs
//     the loop and one elected lane issues (warp-uniform descriptors issue
//     far faster than a loop inside a single-lane branch);
//   * promotion warpgroup: reads each unit's fp32 group partial with
//     tcgen05.ld and adds s * partial to register accumulators -- the FP16
//     scale is converted exactly to fp32 and never rounded to bf16 -- and
//     finishes tiles.
// Every hand-off is an mbarrier per unit (A operands) or per pair of units
// (accumulators), so no role waits for a batch of another's work.
//
// M == 1: the activation row of every problem the CTA's units belong to
// (2K bytes each) is copied once into shared memory and used as B in the
// no-swizzle layout: row 0 of every core matrix is the real row, rows
// 1..15 are whatever bytes follow it (they only feed accumulator columns
// 1..15, which nobody reads), and only column 0 of each unit's accumulator
// is promoted.
// M in 2..16: each stage also carries its units' 16-row X tiles, copied by
// TMA (128-byte swizzle, rows >= M zero-filled).
//
// One launch may serve a group of independent linears (the same M, each
// with its own X, weights and outputs): their units are concatenated, each
// problem's in (row tile, group) order, and the CTAs split the whole
// sequence, so the fixed costs of a launch (start-up, pipeline fill, the
// last tiles' reductions) are paid once for the group.
//
// Work split: CTA v owns the contiguous unit range [U*v/V, U*(v+1)/V) of the
// sequence.  A tile whose groups span two or more CTAs is finished by the
// last of them to arrive (per 32-row quarter), which sums the partials in
// CTA order (deterministic; no waiting on other CTAs).
// Every mbarrier wait is bounded; on a timeout the kernel raises the
// workspace error word, drains its own copies and MMAs, frees its tensor
// memory and returns.

#include <cuda.h>

#include <mutex>

#include "tern_common.cuh"
#include "tern_internal.h"
#include "tern_sm100.cuh"

namespace tern {
namespace {

// warp roles
// The MMA warps come first: a warp scheduler that has to choose among ready
// warps favours the older (lower) ones, and the decode warps, always ready
// with long runs of independent integer and FMA work, would otherwise hold
// the issue slots of their sub-partition for hundreds of cycles at a time.
// Warp w reaches tensor-memory lanes 32 (w mod 4) .. +31, so each
// warpgroup of decode or promotion warps starts at a multiple of 4.
// MMA warp m (warps 0, 1 and 3) issues units m, m+3, ...: a warp's MMA
// issue is slow next to busy decoders, so it is spread over three warps.
constexpr int kMaxMmaWarps = 3;
constexpr int kProducerWarp = 2;
constexpr int kAllocWarp = 0;
constexpr int kDecWarp0 = 4;
constexpr int kDecWarps = 8;                    // 2 streams x 1 warpgroup (whole units)
constexpr int kPromWarp0 = kDecWarp0 + kDecWarps;   // 4 warps
constexpr int kThreads = (kPromWarp0 + 4) * 32;
__device__ __forceinline__ int mma_index(int warp) { return warp < 2 ? warp : warp == 3 ? 2 : -1; }
// tensor memory: each decode stream has its own A ring; accumulators come
// in pairs of 16-column slots (one even unit, one odd unit)
constexpr int kTmemCols = 512;
constexpr int kAQ = 3;                          // A ring per stream (units)
constexpr int kACols = 64;                      // 128 bf16 per row = 64 columns per unit
constexpr int kDCol0 = 2 * kAQ * kACols;        // accumulators after the A rings
constexpr int kNtok = 16;                       // UMMA N
constexpr int kDP = 4;                          // accumulator ring: pairs of 16-column slots
static_assert(kDCol0 + 2 * kDP * kNtok <= kTmemCols, "tensor-memory budget");
// shared memory
constexpr int kPS = 8;                          // units per stage
constexpr int kSmemLimit = 232448;              // 227 KB opt-in per CTA
constexpr int kCtrlBytes = 1024;
constexpr int kMaxStages = 48;

template <bool ONE>
struct SCfg {
    static constexpr int MmaWarps = 3;
    static constexpr int NCOL = ONE ? 1 : kNtok;        // token columns promoted per unit
    static constexpr int XUnit = ONE ? 0 : kNtok * kGroup * 2;   // one unit's X tile
    static constexpr int OffCodes = kPS * XUnit;         // X tiles first (1024-byte aligned)
    static constexpr int OffScales = OffCodes + kPS * kUnitCodeBytes;
    static constexpr int StageBytes = static_cast<int>(round_up(OffScales + kPS * kUnitScaleBytes, ONE ? 16 : 1024));
    // a stage is released by every decode warp, the promotion warps (they
    // read the scales) and, when X travels in the stage, every MMA warp
    static constexpr int EmptyCount = kDecWarps + 4 + (ONE ? 0 : MmaWarps);
};

// control block offsets
constexpr int kBarAFull = 0;                                 // [2][kAQ]
constexpr int kBarAEmpty = kBarAFull + 8 * 2 * kAQ;          // [2][kAQ]
constexpr int kBarDFull = kBarAEmpty + 8 * 2 * kAQ;          // [kDP]
constexpr int kBarDEmpty = kBarDFull + 8 * kDP;              // [kDP]
constexpr int kBarX = kBarDEmpty + 8 * kDP;                  // [kMaxGroup] activation rows copied (M == 1)
constexpr int kBarDrain = kBarX + 8 * kMaxGroup;             // [kMaxMmaWarps]
constexpr int kTmemPtr = kBarDrain + 8 * kMaxMmaWarps;
constexpr int kAbort = kTmemPtr + 4;
constexpr int kBarStages = 256;                              // full[S], empty[S]
static_assert(kAbort + 4 <= kBarStages, "control block");
static_assert(kBarStages + 16 * kMaxStages <= kCtrlBytes, "control block");
static_assert(kPS >= kMaxMmaWarps, "with activation tiles in the stages, every MMA warp has units in every full stage");
// A slot of stream q is used by units j, j + 2 kAQ, ...: the same MMA warp
// must issue all of them, or a warp could test the slot's barrier two
// phases ahead of its decoder and take the older phase (same parity) as the
// one it waits for.  (The accumulator pairs need no such rule: before a
// warp reaches pair k + 2 kDP it has waited for a pair after k.)
static_assert((2 * kAQ) % kMaxMmaWarps == 0, "A ring depth and MMA warp count");

// M == 1: shared memory for a problem's activation row (2K bytes) and 256
// bytes the tensor cores may read past its end.  The rows of the problems a
// CTA's units belong to lie one after another before the stages.
__host__ __device__ constexpr int64_t x_smem_bytes(int64_t K) { return round_up(2 * K + 256, 1024); }

// One linear of the launch's group.
struct StreamProb {
    const uint8_t* codes;      // its units' codes (tiled layout)
    const uint8_t* scales;     // per unit: 128 FP16 scales, or (s8) 128 int8 scales
    const uint16_t* x;         // M == 1: the activation row
    int64_t u_begin;           // its first unit in the launch's unit sequence
    int64_t tile0;             // its first tile in the launch's tile counters
    int64_t N;
    int32_t R;                 // 128-row tiles
    int32_t G;                 // groups per row
    OutputSplit out;
};

struct StreamArgs {
    const float* row_factor;   // s8: per row, the factor of its int8 scales ([R * 128])
    int s8;                    // (s8 and zflags: single-problem launches only)
    int scale_unit;            // bytes of one unit's scales: 256, or 128 (s8)
    const uint8_t* zflags;     // optional, per unit: 1 = every weight of the unit is 0 (skipped)
    int M;
    int P;                     // problems in the group
    int stages;
    uint32_t x_smem;           // M == 1: shared memory before the stages for the CTA's activation rows
    int64_t U;                 // units of all problems
    int64_t V;                 // workers = CTAs
    int* err;                  // workspace error word
    int* counters;             // [tiles of all problems][4 row quarters]
    float* slots;              // [2V][NCOL][128]
    StreamProb prob[kMaxGroup];
};

// Tensor maps of the problems' activations (M > 1).
struct XMaps {
    CUtensorMap map[kMaxGroup];
};

// Problem that holds unit u of the sequence (problems in order, P small).
__device__ __forceinline__ int problem_of(const StreamArgs& a, int64_t u) {
    int p = 0;
    while (p + 1 < a.P && u >= a.prob[p + 1].u_begin) ++p;
    return p;
}

__device__ __forceinline__ int64_t owner_worker(int64_t u, int64_t U, int64_t V) {
    return ((u + 1) * V - 1) / U;
}

// Finish tile b whose group partials this CTA holds in acc (thread = row r
// of the tile, acc[m] = token m).  `whole`: this CTA covered every group of
// the tile and owns the result.  Otherwise each warp publishes its 32 rows'
// partials in the CTA's slot, and the last contributing CTA to arrive for
// that row quarter sums all partials in CTA order.
template <int NCOL>
__device__ __forceinline__ void flush_tile(const StreamArgs& a, int64_t v, int p, int64_t b, bool first,
                                           bool whole, float (&acc)[NCOL], int r, bool s8, float row_f) {
    const StreamProb& pr = a.prob[p];
    const int lane = r & 31, quad = r >> 5;
    const int64_t row = b * kTileRows + r;
    const int mvalid = a.M < NCOL ? a.M : NCOL;
    if (s8) {
        // int8 scales: the group sums were weighted by q; the row's factor
        // (row_f, loaded when the tile began) once
#pragma unroll
        for (int m = 0; m < NCOL; ++m) acc[m] *= row_f;
    }
    const bool live = row < pr.N;
    const RowOut o = row_out(pr.out, live ? row : 0);
    if (whole) {
#pragma unroll
        for (int m = 0; m < NCOL; ++m)
            if (m < mvalid) store_out(pr.out, o, m, row, acc[m], live);
        return;
    }
    const int64_t slot = 2 * v + (first ? 0 : 1);
    float* sp = a.slots + slot * (kTileRows * NCOL) + r;
#pragma unroll
    for (int m = 0; m < NCOL; ++m)
        if (m < mvalid) sp[m * kTileRows] = acc[m];
    __syncwarp();
    const int64_t t0 = pr.u_begin + b * pr.G;   // the tile's first unit in the sequence
    const int64_t w_first = owner_worker(t0, a.U, a.V);
    const int64_t w_last = owner_worker(t0 + pr.G - 1, a.U, a.V);
    int* counter = a.counters + (pr.tile0 + b) * 4 + quad;
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
#pragma unroll
    for (int m = 0; m < NCOL; ++m)
        if (m < mvalid) store_out(pr.out, o, m, row, sum[m], live);
    if (lane == 0) *counter = 0;   // leave the workspace zeroed
}

// Warp-uniform bounded wait (every lane observes the barrier itself).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
    const bool got = mbar_wait(bar, parity, abort);
    return __all_sync(0xffffffffu, got);
}

// Each lane with `active` set waits for its own barrier; the warp goes on
// when all have completed.  The common case costs one test and one vote:
// while an MMA warp waits, its share of the tensor pipe stands idle.
__device__ __forceinline__ bool vote_wait(uint32_t bar, uint32_t parity, bool active, volatile int* abort) {
    if (__all_sync(0xffffffffu, !active || mbar_test_wait(bar, parity))) return true;
    const bool got = !active || mbar_wait(bar, parity, abort);
    return __all_sync(0xffffffffu, got);
}

// EXT: 0 plain weights; 1 int8 scales (a.s8); 2 zero-unit flags
// (a.zflags).  Each form is its own instantiation, so that the scale width
// and the flag checks are compile-time on the hot paths.
template <bool ONE, bool XF16, int EXT>
__global__ void __launch_bounds__(kThreads, 1)
stream_kernel(const __grid_constant__ XMaps xmaps, const StreamArgs a) {
    using C = SCfg<ONE>;
    constexpr bool s8 = EXT == 1;
    const uint8_t* const zflags = EXT == 2 ? a.zflags : nullptr;
    constexpr int scale_unit = s8 ? kUnitScaleBytesS8 : kUnitScaleBytes;
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

    // this CTA's worker: a contiguous unit range
    const int64_t v = blockIdx.x;
    const int64_t u0 = a.U * v / a.V;
    const int32_t n = static_cast<int32_t>(a.U * (v + 1) / a.V - u0);
    const int32_t nst = (n + kPS - 1) / kPS;   // stages of this worker

    // the producer's lane 0 starts the weight copies of the first stages at
    // once (they do not depend on earlier kernels): their memory latency then
    // overlaps the rest of the setup
    auto load_weights = [&](int32_t f, uint32_t st, uint32_t bar) {
        const int64_t uf = u0 + (int64_t)f * kPS;
        const int32_t cnt = n - f * kPS < kPS ? n - f * kPS : kPS;
        if (zflags == nullptr) {
            mbar_arrive_expect_tx(bar, cnt * (kUnitCodeBytes + scale_unit + C::XUnit));
            // one pair of copies per problem the stage's units belong to
            int p = problem_of(a, uf);
            for (int32_t i = 0; i < cnt; ++p) {
                const StreamProb& pr = a.prob[p];
                const int64_t l = uf + i - pr.u_begin;
                const int64_t left = (int64_t)pr.R * pr.G - l;
                const int32_t run = cnt - i < left ? cnt - i : static_cast<int32_t>(left);
                bulk_load(st + C::OffCodes + i * kUnitCodeBytes, pr.codes + l * kUnitCodeBytes, run * kUnitCodeBytes,
                          bar);
                bulk_load(st + C::OffScales + i * scale_unit, pr.scales + l * scale_unit, run * scale_unit, bar);
                i += run;
            }
        } else {
            // (single problem)
            // one pair of copies from the stage's first to its last non-zero
            // unit (zero units between them come along): a CTA's copy engine
            // completes few copies per microsecond, so a copy per run of
            // non-zero units would cost more than the bytes it saves
            uint32_t live = 0;
            for (int32_t i = 0; i < cnt; ++i) live |= (__ldg(zflags + uf + i) ? 0u : 1u) << i;
            if (live == 0) {
                mbar_arrive_expect_tx(bar, cnt * C::XUnit);
            } else {
                const int32_t i0 = __ffs(live) - 1, i1 = 32 - __clz(live);   // [i0, i1)
                mbar_arrive_expect_tx(bar, (i1 - i0) * (kUnitCodeBytes + scale_unit) + cnt * C::XUnit);
                bulk_load(st + C::OffCodes + i0 * kUnitCodeBytes, a.prob[0].codes + (uf + i0) * kUnitCodeBytes,
                          (i1 - i0) * kUnitCodeBytes, bar);
                bulk_load(st + C::OffScales + i0 * scale_unit, a.prob[0].scales + (uf + i0) * scale_unit,
                          (i1 - i0) * scale_unit, bar);
            }
        }
    };
    const int32_t pre = nst < S ? nst : S;
    if (threadIdx.x == kProducerWarp * 32) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, C::EmptyCount);
        }
        mbar_fence_init();
        fence_proxy_async_smem();   // the copies below complete on these barriers
        for (int32_t f = 0; f < pre; ++f) load_weights(f, ring + f * C::StageBytes, bar_full + 8 * f);
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2 * kAQ; ++i) {
            mbar_init(cb + kBarAFull + 8 * i, kDecWarps / 2);   // the stream's 4 warps
            mbar_init(cb + kBarAEmpty + 8 * i, 1);
        }
        for (int i = 0; i < kDP; ++i) {
            mbar_init(cb + kBarDFull + 8 * i, 2);                // both MMA warps
            mbar_init(cb + kBarDEmpty + 8 * i, 4);               // the promotion warps
        }
        for (int i = 0; i < kMaxGroup; ++i) mbar_init(cb + kBarX + 8 * i, 1);
        for (int i = 0; i < kMaxMmaWarps; ++i) mbar_init(cb + kBarDrain + 8 * i, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == kAllocWarp) {
        tmem_alloc(smem_u32(tmem_base_ptr), kTmemCols);
        tmem_relinquish();
    }
    if (!ONE && warp == kProducerWarp && lane < a.P) prefetch_tensormap(&xmaps.map[lane]);
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_base_ptr;
    grid_launch_dependents();

    if (warp == kProducerWarp) {
        // ---------------------------------------------------------- producer
        // the whole warp runs the loop; lane 0 issues the copies
        grid_dependency_wait();
        if (ONE && n > 0) {
            // the activation rows of the problems this CTA's units belong to
            const int pf = problem_of(a, u0), pl = problem_of(a, u0 + n - 1);
            uint32_t off = 0;
            for (int p = pf; p <= pl; ++p) {
                const uint32_t bytes = static_cast<uint32_t>(a.prob[p].G) * kGroup * 2;
                if (lane == 0) {
                    mbar_arrive_expect_tx(cb + kBarX + 8 * (p - pf), bytes);
                    bulk_load(sbase + off, a.prob[p].x, bytes, cb + kBarX + 8 * (p - pf));
                }
                off += static_cast<uint32_t>(x_smem_bytes((int64_t)a.prob[p].G * kGroup));
            }
            __syncwarp();
        }
        // problem and group of the next unit whose activation tile is copied (M > 1)
        int px = problem_of(a, u0);
        int32_t gx = static_cast<int32_t>((u0 - a.prob[px].u_begin) % a.prob[px].G);
        int32_t bx = static_cast<int32_t>((u0 - a.prob[px].u_begin) / a.prob[px].G);
        int s = 0;
        uint32_t round = 0;   // completed passes over the ring
        for (int32_t f = 0; f < nst; ++f) {
            const uint32_t st = ring + s * C::StageBytes;
            if (f >= pre) {
                if (!warp_wait(bar_empty + 8 * s, (round - 1) & 1u, abort_flag)) break;
                if (lane == 0) load_weights(f, st, bar_full + 8 * s);
                __syncwarp();
            }
            if (!ONE) {
                const int32_t cnt = n - f * kPS < kPS ? n - f * kPS : kPS;
                for (int32_t i = 0; i < cnt; ++i) {
                    const StreamProb& pr = a.prob[px];
                    if (lane == 0) {
                        tma_load_2d(st + i * C::XUnit, &xmaps.map[px], gx * kGroup, 0, bar_full + 8 * s);
                        tma_load_2d(st + i * C::XUnit + kNtok * 128, &xmaps.map[px], gx * kGroup + 64, 0,
                                    bar_full + 8 * s);
                    }
                    __syncwarp();
                    if (++gx == pr.G) {
                        gx = 0;
                        if (++bx == pr.R) {
                            bx = 0;
                            ++px;
                        }
                    }
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
            if (ONE && n > 0)
                for (int p = problem_of(a, u0); p <= problem_of(a, u0 + n - 1); ++p)
                    (void)mbar_wait(cb + kBarX + 8 * (p - problem_of(a, u0)), 0, &no_abort);
        }
    } else if (mma_index(warp) >= 0 && mma_index(warp) < C::MmaWarps) {
        // --------------------------------------------------------------- MMA
        // MMA warp m issues units j = m, m + 3, ... (stream j mod 2, that
        // stream's unit j / 2).  The whole warp runs the loop with
        // warp-uniform descriptors; one elected lane issues the MMAs and
        // commits.  Each unit's eight MMAs start its own accumulator, so the
        // order between MMA warps does not matter.
        const int m = mma_index(warp);
        constexpr int kMmaWarps = C::MmaWarps;
        constexpr uint32_t idesc = XF16 ? idesc_fp16_f32(128, kNtok) : idesc_bf16_f32(128, kNtok);
        bool ok = true;
        // B descriptors: M == 1 the problem's resident row (+16 per group,
        // +2 per K-step); else the unit's X tile in the stage
        const uint64_t bdesc_x = smem_desc_kmajor_noswz(sbase, 16, 16);
        const uint64_t bdesc_ring = smem_desc_kmajor_sw128(ring);
        // M == 1: one problem at a time, its row offset and group count
        // fixed over the inner loop (B comes from the stage otherwise)
        const int pf = problem_of(a, u0);
        const int pl = ONE && n > 0 ? problem_of(a, u0 + n - 1) : pf;
        uint32_t xoff = 0;
        // stage of unit j (M > 1): tracked, not divided
        int us = m, s = 0;
        uint32_t full_ph = 0;
        int32_t j = m;
        for (int p = pf; p <= pl && ok; ++p) {
            const int32_t G = a.prob[p].G;
            const int64_t pend = a.prob[p].u_begin + (int64_t)a.prob[p].R * G - u0;   // the problem's end in this CTA
            const int32_t jend = p == pl ? n : static_cast<int32_t>(pend < n ? pend : n);
            int32_t g = static_cast<int32_t>((u0 + j - a.prob[p].u_begin) % G);   // group of unit j
            const uint64_t bdesc_p = bdesc_x + (xoff >> 4);
            bool first = true;   // this warp's first unit of the problem: wait for its row
            for (; j < jend && ok; j += kMmaWarps) {
                const int q = j & 1;                 // decode stream
                const int32_t k = j >> 1;            // pair = the stream's unit index
                const int al = k % kAQ, dp = k % kDP;
                const uint32_t a_ph = (k / kAQ) & 1u, d_ph = (k / kDP) & 1u;
                // one vote: D pair free (lane 1), stage full (lane 2), A slot
                // full (lane 3), the problem's activation row copied (lane 4)
                uint32_t bar = 0, par = 0;
                bool act = false;
                if (lane == 1) {
                    act = k >= kDP;
                    bar = cb + kBarDEmpty + 8 * dp;
                    par = d_ph ^ 1u;
                } else if (lane == 2) {
                    act = !ONE && us < kMmaWarps;
                    bar = bar_full + 8 * s;
                    par = full_ph;
                } else if (lane == 3) {
                    act = true;
                    bar = cb + kBarAFull + 8 * (kAQ * q + al);
                    par = a_ph;
                } else if (lane == 4) {
                    act = ONE && first;
                    bar = cb + kBarX + 8 * (p - pf);
                    par = 0;
                }
                if (!(ok = vote_wait(bar, par, act, abort_flag))) break;
                tc_fence_after_sync();
                const uint32_t a_tm = tmem + (q * kAQ + al) * kACols;
                const uint32_t d_tm = tmem + kDCol0 + (2 * dp + q) * kNtok;
                first = false;
                const uint64_t b0 = ONE ? bdesc_p + 16u * (uint32_t)g
                                        : bdesc_ring + ((uint32_t)(s * C::StageBytes + us * C::XUnit) >> 4);
                const bool zero = zflags != nullptr && __ldg(zflags + u0 + j) != 0;
                if (elect_one()) {
                    if (!zero) {
    #pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            // M == 1: +32 bytes per K-step; else +32 bytes within a
                            // 64-wide box and +2048 bytes to the second box
                            const uint32_t step = ONE ? 2 * kk : (kk >> 2) * (kNtok * 128 / 16) + 2 * (kk & 3);
                            umma_bf16_tmem_a(d_tm, a_tm + 8 * kk, b0 + step, idesc, kk > 0 ? 1u : 0u);
                        }
                    }
                    umma_commit(cb + kBarAEmpty + 8 * (kAQ * q + al));
                    umma_commit(cb + kBarDFull + 8 * dp);
                    if (!ONE && (us + kMmaWarps >= kPS || j + kMmaWarps >= n)) umma_commit(bar_empty + 8 * s);
                }
                __syncwarp();
                g += kMmaWarps;
                while (g >= G) g -= G;
                if (!ONE && (us += kMmaWarps) >= kPS) {
                    us -= kPS;
                    if (++s == S) {
                        s = 0;
                        full_ph ^= 1u;
                    }
                }
            }
            xoff += static_cast<uint32_t>(x_smem_bytes((int64_t)G * kGroup));
        }
        // odd n: the last pair has no stream-1 unit; the warp that would
        // have issued it still signals the pair's accumulators -- after the
        // slot's previous pair has been consumed, so that the arrival cannot
        // count towards that phase
        if (ok && (n & 1) && n % kMmaWarps == m) {
            const int32_t k = n >> 1;
            const int dp = k % kDP;
            const uint32_t d_ph = (k / kDP) & 1u;
            if (vote_wait(cb + kBarDEmpty + 8 * dp, d_ph ^ 1u, lane == 1 && k >= kDP, abort_flag)) {
                if (elect_one()) umma_commit(cb + kBarDFull + 8 * dp);
                __syncwarp();
            }
        }
        // every MMA this warp issued has completed before tensor memory is freed
        if (elect_one()) umma_commit(cb + kBarDrain + 8 * m);
        __syncwarp();
        volatile int no_abort = 0;
        (void)mbar_wait(cb + kBarDrain + 8 * m, 0, &no_abort);
    } else if (warp >= kDecWarp0 && warp < kDecWarp0 + kDecWarps) {
        // ---------------------------------------------------- decode streams
        // stream q (one warpgroup) decodes units j = q, q+2, ...: each
        // thread the 128 weights of its row
        const int q = (warp - kDecWarp0) >> 2;
        const int r = threadIdx.x & 127;   // weight row in the tile = tensor-memory lane
        const uint32_t tm = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + q * kAQ * kACols;
        const DecodeConsts dk = XF16 ? decode_consts_fp16() : decode_consts_bf16();
        const int codes_off = C::OffCodes + 16 * r;   // + unit in stage * 4096 (+ 2048 second half)
        const uint32_t bar_afull = cb + kBarAFull + 8 * kAQ * q;
        const uint32_t bar_aempty = cb + kBarAEmpty + 8 * kAQ * q;
        int s = 0, al = 0;
        uint32_t full_ph = 0, a_ph = 0;
        for (int32_t j = q; j < n; j += 2) {
            const int us = j % kPS;
            if (us < 2 && !warp_wait(bar_full + 8 * s, full_ph, abort_flag)) break;   // first unit of the stage
            const bool zero = zflags != nullptr && __ldg(zflags + u0 + j) != 0;   // nothing to decode
            const uint8_t* cp = ring_ptr + s * C::StageBytes + codes_off + us * kUnitCodeBytes;
            uint4 c0 = make_uint4(0, 0, 0, 0), c1 = c0;
            if (!zero) {
                c0 = lds_v4(cp);
                c1 = lds_v4(cp + 2048);
            }
            if (us >= kPS - 2 || j + 2 >= n) {   // this stream's last unit of the stage
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_empty + 8 * s);
                if (++s == S) {
                    s = 0;
                    full_ph ^= 1u;
                }
            }
            if (j >= 2 * kAQ) {
                if (!warp_wait(bar_aempty + 8 * al, a_ph ^ 1u, abort_flag)) break;
                tc_fence_after_sync();
            }
            if (!zero) {
                // two halves of 32 columns: the first half's store runs while
                // the second half decodes (the empty asm keeps the compiler
                // from moving that decode ahead of the first store)
                uint32_t p[64];
                const uint32_t cw[4] = {c0.x, c0.y, c0.z, c0.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (XF16)
                        decode_word_f16(cw[i], dk, p + 8 * i);
                    else
                        decode_word_bf16(cw[i], dk, p + 8 * i);
                }
                tmem_st_32x32b_x32(tm + al * kACols, p);
                asm volatile("" : "+r"(c1.x), "+r"(c1.y), "+r"(c1.z), "+r"(c1.w));
                const uint32_t cw2[4] = {c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (XF16)
                        decode_word_f16(cw2[i], dk, p + 32 + 8 * i);
                    else
                        decode_word_bf16(cw2[i], dk, p + 32 + 8 * i);
                }
                tmem_st_32x32b_x32(tm + al * kACols + 32, p + 32);
            }
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_afull + 8 * al);
            if (++al == kAQ) {
                al = 0;
                a_ph ^= 1u;
            }
        }
    } else if (warp >= kPromWarp0) {
        // ------------------------------------------------------- promotion
        const int r = threadIdx.x & 127;   // weight row in the tile = tensor-memory lane
        const uint32_t tm = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + kDCol0;
        const int scale_off = C::OffScales + (s8 ? 1 : 2) * r;   // + unit in stage * scale_unit
        // problem, tile and group of the next unit
        int pp = problem_of(a, u0);
        const int first_p = pp;
        int32_t G = a.prob[pp].G, R = a.prob[pp].R;
        const int64_t first_tile = (u0 - a.prob[pp].u_begin) / G;
        const int32_t first_g = static_cast<int32_t>((u0 - a.prob[pp].u_begin) % G);
        int64_t pb = first_tile;
        int32_t pg = first_g;
        // int8 scales (one problem): the current tile's row factor, loaded a
        // tile ahead of its use
        float row_f = s8 && pb < R ? a.row_factor[pb * kTileRows + r] : 1.f;
        float acc[NCOL];
#pragma unroll
        for (int m = 0; m < NCOL; ++m) acc[m] = 0.f;
        grid_dependency_wait();   // outputs and workspace belong to earlier kernels until now
        int s = 0, us = 0, dp = 0;
        uint32_t full_ph = 0, d_ph = 0;
        for (int32_t f = 0; f < n; f += 2) {
            const bool two = f + 1 < n;
            // the stage's copies completed long ago (its units were decoded);
            // observing its barrier makes the scales visible to these threads
            if (us == 0 && !warp_wait(bar_full + 8 * s, full_ph, abort_flag)) break;
            if (!warp_wait(cb + kBarDFull + 8 * dp, d_ph, abort_flag)) break;
            tc_fence_after_sync();
            uint32_t d[2 * NCOL];
            if (ONE) {
                tmem_ld_32x32b_x1(tm + 2 * dp * kNtok, d[0]);
                tmem_ld_32x32b_x1(tm + (2 * dp + 1) * kNtok, d[1]);
            } else {
                tmem_ld_32x32b_x16(tm + 2 * dp * kNtok, *reinterpret_cast<uint32_t(*)[16]>(d));
                tmem_ld_32x32b_x16(tm + (2 * dp + 1) * kNtok, *reinterpret_cast<uint32_t(*)[16]>(d + NCOL));
            }
            const uint8_t* sp = ring_ptr + s * C::StageBytes + scale_off + us * scale_unit;
            float sc0, sc1;
            if (s8) {
                sc0 = static_cast<float>(*reinterpret_cast<const int8_t*>(sp));
                sc1 = two ? static_cast<float>(*reinterpret_cast<const int8_t*>(sp + scale_unit)) : 0.f;
            } else {
                sc0 = fp16_bits_to_float(*reinterpret_cast<const uint16_t*>(sp));
                sc1 = two ? fp16_bits_to_float(*reinterpret_cast<const uint16_t*>(sp + scale_unit)) : 0.f;
            }
            tmem_ld_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(cb + kBarDEmpty + 8 * dp);
            us += 2;
            if (us == kPS || f + 2 >= n) {   // done with this stage's scales
                if (lane == 0) mbar_arrive(bar_empty + 8 * s);
                us = 0;
                if (++s == S) {
                    s = 0;
                    full_ph ^= 1u;
                }
            }
            if (++dp == kDP) {
                dp = 0;
                d_ph ^= 1u;
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                if (i == 1 && !two) break;
                const float sc = i == 0 ? sc0 : sc1;
                const int32_t u = f + i;
                if (zflags == nullptr || __ldg(zflags + u0 + u) == 0)
#pragma unroll
                    for (int m = 0; m < NCOL; ++m) acc[m] = fmaf(sc, __uint_as_float(d[i * NCOL + m]), acc[m]);
                if (pg == G - 1 || u == n - 1) {
                    const bool first = pp == first_p && pb == first_tile;
                    const bool whole = (!first || first_g == 0) && pg == G - 1;
                    flush_tile<NCOL>(a, v, pp, pb, first, whole, acc, r, s8, row_f);
#pragma unroll
                    for (int m = 0; m < NCOL; ++m) acc[m] = 0.f;
                }
                if (++pg == G) {
                    pg = 0;
                    if (++pb == R && pp + 1 < a.P) {
                        pb = 0;
                        ++pp;
                        G = a.prob[pp].G;
                        R = a.prob[pp].R;
                    }
                    if (s8 && pb < R) row_f = a.row_factor[pb * kTileRows + r];
                }
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before_sync();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) atomicOr(a.err, 1);
    if (warp == kAllocWarp) {
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

template <bool ONE, bool XF16, int EXT>
cudaError_t set_smem_limit() {
    static cudaError_t status = cudaErrorUnknown;
    static std::once_flag once;
    std::call_once(once, [] {
        status = cudaFuncSetAttribute(stream_kernel<ONE, XF16, EXT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      kSmemLimit);
    });
    return status;
}

template <bool ONE, bool XF16, int EXT>
cudaError_t launch_one(const StreamProblem* probs, const StreamArgs& a, const StreamPlan& plan,
                       cudaStream_t stream) {
    XMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (!ONE) {
        EncodeTiledFn enc = encode_tiled_fn();
        if (enc == nullptr) return cudaErrorNotSupported;
        for (int p = 0; p < a.P; ++p) {
            const cuuint64_t dims[2] = {static_cast<cuuint64_t>(probs[p].K), static_cast<cuuint64_t>(a.M)};
            const cuuint64_t strides[1] = {static_cast<cuuint64_t>(probs[p].ldx) * 2};
            const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kNtok)};
            const cuuint32_t estr[2] = {1, 1};
            if (enc(&maps.map[p], XF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<uint16_t*>(probs[p].x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return cudaErrorInvalidValue;
        }
    }
    cudaError_t e = set_smem_limit<ONE, XF16, EXT>();
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
    return cudaLaunchKernelEx(&cfg, stream_kernel<ONE, XF16, EXT>, maps, a);
}

}  // namespace

StreamPlan plan_stream(int64_t M, const int64_t* N, const int64_t* K, int P, int sm_count) {
    StreamPlan p = {};
    if (sm_count <= 0) sm_count = 152;
    p.U = 0;
    p.tiles = 0;
    for (int i = 0; i < P; ++i) {
        const int64_t R = ceil_div(N[i], kTileRows);
        p.U += R * (K[i] / kGroup);
        p.tiles += R;
    }
    p.V = p.U < sm_count ? p.U : sm_count;   // one worker per CTA, one CTA per SM
    p.grid = p.V;
    // M == 1 keeps the activation rows of each CTA's problems in shared
    // memory when at least three stages still fit beside the largest set
    int64_t x_smem = 0;
    if (M == 1) {
        int64_t begin[kMaxGroup + 1];
        begin[0] = 0;
        for (int i = 0; i < P; ++i) begin[i + 1] = begin[i] + ceil_div(N[i], kTileRows) * (K[i] / kGroup);
        for (int64_t v = 0; v < p.V; ++v) {
            const int64_t u0 = p.U * v / p.V, u1 = p.U * (v + 1) / p.V;
            int64_t bytes = 0;
            for (int i = 0; i < P; ++i)
                if (begin[i] < u1 && begin[i + 1] > u0) bytes += x_smem_bytes(K[i]);
            if (bytes > x_smem) x_smem = bytes;
        }
    }
    p.one = M == 1 && kSmemLimit - 1024 - kCtrlBytes - x_smem >= 3 * SCfg<true>::StageBytes;
    p.x_smem = p.one ? x_smem : 0;
    const int64_t stage_bytes = p.one ? SCfg<true>::StageBytes : SCfg<false>::StageBytes;
    int64_t stages = (kSmemLimit - 1024 - kCtrlBytes - p.x_smem) / stage_bytes;
    if (stages > kMaxStages) stages = kMaxStages;
    p.stages = static_cast<int>(stages);
    p.smem = static_cast<size_t>(1024 + p.x_smem + stages * stage_bytes + kCtrlBytes);
    const int64_t ncol = p.one ? SCfg<true>::NCOL : SCfg<false>::NCOL;
    const size_t counters = static_cast<size_t>(round_up(p.tiles * 4 * 4, 256));
    p.ws_bytes = kWorkspaceErrBytes + counters + static_cast<size_t>(2 * p.V * kTileRows * ncol) * sizeof(float);
    return p;
}

cudaError_t launch_stream(const StreamProblem* probs, int P, bool x_f16, bool s8, const uint8_t* zflags, int64_t M,
                          void* ws, const StreamPlan& plan, cudaStream_t stream) {
    if (P < 1 || P > kMaxGroup || ((s8 || zflags != nullptr) && P != 1)) return cudaErrorInvalidValue;
    StreamArgs a = {};
    a.zflags = zflags;
    a.s8 = s8 ? 1 : 0;
    a.scale_unit = s8 ? kUnitScaleBytesS8 : kUnitScaleBytes;
    a.M = static_cast<int>(M);
    a.P = P;
    a.stages = plan.stages;
    a.x_smem = static_cast<uint32_t>(plan.x_smem);
    a.U = plan.U;
    a.V = plan.V;
    int64_t u = 0, tile = 0;
    for (int p = 0; p < P; ++p) {
        StreamProb& pr = a.prob[p];
        const int64_t R = ceil_div(probs[p].N, kTileRows), G = probs[p].K / kGroup;
        pr.codes = probs[p].tiled;
        pr.scales = probs[p].tiled + R * G * kUnitCodeBytes;
        pr.x = probs[p].x;
        pr.u_begin = u;
        pr.tile0 = tile;
        pr.N = probs[p].N;
        pr.R = static_cast<int32_t>(R);
        pr.G = static_cast<int32_t>(G);
        pr.out = probs[p].out;
        u += R * G;
        tile += R;
    }
    if (s8) {
        const int64_t U0 = a.prob[0].R * (int64_t)a.prob[0].G;
        a.row_factor = reinterpret_cast<const float*>(probs[0].tiled + U0 * (kUnitCodeBytes + kUnitScaleBytesS8));
    }
    uint8_t* w = static_cast<uint8_t*>(ws);
    a.err = reinterpret_cast<int*>(w);
    a.counters = reinterpret_cast<int*>(w + kWorkspaceErrBytes);
    a.slots = reinterpret_cast<float*>(w + kWorkspaceErrBytes + static_cast<size_t>(round_up(plan.tiles * 4 * 4, 256)));
    if (s8) {
        if (x_f16)
            return plan.one ? launch_one<true, true, 1>(probs, a, plan, stream)
                            : launch_one<false, true, 1>(probs, a, plan, stream);
        return plan.one ? launch_one<true, false, 1>(probs, a, plan, stream)
                        : launch_one<false, false, 1>(probs, a, plan, stream);
    }
    if (zflags != nullptr) {
        if (x_f16)
            return plan.one ? launch_one<true, true, 2>(probs, a, plan, stream)
                            : launch_one<false, true, 2>(probs, a, plan, stream);
        return plan.one ? launch_one<true, false, 2>(probs, a, plan, stream)
                        : launch_one<false, false, 2>(probs, a, plan, stream);
    }
    if (x_f16)
        return plan.one ? launch_one<true, true, 0>(probs, a, plan, stream)
                        : launch_one<false, true, 0>(probs, a, plan, stream);
    return plan.one ? launch_one<true, false, 0>(probs, a, plan, stream)
                    : launch_one<false, false, 0>(probs, a, plan, stream);
}

}  // namespace tern
