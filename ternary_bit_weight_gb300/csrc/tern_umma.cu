// Tensor-core (tcgen05) kernel of libtern: Y[M,N] = X[M,K] . (s (.) T)^T for
// any M, streaming the tiled 2-bit weights once per token tile.
//
// Method ("Ternary embedding model in vLLM", 2kiu.com/news/5082861, §4.2,
// §4.3): the weights stay packed in memory and are decoded on chip; signs
// are summed inside each 128-wide scale group and the FP16 scale is applied
// once per group.  The page's CUDA-core kernel is replaced by tcgen05:
//
//   * work unit = one 128-row x 128-weight block of the tiled layout
//     (4 KB of codes + 256 B of scales) for one tile of NTOK tokens;
//   * producer warp: a ring of shared-memory stages filled by bulk copies
//     (codes, scales) and a 2-D TMA copy of the X tile (128-byte swizzle,
//     rows past M zero-filled);
//   * decode warpgroups (one thread per weight row = one tensor-memory
//     lane): each 16-weight code word becomes eight exact bf16 pairs
//     t in {-1,0,+1} (one LOP3 + one bf16x2 FMA per pair) written with
//     tcgen05.st as the A operand of the unit (64 columns);
//   * MMA warp: eight tcgen05.mma (M = 128, N = NTOK, K = 16, bf16 -> fp32)
//     per unit, A from tensor memory, B = X from shared memory, into a
//     double-buffered per-unit accumulator in tensor memory;
//   * promotion: the decode threads read the unit's fp32 group partial with
//     tcgen05.ld and add s * partial to their register accumulators -- the
//     FP16 scale is converted exactly to fp32 and never rounded to bf16.
//
// Work split: each decode warpgroup is an independent worker owning the
// contiguous unit range [U*v/V, U*(v+1)/V) of all U units, in (token tile,
// row tile, group) order.  A tile whose groups span two or more workers is
// finished by the last of them to arrive, which sums the partials in worker
// order (deterministic; no waiting on other CTAs).  Every mbarrier wait is
// bounded; on a timeout the kernel raises an error word in the workspace,
// drains its own copies and MMAs, frees its tensor memory and returns.

#include <cuda.h>

#include <mutex>

#include "tern_common.cuh"
#include "tern_internal.h"
#include "tern_sm100.cuh"

namespace tern {
namespace {

constexpr int kNWG = 2;                          // decode warpgroups (workers) per CTA
constexpr int kDecWarps = 4 * kNWG;
constexpr int kProducerWarp = kDecWarps;
constexpr int kMmaWarp = kDecWarps + 1;
constexpr int kUThreads = (kDecWarps + 2) * 32;

template <int NTOK>
struct Cfg {
    static constexpr int kDBuf = NTOK <= 64 ? 2 : 1;
    // decoded A lives in a ring of 32-column half-unit buffers per worker
    static constexpr int kAHalves = (NTOK == 16 || NTOK >= 64) ? 3 : 2;
    static constexpr int kAColsW = 32 * kAHalves;
    static constexpr int kColsUsed = kNWG * kAColsW + kNWG * kDBuf * NTOK;
    static constexpr int kTmemCols = kColsUsed <= 256 ? 256 : 512;
    static constexpr int kCtasPerSm = kTmemCols <= 256 ? 2 : 1;
    static constexpr int kXBox = NTOK * 128;                 // one 64-wide X box
    static constexpr int kXUnit = 2 * kXBox;                 // one unit's X tile
    static constexpr int kOffCodes = kNWG * kXUnit;
    static constexpr int kOffScales = kOffCodes + kNWG * kUnitCodeBytes;
    static constexpr int kStageBytes = (kOffScales + kNWG * kUnitScaleBytes + 1023) / 1024 * 1024;
    static constexpr int kSmemBudget = kCtasPerSm == 2 ? 110 * 1024 : 224 * 1024;
    static constexpr int kStages = (kSmemBudget - 2048) / kStageBytes;
    static_assert(kStages >= 2, "stage ring too small");
    // control block: barriers, tensor-memory base, abort flag
    static constexpr int kOffCtrl = kStages * kStageBytes;
    static constexpr int kCtrlBytes = 1024;
    static constexpr int kSmemBytes = 1024 /*alignment slack*/ + kOffCtrl + kCtrlBytes;
};

struct UmmaArgs {
    const uint8_t* codes;
    const uint8_t* scales;
    int M;
    int64_t N;
    int64_t R;               // 128-row tiles
    int64_t G;               // groups per row
    int64_t U;               // units = token tiles x R x G
    int64_t V;               // workers (<= U)
    OutputSplit out;
    int* err;                // workspace error word
    int* counters;           // [token tiles x R][4 row quarters]
    float* slots;            // [2V][NTOK][128] (column-major per slot)
};

__device__ __forceinline__ int64_t owner_worker(int64_t u, int64_t U, int64_t V) {
    return ((u + 1) * V - 1) / U;
}

// Finish a tile whose group partials this worker holds in acc (thread =
// row r of the tile, acc[m] = token m of the tile).  `whole`: this worker
// covered every group of the tile, so it owns the result.  Otherwise each
// warp (32 rows) publishes the valid token columns of its partial and the
// last contributing worker to arrive for that row quarter sums all
// partials in worker order.  Slots are column-major ([slot][token][128
// rows]) so a warp's column is one contiguous 128-byte run.
template <int NTOK>
__device__ __forceinline__ void flush_tile(const UmmaArgs& a, int64_t v, int64_t tile_id,
                                           int64_t first_tile, bool whole, float (&acc)[NTOK],
                                           int mvalid, int r) {
    const int lane = r & 31, quad = r >> 5;
    const int64_t tt = tile_id / a.R, b = tile_id - tt * a.R;
    const int64_t row = b * kTileRows + r;
    const int m0 = static_cast<int>(tt * NTOK);
    if (whole) {
        if (row < a.N)
#pragma unroll
            for (int m = 0; m < NTOK; ++m)
                if (m < mvalid) store_y(a.out, m0 + m, row, acc[m]);
        return;
    }
    const int64_t slot = 2 * v + (tile_id == first_tile ? 0 : 1);
    float* sp = a.slots + slot * (kTileRows * NTOK) + r;
#pragma unroll
    for (int m = 0; m < NTOK; ++m)
        if (m < mvalid) sp[m * kTileRows] = acc[m];
    __syncwarp();
    const int64_t t0 = tile_id * a.G;
    const int64_t w_first = owner_worker(t0, a.U, a.V);
    const int64_t w_last = owner_worker(t0 + a.G - 1, a.U, a.V);
    int* counter = a.counters + tile_id * 4 + quad;
    int last = 0;
    if (lane == 0) {
        __threadfence();   // publish the warp's slot writes (ordered by the warp barrier)
        last = atomicAdd(counter, 1) == static_cast<int>(w_last - w_first);
        if (last) __threadfence();
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __syncwarp();   // order the lanes' loads after lane 0's acquire
    // the first contributor's range starts before this tile (its partial
    // is its "last tile" slot) unless it starts exactly at the tile start
    const int first_side = (a.U * w_first < t0 * a.V) ? 1 : 0;
#pragma unroll
    for (int m = 0; m < NTOK; ++m) acc[m] = 0.f;
    for (int64_t ww = w_first; ww <= w_last; ++ww) {
        const int64_t sl = 2 * ww + (ww == w_first ? first_side : 0);
        const float* src = a.slots + sl * (kTileRows * NTOK) + r;
#pragma unroll
        for (int m = 0; m < NTOK; ++m)
            if (m < mvalid) acc[m] += __ldcg(src + m * kTileRows);
    }
    if (row < a.N)
#pragma unroll
        for (int m = 0; m < NTOK; ++m)
            if (m < mvalid) store_y(a.out, m0 + m, row, acc[m]);
    if (lane == 0) *counter = 0;   // leave the workspace zeroed
}

// Warp-uniform bounded wait (every lane observes the barrier itself).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
    const bool got = mbar_wait(bar, parity, abort);
    return __all_sync(0xffffffffu, got);
}

// Position of a unit in (token tile, row tile, group) order, advanced by
// increments so the per-unit loops do no integer division.
struct UnitCursor {
    int32_t g;    // group along K
    int32_t b;    // 128-row tile
    int32_t tt;   // token tile
    int32_t cu;   // unit of the tiled weight: b * G + g
};

__device__ __forceinline__ UnitCursor cursor_at(int64_t u, int64_t R, int64_t G) {
    const int64_t RG = R * G;
    UnitCursor c;
    c.tt = static_cast<int32_t>(u / RG);
    const int64_t rem = u - (int64_t)c.tt * RG;
    c.b = static_cast<int32_t>(rem / G);
    c.g = static_cast<int32_t>(rem - (int64_t)c.b * G);
    c.cu = static_cast<int32_t>(rem);
    return c;
}

__device__ __forceinline__ void cursor_next(UnitCursor& c, int32_t R, int32_t G) {
    ++c.cu;
    if (++c.g == G) {
        c.g = 0;
        if (++c.b == R) {
            c.b = 0;
            ++c.tt;
            c.cu = 0;
        }
    }
}

template <int NTOK, int MV>
__global__ void __launch_bounds__(kUThreads, Cfg<NTOK>::kCtasPerSm)
umma_kernel(const __grid_constant__ CUtensorMap xmap, const UmmaArgs a) {
    // MV: token columns promoted per unit (1 when M == 1, else NTOK)
    using C = Cfg<NTOK>;
    constexpr int AH = C::kAHalves;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base (swizzle atoms)
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);

    // control block
    uint8_t* ctrl = smem + C::kOffCtrl;
    const uint32_t cbase = sbase + C::kOffCtrl;
    const uint32_t bar_full = cbase;                                  // [kStages]
    const uint32_t bar_empty = bar_full + 8 * C::kStages;             // [kStages]
    const uint32_t bar_afull = bar_empty + 8 * C::kStages;            // [kNWG][AH]
    const uint32_t bar_aempty = bar_afull + 8 * kNWG * AH;            // [kNWG][AH]
    const uint32_t bar_dfull = bar_aempty + 8 * kNWG * AH;            // [kNWG][kDBuf]
    const uint32_t bar_dempty = bar_dfull + 8 * kNWG * C::kDBuf;      // [kNWG][kDBuf]
    const uint32_t bar_drain = bar_dempty + 8 * kNWG * C::kDBuf;
    uint32_t* tmem_base_ptr = reinterpret_cast<uint32_t*>(ctrl + 512);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 516);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // workers of this CTA: contiguous unit ranges
    int64_t w_u0[kNWG];
    int32_t w_n[kNWG];
    int32_t max_n = 0;
#pragma unroll
    for (int w = 0; w < kNWG; ++w) {
        const int64_t v = (int64_t)blockIdx.x * kNWG + w;
        w_u0[w] = v < a.V ? a.U * v / a.V : 0;
        w_n[w] = v < a.V ? static_cast<int32_t>(a.U * (v + 1) / a.V - w_u0[w]) : 0;
        max_n = w_n[w] > max_n ? w_n[w] : max_n;
    }
    const int32_t R32 = static_cast<int32_t>(a.R), G32 = static_cast<int32_t>(a.G);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int w = 0; w < kNWG; ++w) {
            for (int q = 0; q < AH; ++q) {
                mbar_init(bar_afull + 8 * (AH * w + q), 4);
                mbar_init(bar_aempty + 8 * (AH * w + q), 1);
            }
            for (int b = 0; b < C::kDBuf; ++b) {
                mbar_init(bar_dfull + 8 * (w * C::kDBuf + b), 1);
                mbar_init(bar_dempty + 8 * (w * C::kDBuf + b), 4);
            }
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_base_ptr), C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) prefetch_tensormap(&xmap);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_base_ptr;
    grid_launch_dependents();

    if (warp == kProducerWarp) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            constexpr uint32_t kUnitBytes = kUnitCodeBytes + kUnitScaleBytes + C::kXUnit;
            UnitCursor cw[kNWG], cx[kNWG];   // next unit for weights / for X
#pragma unroll
            for (int w = 0; w < kNWG; ++w) cw[w] = cx[w] = cursor_at(w_u0[w], a.R, a.G);
            bool ok = true;
            // the weights of the first stages do not depend on earlier kernels
            const int32_t pre = max_n < C::kStages ? max_n : C::kStages;
            for (int32_t f = 0; f < pre; ++f) {
                const uint32_t st = sbase + f * C::kStageBytes;
                uint32_t bytes = 0;
#pragma unroll
                for (int w = 0; w < kNWG; ++w) bytes += f < w_n[w] ? kUnitBytes : 0u;
                mbar_arrive_expect_tx(bar_full + 8 * f, bytes);
#pragma unroll
                for (int w = 0; w < kNWG; ++w) {
                    if (f >= w_n[w]) continue;
                    bulk_load(st + C::kOffCodes + w * kUnitCodeBytes,
                              a.codes + (int64_t)cw[w].cu * kUnitCodeBytes, kUnitCodeBytes, bar_full + 8 * f);
                    bulk_load(st + C::kOffScales + w * kUnitScaleBytes,
                              a.scales + (int64_t)cw[w].cu * kUnitScaleBytes, kUnitScaleBytes, bar_full + 8 * f);
                    cursor_next(cw[w], R32, G32);
                }
            }
            grid_dependency_wait();
            int s = 0;
            uint32_t round = 0;   // completed passes over the ring
            for (int32_t f = 0; f < max_n && ok; ++f) {
                const uint32_t st = sbase + s * C::kStageBytes;
                if (f >= pre) {
                    if (!mbar_wait(bar_empty + 8 * s, (round - 1) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint32_t bytes = 0;
#pragma unroll
                    for (int w = 0; w < kNWG; ++w) bytes += f < w_n[w] ? kUnitBytes : 0u;
                    mbar_arrive_expect_tx(bar_full + 8 * s, bytes);
#pragma unroll
                    for (int w = 0; w < kNWG; ++w) {
                        if (f >= w_n[w]) continue;
                        bulk_load(st + C::kOffCodes + w * kUnitCodeBytes,
                                  a.codes + (int64_t)cw[w].cu * kUnitCodeBytes, kUnitCodeBytes, bar_full + 8 * s);
                        bulk_load(st + C::kOffScales + w * kUnitScaleBytes,
                                  a.scales + (int64_t)cw[w].cu * kUnitScaleBytes, kUnitScaleBytes,
                                  bar_full + 8 * s);
                        cursor_next(cw[w], R32, G32);
                    }
                }
#pragma unroll
                for (int w = 0; w < kNWG; ++w) {
                    if (f >= w_n[w]) continue;
                    const uint32_t xs = st + w * C::kXUnit;
                    const int32_t k0 = cx[w].g * kGroup, row = cx[w].tt * NTOK;
                    tma_load_2d(xs, &xmap, k0, row, bar_full + 8 * s);
                    tma_load_2d(xs + C::kXBox, &xmap, k0 + 64, row, bar_full + 8 * s);
                    cursor_next(cx[w], R32, G32);
                }
                if (++s == C::kStages) {
                    s = 0;
                    ++round;
                }
            }
            if (*abort_flag) {
                // drain the copies this CTA may still have in flight (bounded)
                volatile int no_abort = 0;
                for (int t = 0; t < C::kStages; ++t) {
                    (void)mbar_wait(bar_full + 8 * t, 0, &no_abort);
                    (void)mbar_wait(bar_full + 8 * t, 1, &no_abort);
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------- MMA
        grid_dependency_wait();
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, NTOK);
            bool ok = true;
            int s = 0;
            uint32_t full_ph = 0;
            int abuf[kNWG];          // next A half-buffer per worker
            uint32_t around[kNWG];   // its completion parity
#pragma unroll
            for (int w = 0; w < kNWG; ++w) { abuf[w] = 0; around[w] = 0; }
            for (int32_t f = 0; f < max_n && ok; ++f) {
                const uint32_t st = sbase + s * C::kStageBytes;
                if (!mbar_wait(bar_full + 8 * s, full_ph, abort_flag)) {
                    ok = false;
                    break;
                }
                const int db = C::kDBuf == 2 ? (f & 1) : 0;
                const uint32_t dempty_ph = C::kDBuf == 2 ? (((f >> 1) & 1) ^ 1u) : ((f & 1) ^ 1u);
                // half h of every worker, then the next half: each half's four
                // MMAs start as soon as its decoded A is in tensor memory
#pragma unroll
                for (int h = 0; h < 2; ++h) {
#pragma unroll
                    for (int w = 0; w < kNWG; ++w) {
                        if (!ok || f >= w_n[w]) continue;
                        const int q = abuf[w];
                        if (!mbar_wait(bar_afull + 8 * (AH * w + q), around[w], abort_flag)) {
                            ok = false;
                            break;
                        }
                        if (h == 0 && f >= C::kDBuf &&
                            !mbar_wait(bar_dempty + 8 * (w * C::kDBuf + db), dempty_ph, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        const uint32_t a_tm = tmem + w * C::kAColsW + 32 * q;
                        const uint32_t d_tm = tmem + kNWG * C::kAColsW + (w * C::kDBuf + db) * NTOK;
                        const uint64_t bdesc0 = smem_desc_kmajor_sw128(st + w * C::kXUnit + h * C::kXBox);
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj)   // +32 bytes per K-step = +2 in the address field
                            umma_bf16_tmem_a(d_tm, a_tm + 8 * jj, bdesc0 + 2 * jj, idesc, (h | jj) != 0 ? 1u : 0u);
                        umma_commit(bar_aempty + 8 * (AH * w + q));
                        if (h == 1) umma_commit(bar_dfull + 8 * (w * C::kDBuf + db));
                        if (++abuf[w] == AH) {
                            abuf[w] = 0;
                            around[w] ^= 1u;
                        }
                    }
                }
                if (ok) umma_commit(bar_empty + 8 * s);
                if (++s == C::kStages) {
                    s = 0;
                    full_ph ^= 1u;
                }
            }
            // every MMA issued has completed before tensor memory is freed
            umma_commit(bar_drain);
            volatile int no_abort = 0;
            (void)mbar_wait(bar_drain, 0, &no_abort);
        }
    } else {
        // ------------------------------------------------ decode workers
        grid_dependency_wait();
        const int wg = warp >> 2;
        const int r = threadIdx.x & 127;               // weight row in the tile = TMEM lane
        const int64_t v = (int64_t)blockIdx.x * kNWG + wg;
        const int32_t n = w_n[wg == 0 ? 0 : 1];
        const int64_t u0 = w_u0[wg == 0 ? 0 : 1];
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t a_tm0 = tmem + lane_off + wg * C::kAColsW;
        const uint32_t d_tm0 = tmem + lane_off + kNWG * C::kAColsW + wg * C::kDBuf * NTOK;
        const uint32_t bar_afull_w = bar_afull + 8 * AH * wg;
        const uint32_t bar_aempty_w = bar_aempty + 8 * AH * wg;
        if (n > 0) {
            UnitCursor cur = cursor_at(u0, a.R, a.G);    // unit j
            UnitCursor prev = cur;                        // unit j - 1
            const int64_t first_tile = (int64_t)cur.tt * a.R + cur.b;
            bool whole = cur.g == 0;
            float acc[NTOK];
#pragma unroll
            for (int m = 0; m < NTOK; ++m) acc[m] = 0.f;
            float s_prev = 0.f;
            bool ok = true;
            int s = 0;
            uint32_t full_ph = 0;
            int q = 0;               // next A half-buffer
            uint32_t qround = 0;     // completions of that buffer so far (parity)
            int32_t halves = 0;      // half-units decoded so far
            const uint8_t* codes_base = smem + C::kOffCodes + wg * kUnitCodeBytes + 16 * r;
            const uint8_t* scale_base = smem + C::kOffScales + wg * kUnitScaleBytes + 2 * r;
            for (int32_t j = 0; j <= n && ok; ++j) {
                float s_cur = 0.f;
                if (j < n) {
                    // ---- decode unit j into two A half-buffers
                    if (!warp_wait(bar_full + 8 * s, full_ph, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint4 c0 = lds_v4(codes_base + s * C::kStageBytes);
                    const uint4 c1 = lds_v4(codes_base + s * C::kStageBytes + 2048);
                    s_cur = fp16_bits_to_float(*reinterpret_cast<const uint16_t*>(scale_base + s * C::kStageBytes));
                    if (++s == C::kStages) {
                        s = 0;
                        full_ph ^= 1u;
                    }
                    const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (halves >= AH) {
                            // the MMAs that last read this buffer have completed
                            if (!warp_wait(bar_aempty_w + 8 * q, qround ^ 1u, abort_flag)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after_sync();
                        }
                        const uint32_t a_tm = a_tm0 + 32 * q;
#pragma unroll
                        for (int w4 = 0; w4 < 4; ++w4) {
                            uint32_t pairs[8];
                            decode_word_bf16(words[4 * h + w4], pairs);
                            tmem_st_32x32b_x8(a_tm + 8 * w4, pairs);
                        }
                        tmem_st_wait();
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar_afull_w + 8 * q);
                        ++halves;
                        if (++q == AH) {
                            q = 0;
                            qround ^= 1u;
                        }
                    }
                    if (!ok) break;
                }
                if (j >= 1) {
                    // ---- promote unit j-1: acc += s * group partial
                    const int jp = j - 1;
                    const int db = C::kDBuf == 2 ? (jp & 1) : 0;
                    const uint32_t dfull_ph = C::kDBuf == 2 ? ((jp >> 1) & 1) : (jp & 1);
                    if (!warp_wait(bar_dfull + 8 * (wg * C::kDBuf + db), dfull_ph, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t d_tm = d_tm0 + db * NTOK;
                    if (MV == 1) {
                        uint32_t d0;
                        tmem_ld_32x32b_x1(d_tm, d0);
                        tmem_ld_wait();
                        acc[0] = fmaf(s_prev, __uint_as_float(d0), acc[0]);
                    } else {
#pragma unroll
                        for (int c = 0; c < NTOK; c += 16) {
                            uint32_t d[16];
                            tmem_ld_32x32b_x16(d_tm + c, d);
                            tmem_ld_wait();
#pragma unroll
                            for (int m = 0; m < 16; ++m) acc[c + m] = fmaf(s_prev, __uint_as_float(d[m]), acc[c + m]);
                        }
                    }
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_dempty + 8 * (wg * C::kDBuf + db));
                    // tile finished (next unit in another tile, or no next unit)?
                    const bool tile_end = (j == n) || cur.b != prev.b || cur.tt != prev.tt;
                    if (tile_end) {
                        const int64_t tile_id = (int64_t)prev.tt * a.R + prev.b;
                        const int mvalid =
                            MV == 1 ? 1 : ((a.M - prev.tt * NTOK) < NTOK ? (a.M - prev.tt * NTOK) : NTOK);
                        flush_tile<NTOK>(a, v, tile_id, first_tile, whole && prev.g == G32 - 1, acc, mvalid, r);
#pragma unroll
                        for (int m = 0; m < NTOK; ++m) acc[m] = 0.f;
                        whole = true;
                    }
                }
                s_prev = s_cur;
                prev = cur;
                if (j < n) cursor_next(cur, R32, G32);
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before_sync();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) atomicOr(a.err, 1);
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::kTmemCols);
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

template <int NTOK, int MV>
cudaError_t launch_ntok(const uint16_t* X, int64_t ldx, const UmmaArgs& a, const UmmaPlan& plan,
                        cudaStream_t stream) {
    using C = Cfg<NTOK>;
    EncodeTiledFn enc = encode_tiled_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    CUtensorMap map;
    const int64_t K = a.G * kGroup;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(a.M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldx) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(NTOK)};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(X), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;

    cudaError_t e = cudaFuncSetAttribute(umma_kernel<NTOK, MV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.grid));
    cfg.blockDim = dim3(kUThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, umma_kernel<NTOK, MV>, map, a);
}

template <int NTOK>
void fill_plan(UmmaPlan& p, int64_t M, int64_t N, int64_t K, int sms) {
    using C = Cfg<NTOK>;
    p.ntok = NTOK;
    p.R = ceil_div(N, kTileRows);
    p.G = K / kGroup;
    p.token_tiles = ceil_div(M, NTOK);
    p.U = p.token_tiles * p.R * p.G;
    int64_t workers = (int64_t)sms * C::kCtasPerSm * kNWG;
    if (workers > p.U) workers = p.U;
    p.V = workers;
    p.grid = ceil_div(workers, kNWG);
    p.smem = C::kSmemBytes;
    const size_t counters = (size_t)ceil_div(p.token_tiles * p.R * 4 * 4, 256) * 256;
    p.ws_bytes = kWorkspaceErrBytes + counters + (size_t)2 * p.V * kTileRows * NTOK * sizeof(float);
}

}  // namespace

UmmaPlan plan_umma(int64_t M, int64_t N, int64_t K, int sm_count) {
    UmmaPlan p = {};
    if (sm_count <= 0) sm_count = 152;
    if (M <= 16)
        fill_plan<16>(p, M, N, K, sm_count);
    else if (M <= 32)
        fill_plan<32>(p, M, N, K, sm_count);
    else if (M <= 64)
        fill_plan<64>(p, M, N, K, sm_count);
    else
        fill_plan<128>(p, M, N, K, sm_count);
    return p;
}

cudaError_t launch_umma(const uint16_t* X, int64_t ldx, const uint8_t* tiled, int64_t M, int64_t N,
                        int64_t K, const OutputSplit& out, void* ws, const UmmaPlan& plan,
                        cudaStream_t stream) {
    UmmaArgs a = {};
    a.codes = tiled;
    a.scales = tiled + plan.R * plan.G * kUnitCodeBytes;
    a.M = static_cast<int>(M);
    a.N = N;
    a.R = plan.R;
    a.G = plan.G;
    a.U = plan.U;
    a.V = plan.V;
    a.out = out;
    uint8_t* w = static_cast<uint8_t*>(ws);
    a.err = reinterpret_cast<int*>(w);
    a.counters = reinterpret_cast<int*>(w + kWorkspaceErrBytes);
    a.slots = reinterpret_cast<float*>(w + kWorkspaceErrBytes +
                                       (size_t)ceil_div(plan.token_tiles * plan.R * 4 * 4, 256) * 256);
    switch (plan.ntok) {
        case 16:
            return M == 1 ? launch_ntok<16, 1>(X, ldx, a, plan, stream)
                          : launch_ntok<16, 16>(X, ldx, a, plan, stream);
        case 32: return launch_ntok<32, 32>(X, ldx, a, plan, stream);
        case 64: return launch_ntok<64, 64>(X, ldx, a, plan, stream);
        default: return launch_ntok<128, 128>(X, ldx, a, plan, stream);
    }
}

}  // namespace tern
