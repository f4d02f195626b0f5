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
constexpr int kACols = 64;                       // tensor-memory columns of one unit's A
constexpr int kWorkspaceErr = 256;               // error word + padding at the workspace start

template <int NTOK>
struct Cfg {
    static constexpr int kDBuf = NTOK <= 64 ? 2 : 1;
    static constexpr int kColsUsed = kNWG * kACols + kNWG * kDBuf * NTOK;
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
    float* slots;            // [2V][128][NTOK]
};

__device__ __forceinline__ void store_y(const OutputSplit& out, int m, int64_t n, float v) {
    int j = 0;
#pragma unroll
    for (int i = 1; i < kMaxOutputs; ++i) j += (i < out.n_out && n >= out.offset[i]);
    out.y[j][(int64_t)m * out.ldy[j] + (n - out.offset[j])] = v;
}

__device__ __forceinline__ int64_t owner_worker(int64_t u, int64_t U, int64_t V) {
    return ((u + 1) * V - 1) / U;
}

// Finish a tile whose group partials this worker holds in acc (thread =
// row r of the tile, acc[m] = token m of the tile).  `whole`: this worker
// covered every group of the tile, so it owns the result.  Otherwise each
// warp (32 rows) publishes its partial and the last contributing worker to
// arrive for that row quarter sums all partials in worker order.
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
    float4* sp = reinterpret_cast<float4*>(a.slots + (slot * kTileRows + r) * NTOK);
#pragma unroll
    for (int m = 0; m < NTOK; m += 4) sp[m / 4] = make_float4(acc[m], acc[m + 1], acc[m + 2], acc[m + 3]);
    __threadfence();
    __syncwarp();
    const int64_t w_first = owner_worker(tile_id * a.G, a.U, a.V);
    const int64_t w_last = owner_worker(tile_id * a.G + a.G - 1, a.U, a.V);
    int* counter = a.counters + tile_id * 4 + quad;
    int last = 0;
    if (lane == 0) last = atomicAdd(counter, 1) == static_cast<int>(w_last - w_first);
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __threadfence();
    // sum the partials in worker order (this worker's own included)
#pragma unroll
    for (int m = 0; m < NTOK; ++m) acc[m] = 0.f;
    for (int64_t ww = w_first; ww <= w_last; ++ww) {
        const int64_t ww_first_tile = (a.U * ww / a.V) / a.G;
        const int64_t sl = 2 * ww + (tile_id == ww_first_tile ? 0 : 1);
        const float4* src = reinterpret_cast<const float4*>(a.slots + (sl * kTileRows + r) * NTOK);
#pragma unroll
        for (int m = 0; m < NTOK; m += 4) {
            const float4 q = __ldcg(src + m / 4);
            acc[m] += q.x; acc[m + 1] += q.y; acc[m + 2] += q.z; acc[m + 3] += q.w;
        }
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

template <int NTOK>
__global__ void __launch_bounds__(kUThreads, Cfg<NTOK>::kCtasPerSm)
umma_kernel(const __grid_constant__ CUtensorMap xmap, const UmmaArgs a) {
    using C = Cfg<NTOK>;
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
    const uint32_t bar_afull = bar_empty + 8 * C::kStages;            // [kNWG]
    const uint32_t bar_dfull = bar_afull + 8 * kNWG;                  // [kNWG][kDBuf]
    const uint32_t bar_dempty = bar_dfull + 8 * kNWG * C::kDBuf;      // [kNWG][kDBuf]
    const uint32_t bar_drain = bar_dempty + 8 * kNWG * C::kDBuf;
    uint32_t* tmem_base_ptr = reinterpret_cast<uint32_t*>(ctrl + 512);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 516);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // workers of this CTA
    int64_t w_u0[kNWG], w_n[kNWG];
    int64_t max_n = 0;
#pragma unroll
    for (int w = 0; w < kNWG; ++w) {
        const int64_t v = (int64_t)blockIdx.x * kNWG + w;
        if (v < a.V) {
            w_u0[w] = a.U * v / a.V;
            w_n[w] = a.U * (v + 1) / a.V - w_u0[w];
        } else {
            w_u0[w] = 0;
            w_n[w] = 0;
        }
        max_n = w_n[w] > max_n ? w_n[w] : max_n;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int w = 0; w < kNWG; ++w) {
            mbar_init(bar_afull + 8 * w, 4);
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
            const uint32_t xbytes = C::kXUnit;
            int64_t issued = 0;
            bool ok = true;
            // weights of the first stages do not depend on earlier kernels
            const int64_t pre = max_n < C::kStages ? max_n : C::kStages;
            for (int64_t f = 0; f < pre; ++f) {
                const int s = static_cast<int>(f);
                uint32_t bytes = 0;
                for (int w = 0; w < kNWG; ++w)
                    if (f < w_n[w]) bytes += kUnitCodeBytes + kUnitScaleBytes + xbytes;
                mbar_arrive_expect_tx(bar_full + 8 * s, bytes);
                for (int w = 0; w < kNWG; ++w) {
                    if (f >= w_n[w]) continue;
                    const int64_t u = w_u0[w] + f;
                    const int64_t cu = u % (a.R * a.G);
                    const uint32_t st = sbase + s * C::kStageBytes;
                    bulk_load(st + C::kOffCodes + w * kUnitCodeBytes, a.codes + cu * kUnitCodeBytes,
                              kUnitCodeBytes, bar_full + 8 * s);
                    bulk_load(st + C::kOffScales + w * kUnitScaleBytes, a.scales + cu * kUnitScaleBytes,
                              kUnitScaleBytes, bar_full + 8 * s);
                }
                issued = f + 1;
            }
            grid_dependency_wait();
            for (int64_t f = 0; f < max_n && ok; ++f) {
                const int s = static_cast<int>(f % C::kStages);
                const uint32_t st = sbase + s * C::kStageBytes;
                if (f >= pre) {
                    if (!mbar_wait(bar_empty + 8 * s, static_cast<uint32_t>((f / C::kStages - 1) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint32_t bytes = 0;
                    for (int w = 0; w < kNWG; ++w)
                        if (f < w_n[w]) bytes += kUnitCodeBytes + kUnitScaleBytes + xbytes;
                    mbar_arrive_expect_tx(bar_full + 8 * s, bytes);
                    for (int w = 0; w < kNWG; ++w) {
                        if (f >= w_n[w]) continue;
                        const int64_t u = w_u0[w] + f;
                        const int64_t cu = u % (a.R * a.G);
                        bulk_load(st + C::kOffCodes + w * kUnitCodeBytes, a.codes + cu * kUnitCodeBytes,
                                  kUnitCodeBytes, bar_full + 8 * s);
                        bulk_load(st + C::kOffScales + w * kUnitScaleBytes,
                                  a.scales + cu * kUnitScaleBytes, kUnitScaleBytes, bar_full + 8 * s);
                    }
                    issued = f + 1;
                }
                for (int w = 0; w < kNWG; ++w) {
                    if (f >= w_n[w]) continue;
                    const int64_t u = w_u0[w] + f;
                    const int64_t tt = u / (a.R * a.G);
                    const int64_t g = u % a.G;
                    const uint32_t xs = st + w * C::kXUnit;
                    const int32_t row = static_cast<int32_t>(tt * NTOK);
                    tma_load_2d(xs, &xmap, static_cast<int32_t>(g * kGroup), row, bar_full + 8 * s);
                    tma_load_2d(xs + C::kXBox, &xmap, static_cast<int32_t>(g * kGroup + 64), row,
                                bar_full + 8 * s);
                }
            }
            if (*abort_flag) {
                // drain the copies this CTA still has in flight (bounded)
                volatile int no_abort = 0;
                for (int64_t f = issued - C::kStages < 0 ? 0 : issued - C::kStages; f < issued; ++f)
                    (void)mbar_wait(bar_full + 8 * static_cast<int>(f % C::kStages),
                                    static_cast<uint32_t>((f / C::kStages) & 1), &no_abort);
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------- MMA
        grid_dependency_wait();
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, NTOK);
            bool ok = true;
            for (int64_t f = 0; f < max_n && ok; ++f) {
                const int s = static_cast<int>(f % C::kStages);
                const uint32_t st = sbase + s * C::kStageBytes;
                if (!mbar_wait(bar_full + 8 * s, static_cast<uint32_t>((f / C::kStages) & 1), abort_flag)) {
                    ok = false;
                    break;
                }
                for (int w = 0; w < kNWG && ok; ++w) {
                    if (f >= w_n[w]) continue;
                    const int db = static_cast<int>(f % C::kDBuf);
                    if (!mbar_wait(bar_afull + 8 * w, static_cast<uint32_t>(f & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (f >= C::kDBuf &&
                        !mbar_wait(bar_dempty + 8 * (w * C::kDBuf + db),
                                   static_cast<uint32_t>((f / C::kDBuf - 1) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a_tm = tmem + w * kACols;
                    const uint32_t d_tm = tmem + kNWG * kACols + (w * C::kDBuf + db) * NTOK;
                    const uint32_t xs = st + w * C::kXUnit;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint64_t bdesc =
                            smem_desc_kmajor_sw128(xs + (j >> 2) * C::kXBox + 32 * (j & 3));
                        umma_bf16_tmem_a(d_tm, a_tm + 8 * j, bdesc, idesc, j > 0 ? 1u : 0u);
                    }
                    umma_commit(bar_dfull + 8 * (w * C::kDBuf + db));
                }
                if (ok) umma_commit(bar_empty + 8 * s);
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
        const int64_t u0 = v < a.V ? a.U * v / a.V : 0;
        const int64_t n = v < a.V ? a.U * (v + 1) / a.V - u0 : 0;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t a_tm = tmem + lane_off + wg * kACols;
        const int64_t RG = a.R * a.G;
        if (n > 0) {
            const int64_t first_tile = u0 / a.G;
            int64_t tile_cur = first_tile;
            bool whole = (u0 % a.G) == 0;
            float acc[NTOK];
#pragma unroll
            for (int m = 0; m < NTOK; ++m) acc[m] = 0.f;
            float s_prev = 0.f;
            int mvalid = 0;
            bool ok = true;
            for (int64_t j = 0; j <= n && ok; ++j) {
                // decode unit j (if any) into A
                float s_cur = 0.f;
                if (j < n) {
                    const int s = static_cast<int>(j % C::kStages);
                    const uint8_t* st = smem + s * C::kStageBytes;
                    if (!warp_wait(bar_full + 8 * s, static_cast<uint32_t>((j / C::kStages) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint4 c0 = lds_v4(st + C::kOffCodes + wg * kUnitCodeBytes + 16 * r);
                    const uint4 c1 = lds_v4(st + C::kOffCodes + wg * kUnitCodeBytes + 2048 + 16 * r);
                    s_cur = fp16_bits_to_float(
                        *reinterpret_cast<const uint16_t*>(st + C::kOffScales + wg * kUnitScaleBytes + 2 * r));
                    if (j >= 1) {
                        // MMA of unit j-1 complete: A is free and its partial is ready
                        const int db = static_cast<int>((j - 1) % C::kDBuf);
                        if (!warp_wait(bar_dfull + 8 * (wg * C::kDBuf + db),
                                       static_cast<uint32_t>(((j - 1) / C::kDBuf) & 1), abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                    }
                    const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        uint32_t pairs[8];
                        decode_word(words[q], pairs);
                        tmem_st_32x32b_x8(a_tm + 8 * q, pairs);
                    }
                    tmem_st_wait();
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_afull + 8 * wg);
                } else {
                    // final unit's partial
                    const int db = static_cast<int>((j - 1) % C::kDBuf);
                    if (!warp_wait(bar_dfull + 8 * (wg * C::kDBuf + db),
                                   static_cast<uint32_t>(((j - 1) / C::kDBuf) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                }
                if (j >= 1) {
                    // promote unit j-1: acc += s * partial
                    const int64_t up = u0 + j - 1;
                    const int64_t tt = up / RG;
                    mvalid = static_cast<int>((a.M - tt * NTOK) < NTOK ? (a.M - tt * NTOK) : NTOK);
                    const int db = static_cast<int>((j - 1) % C::kDBuf);
                    const uint32_t d_tm = tmem + lane_off + kNWG * kACols + (wg * C::kDBuf + db) * NTOK;
#pragma unroll
                    for (int c = 0; c < NTOK; c += 16) {
                        uint32_t d[16];
                        tmem_ld_32x32b_x16(d_tm + c, d);
                        tmem_ld_wait();
#pragma unroll
                        for (int m = 0; m < 16; ++m) acc[c + m] = fmaf(s_prev, __uint_as_float(d[m]), acc[c + m]);
                    }
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_dempty + 8 * (wg * C::kDBuf + db));
                    // tile finished?
                    const int64_t tile_next = (j < n) ? (u0 + j) / a.G : -1;
                    if (tile_next != tile_cur) {
                        const bool whole_tile = whole && ((up % a.G) == a.G - 1);
                        flush_tile<NTOK>(a, v, tile_cur, first_tile, whole_tile, acc, mvalid, r);
#pragma unroll
                        for (int m = 0; m < NTOK; ++m) acc[m] = 0.f;
                        tile_cur = tile_next;
                        whole = true;
                    }
                }
                s_prev = s_cur;
            }
            (void)mvalid;
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

template <int NTOK>
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

    cudaError_t e = cudaFuncSetAttribute(umma_kernel<NTOK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
    return cudaLaunchKernelEx(&cfg, umma_kernel<NTOK>, map, a);
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
    p.ws_bytes = kWorkspaceErr + counters + (size_t)2 * p.V * kTileRows * NTOK * sizeof(float);
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
    a.counters = reinterpret_cast<int*>(w + kWorkspaceErr);
    a.slots = reinterpret_cast<float*>(w + kWorkspaceErr +
                                       (size_t)ceil_div(plan.token_tiles * plan.R * 4 * 4, 256) * 256);
    switch (plan.ntok) {
        case 16: return launch_ntok<16>(X, ldx, a, plan, stream);
        case 32: return launch_ntok<32>(X, ldx, a, plan, stream);
        case 64: return launch_ntok<64>(X, ldx, a, plan, stream);
        default: return launch_ntok<128>(X, ldx, a, plan, stream);
    }
}

}  // namespace tern
