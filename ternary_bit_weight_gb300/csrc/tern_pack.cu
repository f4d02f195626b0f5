// Byte-format kernels of libtern: pack, unpack, repack (disk -> tiled, also
// into the GLU-interleaved layout) and unrepack (tiled -> disk).  All are
// memory-bound single passes and bit-exact by construction: pack, unpack and
// unrepack with one thread per 32-bit output word, repack with one thread
// per (unit, row) so that its reads are whole DRAM sectors and its writes
// whole 512-byte runs per warp.  Every thread
// fences its writes before exiting, so that a following linear-layer kernel
// that starts early (programmatic dependent launch) and streams weights
// before its grid dependency resolves sees them.
//
// Packing rule ("Ternary embedding model in vLLM", 2kiu.com/news/5082861,
// §3.1): 2-bit codes 00 -> 0, 01 -> +1, 10 -> -1, 11 -> reserved read as 0;
// four codes per byte, first weight in the lowest two bits.  The tiled
// layout is the library's own (documented in include/tern.h).

#include "tern_common.cuh"
#include "tern_internal.h"

namespace tern {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void count_errors(int32_t* err, int bad) {
    if (err == nullptr) return;
    const unsigned active = __activemask();
    const int total = __reduce_add_sync(active, bad);
    if (total != 0 && (threadIdx.x & 31) == (__ffs(active) - 1)) atomicAdd(err, total);
}

// Code of one int8 ternary value; values outside {-1,0,+1} give 00 and count.
__device__ __forceinline__ uint32_t code_of(int8_t v, int& bad) {
    bad += (v < -1 || v > 1);
    return v == 1 ? 1u : (v == -1 ? 2u : 0u);
}

// One output word = 16 ternary values (one uint4 of int8) -> 4 packed bytes.
__global__ void __launch_bounds__(kThreads)
pack_words_kernel(const uint4* __restrict__ t, int64_t words, uint32_t* __restrict__ packed,
                  int32_t* err) {
    int bad = 0;
    for (int64_t i = blockIdx.x * (int64_t)kThreads + threadIdx.x; i < words;
         i += (int64_t)gridDim.x * kThreads) {
        const uint4 v = t[i];
        const uint32_t part[4] = {v.x, v.y, v.z, v.w};
        uint32_t out = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j)
            out |= code_of(static_cast<int8_t>(part[j >> 2] >> (8 * (j & 3))), bad) << (2 * j);
        packed[i] = out;
    }
    __threadfence();   // writes visible GPU-wide before exit (early-starting successors)
    count_errors(err, bad);
}

// Fallback for unaligned or ragged data: one packed byte per iteration.
__global__ void __launch_bounds__(kThreads)
pack_bytes_kernel(const int8_t* __restrict__ t, int64_t first_byte, int64_t bytes,
                  uint8_t* __restrict__ packed, int32_t* err) {
    int bad = 0;
    for (int64_t i = first_byte + blockIdx.x * (int64_t)kThreads + threadIdx.x; i < bytes;
         i += (int64_t)gridDim.x * kThreads) {
        uint32_t out = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) out |= code_of(t[4 * i + j], bad) << (2 * j);
        packed[i] = static_cast<uint8_t>(out);
    }
    __threadfence();   // writes visible GPU-wide before exit (early-starting successors)
    count_errors(err, bad);
}

__device__ __forceinline__ int8_t value_of(uint32_t code) {
    return code == 1u ? int8_t(1) : (code == 2u ? int8_t(-1) : int8_t(0));
}

// One packed word (16 codes) -> 16 int8 values.
__global__ void __launch_bounds__(kThreads)
unpack_words_kernel(const uint32_t* __restrict__ packed, int64_t words, uint4* __restrict__ t,
                    int32_t* err) {
    int bad = 0;
    for (int64_t i = blockIdx.x * (int64_t)kThreads + threadIdx.x; i < words;
         i += (int64_t)gridDim.x * kThreads) {
        const uint32_t w = packed[i];
        bad += __popc(w & (w >> 1) & 0x55555555u);   // code 11
        uint32_t part[4] = {0, 0, 0, 0};
#pragma unroll
        for (int j = 0; j < 16; ++j)
            part[j >> 2] |= (uint32_t)(uint8_t)value_of((w >> (2 * j)) & 3u) << (8 * (j & 3));
        t[i] = make_uint4(part[0], part[1], part[2], part[3]);
    }
    __threadfence();   // writes visible GPU-wide before exit (early-starting successors)
    count_errors(err, bad);
}

__global__ void __launch_bounds__(kThreads)
unpack_bytes_kernel(const uint8_t* __restrict__ packed, int64_t first_byte, int64_t bytes,
                    int8_t* __restrict__ t, int32_t* err) {
    int bad = 0;
    for (int64_t i = first_byte + blockIdx.x * (int64_t)kThreads + threadIdx.x; i < bytes;
         i += (int64_t)gridDim.x * kThreads) {
        const uint32_t b = packed[i];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t c = (b >> (2 * j)) & 3u;
            bad += (c == 3u);
            t[4 * i + j] = value_of(c);
        }
    }
    __threadfence();   // writes visible GPU-wide before exit (early-starting successors)
    count_errors(err, bad);
}

// Disk word (16 codes of weights k0..k0+15, code j at bits 2j) -> tiled word
// (biased v = t + 1, weight k0+2i at bits 2i, k0+2i+1 at bits 16+2i).
__device__ __forceinline__ uint32_t disk_to_tiled_word(uint32_t src, int& bad) {
    const uint32_t lo = src & 0x55555555u;          // code bit 0 of each field
    const uint32_t hi = (src >> 1) & 0x55555555u;   // code bit 1
    bad += __popc(lo & hi);
    // v = t + 1: code 01 (+1) -> 10, code 10 (-1) -> 00, codes 00/11 -> 01
    const uint32_t v_bit1 = lo & ~hi;
    const uint32_t v_bit0 = ~(lo ^ hi) & 0x55555555u;
    uint32_t v = v_bit0 | (v_bit1 << 1);
    // Field i (weight k0+i) moves to field (i mod 2)*8 + i/2: a rotation of
    // the four bits of the field index, done as three exchanges of adjacent
    // index bits (bits 0-1, 1-2, 2-3), each one masked swap of fields.
    auto swap_fields = [](uint32_t x, uint32_t mask, int shift) {
        const uint32_t t = ((x >> shift) ^ x) & mask;
        return x ^ t ^ (t << shift);
    };
    v = swap_fields(v, 0x0C0C0C0Cu, 2);
    v = swap_fields(v, 0x00F000F0u, 4);
    v = swap_fields(v, 0x0000FF00u, 8);
    return v;
}

// Tiled word -> disk word (inverse of the above; v = 3 gives code 00 and counts).
__device__ __forceinline__ uint32_t tiled_to_disk_word(uint32_t w, int& bad) {
    uint32_t out = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const uint32_t v = (w >> (16 * e + 2 * i)) & 3u;
            bad += (v == 3u);
            const uint32_t code = v == 0u ? 2u : (v == 2u ? 1u : 0u);
            out |= code << (2 * (2 * i + e));
        }
    }
    return out;
}

// Position of tiled code word `idx`: row n and first weight k0.
__device__ __forceinline__ void tiled_word_coords(int64_t idx, int64_t G, int64_t& n, int64_t& k0) {
    const int64_t unit = idx >> 10;            // 1024 words per 128x128 unit
    const int within = static_cast<int>(idx & 1023);
    const int h = within >> 9, r = (within >> 2) & 127, q = within & 3;
    const int64_t b = unit / G, g = unit - b * G;
    n = kTileRows * b + r;
    k0 = kGroup * g + 64 * h + 16 * q;
}

// Scale word `j` (two fp16 scales): rows n_lo, n_lo + 1 of group g.
__device__ __forceinline__ void tiled_scale_coords(int64_t j, int64_t G, int64_t& n_lo, int64_t& g) {
    const int64_t unit = j >> 6;               // 64 words per unit
    const int r2 = static_cast<int>(j & 63);
    const int64_t b = unit / G;
    g = unit - b * G;
    n_lo = kTileRows * b + 2 * r2;
}

// Where the tiled rows come from: row n of one source, or (GLU) blocks of
// 16 rows taken alternately from the gate and the up source, so that tiled
// row n is gate row 16*(n/32) + n%32 when n%32 < 16 and the up row of the
// same index otherwise.
struct RepackSrc {
    const uint8_t* packed[2];
    const uint16_t* scales[2];
    const int8_t* q8;   // s8: int8 scales [rows, G] and per-row factors [rows]
    const float* f;
    int64_t rows;   // rows per source
    int glu;
    int s8;
};

__device__ __forceinline__ bool source_row(const RepackSrc& s, int64_t n, int& which, int64_t& row) {
    if (!s.glu) {
        which = 0;
        row = n;
    } else {
        const int j = static_cast<int>(n & 31);
        which = j >> 4;
        row = (n >> 5) * 16 + (j & 15);
    }
    return row < s.rows;
}

// One thread per (row, run of up to kRunGroups groups): the row's disk bytes
// of those groups (contiguous, 32 per group) become the row's two 16-byte
// runs in each of the units (a warp of 32 rows writes 512 contiguous bytes
// per run), and its scales.  Reading a whole run per thread keeps the
// warp's reads in long contiguous pieces of each row.  VEC: the sources are
// 16-byte aligned, so each group's 32 bytes come in two vector loads.
constexpr int kRunGroups = 2;

__host__ __device__ constexpr int64_t repack_items(int64_t units, int64_t K) {
    return units / (K / kGroup) * kTileRows * ceil_div(K / kGroup, kRunGroups);
}

// One repack of a launch: a weight (or, GLU, a pair of them) into its
// tiled buffer; a launch serves up to kMaxGroup of them, their items one
// after another.
struct RepackJob {
    RepackSrc src;
    uint8_t* tiled;
    int64_t K;
    int64_t units;
    int64_t item_begin;
};
struct RepackJobs {
    RepackJob job[kMaxGroup];
    int count;
    int64_t items;
};

template <bool VEC>
__global__ void __launch_bounds__(kThreads)
repack_kernel(const RepackJobs jobs, int32_t* err) {
    int bad = 0;
    int p = 0;   // job of item i (items rise along the loop)
    for (int64_t i = blockIdx.x * (int64_t)kThreads + threadIdx.x; i < jobs.items;
         i += (int64_t)gridDim.x * kThreads) {
        while (p + 1 < jobs.count && i >= jobs.job[p + 1].item_begin) ++p;
        const RepackJob& J = jobs.job[p];
        const RepackSrc& src = J.src;
        const int64_t K = J.K, units = J.units;
        uint8_t* const tiled = J.tiled;
        const int64_t G = K / kGroup;
        const int64_t GB = ceil_div(G, kRunGroups);   // runs per row
        const int64_t row_bytes = K / 4;
        uint16_t* tscales = reinterpret_cast<uint16_t*>(tiled + units * kUnitCodeBytes);
        int8_t* tscales8 = reinterpret_cast<int8_t*>(tiled + units * kUnitCodeBytes);
        float* tfactor = reinterpret_cast<float*>(tiled + units * (kUnitCodeBytes + kUnitScaleBytesS8));
        const int64_t li = i - J.item_begin;
        const int r = static_cast<int>(li & 127);
        const int64_t tb = li >> 7;                   // (tile, run)
        const int64_t b = tb / GB, gb = tb - b * GB;
        const int64_t g0 = gb * kRunGroups;
        const int ng = static_cast<int>(G - g0 < kRunGroups ? G - g0 : kRunGroups);
        int which;
        int64_t row;
        const bool valid = source_row(src, b * kTileRows + r, which, row);
        uint32_t w[kRunGroups][8];
        uint16_t sc[kRunGroups];
#pragma unroll
        for (int q = 0; q < kRunGroups; ++q) {
            sc[q] = 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) w[q][e] = 0;   // padding rows: code 00, weight 0
        }
        if (valid) {
            const uint8_t* p = (which ? src.packed[1] : src.packed[0]) + row * row_bytes + 32 * g0;
            const uint16_t* sp = (which ? src.scales[1] : src.scales[0]) + row * G + g0;
#pragma unroll
            for (int q = 0; q < kRunGroups; ++q) {
                if (q < ng) {
                    if (VEC) {
                        const uint4 a = __ldg(reinterpret_cast<const uint4*>(p + 32 * q));
                        const uint4 c = __ldg(reinterpret_cast<const uint4*>(p + 32 * q) + 1);
                        w[q][0] = a.x; w[q][1] = a.y; w[q][2] = a.z; w[q][3] = a.w;
                        w[q][4] = c.x; w[q][5] = c.y; w[q][6] = c.z; w[q][7] = c.w;
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) w[q][e] = __ldg(reinterpret_cast<const uint32_t*>(p + 32 * q) + e);
                    }
                    if (!src.s8) sc[q] = __ldg(sp + q);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kRunGroups; ++q) {
            if (q < ng) {
                const int64_t unit = b * G + g0 + q;
                uint8_t* u = tiled + unit * kUnitCodeBytes + 16 * r;
                *reinterpret_cast<uint4*>(u) = make_uint4(disk_to_tiled_word(w[q][0], bad), disk_to_tiled_word(w[q][1], bad),
                                                          disk_to_tiled_word(w[q][2], bad), disk_to_tiled_word(w[q][3], bad));
                *reinterpret_cast<uint4*>(u + 2048) =
                    make_uint4(disk_to_tiled_word(w[q][4], bad), disk_to_tiled_word(w[q][5], bad),
                               disk_to_tiled_word(w[q][6], bad), disk_to_tiled_word(w[q][7], bad));
                if (src.s8) {
                    tscales8[unit * kTileRows + r] = valid ? src.q8[row * G + g0 + q] : int8_t(0);
                } else {
                    tscales[unit * kTileRows + r] = sc[q];
                }
            }
        }
        if (src.s8 && gb == 0) tfactor[b * kTileRows + r] = valid ? src.f[row] : 0.f;
    }
    __threadfence();   // writes visible GPU-wide before exit (early-starting successors)
    count_errors(err, bad);
}

__global__ void __launch_bounds__(kThreads)
unrepack_kernel(const uint32_t* __restrict__ tiled, int64_t N, int64_t K, int64_t code_words,
                int64_t scale_words, uint8_t* __restrict__ packed, uint16_t* __restrict__ scales,
                int32_t* err) {
    const int64_t G = K / kGroup;
    int bad = 0;
    for (int64_t i = blockIdx.x * (int64_t)kThreads + threadIdx.x; i < code_words + scale_words;
         i += (int64_t)gridDim.x * kThreads) {
        if (i < code_words) {
            int64_t n, k0;
            tiled_word_coords(i, G, n, k0);
            if (n < N) {
                const uint32_t w = tiled[i];
                *reinterpret_cast<uint32_t*>(packed + n * (K / 4) + k0 / 4) = tiled_to_disk_word(w, bad);
            }
        } else {
            int64_t n_lo, g;
            tiled_scale_coords(i - code_words, G, n_lo, g);
            const uint32_t w = tiled[i];
            if (n_lo < N) scales[n_lo * G + g] = static_cast<uint16_t>(w & 0xFFFFu);
            if (n_lo + 1 < N) scales[(n_lo + 1) * G + g] = static_cast<uint16_t>(w >> 16);
        }
    }
    __threadfence();   // writes visible GPU-wide before exit (early-starting successors)
    count_errors(err, bad);
}

template <typename Kernel, typename... Args>
cudaError_t launch_flat(Kernel kernel, int64_t items, cudaStream_t stream, Args... args) {
    if (items <= 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // grid-stride loops: enough blocks to fill every SM several times over
    const int64_t want = ceil_div(items, kThreads);
    const int64_t cap = (int64_t)sms * 32;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(want < cap ? want : cap));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// P repacks in one launch: source, tiled buffer, tiled rows and K of each.
cudaError_t launch_repack_jobs(const RepackSrc* srcs, uint8_t* const* tiled, const int64_t* rows, const int64_t* K,
                               int P, int32_t* err, cudaStream_t stream) {
    if (P < 1 || P > kMaxGroup) return cudaErrorInvalidValue;
    RepackJobs jobs = {};
    jobs.count = P;
    bool vec = true;
    int64_t items = 0;
    for (int i = 0; i < P; ++i) {
        RepackJob& J = jobs.job[i];
        J.src = srcs[i];
        J.tiled = tiled[i];
        J.K = K[i];
        J.units = ceil_div(rows[i], kTileRows) * (K[i] / kGroup);
        J.item_begin = items;
        items += repack_items(J.units, K[i]);
        vec = vec && ((reinterpret_cast<uintptr_t>(srcs[i].packed[0]) | reinterpret_cast<uintptr_t>(srcs[i].packed[1])) &
                      15) == 0;
    }
    jobs.items = items;
    return vec ? launch_flat(repack_kernel<true>, items, stream, jobs, err)
               : launch_flat(repack_kernel<false>, items, stream, jobs, err);
}

}  // namespace

cudaError_t launch_pack(const int8_t* t, int64_t count, uint8_t* packed, int32_t* err,
                        cudaStream_t stream) {
    const int64_t bytes = count / 4;
    int64_t words = 0;
    if ((reinterpret_cast<uintptr_t>(t) & 15) == 0 && (reinterpret_cast<uintptr_t>(packed) & 3) == 0)
        words = count / 16;
    cudaError_t e = launch_flat(pack_words_kernel, words, stream, reinterpret_cast<const uint4*>(t),
                                words, reinterpret_cast<uint32_t*>(packed), err);
    if (e != cudaSuccess) return e;
    return launch_flat(pack_bytes_kernel, bytes - 4 * words, stream, t, 4 * words, bytes, packed, err);
}

cudaError_t launch_unpack(const uint8_t* packed, int64_t count, int8_t* t, int32_t* err,
                          cudaStream_t stream) {
    const int64_t bytes = count / 4;
    int64_t words = 0;
    if ((reinterpret_cast<uintptr_t>(t) & 15) == 0 && (reinterpret_cast<uintptr_t>(packed) & 3) == 0)
        words = count / 16;
    cudaError_t e = launch_flat(unpack_words_kernel, words, stream,
                                reinterpret_cast<const uint32_t*>(packed), words,
                                reinterpret_cast<uint4*>(t), err);
    if (e != cudaSuccess) return e;
    return launch_flat(unpack_bytes_kernel, bytes - 4 * words, stream, packed, 4 * words, bytes, t, err);
}

cudaError_t launch_repack_grouped(const uint8_t* const* packed, const uint16_t* const* scales, const int64_t* N,
                                  const int64_t* K, uint8_t* const* tiled, int P, int32_t* err, cudaStream_t stream) {
    RepackSrc src[kMaxGroup] = {};
    if (P < 1 || P > kMaxGroup) return cudaErrorInvalidValue;
    for (int i = 0; i < P; ++i) {
        src[i].packed[0] = src[i].packed[1] = packed[i];
        src[i].scales[0] = src[i].scales[1] = scales[i];
        src[i].rows = N[i];
    }
    return launch_repack_jobs(src, tiled, N, K, P, err, stream);
}

cudaError_t launch_repack(const uint8_t* packed, const uint16_t* scales, int64_t N, int64_t K,
                          uint8_t* tiled, int32_t* err, cudaStream_t stream) {
    RepackSrc src = {};
    src.packed[0] = src.packed[1] = packed;
    src.scales[0] = src.scales[1] = scales;
    src.rows = N;
    src.glu = 0;
    return launch_repack_jobs(&src, &tiled, &N, &K, 1, err, stream);
}

// One warp per unit: 1024 code words, 32 per lane, one vote.
__global__ void __launch_bounds__(kThreads)
zero_units_kernel(const uint4* __restrict__ codes, int64_t units, uint8_t* __restrict__ flags) {
    const int lane = threadIdx.x & 31;
    for (int64_t u = (blockIdx.x * (int64_t)kThreads + threadIdx.x) >> 5; u < units;
         u += ((int64_t)gridDim.x * kThreads) >> 5) {
        const uint4* p = codes + u * (kUnitCodeBytes / 16);
        bool zero = true;
#pragma unroll
        for (int i = 0; i < kUnitCodeBytes / 16 / 32; ++i) {
            const uint4 v = __ldg(p + i * 32 + lane);
            zero = zero && v.x == 0x55555555u && v.y == 0x55555555u && v.z == 0x55555555u && v.w == 0x55555555u;
        }
        zero = __all_sync(0xffffffffu, zero);
        if (lane == 0) flags[u] = zero ? 1 : 0;
    }
    __threadfence();
}

cudaError_t launch_zero_units(const uint8_t* tiled, int64_t units, uint8_t* flags, cudaStream_t stream) {
    return launch_flat(zero_units_kernel, units * 32, stream, reinterpret_cast<const uint4*>(tiled), units, flags);
}

cudaError_t launch_repack_s8(const uint8_t* packed, const int8_t* q8, const float* f, int64_t N, int64_t K,
                             uint8_t* tiled, int32_t* err, cudaStream_t stream) {
    RepackSrc src = {};
    src.packed[0] = src.packed[1] = packed;
    src.q8 = q8;
    src.f = f;
    src.rows = N;
    src.s8 = 1;
    return launch_repack_jobs(&src, &tiled, &N, &K, 1, err, stream);
}

// FP16 scales -> int8 scales and per-row factors, in fp32 with ties to
// even: f = max_g |s| / 127, q = rint(s * (127 / max_g |s|)).
__global__ void __launch_bounds__(kThreads)
quantize_scales_kernel(const uint16_t* __restrict__ scales, int64_t N, int64_t G, int8_t* __restrict__ q8,
                       float* __restrict__ f) {
    for (int64_t n = blockIdx.x * (int64_t)kThreads + threadIdx.x; n < N; n += (int64_t)gridDim.x * kThreads) {
        float mx = 0.f;
        for (int64_t g = 0; g < G; ++g) mx = fmaxf(mx, fabsf(fp16_bits_to_float(scales[n * G + g])));
        const float inv = mx > 0.f ? 127.0f / mx : 0.f;
        f[n] = mx / 127.0f;
        for (int64_t g = 0; g < G; ++g) {
            float q = rintf(fp16_bits_to_float(scales[n * G + g]) * inv);
            q = fminf(fmaxf(q, -127.f), 127.f);
            q8[n * G + g] = static_cast<int8_t>(q);
        }
    }
    __threadfence();
}

cudaError_t launch_quantize_scales(const uint16_t* scales, int64_t N, int64_t K, int8_t* q8, float* f,
                                   cudaStream_t stream) {
    return launch_flat(quantize_scales_kernel, N, stream, scales, N, K / kGroup, q8, f);
}

cudaError_t launch_repack_glu(const uint8_t* packed_gate, const uint16_t* scales_gate, const uint8_t* packed_up,
                              const uint16_t* scales_up, int64_t I, int64_t K, uint8_t* tiled, int32_t* err,
                              cudaStream_t stream) {
    RepackSrc src = {};
    src.packed[0] = packed_gate;
    src.packed[1] = packed_up;
    src.scales[0] = scales_gate;
    src.scales[1] = scales_up;
    src.rows = I;
    src.glu = 1;
    const int64_t rows = glu_rows(I);
    return launch_repack_jobs(&src, &tiled, &rows, &K, 1, err, stream);
}

cudaError_t launch_unrepack(const uint8_t* tiled, int64_t N, int64_t K, uint8_t* packed,
                            uint16_t* scales, int32_t* err, cudaStream_t stream) {
    const int64_t R = ceil_div(N, kTileRows), G = K / kGroup;
    const int64_t code_words = R * G * (kUnitCodeBytes / 4);
    const int64_t scale_words = R * G * (kUnitScaleBytes / 4);
    return launch_flat(unrepack_kernel, code_words + scale_words, stream,
                       reinterpret_cast<const uint32_t*>(tiled), N, K, code_words, scale_words,
                       packed, scales, err);
}

}  // namespace tern
