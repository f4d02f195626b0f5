// Internal device helpers shared by libtern's kernels (sm_103a only).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace tern {

constexpr int kGroup = 128;            // weights per FP16 scale along K
constexpr int kTileRows = 128;         // rows per tile of the tiled layout
constexpr int kUnitCodeBytes = 4096;   // 128 rows x 128 weights x 2 bits
constexpr int kUnitScaleBytes = 256;   // 128 FP16 scales

__host__ __device__ constexpr int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------- loads

// Loads of data read exactly once (weights): cache-streaming (evict-first).
// Plain load intrinsics let the compiler schedule them as loads (issued as
// early as the prefetch ring allows), which opaque asm would not.
__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
    return __ldcs(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ uint32_t ldg_stream_u32(const void* p) {
    return __ldcs(reinterpret_cast<const unsigned int*>(p));
}

__device__ __forceinline__ uint4 lds_v4(const void* smem_ptr) {
    return *reinterpret_cast<const uint4*>(smem_ptr);
}

// ------------------------------------------------- programmatic launch

// Block until the grids this one depends on have completed and their
// memory is visible (no-op when launched without programmatic dependence).
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Allow the next grid on the stream to be scheduled once every block of
// this grid has called this (or exited).
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;");
}

// ------------------------------------------------------- tensor cores

// D += A(16x16 bf16, row) * B(16x8 bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma_bf16_m16n8k16(float (&d)[4], uint32_t a0, uint32_t a1,
                                                  uint32_t a2, uint32_t a3, uint32_t b0,
                                                  uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Same with C = 0 (the first MMA of a chain): no register zeroing needed.
__device__ __forceinline__ void mma_bf16_m16n8k16_zc(float (&d)[4], uint32_t a0, uint32_t a1,
                                                     uint32_t a2, uint32_t a3, uint32_t b0,
                                                     uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// ------------------------------------------------------ code decoding
//
// A tiled code word covers 16 consecutive weights of one row: weight k0+2i
// at bits 2i..2i+1, weight k0+2i+1 at bits 16+2i..17+2i, value v = t + 1.
// Pair i becomes one bf16x2 register (low half = the even weight):
//   r = (w >> s) & (3 << p | 3 << 16+p) | bf16x2(128, 128)
// puts v * 2^p into the mantissa of 128.0 in both halves, so each half is
// exactly 128 + v*2^p; then one bf16x2 FMA, exact because every value
// involved fits in 8 significant bits:
//   t = r * 2^-p - (128 * 2^-p + 1) = v - 1.
// Bit positions p = 0, 2, 4 of the 7-bit mantissa hold three pairs, so a
// word is read at shifts 0, 6 and 12.

template <int P>
__device__ __forceinline__ uint32_t decode_pair(uint32_t w) {
    // bf16x2 bit patterns: 2^-p and -(128 * 2^-p + 1) in both halves
    constexpr uint32_t kMul = P == 0 ? 0x3F803F80u : (P == 2 ? 0x3E803E80u : 0x3D803D80u);
    constexpr uint32_t kAdd = P == 0 ? 0xC301C301u : (P == 2 ? 0xC204C204u : 0xC110C110u);
    const uint32_t r = (w & (0x00030003u << P)) | 0x43004300u;
    uint32_t out;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(out) : "r"(r), "r"(kMul), "r"(kAdd));
    return out;
}

// All eight bf16x2 pairs of one code word: out[i] = (t[k0+2i], t[k0+2i+1]).
__device__ __forceinline__ void decode_word(uint32_t w, uint32_t (&out)[8]) {
    const uint32_t w6 = w >> 6, w12 = w >> 12;
    out[0] = decode_pair<0>(w);
    out[1] = decode_pair<2>(w);
    out[2] = decode_pair<4>(w);
    out[3] = decode_pair<0>(w6);
    out[4] = decode_pair<2>(w6);
    out[5] = decode_pair<4>(w6);
    out[6] = decode_pair<0>(w12);
    out[7] = decode_pair<2>(w12);
}

__device__ __forceinline__ float fp16_bits_to_float(uint32_t bits16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

}  // namespace tern
