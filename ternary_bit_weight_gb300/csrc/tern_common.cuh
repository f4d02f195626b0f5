// Internal device helpers shared by libtern's kernels (sm_103a only).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "tern_internal.h"

namespace tern {

constexpr int kGroup = 128;            // weights per FP16 scale along K
constexpr int kTileRows = 128;         // rows per tile of the tiled layout
constexpr int kUnitCodeBytes = 4096;   // 128 rows x 128 weights x 2 bits
constexpr int kUnitScaleBytes = 256;   // 128 FP16 scales
constexpr int kUnitBytes = kUnitCodeBytes + kUnitScaleBytes;
constexpr int kUnitScaleBytesS8 = 128;   // 128 int8 scales (INT8-scale layout)

__host__ __device__ constexpr int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ constexpr int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

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

// ------------------------------------------------------ code decoding
//
// A tiled code word covers 16 consecutive weights of one row: weight k0+2i
// at bits 2i..2i+1, weight k0+2i+1 at bits 16+2i..17+2i, value v = t + 1.
// Pair i becomes one 32-bit register of two 16-bit floats (low half = the
// even weight).  With the word viewed unshifted (pairs 0-3) or shifted
// right by 8 (pairs 4-7), the pair's two fields sit at bit p = 2(i mod 4)
// of each half:
//   r = (w & (3 << p | 3 << 16+p)) | BASE
// where BASE holds, in both halves, the float 128.0 (bf16 0x4300) or
// 1024.0 (fp16 0x6400), whose low mantissa/exponent bits are clear.  The
// field adds v * 2^p * u to the value, u being its unit in the last place
// (bf16: u = 1, p <= 6: bit 7 is the exponent's lowest bit, and 128 + 128
// = 256 is exactly the doubled value, so the field v*64 stays linear;
// fp16: u = 1, p <= 6 sits inside the 10-bit mantissa).  So each half is
// exactly BASE + v * 2^p, and one two-way FMA, exact because every value
// involved fits the format's precision, gives
//   t = r * 2^-p - (BASE * 2^-p + 1) = v - 1.

//
// The four masks, the base and the FMA constants live in registers that the
// compiler cannot see through (an opaque move), and the mask-and-merge is an
// explicit LOP3: with the constants as immediates the compiler splits it
// into two integer operations, and the integer pipe is the decoder's limit.

__device__ __forceinline__ uint32_t opaque_reg(uint32_t v) {
    asm volatile("mov.b32 %0, %0;" : "+r"(v));
    return v;
}

struct DecodeConsts {
    uint32_t mask[4];   // fields of pair p = 2i in both halves
    uint32_t base;
    uint32_t mul[4];    // 2^-p in both halves
    uint32_t add[4];    // -(BASE * 2^-p + 1) in both halves
};

// bf16: BASE = 128.0 (0x4300)
__device__ __forceinline__ DecodeConsts decode_consts_bf16() {
    DecodeConsts k;
    const uint32_t mul[4] = {0x3F803F80u, 0x3E803E80u, 0x3D803D80u, 0x3C803C80u};
    const uint32_t add[4] = {0xC301C301u, 0xC204C204u, 0xC110C110u, 0xC040C040u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        k.mask[i] = opaque_reg(0x00030003u << (2 * i));
        k.mul[i] = opaque_reg(mul[i]);
        k.add[i] = opaque_reg(add[i]);
    }
    k.base = opaque_reg(0x43004300u);
    return k;
}

// fp16: BASE = 1024.0 (0x6400)
__device__ __forceinline__ DecodeConsts decode_consts_fp16() {
    DecodeConsts k;
    const uint32_t mul[4] = {0x3C003C00u, 0x34003400u, 0x2C002C00u, 0x24002400u};
    const uint32_t add[4] = {0xE401E401u, 0xDC04DC04u, 0xD410D410u, 0xCC40CC40u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        k.mask[i] = opaque_reg(0x00030003u << (2 * i));
        k.mul[i] = opaque_reg(mul[i]);
        k.add[i] = opaque_reg(add[i]);
    }
    k.base = opaque_reg(0x64006400u);
    return k;
}

__device__ __forceinline__ uint32_t merge_field(uint32_t w, uint32_t mask, uint32_t base) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "r"(mask), "r"(base));   // (w & mask) | base
    return r;
}

// All eight bf16x2 pairs of one code word: out[i] = (t[k0+2i], t[k0+2i+1]).
__device__ __forceinline__ void decode_word_bf16(uint32_t w, const DecodeConsts& k, uint32_t* out) {
    const uint32_t w8 = w >> 8;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t r = merge_field(h == 0 ? w : w8, k.mask[i], k.base);
            asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(out[4 * h + i]) : "r"(r), "r"(k.mul[i]), "r"(k.add[i]));
        }
    }
}

// All eight fp16x2 pairs of one code word, t exact in fp16 (for fp16
// activations).
__device__ __forceinline__ void decode_word_f16(uint32_t w, const DecodeConsts& k, uint32_t* out) {
    const uint32_t w8 = w >> 8;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t r = merge_field(h == 0 ? w : w8, k.mask[i], k.base);
            asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(out[4 * h + i]) : "r"(r), "r"(k.mul[i]), "r"(k.add[i]));
        }
    }
}

// fp16 variant: t as exact fp16 (+-1, 0), then times the row's FP16 scale
// s (given in both halves): t * s is exactly +-s or 0.
__device__ __forceinline__ void decode_word_fp16_scaled(uint32_t w, uint32_t s2, const DecodeConsts& k, uint32_t* out) {
    const uint32_t w8 = w >> 8;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t r = merge_field(h == 0 ? w : w8, k.mask[i], k.base);
            uint32_t t;
            asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(t) : "r"(r), "r"(k.mul[i]), "r"(k.add[i]));
            asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(out[4 * h + i]) : "r"(t), "r"(s2));
        }
    }
}

__device__ __forceinline__ float fp16_bits_to_float(uint32_t bits16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

// ------------------------------------------------------------- outputs

// Index of the output that holds row n of the concatenated N.
__device__ __forceinline__ int output_of(const OutputSplit& out, int64_t n) {
    int j = 0;
#pragma unroll
    for (int i = 1; i < kMaxOutputs; ++i) j += (i < out.n_out && n >= out.offset[i]);
    return j;
}

// Output row n of the concatenated N: address of element (m = 0, n) and the
// stride between tokens, so that a thread owning one row stores with one
// multiply-add per element.
struct RowOut {
    char* base;
    int64_t ld;
    int otype;   // 0 fp32, 1 bf16, 2 fp16
};
__device__ __forceinline__ RowOut row_out(const OutputSplit& out, int64_t n) {
    const int j = out.glu ? 0 : output_of(out, n);
    RowOut o;
    o.base = static_cast<char*>(out.y[j]) + (n - out.offset[j]) * (out.bf16 ? 2 : 4);
    o.ld = out.ldy[j];
    o.otype = out.bf16;
    return o;
}
__device__ __forceinline__ void store_elem(void* base, int64_t idx, int otype, float v) {
    if (otype == 1)
        static_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v);
    else if (otype == 2)
        static_cast<__half*>(base)[idx] = __float2half_rn(v);
    else
        static_cast<float*>(base)[idx] = v;
}
__device__ __forceinline__ void store_row(const RowOut& o, int m, float v) {
    store_elem(o.base, (int64_t)m * o.ld, o.otype, v);
}

// C final values v[0..C) of tokens m0 .. m0+C-1 of one output row, those
// below the token bound `mend` stored; the whole warp calls together, and
// the output form is decided once for the C stores instead of per element.
template <int C>
__device__ __forceinline__ void store_run(const OutputSplit& out, const RowOut& o, int m0, int mend, int64_t row,
                                          const float (&v)[C], bool live);

// Final value v of output (m, row), the row being lane (row mod 32) of the
// calling warp; every lane of the warp calls with the same m.  `live`: the
// row exists (row < N).  With the GLU layout the partner lane (lane ^ 16)
// holds the matching up (or gate) value, and the gate lane stores
// silu(gate) * up in fp32 at column 16*(row/32) + row%32.
__device__ __forceinline__ void store_out(const OutputSplit& out, const RowOut& o, int m, int64_t row, float v,
                                          bool live) {
    if (out.glu) {
        const float u = __shfl_xor_sync(0xffffffffu, v, 16);
        const int64_t i = (row >> 5) * 16 + (row & 15);
        if ((row & 16) == 0 && i < out.glu_cols) {
            const float h = v / (1.0f + expf(-v)) * u;
            store_elem(out.y[0], (int64_t)m * out.ldy[0] + i, out.bf16, h);
        }
    } else if (live) {
        store_row(o, m, v);
    }
}

template <int C>
__device__ __forceinline__ void store_run(const OutputSplit& out, const RowOut& o, int m0, int mend, int64_t row,
                                          const float (&v)[C], bool live) {
    if (out.glu) {
#pragma unroll
        for (int m = 0; m < C; ++m)
            if (m0 + m < mend) store_out(out, o, m0 + m, row, v[m], live);
        return;
    }
    if (!live) return;
    // streaming stores (evict first): the outputs are not read again here,
    // and L2 is better spent on weights and activation tiles
    if (o.otype == 0) {
        float* p = reinterpret_cast<float*>(o.base) + (int64_t)m0 * o.ld;
#pragma unroll
        for (int m = 0; m < C; ++m)
            if (m0 + m < mend) __stcs(p + (int64_t)m * o.ld, v[m]);
    } else {
        unsigned short* p = reinterpret_cast<unsigned short*>(o.base) + (int64_t)m0 * o.ld;
#pragma unroll
        for (int m = 0; m < C; ++m)
            if (m0 + m < mend) {
                const unsigned short b = o.otype == 1 ? __bfloat16_as_ushort(__float2bfloat16_rn(v[m]))
                                                      : __half_as_ushort(__float2half_rn(v[m]));
                asm volatile("st.global.cs.b16 [%0], %1;" ::"l"(p + (int64_t)m * o.ld), "h"(b) : "memory");
            }
    }
}

}  // namespace tern
