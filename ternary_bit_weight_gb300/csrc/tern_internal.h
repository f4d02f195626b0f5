// Internal host-side interface between libtern's entry points (tern_api.cu)
// and its kernel launchers.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace tern {

// ------------------------------------------------------------ pack family
cudaError_t launch_pack(const int8_t* t, int64_t count, uint8_t* packed, int32_t* err,
                        cudaStream_t stream);
cudaError_t launch_unpack(const uint8_t* packed, int64_t count, int8_t* t, int32_t* err,
                          cudaStream_t stream);
cudaError_t launch_repack(const uint8_t* packed, const uint16_t* scales, int64_t N, int64_t K,
                          uint8_t* tiled, int32_t* err, cudaStream_t stream);
// P (<= kMaxGroup) independent repacks in one launch.
cudaError_t launch_repack_grouped(const uint8_t* const* packed, const uint16_t* const* scales, const int64_t* N,
                                  const int64_t* K, uint8_t* const* tiled, int P, int32_t* err, cudaStream_t stream);
// GLU layout: gate and up rows interleaved in blocks of 16 (tiled row n is
// gate row 16*(n/32) + n%32 when n%32 < 16, else the up row of that index);
// glu_rows(I) combined rows, padded with zero rows.
constexpr int64_t glu_rows(int64_t I) { return 2 * ((I + 15) / 16) * 16; }
cudaError_t launch_repack_glu(const uint8_t* packed_gate, const uint16_t* scales_gate, const uint8_t* packed_up,
                              const uint16_t* scales_up, int64_t I, int64_t K, uint8_t* tiled, int32_t* err,
                              cudaStream_t stream);
// INT8-scale layout: codes as the tiled layout, then per unit 128 int8
// scales, then per row tile 128 fp32 row factors.
cudaError_t launch_repack_s8(const uint8_t* packed, const int8_t* q8, const float* f, int64_t N, int64_t K,
                             uint8_t* tiled, int32_t* err, cudaStream_t stream);
cudaError_t launch_quantize_scales(const uint16_t* scales, int64_t N, int64_t K, int8_t* q8, float* f,
                                   cudaStream_t stream);
// Per unit of the tiled codes: 1 if every weight is zero (every code word
// holds the biased value 1 in all sixteen fields).
cudaError_t launch_zero_units(const uint8_t* tiled, int64_t units, uint8_t* flags, cudaStream_t stream);
cudaError_t launch_unrepack(const uint8_t* tiled, int64_t N, int64_t K, uint8_t* packed,
                            uint16_t* scales, int32_t* err, cudaStream_t stream);

// ---------------------------------------------------------- linear layer
constexpr int kMaxOutputs = 4;
// Largest group of independent problems (linears, repacks) one launch serves.
constexpr int kMaxGroup = 8;

// Where the rows of the concatenated N go: rows [offset[j], offset[j+1])
// to output j, element (m, n) at y[j][m * ldy[j] + n - offset[j]], stored as
// fp32, bf16 or fp16 (rounded to nearest even).
// glu != 0: the rows are the GLU interleave of gate and up (see glu_rows);
// the one output y[0] receives h[m, i] = silu(gate[m, i]) * up[m, i] for
// i < glu_cols at y[0][m * ldy[0] + i].
struct OutputSplit {
    int n_out;
    int bf16;      // 1: bf16 output, 2: fp16 output, 0: fp32
    int glu;
    int64_t glu_cols;
    int64_t offset[kMaxOutputs + 1];
    void* y[kMaxOutputs];
    int64_t ldy[kMaxOutputs];
};

int device_sm_count();

// Largest M served by the streaming (decode) kernel; larger M goes to the
// tensor-core GEMM kernel.
constexpr int64_t kStreamMaxM = 16;

// Streaming kernel plan (M <= 16): persistent CTAs, one per SM, whose
// decode workers each own a contiguous range of 128x128 weight units.
struct StreamPlan {
    bool one;              // M == 1: activation rows resident in shared memory
    int64_t x_smem;        // shared memory for them (the largest set one CTA needs)
    int64_t U;             // units of all problems
    int64_t tiles;         // 128-row tiles of all problems
    int64_t V;             // workers
    int64_t grid;          // CTAs
    int stages;            // shared-memory ring depth
    size_t smem;           // dynamic shared memory per CTA
    size_t ws_bytes;       // workspace: error word, tile counters, partial slots
};


// One linear of a streaming launch: Y = X . W^T with X [M, K] (row stride
// ldx), W in the tiled layout, N outputs rows.
struct StreamProblem {
    const uint16_t* x;
    int64_t ldx;
    const uint8_t* tiled;
    int64_t N;
    int64_t K;
    OutputSplit out;
};

StreamPlan plan_stream(int64_t M, const int64_t* N, const int64_t* K, int P, int sm_count);

// x_f16: X holds fp16 rather than bf16 bits.
// s8: the tiled weights carry int8 scales and per-row factors (INT8-scale layout).
// zflags (optional): per unit, 1 = all its weights are zero; such units are skipped.
// (s8 and zflags need P == 1.)
cudaError_t launch_stream(const StreamProblem* probs, int P, bool x_f16, bool s8, const uint8_t* zflags, int64_t M,
                          void* ws, const StreamPlan& plan, cudaStream_t stream);

// Tensor-core GEMM plan for M > kStreamMaxM: items of 256 weight rows x NT
// tokens x a range of groups along K, persistent CTAs.  One launch serves up
// to kMaxGroup independent linears with the same M (their items
// concatenated).
struct GemmPlan {
    int P;                          // problems
    int64_t T;                      // token tiles
    int NT;                         // tokens per tile
    int64_t R[kMaxGroup];           // 128-row tiles
    int64_t RP[kMaxGroup];          // pairs of row tiles
    int64_t G[kMaxGroup];           // groups along K
    int64_t KS[kMaxGroup];          // splits of K
    int64_t item_begin[kMaxGroup];  // items of the problems before
    int64_t items;
    int64_t grid;
    size_t off_x16[kMaxGroup], off_inv[kMaxGroup], off_partial[kMaxGroup];   // workspace layout
    size_t ws_bytes;
};

GemmPlan plan_gemm(int64_t M, const int64_t* N, const int64_t* K, int P, int sm_count);

// s8 and zflags need P == 1.
cudaError_t launch_gemm(const StreamProblem* probs, int P, bool x_f16, bool s8, const uint8_t* zflags, int64_t M,
                        void* ws, const GemmPlan& plan, cudaStream_t stream);

// int8-activation variant: quantised activations in the code words' field
// order, one CTA per (row tile, K split).
struct I8Plan {
    int64_t R, G, KS;
    size_t ws_bytes;
};
size_t i8_xq_bytes(int64_t M, int64_t K);
I8Plan plan_i8(int64_t M, int64_t N, int64_t K, int sm_count);
cudaError_t launch_quantize_x(const uint16_t* X, bool x_f16, int64_t ldx, int64_t M, int64_t K, int8_t* xq, float* a,
                              cudaStream_t stream);
cudaError_t launch_i8(const int8_t* xq, const float* a, const uint8_t* tiled, int64_t M, int64_t N,
                      const OutputSplit& out, void* ws, const I8Plan& plan, cudaStream_t stream);

// Size of the error word + padding at the start of every linear workspace.
constexpr size_t kWorkspaceErrBytes = 256;

}  // namespace tern
