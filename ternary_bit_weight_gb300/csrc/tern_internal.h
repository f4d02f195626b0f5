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
cudaError_t launch_unrepack(const uint8_t* tiled, int64_t N, int64_t K, uint8_t* packed,
                            uint16_t* scales, int32_t* err, cudaStream_t stream);

// ---------------------------------------------------------- linear layer
constexpr int kMaxOutputs = 4;

struct OutputSplit {
    int n_out;
    int64_t offset[kMaxOutputs + 1];  // row offsets into the concatenated N
    float* y[kMaxOutputs];
    int64_t ldy[kMaxOutputs];
};

// Decode (small-M) plan.  kStream: persistent CTAs, X resident in shared
// memory, each warp streams a contiguous run of 16x128 blocks.  kSplit: one
// CTA per (128-row block, K range), X slice per CTA.
struct DecodePlan {
    enum Kind { kStream = 0, kSplit = 1 };
    Kind kind;
    int mt;            // n8 token tiles per MMA row tile (1: M<=8, 2: M<=16)
    int splits;        // S (kSplit)
    int64_t n_rb;      // 128-row blocks
    int64_t groups;    // K / 128
    int64_t max_gps;   // largest number of groups in one split
    int64_t grid;      // CTAs
    int64_t warps;     // working warps
    size_t smem;       // dynamic shared memory per CTA
    size_t ws_bytes;   // workspace: counters + partials
};

int device_sm_count();
DecodePlan plan_decode(int64_t M, int64_t N, int64_t K, int sm_count);

// Largest M the decode kernel handles in one launch.
constexpr int64_t kDecodeMaxM = 16;

cudaError_t launch_decode(const uint16_t* X, int64_t ldx, const uint8_t* tiled, int64_t M,
                          int64_t N, int64_t K, const OutputSplit& out, void* ws,
                          const DecodePlan& plan, cudaStream_t stream);

// Tensor-core (tcgen05) plan: token tiles of `ntok`, persistent CTAs whose
// decode warpgroups each stream a contiguous range of 128x128 units.
struct UmmaPlan {
    int ntok;              // tokens per tile (UMMA N): 16, 32, 64 or 128
    int64_t R;             // 128-row tiles
    int64_t G;             // groups per row
    int64_t token_tiles;
    int64_t U;             // units = token_tiles x R x G
    int64_t V;             // workers
    int64_t grid;          // CTAs
    size_t smem;           // dynamic shared memory per CTA
    size_t ws_bytes;       // workspace: error word, tile counters, partial slots
};

UmmaPlan plan_umma(int64_t M, int64_t N, int64_t K, int sm_count);

cudaError_t launch_umma(const uint16_t* X, int64_t ldx, const uint8_t* tiled, int64_t M, int64_t N,
                        int64_t K, const OutputSplit& out, void* ws, const UmmaPlan& plan,
                        cudaStream_t stream);

}  // namespace tern
