// tern_linear_noalloc: tern_linear for callers that cannot allocate device
// memory (no counterpart in the source pages).
//
// Some callers cannot call cudaMalloc: code that runs while a CUDA graph is
// being captured (allocation is not allowed there), or a plug-in whose
// device memory is owned by a host framework's allocator that it cannot
// reach.  For them this entry point supplies the layer's split-K scratch
// itself, from one file-scope device array of fixed size.  The array lives
// in every GPU that loads this library until the process exits.
//
// Set-up: the first call on a device, with that device current, looks up
// the array's device address (cudaGetSymbolAddress; the host-side symbol
// is only a stand-in and must never be handed to a kernel) and caches it.
// That first call may load the module, so make it before any stream
// capture.  Every later call reuses the cached address and allocates
// nothing: no cudaMalloc, no cudaFree, no allocating library routine.
//
// All calls share the one array: calls whose kernels may overlap on the GPU
// (different streams, or graphs replayed concurrently) race on it.  Each
// call clears the part it uses before its kernels run.

#include <mutex>

#include "tern.h"
#include "tern_common.cuh"
#include "tern_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;   // 16 MiB per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) uint8_t g_scratch[kScratchBytes];

std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once).
tern_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TERN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TERN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return TERN_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return TERN_OK;
}

}  // namespace

extern "C" tern_status tern_linear_noalloc(const uint16_t* d_X, int64_t ldx, const void* d_tiled,
                                           int64_t M, int64_t N, int64_t K, float* d_Y,
                                           int64_t ldy, void* stream) {
    if (M < 0 || N < 0 || K <= 0 || K % tern::kGroup != 0) return TERN_ERR_SHAPE;
    if (M == 0 || N == 0) return TERN_OK;
    // the argument checks of tern_linear, before anything is enqueued
    if (d_X == nullptr || d_tiled == nullptr || d_Y == nullptr) return TERN_ERR_NULL;
    if (ldx < K || ldy < N) return TERN_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(d_X) & 15) || ldx % 8 || (reinterpret_cast<uintptr_t>(d_tiled) & 15) ||
        (reinterpret_cast<uintptr_t>(d_Y) & 3))
        return TERN_ERR_ALIGN;
    const size_t need = tern_workspace_bytes(M, N, K);
    if (need > kScratchBytes) return TERN_ERR_SIZE;
    void* scratch = nullptr;
    if (need > 0) {
        const tern_status st = scratch_address(&scratch);
        if (st != TERN_OK) return st;
        // counters must start at zero; an earlier call may have left data
        if (cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return TERN_ERR_CUDA;
    }
    return tern_linear(d_X, ldx, d_tiled, M, N, K, d_Y, ldy, scratch, need, stream);
}
