// Host entry points of libtern (the C ABI declared in include/tern.h):
// argument checks, kernel selection and launches.  Nothing here allocates
// memory or keeps state between calls.

#include "tern.h"
#include "tern_common.cuh"
#include "tern_internal.h"

static_assert(tern::kMaxGroup == TERN_MAX_GROUP, "group size limit of the C ABI");

namespace {

using tern::ceil_div;

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

inline tern_status from_cuda(cudaError_t e) { return e == cudaSuccess ? TERN_OK : TERN_ERR_CUDA; }

inline bool valid_group_shape(int64_t N, int64_t K) { return N >= 0 && K > 0 && K % tern::kGroup == 0; }

tern_status run_linear(const uint16_t* X, bool x_f16, int64_t ldx, const void* tiled, int64_t M, int64_t N,
                       int64_t K, const tern::OutputSplit& out, void* ws, size_t ws_bytes,
                       cudaStream_t stream, bool s8 = false, const uint8_t* zflags = nullptr) {
    const int sms = tern::device_sm_count();
    if (sms <= 0) return TERN_ERR_UNSUPPORTED;
    if (ws == nullptr) return TERN_ERR_NULL;
    if (!aligned(ws, 256)) return TERN_ERR_ALIGN;
    const uint8_t* w = static_cast<const uint8_t*>(tiled);
    cudaError_t e;
    if (M <= tern::kStreamMaxM) {
        const tern::StreamPlan plan = tern::plan_stream(M, &N, &K, 1, sms);
        if (ws_bytes < plan.ws_bytes) return TERN_ERR_SIZE;
        tern::StreamProblem prob = {X, ldx, w, N, K, out};
        e = tern::launch_stream(&prob, 1, x_f16, s8, zflags, M, ws, plan, stream);
    } else {
        const tern::GemmPlan plan = tern::plan_gemm(M, &N, &K, 1, sms);
        if (ws_bytes < plan.ws_bytes) return TERN_ERR_SIZE;
        tern::StreamProblem prob = {X, ldx, w, N, K, out};
        e = tern::launch_gemm(&prob, 1, x_f16, s8, zflags, M, ws, plan, stream);
    }
    return e == cudaSuccess ? TERN_OK : TERN_ERR_CUDA;
}

size_t workspace_bytes(int64_t M, int64_t N, int64_t K) {
    const int sms = tern::device_sm_count();
    if (M <= tern::kStreamMaxM) return tern::plan_stream(M, &N, &K, 1, sms).ws_bytes;
    return tern::plan_gemm(M, &N, &K, 1, sms).ws_bytes;
}

tern_status check_x_w(const uint16_t* X, int64_t ldx, const void* tiled, int64_t M, int64_t K) {
    if (X == nullptr || tiled == nullptr) return TERN_ERR_NULL;
    if (ldx < K) return TERN_ERR_SHAPE;
    if (M > (int64_t(1) << 30)) return TERN_ERR_SHAPE;
    if (!aligned(X, 16) || ldx % 8 != 0) return TERN_ERR_ALIGN;
    if (!aligned(tiled, 16)) return TERN_ERR_ALIGN;
    return TERN_OK;
}

}  // namespace

namespace tern {

int device_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

}  // namespace tern

extern "C" {

const char* tern_status_string(int status) {
    switch (status) {
        case TERN_OK: return "TERN_OK";
        case TERN_ERR_NULL: return "TERN_ERR_NULL: a required pointer is NULL";
        case TERN_ERR_SHAPE: return "TERN_ERR_SHAPE: invalid dimension or leading dimension";
        case TERN_ERR_ALIGN: return "TERN_ERR_ALIGN: pointer or leading dimension misaligned";
        case TERN_ERR_SIZE: return "TERN_ERR_SIZE: buffer too small";
        case TERN_ERR_UNSUPPORTED: return "TERN_ERR_UNSUPPORTED: request not supported on this device";
        case TERN_ERR_CUDA: return "TERN_ERR_CUDA: CUDA call or kernel launch failed";
        default: return "TERN_ERR_UNKNOWN";
    }
}

int tern_version(void) { return 10100; }

tern_status tern_pack(const int8_t* d_t, int64_t N, int64_t K, uint8_t* d_packed, int32_t* d_err,
                      void* stream) {
    if (N < 0 || K < 0 || K % 4 != 0) return TERN_ERR_SHAPE;
    if (N == 0 || K == 0) return TERN_OK;
    if (d_t == nullptr || d_packed == nullptr) return TERN_ERR_NULL;
    if (d_err != nullptr && !aligned(d_err, 4)) return TERN_ERR_ALIGN;
    return from_cuda(tern::launch_pack(d_t, N * K, d_packed, d_err, as_stream(stream)));
}

tern_status tern_unpack(const uint8_t* d_packed, int64_t N, int64_t K, int8_t* d_t, int32_t* d_err,
                        void* stream) {
    if (N < 0 || K < 0 || K % 4 != 0) return TERN_ERR_SHAPE;
    if (N == 0 || K == 0) return TERN_OK;
    if (d_t == nullptr || d_packed == nullptr) return TERN_ERR_NULL;
    if (d_err != nullptr && !aligned(d_err, 4)) return TERN_ERR_ALIGN;
    return from_cuda(tern::launch_unpack(d_packed, N * K, d_t, d_err, as_stream(stream)));
}

size_t tern_tiled_bytes(int64_t N, int64_t K) {
    if (!valid_group_shape(N, K)) return 0;
    return (size_t)ceil_div(N, tern::kTileRows) * (size_t)(K / tern::kGroup) *
           (size_t)(tern::kUnitCodeBytes + tern::kUnitScaleBytes);
}

tern_status tern_repack(const uint8_t* d_packed, const uint16_t* d_scales, int64_t N, int64_t K,
                        void* d_tiled, size_t tiled_bytes, int32_t* d_err, void* stream) {
    if (!valid_group_shape(N, K)) return TERN_ERR_SHAPE;
    if (N == 0) return TERN_OK;
    if (d_packed == nullptr || d_scales == nullptr || d_tiled == nullptr) return TERN_ERR_NULL;
    if (!aligned(d_packed, 4) || !aligned(d_scales, 2) || !aligned(d_tiled, 16)) return TERN_ERR_ALIGN;
    if (d_err != nullptr && !aligned(d_err, 4)) return TERN_ERR_ALIGN;
    if (tiled_bytes < tern_tiled_bytes(N, K)) return TERN_ERR_SIZE;
    return from_cuda(tern::launch_repack(d_packed, d_scales, N, K, static_cast<uint8_t*>(d_tiled),
                                         d_err, as_stream(stream)));
}

tern_status tern_repack_grouped(int count, const uint8_t* const* d_packed, const uint16_t* const* d_scales,
                                const int64_t* Ns, const int64_t* Ks, void* const* d_tiled,
                                const size_t* tiled_bytes, int32_t* d_err, void* stream) {
    if (count < 1 || count > tern::kMaxGroup) return TERN_ERR_SHAPE;
    if (d_packed == nullptr || d_scales == nullptr || Ns == nullptr || Ks == nullptr || d_tiled == nullptr ||
        tiled_bytes == nullptr)
        return TERN_ERR_NULL;
    if (d_err != nullptr && !aligned(d_err, 4)) return TERN_ERR_ALIGN;
    const uint8_t* packed[tern::kMaxGroup];
    const uint16_t* scales[tern::kMaxGroup];
    int64_t n[tern::kMaxGroup], k[tern::kMaxGroup];
    uint8_t* tiled[tern::kMaxGroup];
    int P = 0;
    for (int i = 0; i < count; ++i) {
        if (!valid_group_shape(Ns[i], Ks[i])) return TERN_ERR_SHAPE;
        if (Ns[i] == 0) continue;
        if (d_packed[i] == nullptr || d_scales[i] == nullptr || d_tiled[i] == nullptr) return TERN_ERR_NULL;
        if (!aligned(d_packed[i], 4) || !aligned(d_scales[i], 2) || !aligned(d_tiled[i], 16)) return TERN_ERR_ALIGN;
        if (tiled_bytes[i] < tern_tiled_bytes(Ns[i], Ks[i])) return TERN_ERR_SIZE;
        packed[P] = d_packed[i];
        scales[P] = d_scales[i];
        n[P] = Ns[i];
        k[P] = Ks[i];
        tiled[P] = static_cast<uint8_t*>(d_tiled[i]);
        ++P;
    }
    if (P == 0) return TERN_OK;
    return from_cuda(tern::launch_repack_grouped(packed, scales, n, k, tiled, P, d_err, as_stream(stream)));
}

tern_status tern_unrepack(const void* d_tiled, int64_t N, int64_t K, uint8_t* d_packed,
                          uint16_t* d_scales, int32_t* d_err, void* stream) {
    if (!valid_group_shape(N, K)) return TERN_ERR_SHAPE;
    if (N == 0) return TERN_OK;
    if (d_packed == nullptr || d_scales == nullptr || d_tiled == nullptr) return TERN_ERR_NULL;
    if (!aligned(d_packed, 4) || !aligned(d_scales, 2) || !aligned(d_tiled, 16)) return TERN_ERR_ALIGN;
    if (d_err != nullptr && !aligned(d_err, 4)) return TERN_ERR_ALIGN;
    return from_cuda(tern::launch_unrepack(static_cast<const uint8_t*>(d_tiled), N, K, d_packed,
                                           d_scales, d_err, as_stream(stream)));
}

size_t tern_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || !valid_group_shape(N, K) || N == 0) return 0;
    return workspace_bytes(M, N, K);
}

tern_status tern_linear(const uint16_t* d_X, int64_t ldx, const void* d_tiled, int64_t M, int64_t N,
                        int64_t K, float* d_Y, int64_t ldy, void* d_ws, size_t ws_bytes,
                        void* stream) {
    if (M < 0 || !valid_group_shape(N, K)) return TERN_ERR_SHAPE;
    if (M == 0 || N == 0) return TERN_OK;
    tern_status st = check_x_w(d_X, ldx, d_tiled, M, K);
    if (st != TERN_OK) return st;
    if (d_Y == nullptr) return TERN_ERR_NULL;
    if (ldy < N) return TERN_ERR_SHAPE;
    if (!aligned(d_Y, 4)) return TERN_ERR_ALIGN;
    tern::OutputSplit out = {};
    out.n_out = 1;
    out.offset[0] = 0;
    out.offset[1] = N;
    out.y[0] = d_Y;
    out.ldy[0] = ldy;
    return run_linear(d_X, false, ldx, d_tiled, M, N, K, out, d_ws, ws_bytes, as_stream(stream));
}

tern_status tern_linear_multi(const uint16_t* d_X, int64_t ldx, const void* d_tiled, int64_t M,
                              int64_t K, int n_out, const int64_t* n_sizes, float* const* d_Ys,
                              const int64_t* ldys, void* d_ws, size_t ws_bytes, void* stream) {
    return tern_linear_ex(d_X, TERN_X_BF16, ldx, d_tiled, M, K, n_out, n_sizes,
                          reinterpret_cast<void* const*>(d_Ys), ldys, TERN_OUT_F32, d_ws, ws_bytes, stream);
}

static tern_status linear_ex(const void* d_X, int x_type, int64_t ldx, const void* d_tiled, int64_t M,
                             int64_t K, int n_out, const int64_t* n_sizes, void* const* d_Ys,
                             const int64_t* ldys, int out_type, void* d_ws, size_t ws_bytes, void* stream,
                             bool s8, const uint8_t* zflags = nullptr) {
    if (x_type != TERN_X_BF16 && x_type != TERN_X_F16) return TERN_ERR_SHAPE;
    if (out_type != TERN_OUT_F32 && out_type != TERN_OUT_BF16 && out_type != TERN_OUT_F16) return TERN_ERR_SHAPE;
    if (n_out < 1 || n_out > tern::kMaxOutputs) return TERN_ERR_SHAPE;
    if (n_sizes == nullptr || d_Ys == nullptr || ldys == nullptr) return TERN_ERR_NULL;
    tern::OutputSplit out = {};
    out.n_out = n_out;
    out.bf16 = out_type == TERN_OUT_BF16 ? 1 : out_type == TERN_OUT_F16 ? 2 : 0;
    const uintptr_t y_align = out.bf16 ? 2 : 4;
    int64_t N = 0;
    for (int j = 0; j < n_out; ++j) {
        if (n_sizes[j] < 0) return TERN_ERR_SHAPE;
        out.offset[j] = N;
        N += n_sizes[j];
    }
    for (int j = n_out; j <= tern::kMaxOutputs; ++j) out.offset[j] = N;
    if (M < 0 || !valid_group_shape(N, K)) return TERN_ERR_SHAPE;
    if (M == 0 || N == 0) return TERN_OK;
    const uint16_t* X = static_cast<const uint16_t*>(d_X);
    tern_status st = check_x_w(X, ldx, d_tiled, M, K);
    if (st != TERN_OK) return st;
    for (int j = 0; j < n_out; ++j) {
        if (n_sizes[j] == 0) { out.y[j] = nullptr; out.ldy[j] = 0; continue; }
        if (d_Ys[j] == nullptr) return TERN_ERR_NULL;
        if (ldys[j] < n_sizes[j]) return TERN_ERR_SHAPE;
        if (!aligned(d_Ys[j], y_align)) return TERN_ERR_ALIGN;
        out.y[j] = d_Ys[j];
        out.ldy[j] = ldys[j];
    }
    return run_linear(X, x_type == TERN_X_F16, ldx, d_tiled, M, N, K, out, d_ws, ws_bytes, as_stream(stream), s8,
                      zflags);
}

tern_status tern_linear_ex(const void* d_X, int x_type, int64_t ldx, const void* d_tiled, int64_t M,
                           int64_t K, int n_out, const int64_t* n_sizes, void* const* d_Ys,
                           const int64_t* ldys, int out_type, void* d_ws, size_t ws_bytes, void* stream) {
    return linear_ex(d_X, x_type, ldx, d_tiled, M, K, n_out, n_sizes, d_Ys, ldys, out_type, d_ws, ws_bytes, stream,
                     false);
}

size_t tern_grouped_workspace_bytes(int64_t M, int count, const int64_t* Ns, const int64_t* Ks) {
    if (M <= 0 || count < 1 || count > tern::kMaxGroup || Ns == nullptr || Ks == nullptr) return 0;
    int64_t n[tern::kMaxGroup], k[tern::kMaxGroup];
    int P = 0;
    for (int i = 0; i < count; ++i) {
        if (!valid_group_shape(Ns[i], Ks[i])) return 0;
        if (Ns[i] == 0) continue;
        n[P] = Ns[i];
        k[P] = Ks[i];
        ++P;
    }
    if (P == 0) return 256;
    if (M > tern::kStreamMaxM) return tern::plan_gemm(M, n, k, P, tern::device_sm_count()).ws_bytes;
    return tern::plan_stream(M, n, k, P, tern::device_sm_count()).ws_bytes;
}

tern_status tern_linear_grouped(int x_type, int64_t M, int count, const void* const* d_Xs, const int64_t* ldxs,
                                const void* const* d_tiled, const int64_t* Ns, const int64_t* Ks,
                                void* const* d_Ys, const int64_t* ldys, int out_type, void* d_ws,
                                size_t ws_bytes, void* stream) {
    if (x_type != TERN_X_BF16 && x_type != TERN_X_F16) return TERN_ERR_SHAPE;
    if (out_type != TERN_OUT_F32 && out_type != TERN_OUT_BF16 && out_type != TERN_OUT_F16) return TERN_ERR_SHAPE;
    if (count < 1 || count > tern::kMaxGroup || M < 0) return TERN_ERR_SHAPE;
    if (d_Xs == nullptr || ldxs == nullptr || d_tiled == nullptr || Ns == nullptr || Ks == nullptr ||
        d_Ys == nullptr || ldys == nullptr)
        return TERN_ERR_NULL;
    tern::StreamProblem probs[tern::kMaxGroup];
    int64_t n[tern::kMaxGroup], k[tern::kMaxGroup];
    int P = 0;
    const int bf16 = out_type == TERN_OUT_BF16 ? 1 : out_type == TERN_OUT_F16 ? 2 : 0;
    for (int i = 0; i < count; ++i) {
        if (!valid_group_shape(Ns[i], Ks[i])) return TERN_ERR_SHAPE;
        if (Ns[i] == 0 || M == 0) continue;
        const uint16_t* X = static_cast<const uint16_t*>(d_Xs[i]);
        tern_status st = check_x_w(X, ldxs[i], d_tiled[i], M, Ks[i]);
        if (st != TERN_OK) return st;
        if (d_Ys[i] == nullptr) return TERN_ERR_NULL;
        if (ldys[i] < Ns[i]) return TERN_ERR_SHAPE;
        if (!aligned(d_Ys[i], bf16 ? 2 : 4)) return TERN_ERR_ALIGN;
        tern::OutputSplit out = {};
        out.n_out = 1;
        out.bf16 = bf16;
        out.offset[0] = 0;
        for (int j = 1; j <= tern::kMaxOutputs; ++j) out.offset[j] = Ns[i];
        out.y[0] = d_Ys[i];
        out.ldy[0] = ldys[i];
        probs[P] = {X, ldxs[i], static_cast<const uint8_t*>(d_tiled[i]), Ns[i], Ks[i], out};
        n[P] = Ns[i];
        k[P] = Ks[i];
        ++P;
    }
    if (P == 0) return TERN_OK;
    const int sms = tern::device_sm_count();
    if (sms <= 0) return TERN_ERR_UNSUPPORTED;
    if (d_ws == nullptr) return TERN_ERR_NULL;
    if (!aligned(d_ws, 256)) return TERN_ERR_ALIGN;
    if (M > tern::kStreamMaxM) {
        const tern::GemmPlan plan = tern::plan_gemm(M, n, k, P, sms);
        if (ws_bytes < plan.ws_bytes) return TERN_ERR_SIZE;
        return from_cuda(tern::launch_gemm(probs, P, x_type == TERN_X_F16, false, nullptr, M, d_ws, plan,
                                           as_stream(stream)));
    }
    const tern::StreamPlan plan = tern::plan_stream(M, n, k, P, sms);
    if (ws_bytes < plan.ws_bytes) return TERN_ERR_SIZE;
    return from_cuda(tern::launch_stream(probs, P, x_type == TERN_X_F16, false, nullptr, M, d_ws, plan,
                                         as_stream(stream)));
}

size_t tern_unit_count(int64_t N, int64_t K) {
    if (!valid_group_shape(N, K)) return 0;
    return (size_t)ceil_div(N, tern::kTileRows) * (size_t)(K / tern::kGroup);
}

tern_status tern_zero_units(const void* d_tiled, int64_t N, int64_t K, uint8_t* d_flags, void* stream) {
    if (!valid_group_shape(N, K)) return TERN_ERR_SHAPE;
    if (N == 0) return TERN_OK;
    if (d_tiled == nullptr || d_flags == nullptr) return TERN_ERR_NULL;
    if (!aligned(d_tiled, 16)) return TERN_ERR_ALIGN;
    return from_cuda(tern::launch_zero_units(static_cast<const uint8_t*>(d_tiled), (int64_t)tern_unit_count(N, K),
                                             d_flags, as_stream(stream)));
}

tern_status tern_linear_sparse(const void* d_X, int x_type, int64_t ldx, const void* d_tiled,
                               const uint8_t* d_flags, int64_t M, int64_t K, int n_out, const int64_t* n_sizes,
                               void* const* d_Ys, const int64_t* ldys, int out_type, void* d_ws, size_t ws_bytes,
                               void* stream) {
    if (d_flags == nullptr) return TERN_ERR_NULL;
    return linear_ex(d_X, x_type, ldx, d_tiled, M, K, n_out, n_sizes, d_Ys, ldys, out_type, d_ws, ws_bytes, stream,
                     false, d_flags);
}

size_t tern_tiled_s8_bytes(int64_t N, int64_t K) {
    if (!valid_group_shape(N, K)) return 0;
    const size_t R = (size_t)ceil_div(N, tern::kTileRows), G = (size_t)(K / tern::kGroup);
    return R * G * (size_t)(tern::kUnitCodeBytes + tern::kUnitScaleBytesS8) + R * tern::kTileRows * sizeof(float);
}

tern_status tern_quantize_scales(const uint16_t* d_scales, int64_t N, int64_t K, int8_t* d_q8, float* d_f,
                                 void* stream) {
    if (!valid_group_shape(N, K)) return TERN_ERR_SHAPE;
    if (N == 0) return TERN_OK;
    if (d_scales == nullptr || d_q8 == nullptr || d_f == nullptr) return TERN_ERR_NULL;
    if (!aligned(d_scales, 2) || !aligned(d_f, 4)) return TERN_ERR_ALIGN;
    return from_cuda(tern::launch_quantize_scales(d_scales, N, K, d_q8, d_f, as_stream(stream)));
}

tern_status tern_repack_s8(const uint8_t* d_packed, const int8_t* d_q8, const float* d_f, int64_t N, int64_t K,
                           void* d_tiled, size_t tiled_bytes, int32_t* d_err, void* stream) {
    if (!valid_group_shape(N, K)) return TERN_ERR_SHAPE;
    if (N == 0) return TERN_OK;
    if (d_packed == nullptr || d_q8 == nullptr || d_f == nullptr || d_tiled == nullptr) return TERN_ERR_NULL;
    if (!aligned(d_packed, 4) || !aligned(d_f, 4) || !aligned(d_tiled, 16)) return TERN_ERR_ALIGN;
    if (d_err != nullptr && !aligned(d_err, 4)) return TERN_ERR_ALIGN;
    if (tiled_bytes < tern_tiled_s8_bytes(N, K)) return TERN_ERR_SIZE;
    return from_cuda(tern::launch_repack_s8(d_packed, d_q8, d_f, N, K, static_cast<uint8_t*>(d_tiled), d_err,
                                            as_stream(stream)));
}

tern_status tern_linear_s8(const void* d_X, int x_type, int64_t ldx, const void* d_tiled_s8, int64_t M,
                           int64_t K, int n_out, const int64_t* n_sizes, void* const* d_Ys,
                           const int64_t* ldys, int out_type, void* d_ws, size_t ws_bytes, void* stream) {
    return linear_ex(d_X, x_type, ldx, d_tiled_s8, M, K, n_out, n_sizes, d_Ys, ldys, out_type, d_ws, ws_bytes,
                     stream, true);
}

size_t tern_tiled_glu_bytes(int64_t I, int64_t K) {
    if (I < 0) return 0;
    return tern_tiled_bytes(tern::glu_rows(I), K);
}

tern_status tern_repack_glu(const uint8_t* d_packed_gate, const uint16_t* d_scales_gate,
                            const uint8_t* d_packed_up, const uint16_t* d_scales_up, int64_t I, int64_t K,
                            void* d_tiled, size_t tiled_bytes, int32_t* d_err, void* stream) {
    if (!valid_group_shape(I, K)) return TERN_ERR_SHAPE;
    if (I == 0) return TERN_OK;
    if (d_packed_gate == nullptr || d_scales_gate == nullptr || d_packed_up == nullptr ||
        d_scales_up == nullptr || d_tiled == nullptr)
        return TERN_ERR_NULL;
    if (!aligned(d_packed_gate, 4) || !aligned(d_packed_up, 4) || !aligned(d_scales_gate, 2) ||
        !aligned(d_scales_up, 2) || !aligned(d_tiled, 16))
        return TERN_ERR_ALIGN;
    if (d_err != nullptr && !aligned(d_err, 4)) return TERN_ERR_ALIGN;
    if (tiled_bytes < tern_tiled_glu_bytes(I, K)) return TERN_ERR_SIZE;
    return from_cuda(tern::launch_repack_glu(d_packed_gate, d_scales_gate, d_packed_up, d_scales_up, I, K,
                                             static_cast<uint8_t*>(d_tiled), d_err, as_stream(stream)));
}

size_t tern_swiglu_workspace_bytes(int64_t M, int64_t I, int64_t K) {
    if (I <= 0) return 0;
    return tern_workspace_bytes(M, tern::glu_rows(I), K);
}

tern_status tern_linear_swiglu(const void* d_X, int x_type, int64_t ldx, const void* d_tiled_glu, int64_t M,
                               int64_t I, int64_t K, void* d_H, int64_t ldh, int out_type, void* d_ws,
                               size_t ws_bytes, void* stream) {
    if (x_type != TERN_X_BF16 && x_type != TERN_X_F16) return TERN_ERR_SHAPE;
    if (out_type != TERN_OUT_F32 && out_type != TERN_OUT_BF16 && out_type != TERN_OUT_F16) return TERN_ERR_SHAPE;
    if (M < 0 || !valid_group_shape(I, K)) return TERN_ERR_SHAPE;
    if (M == 0 || I == 0) return TERN_OK;
    const uint16_t* X = static_cast<const uint16_t*>(d_X);
    tern_status st = check_x_w(X, ldx, d_tiled_glu, M, K);
    if (st != TERN_OK) return st;
    if (d_H == nullptr) return TERN_ERR_NULL;
    if (ldh < I) return TERN_ERR_SHAPE;
    if (!aligned(d_H, out_type == TERN_OUT_F32 ? 4 : 2)) return TERN_ERR_ALIGN;
    const int64_t N = tern::glu_rows(I);
    tern::OutputSplit out = {};
    out.n_out = 1;
    out.bf16 = out_type == TERN_OUT_BF16 ? 1 : out_type == TERN_OUT_F16 ? 2 : 0;
    out.glu = 1;
    out.glu_cols = I;
    out.offset[0] = 0;
    for (int j = 1; j <= tern::kMaxOutputs; ++j) out.offset[j] = N;
    out.y[0] = d_H;
    out.ldy[0] = ldh;
    return run_linear(X, x_type == TERN_X_F16, ldx, d_tiled_glu, M, N, K, out, d_ws, ws_bytes, as_stream(stream));
}

size_t tern_xq_bytes(int64_t M, int64_t K) {
    if (M < 0 || K <= 0 || K % tern::kGroup != 0) return 0;
    return tern::i8_xq_bytes(M, K);
}

tern_status tern_quantize_x(const void* d_X, int x_type, int64_t ldx, int64_t M, int64_t K, void* d_xq,
                            float* d_a, void* stream) {
    if (x_type != TERN_X_BF16 && x_type != TERN_X_F16) return TERN_ERR_SHAPE;
    if (M < 0 || K <= 0 || K % tern::kGroup != 0 || ldx < K) return TERN_ERR_SHAPE;
    if (M == 0) return TERN_OK;
    if (d_X == nullptr || d_xq == nullptr || d_a == nullptr) return TERN_ERR_NULL;
    if (!aligned(d_X, 2) || !aligned(d_xq, 16) || !aligned(d_a, 4)) return TERN_ERR_ALIGN;
    return from_cuda(tern::launch_quantize_x(static_cast<const uint16_t*>(d_X), x_type == TERN_X_F16, ldx, M, K,
                                             static_cast<int8_t*>(d_xq), d_a, as_stream(stream)));
}

size_t tern_i8_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || !valid_group_shape(N, K) || N == 0) return 0;
    return tern::plan_i8(M, N, K, tern::device_sm_count()).ws_bytes;
}

tern_status tern_linear_i8(const void* d_xq, const float* d_a, const void* d_tiled, int64_t M, int64_t N,
                           int64_t K, void* d_Y, int64_t ldy, int out_type, void* d_ws, size_t ws_bytes,
                           void* stream) {
    if (out_type != TERN_OUT_F32 && out_type != TERN_OUT_BF16 && out_type != TERN_OUT_F16) return TERN_ERR_SHAPE;
    if (M < 0 || !valid_group_shape(N, K)) return TERN_ERR_SHAPE;
    if (M == 0 || N == 0) return TERN_OK;
    if (M > (int64_t(1) << 30)) return TERN_ERR_SHAPE;
    if (d_xq == nullptr || d_a == nullptr || d_tiled == nullptr || d_Y == nullptr || d_ws == nullptr)
        return TERN_ERR_NULL;
    if (ldy < N) return TERN_ERR_SHAPE;
    if (!aligned(d_xq, 16) || !aligned(d_a, 4) || !aligned(d_tiled, 16) || !aligned(d_ws, 256) ||
        !aligned(d_Y, out_type == TERN_OUT_F32 ? 4 : 2))
        return TERN_ERR_ALIGN;
    const int sms = tern::device_sm_count();
    if (sms <= 0) return TERN_ERR_UNSUPPORTED;
    const tern::I8Plan plan = tern::plan_i8(M, N, K, sms);
    if (ws_bytes < plan.ws_bytes) return TERN_ERR_SIZE;
    tern::OutputSplit out = {};
    out.n_out = 1;
    out.bf16 = out_type == TERN_OUT_BF16 ? 1 : out_type == TERN_OUT_F16 ? 2 : 0;
    out.offset[0] = 0;
    for (int j = 1; j <= tern::kMaxOutputs; ++j) out.offset[j] = N;
    out.y[0] = d_Y;
    out.ldy[0] = ldy;
    return from_cuda(tern::launch_i8(static_cast<const int8_t*>(d_xq), d_a, static_cast<const uint8_t*>(d_tiled),
                                     M, N, out, d_ws, plan, as_stream(stream)));
}

tern_status tern_workspace_error(const void* d_ws, int32_t* h_err, void* stream) {
    if (d_ws == nullptr || h_err == nullptr) return TERN_ERR_NULL;
    if (!aligned(d_ws, 256)) return TERN_ERR_ALIGN;
    cudaError_t e = cudaMemcpyAsync(h_err, d_ws, sizeof(int32_t), cudaMemcpyDeviceToHost, as_stream(stream));
    if (e == cudaSuccess) e = cudaStreamSynchronize(as_stream(stream));
    return from_cuda(e);
}

tern_status tern_workspace_reset(void* d_ws, size_t ws_bytes, void* stream) {
    if (d_ws == nullptr) return TERN_ERR_NULL;
    if (!aligned(d_ws, 256)) return TERN_ERR_ALIGN;
    if (ws_bytes == 0) return TERN_OK;
    return from_cuda(cudaMemsetAsync(d_ws, 0, ws_bytes, as_stream(stream)));
}

}  // extern "C"
