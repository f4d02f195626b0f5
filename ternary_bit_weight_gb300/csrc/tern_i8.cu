// int8-activation variant of libtern's linear layer ("Ternary embedding
// model in vLLM", 2kiu.com/news/5082861, §4.1-§4.3, the page's third
// route: signs accumulated as integers inside each 128-wide group, the
// float scale applied once at the group boundary).
//
//   quantize_x_kernel: per token m, a[m] = max_k |x[m,k]| / 127 and
//     q[m,k] = rint(x[m,k] * (127 / max_k |x|)) in [-127, 127] (fp32
//     arithmetic, round to nearest even), stored in the tile order of the
//     code words: per 16 weights k0..k0+15, the bytes of k0, k0+2, ..,
//     k0+14, then k0+1, .., k0+15 -- the order of the fields in a tiled
//     code word, so that one byte of codes meets one 32-bit word of q.
//   i8_kernel (M = 1) / i8_batch_kernel (M > 1): one CTA per (row tile,
//     K split), one thread per weight row.  Four codes (a code byte) become
//     four int8 values and one dp4a multiplies them with four q and adds:
//     the group sum is an exact int32.  It becomes fp32 once per group
//     (exact: |sum| <= 127*128) and is scaled by the group's FP16 scale;
//     y = a[m] * (sum over groups).  At M = 1 the byte is spread into four
//     biased codes v = t + 1 with masks and two multiplies (a shared-memory
//     table lookup per byte conflicts in the banks), sum_k t q = sum_k v q -
//     sum_k q with the last sum computed once per CTA, the CTA's q slice is
//     loaded once and the next group's code words are loaded while the
//     current group is summed; for M > 1, where the dp4a work grows with M,
//     a 256-entry table gives t and q is staged per group.
//   i8_finish_kernel: when K is split, sums the splits' partials in split
//     order (deterministic) and stores y.

#include "tern_common.cuh"
#include "tern_internal.h"

namespace tern {
namespace {

constexpr int kI8Tokens = 16;   // tokens per pass over the weights
constexpr int kI8MaxGroups = 48;   // M = 1: groups per K split (the CTA's q slice)
constexpr int kI8CtasPerSm = 8;    // M = 1: K splits so that several 128-thread CTAs share each SM

// Shared memory of one i8_kernel CTA (M = 1): q over the CTA's groups, and
// their sums.
size_t i8_smem_bytes(int64_t M, int64_t G, int64_t KS) {
    return static_cast<size_t>(M * ceil_div(G, KS) * (kGroup + 4));
}

__global__ void __launch_bounds__(256) quantize_x_kernel(const uint16_t* __restrict__ X, int x_f16, int64_t ldx,
                                                         int K, int8_t* __restrict__ xq, float* __restrict__ a) {
    const int m = blockIdx.x;
    const uint16_t* xr = X + (int64_t)m * ldx;
    auto val = [&](int k) {
        const uint32_t b = xr[k];
        return x_f16 ? __half2float(__ushort_as_half(static_cast<unsigned short>(b))) : __uint_as_float(b << 16);
    };
    float mx = 0.f;
    for (int k = threadIdx.x; k < K; k += 256) mx = fmaxf(mx, fabsf(val(k)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    __shared__ float wmax[8];
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = wmax[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) mx = fmaxf(mx, wmax[i]);
    const float inv = mx > 0.f ? 127.0f / mx : 0.f;
    if (threadIdx.x == 0) a[m] = mx / 127.0f;
    int8_t* qr = xq + (int64_t)m * K;
    for (int k = threadIdx.x; k < K; k += 256) {
        float q = rintf(val(k) * inv);
        q = fminf(fmaxf(q, -127.f), 127.f);
        const int j = k & 15;   // position within the 16-weight word
        const int pos = (k & ~15) + (j & 1) * 8 + (j >> 1);
        qr[pos] = static_cast<int8_t>(q);
    }
}

// Four biased 2-bit codes (one byte, fields at bits 0, 2, 4, 6) -> four
// bytes v0..v3: fields 0 and 2 move by 0 and 12 bits, fields 1 and 3 by 6
// and 18 (the masked fields are far enough apart that the products do not
// carry into one another).
__device__ __forceinline__ uint32_t spread_codes(uint32_t byte) {
    const uint32_t even = (byte & 0x33u) * 0x1001u;     // v0 -> bits 0-1, v2 -> bits 16-17
    const uint32_t odd = (byte & 0xCCu) * 0x40040u;     // v1 -> bits 8-9, v3 -> bits 24-25
    return (even & 0x00030003u) | (odd & 0x03000300u);
}

// M > 1: the dp4a work grows with M while the weight stream does not, and
// this form (a 256-entry table from a code byte to four int8 t, the
// group's q staged per group) measured faster than the single-token form
// below at 16 tokens.
__global__ void __launch_bounds__(128) i8_batch_kernel(const int8_t* __restrict__ xq, const float* __restrict__ a,
                                                 const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales,
                                                 int M, int G, int KS, int64_t N, OutputSplit out,
                                                 float* __restrict__ partial) {
    __shared__ uint32_t lut[256];
    __shared__ __align__(16) int8_t xs[kI8Tokens * kGroup];
    const int r = threadIdx.x;
    const int64_t b = blockIdx.x;
    const int ks = blockIdx.y;
    const int g0 = static_cast<int>((int64_t)G * ks / KS), g1 = static_cast<int>((int64_t)G * (ks + 1) / KS);
    // byte of four biased codes v = t + 1 -> four int8 t
    for (int i = r; i < 256; i += 128) {
        uint32_t w = 0;
#pragma unroll
        for (int f = 0; f < 4; ++f) {
            const int v = (i >> (2 * f)) & 3;
            const int t = v == 0 ? -1 : (v == 2 ? 1 : 0);
            w |= static_cast<uint32_t>(static_cast<uint8_t>(static_cast<int8_t>(t))) << (8 * f);
        }
        lut[i] = w;
    }
    const int64_t row = b * kTileRows + r;
    const bool live = row < N;
    const RowOut o = row_out(out, live ? row : 0);
    for (int m0 = 0; m0 < M; m0 += kI8Tokens) {
        const int mt = M - m0 < kI8Tokens ? M - m0 : kI8Tokens;
        float acc[kI8Tokens];
#pragma unroll
        for (int m = 0; m < kI8Tokens; ++m) acc[m] = 0.f;
        for (int g = g0; g < g1; ++g) {
            __syncthreads();   // the previous group's q (and, first time, the table) are consumed / ready
            for (int i = r; i < mt * (kGroup / 16); i += 128) {
                const int m = i / (kGroup / 16), c = i % (kGroup / 16);
                reinterpret_cast<uint4*>(xs)[m * (kGroup / 16) + c] =
                    *reinterpret_cast<const uint4*>(xq + (int64_t)(m0 + m) * G * kGroup + (int64_t)g * kGroup + 16 * c);
            }
            __syncthreads();
            const uint8_t* u = codes + (b * G + g) * kUnitCodeBytes + 16 * r;
            const uint4 c0 = __ldg(reinterpret_cast<const uint4*>(u));
            const uint4 c1 = __ldg(reinterpret_cast<const uint4*>(u + 2048));
            const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            uint32_t t[32];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) t[4 * i + j] = lut[(w[i] >> (8 * j)) & 0xFFu];
            const float s = fp16_bits_to_float(scales[(b * G + g) * kTileRows + r]);
#pragma unroll
            for (int m = 0; m < kI8Tokens; ++m) {
                if (m >= mt) break;
                const uint4* xw = reinterpret_cast<const uint4*>(xs + m * kGroup);
                int isum = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint4 q = xw[i];
                    isum = __dp4a(static_cast<int>(t[4 * i + 0]), static_cast<int>(q.x), isum);
                    isum = __dp4a(static_cast<int>(t[4 * i + 1]), static_cast<int>(q.y), isum);
                    isum = __dp4a(static_cast<int>(t[4 * i + 2]), static_cast<int>(q.z), isum);
                    isum = __dp4a(static_cast<int>(t[4 * i + 3]), static_cast<int>(q.w), isum);
                }
                acc[m] = fmaf(s, static_cast<float>(isum), acc[m]);
            }
        }
#pragma unroll
        for (int m = 0; m < kI8Tokens; ++m) {
            if (m >= mt) break;
            if (KS == 1)
                store_out(out, o, m0 + m, row, acc[m] * a[m0 + m], live);
            else if (live)
                partial[((int64_t)ks * M + m0 + m) * N + row] = acc[m];
        }
    }
}

// M = 1 (MT = 1): codes spread arithmetically, the CTA's q slice loaded
// once, the next group's codes loaded while the current one is summed.
template <int MT>
__global__ void __launch_bounds__(128) i8_kernel(const int8_t* __restrict__ xq, const float* __restrict__ a,
                                                 const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales,
                                                 int M, int G, int KS, int64_t N, OutputSplit out,
                                                 float* __restrict__ partial) {
    extern __shared__ __align__(16) uint8_t i8_smem[];
    const int r = threadIdx.x;
    const int64_t b = blockIdx.x;
    const int ks = blockIdx.y;
    const int g0 = static_cast<int>((int64_t)G * ks / KS), g1 = static_cast<int>((int64_t)G * (ks + 1) / KS);
    const int ng = g1 - g0;
    const int64_t row = b * kTileRows + r;
    const bool live = row < N;
    const RowOut o = row_out(out, live ? row : 0);
    for (int m0 = 0; m0 < M; m0 += MT) {
        const int mt = M - m0 < MT ? M - m0 : MT;
        // the CTA's q: [token][group][128 bytes], then sum_k q per (token, group)
        int8_t* xs = reinterpret_cast<int8_t*>(i8_smem);
        int* qs = reinterpret_cast<int*>(i8_smem + mt * ng * kGroup);
        __syncthreads();   // the previous token batch is consumed
        for (int i = r; i < mt * ng * (kGroup / 16); i += kTileRows) {
            const int m = i / (ng * (kGroup / 16)), c = i % (ng * (kGroup / 16));
            reinterpret_cast<uint4*>(xs)[i] =
                *reinterpret_cast<const uint4*>(xq + (int64_t)(m0 + m) * G * kGroup + (int64_t)g0 * kGroup + 16 * c);
        }
        __syncthreads();
        for (int i = r; i < mt * ng; i += kTileRows) {
            const uint4* q = reinterpret_cast<const uint4*>(xs + i * kGroup);
            int sum = 0;
#pragma unroll
            for (int j = 0; j < kGroup / 16; ++j) {
                const uint4 w = q[j];
                sum = __dp4a(static_cast<int>(w.x), 0x01010101, sum);
                sum = __dp4a(static_cast<int>(w.y), 0x01010101, sum);
                sum = __dp4a(static_cast<int>(w.z), 0x01010101, sum);
                sum = __dp4a(static_cast<int>(w.w), 0x01010101, sum);
            }
            qs[i] = sum;
        }
        __syncthreads();
        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.f;
        const uint8_t* u = codes + (b * G + g0) * kUnitCodeBytes + 16 * r;
        uint4 c0 = __ldg(reinterpret_cast<const uint4*>(u));
        uint4 c1 = __ldg(reinterpret_cast<const uint4*>(u + 2048));
        for (int gi = 0; gi < ng; ++gi) {
            const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            if (gi + 1 < ng) {   // the next group's code words, while this group is summed
                u += kUnitCodeBytes;
                c0 = __ldg(reinterpret_cast<const uint4*>(u));
                c1 = __ldg(reinterpret_cast<const uint4*>(u + 2048));
            }
            const float s = fp16_bits_to_float(scales[(b * G + g0 + gi) * kTileRows + r]);
            int isum[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) isum[m] = m < mt ? -qs[m * ng + gi] : 0;
            // four weights at a time: spread once, then one dp4a per token
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t v0 = spread_codes(w[i] & 0xFFu), v1 = spread_codes((w[i] >> 8) & 0xFFu);
                const uint32_t v2 = spread_codes((w[i] >> 16) & 0xFFu), v3 = spread_codes(w[i] >> 24);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (m >= mt) continue;
                    const uint4 q = reinterpret_cast<const uint4*>(xs + (m * ng + gi) * kGroup)[i];
                    isum[m] = __dp4a(static_cast<int>(v0), static_cast<int>(q.x), isum[m]);
                    isum[m] = __dp4a(static_cast<int>(v1), static_cast<int>(q.y), isum[m]);
                    isum[m] = __dp4a(static_cast<int>(v2), static_cast<int>(q.z), isum[m]);
                    isum[m] = __dp4a(static_cast<int>(v3), static_cast<int>(q.w), isum[m]);
                }
            }
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (m < mt) acc[m] = fmaf(s, static_cast<float>(isum[m]), acc[m]);
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m >= mt) break;
            if (KS == 1)
                store_out(out, o, m0 + m, row, acc[m] * a[m0 + m], live);
            else if (live)
                partial[((int64_t)ks * M + m0 + m) * N + row] = acc[m];
        }
    }
}

__global__ void __launch_bounds__(256) i8_finish_kernel(const float* __restrict__ partial, const float* __restrict__ a,
                                                        int M, int KS, int64_t N, OutputSplit out) {
    // one warp per 32 consecutive rows of one token: every lane of the warp
    // reaches store_out together (the GLU pairing needs whole warps)
    const int64_t rows = ceil_div(N, 32) * 32;
    for (int64_t i = blockIdx.x * 256LL + threadIdx.x; i < (int64_t)M * rows; i += gridDim.x * 256LL) {
        const int m = static_cast<int>(i / rows);
        const int64_t row = i - (int64_t)m * rows;
        const bool live = row < N;
        float v = 0.f;
        if (live)
            for (int k = 0; k < KS; ++k) v += partial[((int64_t)k * M + m) * N + row];
        store_out(out, row_out(out, live ? row : 0), m, row, v * a[m], live);
    }
}

}  // namespace

size_t i8_xq_bytes(int64_t M, int64_t K) { return static_cast<size_t>(round_up(M * K, 16)); }

cudaError_t launch_quantize_x(const uint16_t* X, bool x_f16, int64_t ldx, int64_t M, int64_t K, int8_t* xq, float* a,
                              cudaStream_t stream) {
    if (M == 0) return cudaSuccess;
    quantize_x_kernel<<<static_cast<unsigned>(M), 256, 0, stream>>>(X, x_f16 ? 1 : 0, ldx, static_cast<int>(K), xq, a);
    return cudaGetLastError();
}

I8Plan plan_i8(int64_t M, int64_t N, int64_t K, int sm_count) {
    I8Plan p = {};
    if (sm_count <= 0) sm_count = 152;
    p.R = ceil_div(N, kTileRows);
    p.G = K / kGroup;
    // M = 1 (bound by the weight stream): enough K splits for several CTAs
    // per SM, each split at least 4 groups and at most kI8MaxGroups long;
    // larger M (bound by the dp4a work): two CTAs per SM
    int64_t ks = ceil_div((M == 1 ? kI8CtasPerSm : 2) * sm_count, p.R);
    if (M == 1) {
        if (ks > p.G / 4) ks = p.G / 4;
        if (ks < ceil_div(p.G, kI8MaxGroups)) ks = ceil_div(p.G, kI8MaxGroups);
    }
    if (ks > p.G) ks = p.G;
    if (ks < 1) ks = 1;
    p.KS = ks;
    p.ws_bytes = kWorkspaceErrBytes + (p.KS > 1 ? static_cast<size_t>(p.KS * M * N) * sizeof(float) : 0);
    return p;
}

cudaError_t launch_i8(const int8_t* xq, const float* a, const uint8_t* tiled, int64_t M, int64_t N,
                      const OutputSplit& out, void* ws, const I8Plan& plan, cudaStream_t stream) {
    float* partial = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kWorkspaceErrBytes);
    const uint8_t* codes = tiled;
    const uint16_t* scales = reinterpret_cast<const uint16_t*>(tiled + plan.R * plan.G * kUnitCodeBytes);
    dim3 grid(static_cast<unsigned>(plan.R), static_cast<unsigned>(plan.KS));
    if (M == 1)
        i8_kernel<1><<<grid, 128, i8_smem_bytes(M, plan.G, plan.KS), stream>>>(
            xq, a, codes, scales, static_cast<int>(M), static_cast<int>(plan.G), static_cast<int>(plan.KS), N, out,
            partial);
    else
        i8_batch_kernel<<<grid, 128, 0, stream>>>(xq, a, codes, scales, static_cast<int>(M), static_cast<int>(plan.G),
                                                  static_cast<int>(plan.KS), N, out, partial);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || plan.KS == 1) return e;
    const int64_t items = M * ceil_div(N, 32) * 32;
    const int64_t blocks = ceil_div(items, 256);
    i8_finish_kernel<<<static_cast<unsigned>(blocks < 152 * 16 ? blocks : 152 * 16), 256, 0, stream>>>(
        partial, a, static_cast<int>(M), static_cast<int>(plan.KS), N, out);
    return cudaGetLastError();
}

}  // namespace tern
