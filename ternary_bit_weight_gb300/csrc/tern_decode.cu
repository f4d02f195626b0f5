// Decode / skinny-batch kernel of libtern: Y[M,N] = X[M,K] . (s (.) T)^T for
// M <= 16, streaming the tiled 2-bit weights at HBM rate.
//
// Method ("Ternary embedding model in vLLM", 2kiu.com/news/5082861, §4.2,
// §4.3): keep the weights packed in memory, decode them in registers, sum
// the sign-selected activations inside each 128-wide scale group and apply
// the FP16 scale once per group.  The page's kernels run one thread per
// output on CUDA cores; here the per-group sum is done by the tensor cores:
//
//   * a warp owns a 16-row tile; each group of 128 weights arrives as one
//     coalesced 512-byte block (one 16-byte load per lane, prefetched
//     several groups ahead in registers);
//   * each lane decodes its 64 codes to exact bf16 values t in {-1,0,+1}
//     (one LOP3 + one bf16x2 FMA per pair, see decode_pair) which are
//     directly the A fragments of mma.m16n8k16 -- weights on the MMA M
//     side, tokens on the N side (8 per n-tile);
//   * the group partial (exact products, fp32 sums) is scaled by the fp32
//     value of the FP16 scale and added to the fp32 accumulator: the scale
//     is never rounded to bf16;
//   * K is split into S ranges when N alone does not fill the GPU; the
//     last CTA of a row block to finish sums the S partials in split order
//     (deterministic, no spin-waiting) and writes Y.
//
// K-slot order inside an MMA: the MMA sums over its 16 k-slots, so any
// consistent permutation of k between A and B is free.  Lane (g, c) of
// MMA j of half h takes physical k = 128*grp + 64h + 16c + 4j + {0,1,2,3}
// for its k-slots {2c, 2c+1, 2c+8, 2c+9}: its A registers then come from one
// 16-weight code word of the tiled layout and its B registers are four
// consecutive activations, one 64-bit shared-memory read.

#include "tern_common.cuh"
#include "tern_internal.h"

namespace tern {
namespace {

constexpr int kWarps = 8;                 // row tiles per CTA (128 rows)
constexpr int kThreads = kWarps * 32;
constexpr int kPrefetch = 8;              // groups in flight per warp
constexpr int kRowsPerBlock = kWarps * kTileRows;
constexpr size_t kMaxSmem = 200 * 1024;

struct DecodeArgs {
    const uint16_t* X;
    int64_t ldx;
    const uint8_t* codes;    // tiled code region
    const uint8_t* scales;   // tiled scale region
    int M;
    int64_t N;
    int64_t Np;              // rows padded to 16
    int64_t R;               // row tiles
    int64_t G;               // groups along K
    int64_t n_rb;            // 128-row blocks
    int S;                   // K splits
    OutputSplit out;
    float* part;             // [S][M][Np] split partials (S > 1)
    int* counters;           // [n_rb] arrival counters (S > 1)
};

__device__ __forceinline__ void store_y(const OutputSplit& out, int m, int64_t n, float v) {
    int j = 0;
#pragma unroll
    for (int i = 1; i < kMaxOutputs; ++i) j += (i < out.n_out && n >= out.offset[i]);
    out.y[j][(int64_t)m * out.ldy[j] + (n - out.offset[j])] = v;
}

template <int MT>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(const DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem_raw);
    __shared__ int last_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, cq = lane & 3;
    const int64_t rb = blockIdx.x % a.n_rb;
    const int s = static_cast<int>(blockIdx.x / a.n_rb);
    const int64_t g0 = (int64_t)s * a.G / a.S, g1 = (int64_t)(s + 1) * a.G / a.S;
    const int ng = static_cast<int>(g1 - g0);
    const int64_t tile = rb * kWarps + warp;
    const bool active = tile < a.R;

    // 1. Start streaming this warp's weights: they do not depend on earlier
    //    kernels, so this happens before the grid-dependency wait.
    const uint8_t* cptr = a.codes + ((tile * a.G + g0) * 32 + lane) * 16;
    const uint8_t* sptr = a.scales + ((tile * a.G + g0) * 8 + gq) * 4;
    uint4 cbuf[kPrefetch];
    uint32_t sbuf[kPrefetch];
#pragma unroll
    for (int d = 0; d < kPrefetch; ++d) {
        if (active && d < ng) {
            cbuf[d] = ldg_stream_v4(cptr + (int64_t)d * kCodeBlockBytes);
            sbuf[d] = ldg_stream_u32(sptr + (int64_t)d * kScaleBlockBytes);
        } else {
            cbuf[d] = make_uint4(0, 0, 0, 0);
            sbuf[d] = 0;
        }
    }
    grid_launch_dependents();
    grid_dependency_wait();

    // 2. Stage X[0:M, 128*g0 : 128*g1] in shared memory, row stride ck + 8
    //    (the 16-byte pad spreads the 8 token rows over all banks).
    const int ck = ng * kGroup;
    const int sx = ck + 8;
    {
        const int vec_per_row = ck / 8;
        const int total = a.M * vec_per_row;
        for (int i = threadIdx.x; i < total; i += kThreads) {
            const int m = i / vec_per_row, j = i - m * vec_per_row;
            const uint4 v = *reinterpret_cast<const uint4*>(a.X + (int64_t)m * a.ldx + g0 * kGroup + 8 * j);
            *reinterpret_cast<uint4*>(xs + m * sx + 8 * j) = v;
        }
    }
    __syncthreads();

    // 3. Main loop over this split's groups.
    float acc[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;

    if (active) {
        for (int base = 0; base < ng; base += kPrefetch) {
#pragma unroll
            for (int d = 0; d < kPrefetch; ++d) {
                const int gi = base + d;
                if (gi < ng) {
                    const uint4 cw = cbuf[d];
                    const uint32_t sw = sbuf[d];
                    if (gi + kPrefetch < ng) {
                        cbuf[d] = ldg_stream_v4(cptr + (int64_t)(gi + kPrefetch) * kCodeBlockBytes);
                        sbuf[d] = ldg_stream_u32(sptr + (int64_t)(gi + kPrefetch) * kScaleBlockBytes);
                    }
                    // two independent MMA chains (one per 64-wide half)
                    float cg[2][MT][4];
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                            for (int e = 0; e < 4; ++e) cg[h][mt][e] = 0.f;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t lo[8], hi[8];
                        decode_word(h ? cw.z : cw.x, lo);   // row gq
                        decode_word(h ? cw.w : cw.y, hi);   // row gq + 8
                        uint32_t xb[MT][8];
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            const int m = mt * 8 + gq;
                            if (m < a.M) {
                                const uint16_t* p = xs + m * sx + gi * kGroup + 64 * h + 16 * cq;
                                const uint4 v0 = lds_v4(p), v1 = lds_v4(p + 8);
                                xb[mt][0] = v0.x; xb[mt][1] = v0.y; xb[mt][2] = v0.z; xb[mt][3] = v0.w;
                                xb[mt][4] = v1.x; xb[mt][5] = v1.y; xb[mt][6] = v1.z; xb[mt][7] = v1.w;
                            } else {
#pragma unroll
                                for (int e = 0; e < 8; ++e) xb[mt][e] = 0u;
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int mt = 0; mt < MT; ++mt)
                                mma_bf16_m16n8k16(cg[h][mt], lo[2 * j], hi[2 * j], lo[2 * j + 1],
                                                  hi[2 * j + 1], xb[mt][2 * j], xb[mt][2 * j + 1]);
                    }
                    const float s_lo = fp16_bits_to_float(sw), s_hi = fp16_bits_to_float(sw >> 16);
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        acc[mt][0] = fmaf(s_lo, cg[0][mt][0] + cg[1][mt][0], acc[mt][0]);
                        acc[mt][1] = fmaf(s_lo, cg[0][mt][1] + cg[1][mt][1], acc[mt][1]);
                        acc[mt][2] = fmaf(s_hi, cg[0][mt][2] + cg[1][mt][2], acc[mt][2]);
                        acc[mt][3] = fmaf(s_hi, cg[0][mt][3] + cg[1][mt][3], acc[mt][3]);
                    }
                }
            }
        }
    }

    // 4. Epilogue.  Fragment element e of n-tile mt: row 16*tile + gq + 8*(e/2),
    //    token 8*mt + 2*cq + (e%2).
    if (a.S == 1) {
        if (active) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int m = mt * 8 + 2 * cq + (e & 1);
                    const int64_t n = tile * kTileRows + gq + 8 * (e >> 1);
                    if (m < a.M && n < a.N) store_y(a.out, m, n, acc[mt][e]);
                }
        }
        return;
    }

    if (active) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int m = mt * 8 + 2 * cq + (e & 1);
                const int64_t n = tile * kTileRows + gq + 8 * (e >> 1);
                if (m < a.M) a.part[((int64_t)s * a.M + m) * a.Np + n] = acc[mt][e];
            }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last_flag = (atomicAdd(a.counters + rb, 1) == a.S - 1);
    __syncthreads();
    if (!last_flag) return;
    __threadfence();
    // Last CTA of this row block: sum the S partials in split order.
    const int64_t row0 = rb * kRowsPerBlock;
    const int rows = static_cast<int>((a.Np - row0) < kRowsPerBlock ? (a.Np - row0) : kRowsPerBlock);
    for (int i = threadIdx.x; i < rows * a.M; i += kThreads) {
        const int m = i / rows;
        const int64_t n = row0 + (i - m * rows);
        if (n >= a.N) continue;
        float v = 0.f;
        for (int k = 0; k < a.S; ++k) v += __ldcg(a.part + ((int64_t)k * a.M + m) * a.Np + n);
        store_y(a.out, m, n, v);
    }
    if (threadIdx.x == 0) a.counters[rb] = 0;   // leave the workspace zeroed
}

}  // namespace

int device_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

DecodePlan plan_decode(int64_t M, int64_t N, int64_t K, int sm_count) {
    DecodePlan p = {};
    if (sm_count <= 0) sm_count = 152;
    p.mt = M <= 8 ? 1 : 2;
    const int64_t R = ceil_div(N, kTileRows);
    const int64_t Np = R * kTileRows;
    p.n_rb = ceil_div(R, kWarps);
    p.groups = K / kGroup;
    const int64_t slots = (int64_t)sm_count * 2;   // two 256-thread CTAs per SM
    // Pick the split count that minimises (waves x groups per CTA + a fixed
    // start-up cost of ~2 groups), subject to the X slice fitting in smem.
    double best = 1e300;
    int best_s = 1;
    const int64_t s_max = p.groups < 256 ? p.groups : 256;
    for (int64_t S = 1; S <= s_max; ++S) {
        const int64_t gps = ceil_div(p.groups, S);
        const size_t smem = (size_t)M * (size_t)(gps * kGroup + 8) * 2;
        if (smem > kMaxSmem) continue;
        const int64_t waves = ceil_div(p.n_rb * S, slots);
        const double cost = (double)waves * ((double)gps + 2.0);
        if (cost < best - 1e-9) { best = cost; best_s = static_cast<int>(S); }
    }
    p.splits = best_s;
    p.max_gps = ceil_div(p.groups, best_s);
    p.smem = (size_t)M * (size_t)(p.max_gps * kGroup + 8) * 2;
    if (p.splits > 1) {
        const size_t counters = (size_t)ceil_div(p.n_rb * 4, 256) * 256;
        p.ws_bytes = counters + (size_t)p.splits * (size_t)M * (size_t)Np * 4;
    } else {
        p.ws_bytes = 0;
    }
    return p;
}

cudaError_t launch_decode(const uint16_t* X, int64_t ldx, const uint8_t* tiled, int64_t M,
                          int64_t N, int64_t K, const OutputSplit& out, void* ws,
                          const DecodePlan& plan, cudaStream_t stream) {
    DecodeArgs a = {};
    a.X = X;
    a.ldx = ldx;
    a.R = ceil_div(N, kTileRows);
    a.G = K / kGroup;
    a.codes = tiled;
    a.scales = tiled + a.R * a.G * kCodeBlockBytes;
    a.M = static_cast<int>(M);
    a.N = N;
    a.Np = a.R * kTileRows;
    a.n_rb = plan.n_rb;
    a.S = plan.splits;
    a.out = out;
    if (plan.splits > 1) {
        const size_t counters = (size_t)ceil_div(plan.n_rb * 4, 256) * 256;
        a.counters = static_cast<int*>(ws);
        a.part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + counters);
    }

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.n_rb * plan.splits));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;

    cudaError_t e;
    if (plan.mt == 1) {
        e = cudaFuncSetAttribute(decode_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kMaxSmem));
        if (e != cudaSuccess) return e;
        return cudaLaunchKernelEx(&cfg, decode_kernel<1>, a);
    }
    e = cudaFuncSetAttribute(decode_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kMaxSmem));
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, decode_kernel<2>, a);
}

}  // namespace tern
