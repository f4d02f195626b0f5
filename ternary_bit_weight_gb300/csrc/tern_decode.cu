// Decode / skinny-batch kernels of libtern: Y[M,N] = X[M,K] . (s (.) T)^T for
// M <= 16, streaming the tiled 2-bit weights at HBM rate.
//
// Method ("Ternary embedding model in vLLM", 2kiu.com/news/5082861, §4.2,
// §4.3): keep the weights packed in memory, decode them in registers, sum
// the sign-selected activations inside each 128-wide scale group and apply
// the FP16 scale once per group.  The page's kernels run one thread per
// output on CUDA cores; here the per-group sum is done by the tensor cores:
//
//   * a warp works on 16-row tiles; each group of 128 weights of a tile
//     arrives as one coalesced 512-byte block (one 16-byte load per lane,
//     prefetched eight groups ahead in registers);
//   * each lane decodes its 64 codes to exact bf16 values t in {-1,0,+1}
//     (one LOP3 + one bf16x2 FMA per pair, see decode_pair) which are
//     directly the A fragments of mma.m16n8k16 -- weights on the MMA M
//     side, tokens on the N side (8 per n-tile);
//   * the group partial (exact products, fp32 sums) is scaled by the fp32
//     value of the FP16 scale and added to the fp32 accumulator: the scale
//     is never rounded to bf16.
//
// K-slot order inside an MMA: the MMA sums over its 16 k-slots, so any
// consistent permutation of k between A and B is free.  Lane (g, c) of
// MMA j of half h takes physical k = 128*grp + 64h + 16c + 4j + {0,1,2,3}
// for its k-slots {2c, 2c+1, 2c+8, 2c+9}: its A registers then come from one
// 16-weight code word of the tiled layout and its B registers are four
// consecutive activations.
//
// Work split: one CTA of 8 warps per (128-row tile, K range); warp w owns
// rows 16w..16w+15 of the tile.  When N alone does not fill the GPU, K is
// split into S ranges and the last CTA of a tile to finish sums the S
// partials in split order (deterministic, no spin-waiting).

#include "tern_common.cuh"
#include "tern_internal.h"

namespace tern {
namespace {

constexpr int kWarps = 8;                 // warps per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kPrefetch = 8;              // groups in flight per warp
constexpr int kRowsPerBlock = kTileRows;   // one 128-row tile per CTA
constexpr int kSubRows = 16;               // rows per warp (one m16 fragment)
constexpr size_t kSplitMaxSmem = 200 * 1024;
constexpr int kZeroBytes = 32;

__device__ __forceinline__ void store_y(const OutputSplit& out, int m, int64_t n, float v) {
    int j = 0;
#pragma unroll
    for (int i = 1; i < kMaxOutputs; ++i) j += (i < out.n_out && n >= out.offset[i]);
    out.y[j][(int64_t)m * out.ldy[j] + (n - out.offset[j])] = v;
}

// Shared-memory byte offsets of one lane's activation fragments.  Token rows
// >= M point at a zero block with zero strides, so every lane issues the
// same loads (no divergence) and padding tokens contribute exact zeros.
template <int MT>
struct XLanes {
    uint32_t base[MT];      // group 0, half 0
    uint32_t gstride[MT];   // per group (256 bytes, or 0)
    uint32_t hstride[MT];   // per 64-wide half (128 bytes, or 0)
};

template <int MT>
__device__ __forceinline__ XLanes<MT> x_lanes(int M, uint32_t row_bytes, uint32_t zero_off, int gq,
                                              int cq) {
    XLanes<MT> xl;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        const int m = mt * 8 + gq;
        const bool valid = m < M;
        xl.base[mt] = valid ? (uint32_t)m * row_bytes + 32u * cq : zero_off;
        xl.gstride[mt] = valid ? 256u : 0u;
        xl.hstride[mt] = valid ? 128u : 0u;
    }
    return xl;
}

// One 16x128 tile-group: decode, 8 MMAs per n-tile in two chains, promote.
template <int MT>
__device__ __forceinline__ void group_mac(const uint4 cw, uint32_t sw, const uint8_t* smem,
                                          const XLanes<MT>& xl, uint32_t g, float (&acc)[MT][4]) {
    float cg[2][MT][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t lo[8], hi[8];
        decode_word(h ? cw.z : cw.x, lo);   // row gq
        decode_word(h ? cw.w : cw.y, hi);   // row gq + 8
        uint32_t xb[MT][8];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const uint8_t* p = smem + xl.base[mt] + g * xl.gstride[mt] + h * xl.hstride[mt];
            const uint4 v0 = lds_v4(p), v1 = lds_v4(p + 16);
            xb[mt][0] = v0.x; xb[mt][1] = v0.y; xb[mt][2] = v0.z; xb[mt][3] = v0.w;
            xb[mt][4] = v1.x; xb[mt][5] = v1.y; xb[mt][6] = v1.z; xb[mt][7] = v1.w;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
            mma_bf16_m16n8k16_zc(cg[h][mt], lo[0], hi[0], lo[1], hi[1], xb[mt][0], xb[mt][1]);
#pragma unroll
        for (int j = 1; j < 4; ++j)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
                mma_bf16_m16n8k16(cg[h][mt], lo[2 * j], hi[2 * j], lo[2 * j + 1], hi[2 * j + 1],
                                  xb[mt][2 * j], xb[mt][2 * j + 1]);
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

// Write a finished 16-row sub-tile's fragments: element e of n-tile mt is
// row row0 + gq + 8*(e/2), token 8*mt + 2*cq + (e%2).
template <int MT>
__device__ __forceinline__ void store_tile(const OutputSplit& out, int M, int64_t N, int64_t row0,
                                           const float (&acc)[MT][4], int gq, int cq) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int m = mt * 8 + 2 * cq + (e & 1);
            const int64_t n = row0 + gq + 8 * (e >> 1);
            if (m < M && n < N) store_y(out, m, n, acc[mt][e]);
        }
}

// Stage rows [0, M) of X columns [k0, k0 + ck) in shared memory with row
// stride ck + 8 elements (the 16-byte pad spreads token rows over all
// banks), followed by a 32-byte zero block.  Returns the zero block offset.
__device__ __forceinline__ uint32_t stage_x(uint8_t* smem, const uint16_t* X, int64_t ldx, int M,
                                            int64_t k0, int ck) {
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
    const int sx = ck + 8;
    const int vec_per_row = ck / 8;
    const int total = M * vec_per_row;
    for (int i = threadIdx.x; i < total; i += kThreads) {
        const int m = i / vec_per_row, j = i - m * vec_per_row;
        const uint4 v = *reinterpret_cast<const uint4*>(X + (int64_t)m * ldx + k0 + 8 * j);
        *reinterpret_cast<uint4*>(xs + m * sx + 8 * j) = v;
    }
    const uint32_t zero_off = (uint32_t)M * (uint32_t)sx * 2u;
    if (threadIdx.x < kZeroBytes / 16)
        *reinterpret_cast<uint4*>(smem + zero_off + 16 * threadIdx.x) = make_uint4(0, 0, 0, 0);
    return zero_off;
}

// ------------------------------------------------------------ split kernel

struct SplitArgs {
    const uint16_t* X;
    int64_t ldx;
    const uint8_t* codes;
    const uint8_t* scales;
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

// Four 32-bit code words of one lane for one group: rows gq and gq + 8 of
// the warp's 16 rows, halves 0 and 1, word cq (the tiled unit layout).
__device__ __forceinline__ uint4 load_lane_codes(const uint8_t* p) {
    uint4 c;
    c.x = ldg_stream_u32(p);
    c.y = ldg_stream_u32(p + 128);
    c.z = ldg_stream_u32(p + 2048);
    c.w = ldg_stream_u32(p + 2048 + 128);
    return c;
}

__device__ __forceinline__ uint32_t load_lane_scales(const uint8_t* p) {
    const uint32_t lo = __ldcs(reinterpret_cast<const unsigned short*>(p));
    const uint32_t hi = __ldcs(reinterpret_cast<const unsigned short*>(p + 16));
    return lo | (hi << 16);
}

template <int MT>
__global__ void __launch_bounds__(kThreads, 2) split_kernel(const SplitArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int last_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, cq = lane & 3;
    const int64_t rb = blockIdx.x % a.n_rb;
    const int s = static_cast<int>(blockIdx.x / a.n_rb);
    const int64_t g0 = (int64_t)s * a.G / a.S, g1 = (int64_t)(s + 1) * a.G / a.S;
    const int ng = static_cast<int>(g1 - g0);
    const int64_t row0 = rb * kTileRows + kSubRows * warp;
    const bool active = row0 < a.N;

    const uint8_t* cptr = a.codes + (rb * a.G + g0) * kUnitCodeBytes + 16 * (kSubRows * warp + gq) + 4 * cq;
    const uint8_t* sptr = a.scales + (rb * a.G + g0) * kUnitScaleBytes + 2 * (kSubRows * warp + gq);
    uint4 cbuf[kPrefetch];
    uint32_t sbuf[kPrefetch];
#pragma unroll
    for (int d = 0; d < kPrefetch; ++d) {
        if (active && d < ng) {
            cbuf[d] = load_lane_codes(cptr + d * kUnitCodeBytes);
            sbuf[d] = load_lane_scales(sptr + d * kUnitScaleBytes);
        } else {
            cbuf[d] = make_uint4(0, 0, 0, 0);
            sbuf[d] = 0;
        }
    }
    grid_launch_dependents();
    grid_dependency_wait();

    const int ck = ng * kGroup;
    const uint32_t zero_off = stage_x(smem, a.X, a.ldx, a.M, g0 * kGroup, ck);
    __syncthreads();
    const XLanes<MT> xl = x_lanes<MT>(a.M, (uint32_t)(ck + 8) * 2u, zero_off, gq, cq);

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
                        cbuf[d] = load_lane_codes(cptr + (int64_t)(gi + kPrefetch) * kUnitCodeBytes);
                        sbuf[d] = load_lane_scales(sptr + (int64_t)(gi + kPrefetch) * kUnitScaleBytes);
                    }
                    group_mac<MT>(cw, sw, smem, xl, (uint32_t)gi, acc);
                }
            }
        }
    }

    if (a.S == 1) {
        if (active) store_tile<MT>(a.out, a.M, a.N, row0, acc, gq, cq);
        return;
    }

    if (active) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int m = mt * 8 + 2 * cq + (e & 1);
                const int64_t n = row0 + gq + 8 * (e >> 1);
                if (m < a.M) a.part[((int64_t)s * a.M + m) * a.Np + n] = acc[mt][e];
            }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last_flag = (atomicAdd(a.counters + rb, 1) == a.S - 1);
    __syncthreads();
    if (!last_flag) return;
    __threadfence();
    // Last CTA of this row tile: sum the S partials in split order.
    const int64_t t0 = rb * kRowsPerBlock;
    for (int i = threadIdx.x; i < kRowsPerBlock * a.M; i += kThreads) {
        const int m = i / kRowsPerBlock;
        const int64_t n = t0 + (i - m * kRowsPerBlock);
        if (n >= a.N) continue;
        float v = 0.f;
        for (int k = 0; k < a.S; ++k) v += __ldcg(a.part + ((int64_t)k * a.M + m) * a.Np + n);
        store_y(a.out, m, n, v);
    }
    if (threadIdx.x == 0) a.counters[rb] = 0;   // leave the workspace zeroed
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

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
    p.groups = K / kGroup;
    p.n_rb = R;

    p.kind = DecodePlan::kSplit;
    const int64_t slots = (int64_t)sm_count * 2;   // two 256-thread CTAs per SM
    // Pick the split count that minimises (waves x groups per CTA + a fixed
    // start-up cost of ~2 groups), subject to the X slice fitting in smem.
    double best = 1e300;
    int best_s = 1;
    const int64_t s_max = p.groups < 256 ? p.groups : 256;
    for (int64_t S = 1; S <= s_max; ++S) {
        const int64_t gps = ceil_div(p.groups, S);
        const size_t smem = (size_t)M * (size_t)(gps * kGroup + 8) * 2 + kZeroBytes;
        if (smem > kSplitMaxSmem) continue;
        const int64_t waves = ceil_div(p.n_rb * S, slots);
        const double cost = (double)waves * ((double)gps + 2.0);
        if (cost < best - 1e-9) { best = cost; best_s = static_cast<int>(S); }
    }
    p.splits = best_s;
    p.max_gps = ceil_div(p.groups, best_s);
    p.smem = (size_t)M * (size_t)(p.max_gps * kGroup + 8) * 2 + kZeroBytes;
    p.grid = p.n_rb * p.splits;
    p.warps = p.grid * kWarps;
    if (p.splits > 1)
        p.ws_bytes = align256((size_t)p.n_rb * 4) + (size_t)p.splits * (size_t)M * (size_t)Np * 4;
    else
        p.ws_bytes = 0;
    return p;
}

namespace {

template <typename Kernel, typename Args>
cudaError_t launch_pdl(Kernel kernel, const Args& a, int64_t grid, size_t smem, size_t max_smem,
                       cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(max_smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace

cudaError_t launch_decode(const uint16_t* X, int64_t ldx, const uint8_t* tiled, int64_t M,
                          int64_t N, int64_t K, const OutputSplit& out, void* ws,
                          const DecodePlan& plan, cudaStream_t stream) {
    const int64_t R = ceil_div(N, kTileRows), G = K / kGroup;
    const uint8_t* codes = tiled;
    const uint8_t* scales = tiled + R * G * kUnitCodeBytes;

    SplitArgs a = {};
    a.X = X;
    a.ldx = ldx;
    a.codes = codes;
    a.scales = scales;
    a.R = R;
    a.G = G;
    a.M = static_cast<int>(M);
    a.N = N;
    a.Np = R * kTileRows;
    a.n_rb = plan.n_rb;
    a.S = plan.splits;
    a.out = out;
    if (plan.splits > 1) {
        a.counters = static_cast<int*>(ws);
        a.part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + align256((size_t)plan.n_rb * 4));
    }
    if (plan.mt == 1)
        return launch_pdl(split_kernel<1>, a, plan.grid, plan.smem, kSplitMaxSmem, stream);
    return launch_pdl(split_kernel<2>, a, plan.grid, plan.smem, kSplitMaxSmem, stream);
}

}  // namespace tern
