/*
 * CPU oracle for the ternary-weight linear layer -- TEST INFRASTRUCTURE.
 *
 * Plain, slow, obviously correct C.  Only the tests, the package's smoke
 * check and the benchmark's CPU-baseline leg load it; the product path
 * never does.  It shares no code, header, table or helper with the CUDA
 * library: it is written separately from the method's description.
 *
 * Sources (web pages, cited by a short name, address and section):
 *   [EMB]  "Ternary embedding model in vLLM", 2kiu.com/news/5082861
 *          §1.1  weights in {-1,0,+1}, one FP16 scale per 128 weights
 *          §3.1  the packing rule: 2-bit codes 00->0, 01->+1, 10->-1,
 *                11->reserved, read as 0; four codes per uint8, little-endian,
 *                first weight in the lowest two bits; scale blocks cut
 *                contiguously along K; the unpack routine (shifts 0,2,4,6)
 *          §4.2  shapes: x [M,K], packed w [N,K/4] uint8, scale [N,K/128]
 *                half, y = x . W^T; the page's kernel reads half-precision
 *                (fp16) activations
 *   [B27]  "Porting ternary Bonsai 2 27B to vLLM", m.xxqk.cn/news/594847
 *          §5.2  scales are little-endian FP16
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - pack of a value outside {-1,0,+1} writes code 00 and is counted;
 *   - the layer is the plain definition Y[m,n] = sum_k x[m,k] * t[n,k] *
 *     s[n, k/128], computed here with fp64 accumulation in k order;
 *   - the GPU tile layout ("tiled") is this library's own format (the pages
 *     only say the disk and GPU layouts must be reconciled, [EMB] §3).
 *     Its index map is written out in orc_repack below.
 *
 * Parity pins for every function live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ scalars */

/* IEEE binary16 bits -> double, from the format's definition. */
double orc_fp16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-14 * 2^-10 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1.0 + (double)f / 1024.0, e - 15);
    return sign ? -v : v;
}

/* bfloat16 bits -> double: the top half of an IEEE binary32. */
double orc_bf16_to_double(uint16_t b) {
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xFF;
    int f = b & 0x7F;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);                /* f * 2^-126 * 2^-7 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1.0 + (double)f / 128.0, e - 127);
    return sign ? -v : v;
}

/* [EMB] §3.1: 00 -> 0, 01 -> +1, 10 -> -1, 11 -> reserved, read as 0. */
int orc_code_to_ternary(unsigned code) {
    switch (code & 3u) {
        case 1: return 1;
        case 2: return -1;
        default: return 0;
    }
}

static unsigned ternary_to_code(int t, int64_t* invalid) {
    if (t == 1) return 1u;
    if (t == -1) return 2u;
    if (t != 0) ++*invalid;
    return 0u;
}

/* Weight (n,k) of an on-disk packed [N, K/4] matrix: byte k/4 of row n,
   bits 2*(k%4) and 2*(k%4)+1 ([EMB] §3.1, first weight lowest). */
static unsigned packed_code(const uint8_t* packed, int64_t K, int64_t n, int64_t k) {
    uint8_t byte = packed[n * (K / 4) + k / 4];
    return (byte >> (2 * (k % 4))) & 3u;
}

/* ------------------------------------------------------------- pack/unpack */

/* t int8 [N,K] -> packed uint8 [N,K/4].  K must be a multiple of 4.
   Returns the number of entries outside {-1,0,+1} (written as code 00). */
int64_t orc_pack(const int8_t* t, int64_t N, int64_t K, uint8_t* packed) {
    int64_t invalid = 0;
    #pragma omp parallel for schedule(static) reduction(+:invalid)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t kb = 0; kb < K / 4; ++kb) {
            unsigned byte = 0;
            for (int j = 0; j < 4; ++j) {
                unsigned code = ternary_to_code(t[n * K + 4 * kb + j], &invalid);
                byte |= code << (2 * j);
            }
            packed[n * (K / 4) + kb] = (uint8_t)byte;
        }
    }
    return invalid;
}

/* packed uint8 [N,K/4] -> t int8 [N,K].  Returns the number of code-11 entries. */
int64_t orc_unpack(const uint8_t* packed, int64_t N, int64_t K, int8_t* t) {
    int64_t reserved = 0;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            unsigned code = packed_code(packed, K, n, k);
            if (code == 3u) ++reserved;
            t[n * K + k] = (int8_t)orc_code_to_ternary(code);
        }
    return reserved;
}

/* ------------------------------------------------------------ tiled layout
 *
 * The GPU tile layout.  Rows are padded to Np = 128*ceil(N/128) (padding
 * rows hold weight 0 and scale 0).  With G = K/128 groups and R = Np/128
 * row tiles, a unit is one 128-row x 128-weight block:
 *
 *   codes:  R*G units of 4096 bytes; unit (b,g) starts at (b*G + g)*4096.
 *           Inside a unit, half h (0,1) starts at 2048*h, row r (0..127)
 *           of the tile at 16*r within the half, and the row's 16 bytes
 *           are four little-endian 32-bit words; word q covers the weights
 *           k0..k0+15 with k0 = 128g + 64h + 16q.
 *           In a word, weight k0+2i sits at bits 2i..2i+1 and weight
 *           k0+2i+1 at bits 16+2i..17+2i (i in 0..7).
 *           The stored value is the biased code v = t + 1 in {0,1,2}.
 *   scales: R*G units of 256 bytes from byte R*G*4096; unit (b,g) starts
 *           at R*G*4096 + (b*G + g)*256 and holds the 128 fp16 scales
 *           s[128b + r][g], r = 0..127, little-endian.
 *
 *   total:  R*G*4352 bytes.
 */

int64_t orc_tiled_bytes(int64_t N, int64_t K) {
    int64_t R = (N + 127) / 128, G = K / 128;
    return R * G * 4352;
}

static void put_u32(uint8_t* p, uint32_t w) {
    p[0] = (uint8_t)w; p[1] = (uint8_t)(w >> 8); p[2] = (uint8_t)(w >> 16); p[3] = (uint8_t)(w >> 24);
}

static uint32_t get_u32(const uint8_t* p) {
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

/* Byte offset of the 32-bit code word that holds weight (n, k), and the bit
   position of that weight inside it. */
static void tiled_code_position(int64_t K, int64_t n, int64_t k, int64_t* word_off, int* bit) {
    int64_t G = K / 128;
    int64_t b = n / 128, r = n % 128;
    int64_t g = k / 128, kk = k % 128;
    int64_t h = kk / 64, q = (kk % 64) / 16, j = kk % 16;
    *word_off = (b * G + g) * 4096 + 2048 * h + 16 * r + 4 * q;
    *bit = (int)(16 * (j % 2) + 2 * (j / 2));
}

/* Byte offset of the fp16 scale of row n, group g. */
static int64_t tiled_scale_position(int64_t N, int64_t K, int64_t n, int64_t g) {
    int64_t R = (N + 127) / 128, G = K / 128;
    int64_t b = n / 128, r = n % 128;
    return R * G * 4096 + (b * G + g) * 256 + 2 * r;
}

/* on-disk packed [N,K/4] + fp16 scales [N,K/128] -> tiled.
   Returns the number of reserved code-11 entries (stored as weight 0). */
int64_t orc_repack(const uint8_t* packed, const uint16_t* scales, int64_t N, int64_t K,
                   uint8_t* tiled) {
    int64_t reserved = 0;
    int64_t Np = (N + 127) / 128 * 128, G = K / 128;
    memset(tiled, 0, (size_t)orc_tiled_bytes(N, K));
    for (int64_t n = 0; n < Np; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            int t = 0;
            if (n < N) {
                unsigned code = packed_code(packed, K, n, k);
                if (code == 3u) ++reserved;
                t = orc_code_to_ternary(code);
            }
            int64_t off; int bit;
            tiled_code_position(K, n, k, &off, &bit);
            uint32_t w = get_u32(tiled + off);
            w |= (uint32_t)(t + 1) << bit;
            put_u32(tiled + off, w);
        }
        for (int64_t g = 0; g < G; ++g) {
            uint16_t s = n < N ? scales[n * G + g] : 0;
            int64_t off = tiled_scale_position(N, K, n, g);
            tiled[off] = (uint8_t)(s & 0xFF);
            tiled[off + 1] = (uint8_t)(s >> 8);
        }
    }
    return reserved;
}

/* tiled -> on-disk packed [N,K/4] + fp16 scales [N,K/128] (rows < N only).
   Returns the number of biased codes equal to 3 (invalid; written as 00). */
int64_t orc_unrepack(const uint8_t* tiled, int64_t N, int64_t K,
                     uint8_t* packed, uint16_t* scales) {
    int64_t invalid = 0, G = K / 128;
    memset(packed, 0, (size_t)(N * (K / 4)));
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            int64_t off; int bit;
            tiled_code_position(K, n, k, &off, &bit);
            unsigned v = (get_u32(tiled + off) >> bit) & 3u;
            unsigned code;
            if (v == 0) code = 2u;        /* t = -1 */
            else if (v == 2) code = 1u;   /* t = +1 */
            else { code = 0u; if (v == 3) ++invalid; }
            packed[n * (K / 4) + k / 4] |= (uint8_t)(code << (2 * (k % 4)));
        }
        for (int64_t g = 0; g < G; ++g) {
            int64_t off = tiled_scale_position(N, K, n, g);
            scales[n * G + g] = (uint16_t)(tiled[off] | (tiled[off + 1] << 8));
        }
    }
    return invalid;
}

/* ------------------------------------------------------------------ linear */

/* One output: y = sum_k x[k] * t[n,k] * s[n,k/128] in fp64, k ascending, and
   the tolerance scale sum_k |x[k] * t[n,k] * s[n,k/128]|.  x_f16: the
   activations are fp16 bits, else bf16 bits. */
static void dot_row(const uint16_t* xrow, int x_f16, const uint8_t* packed, const uint16_t* scales,
                    int64_t K, int64_t n, double* y, double* bound) {
    double acc = 0.0, mag = 0.0;
    int64_t G = K / 128;
    for (int64_t k = 0; k < K; ++k) {
        double x = x_f16 ? orc_fp16_to_double(xrow[k]) : orc_bf16_to_double(xrow[k]);
        double w = (double)orc_code_to_ternary(packed_code(packed, K, n, k))
                 * orc_fp16_to_double(scales[n * G + k / 128]);
        acc += x * w;
        mag += fabs(x * w);
    }
    *y = acc;
    *bound = mag;
}

/* Y[m,n] (row stride N) and its bound for all m < M, n < N.
   X is bf16 bits [M, ldx]; packed [N, K/4]; scales fp16 bits [N, K/128]. */
void orc_linear_x(const uint16_t* X, int x_f16, int64_t ldx, const uint8_t* packed,
                  const uint16_t* scales, int64_t M, int64_t N, int64_t K,
                  double* Y, double* bound) {
    #pragma omp parallel for schedule(dynamic, 16) collapse(2)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            dot_row(X + m * ldx, x_f16, packed, scales, K, n, &Y[m * N + n], &bound[m * N + n]);
}

void orc_linear(const uint16_t* X, int64_t ldx, const uint8_t* packed,
                const uint16_t* scales, int64_t M, int64_t N, int64_t K,
                double* Y, double* bound) {
    orc_linear_x(X, 0, ldx, packed, scales, M, N, K, Y, bound);
}

/* Same as orc_linear_x for a list of output columns: Y[m, j] for n = cols[j]. */
void orc_linear_cols_x(const uint16_t* X, int x_f16, int64_t ldx, const uint8_t* packed,
                       const uint16_t* scales, int64_t M, int64_t N, int64_t K,
                       const int64_t* cols, int64_t ncols, double* Y, double* bound) {
    (void)N;
    #pragma omp parallel for schedule(dynamic, 4) collapse(2)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t j = 0; j < ncols; ++j)
            dot_row(X + m * ldx, x_f16, packed, scales, K, cols[j], &Y[m * ncols + j], &bound[m * ncols + j]);
}

void orc_linear_cols(const uint16_t* X, int64_t ldx, const uint8_t* packed,
                     const uint16_t* scales, int64_t M, int64_t N, int64_t K,
                     const int64_t* cols, int64_t ncols, double* Y, double* bound) {
    orc_linear_cols_x(X, 0, ldx, packed, scales, M, N, K, cols, ncols, Y, bound);
}

/* ------------------------------------------------------ INT8 group scales */

/* The reading taken for "compress the FP16 scales to INT8" ("Ternary
   embedding model in vLLM" §6, an outlook without a format): per row one
   fp32 factor f = max_g |s| / 127 and per group q = rint(s * (127 / max_g |s|))
   in [-127, 127], in fp32 with ties to even. */
void orc_quantize_scales(const uint16_t* scales, int64_t N, int64_t K, int8_t* q8, float* f) {
    int64_t G = K / 128;
    for (int64_t n = 0; n < N; ++n) {
        float mx = 0.0f;
        for (int64_t g = 0; g < G; ++g) {
            float v = (float)orc_fp16_to_double(scales[n * G + g]);
            if (fabsf(v) > mx) mx = fabsf(v);
        }
        float inv = mx > 0.0f ? 127.0f / mx : 0.0f;
        f[n] = mx / 127.0f;
        for (int64_t g = 0; g < G; ++g) {
            float r = rintf((float)orc_fp16_to_double(scales[n * G + g]) * inv);
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            q8[n * G + g] = (int8_t)r;
        }
    }
}

/* Y[m,n] = sum_k x[m,k] * t[n,k] * q8[n,k/128] * f[n] in fp64 (X bf16 bits),
   and the bound sum_k |x t q8 f|. */
void orc_linear_s8(const uint16_t* X, int64_t ldx, const uint8_t* packed, const int8_t* q8,
                   const float* f, int64_t M, int64_t N, int64_t K, double* Y, double* bound) {
    int64_t G = K / 128;
    #pragma omp parallel for schedule(dynamic, 16) collapse(2)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double x = orc_bf16_to_double(X[m * ldx + k]);
                double w = (double)orc_code_to_ternary(packed_code(packed, K, n, k))
                         * (double)q8[n * G + k / 128] * (double)f[n];
                acc += x * w;
                mag += fabs(x * w);
            }
            Y[m * N + n] = acc;
            bound[m * N + n] = mag;
        }
}

/* --------------------------------------------------- int8 activations */

/* Per-token absmax quantisation (the reading taken for the page's third
   route, "Ternary embedding model in vLLM" §4.1-§4.3, which leaves the
   quantiser open): in fp32, as the kernel does it, so that both sides take
   every rounding decision in the same precision:
     mx = max_k |x|, a = mx / 127, q = rint(x * (127 / mx)) in [-127, 127];
   rint rounds ties to even (the default rounding mode).  q in natural
   k order, [M, K]. */
void orc_quantize_x(const uint16_t* X, int x_f16, int64_t ldx, int64_t M, int64_t K,
                    int8_t* q, float* a) {
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t* xr = X + m * ldx;
        float mx = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float v = (float)(x_f16 ? orc_fp16_to_double(xr[k]) : orc_bf16_to_double(xr[k]));
            if (fabsf(v) > mx) mx = fabsf(v);
        }
        float inv = mx > 0.0f ? 127.0f / mx : 0.0f;
        a[m] = mx / 127.0f;
        for (int64_t k = 0; k < K; ++k) {
            float v = (float)(x_f16 ? orc_fp16_to_double(xr[k]) : orc_bf16_to_double(xr[k]));
            float r = rintf(v * inv);
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            q[m * K + k] = (int8_t)r;
        }
    }
}

/* Y[m,n] = a[m] * sum_g s[n,g] * sum_{k in g} t[n,k] q[m,k] in fp64 (the
   integer group sums are exact), and the bound sum_k |a q t s|. */
void orc_linear_i8(const int8_t* q, const float* a, const uint8_t* packed, const uint16_t* scales,
                   int64_t M, int64_t N, int64_t K, double* Y, double* bound) {
    int64_t G = K / 128;
    #pragma omp parallel for schedule(dynamic, 16) collapse(2)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t g = 0; g < G; ++g) {
                long isum = 0, iabs = 0;
                for (int64_t k = 128 * g; k < 128 * g + 128; ++k) {
                    int t = orc_code_to_ternary(packed_code(packed, K, n, k));
                    isum += (long)t * q[m * K + k];
                    iabs += labs((long)t * q[m * K + k]);
                }
                double s = orc_fp16_to_double(scales[n * G + g]);
                acc += s * (double)isum;
                mag += fabs(s) * (double)iabs;
            }
            Y[m * N + n] = (double)a[m] * acc;
            bound[m * N + n] = (double)a[m] * mag;
        }
}

/* ------------------------------------------------------------------ SwiGLU */

/* silu(g) * u, with silu(g) = g / (1 + e^-g) (the textbook definition of
   the sigmoid-weighted linear unit), elementwise over count values. */
void orc_swiglu(const double* g, const double* u, int64_t count, double* h) {
    for (int64_t i = 0; i < count; ++i) h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
}

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
int orc_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
