/*
 * Seeded synthetic inputs for the ternary linear layer: ternary codes,
 * FP16 group scales and BF16 activations.
 *
 * This module is the one piece shared by the CUDA path's tests/benchmarks
 * and by the CPU oracle.  It holds none of the method's arithmetic (no
 * packing, no decoding, no dot products): it only draws numbers.
 *
 * Generator: counter-based SplitMix64 (G. Steele, D. Lea, C. Flood,
 * "Fast Splittable Pseudorandom Number Generators", OOPSLA 2014), i.e. the
 * i-th draw of a stream is mix(key + (i+1)*gamma) with the published gamma
 * and finaliser constants.  Because every element is a pure function of
 * (seed, stream, index), the output does not depend on the thread count.
 * Uniforms take the top 53 bits.  Normals use the Box-Muller transform
 * (G. Box, M. Muller, Ann. Math. Statist. 1958) on draws 2i and 2i+1,
 * keeping the cosine branch.
 *
 * Rounding to the storage formats (FP16 scales, BF16 activations) is
 * round-to-nearest-even, done once here from the fp64 draw; after that the
 * stored bits are exact inputs for both the GPU path and the oracle.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#define SM64_GAMMA 0x9E3779B97F4A7C15ull

static inline uint64_t sm64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return sm64_mix(sm64_mix(seed + SM64_GAMMA) ^ stream);
}

static inline uint64_t draw(uint64_t key, uint64_t i) {
    return sm64_mix(key + (i + 1) * SM64_GAMMA);
}

static inline double uniform01(uint64_t key, uint64_t i) {
    return (double)(draw(key, i) >> 11) * 0x1.0p-53;
}

static inline double normal01(uint64_t key, uint64_t i) {
    const double two_pi = 6.283185307179586476925286766559;
    double u1 = uniform01(key, 2 * i);
    double u2 = uniform01(key, 2 * i + 1);
    double r = sqrt(-2.0 * log(1.0 - u1)); /* 1-u1 is in (0,1] */
    return r * cos(two_pi * u2);
}

/*
 * Round a finite double to a binary floating format with `sig_bits`
 * significant bits (implicit bit included) and `exp_bits` exponent bits
 * (IEEE-style bias, all-ones exponent is inf/nan), round-to-nearest-even.
 * Returns the raw bit pattern.  Overflow saturates to infinity.
 */
static uint16_t round_to_small_float(double d, int sig_bits, int exp_bits) {
    const int bias = (1 << (exp_bits - 1)) - 1;
    const int mant_bits = sig_bits - 1;
    uint16_t sign = signbit(d) ? (uint16_t)(1u << (exp_bits + mant_bits)) : 0;
    double a = fabs(d);
    if (a == 0.0) return sign;
    int e;
    double m = frexp(a, &e);           /* a = m * 2^e, m in [0.5, 1) */
    int ebiased = e - 1 + bias;        /* a = (2m) * 2^(e-1) */
    uint64_t q;
    if (ebiased >= 1) {
        /* normal: significand 2m in [1,2) with mant_bits fraction bits */
        q = (uint64_t)nearbyint(ldexp(m, sig_bits)); /* in [2^(sig-1), 2^sig] */
        if (q == (1ull << sig_bits)) { q >>= 1; ebiased += 1; }
        if (ebiased >= (1 << exp_bits) - 1)
            return sign | (uint16_t)(((1u << exp_bits) - 1) << mant_bits);
        return sign | (uint16_t)((uint64_t)ebiased << mant_bits)
                    | (uint16_t)(q & ((1ull << mant_bits) - 1));
    }
    /* subnormal: units of 2^(1 - bias - mant_bits) */
    q = (uint64_t)nearbyint(ldexp(a, bias - 1 + mant_bits));
    /* q == 2^mant_bits lands exactly on the smallest normal, which the
       same bit pattern encodes */
    return sign | (uint16_t)q;
}

uint16_t synth_round_fp16(double d) { return round_to_small_float(d, 11, 5); }
uint16_t synth_round_bf16(double d) { return round_to_small_float(d, 8, 8); }

/* Ternary values t in {-1,0,+1}: P(0) = p_zero, P(+1) = P(-1) = (1-p_zero)/2. */
void synth_ternary(uint64_t seed, uint64_t stream, double p_zero,
                   int8_t* out, int64_t start, int64_t n) {
    const uint64_t key = stream_key(seed, stream);
    const double p_neg = 0.5 * (1.0 - p_zero);
    const double p_negzero = p_neg + p_zero;
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double u = uniform01(key, (uint64_t)(start + i));
        out[i] = (int8_t)(u < p_neg ? -1 : (u < p_negzero ? 0 : 1));
    }
}

/* FP16 scales ~ U[lo, hi], rounded RNE. */
void synth_scales_uniform(uint64_t seed, uint64_t stream, double lo, double hi,
                          uint16_t* out, int64_t start, int64_t n) {
    const uint64_t key = stream_key(seed, stream);
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = synth_round_fp16(lo + (hi - lo) * uniform01(key, (uint64_t)(start + i)));
}

/* FP16 scales ~ exp(N(mu, sigma^2)), rounded RNE. */
void synth_scales_lognormal(uint64_t seed, uint64_t stream, double mu, double sigma,
                            uint16_t* out, int64_t start, int64_t n) {
    const uint64_t key = stream_key(seed, stream);
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = synth_round_fp16(exp(mu + sigma * normal01(key, (uint64_t)(start + i))));
}

/* BF16 activations ~ N(0,1), rounded RNE. */
void synth_normal_bf16(uint64_t seed, uint64_t stream, uint16_t* out,
                       int64_t start, int64_t n) {
    const uint64_t key = stream_key(seed, stream);
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = synth_round_bf16(normal01(key, (uint64_t)(start + i)));
}

/* Raw uniform doubles in [0,1), for tests of the generator itself. */
void synth_uniform(uint64_t seed, uint64_t stream, double* out, int64_t n) {
    const uint64_t key = stream_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = uniform01(key, (uint64_t)i);
}

/* Raw SplitMix64 words, for tests of the generator itself. */
void synth_raw(uint64_t seed, uint64_t stream, uint64_t* out, int64_t n) {
    const uint64_t key = stream_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = draw(key, (uint64_t)i);
}

/* Plain sequential SplitMix64 from a state, as published, for a test that
   checks the counter form above against the sequential definition. */
void synth_sequential_splitmix(uint64_t state, uint64_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        state += SM64_GAMMA;
        out[i] = sm64_mix(state);
    }
}

uint64_t synth_stream_key(uint64_t seed, uint64_t stream) {
    return stream_key(seed, stream);
}
