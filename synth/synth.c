/*
 * Seeded synthetic inputs for the GRPO loss workloads.
 *
 * This module holds no arithmetic of the loss itself: it only draws the
 * random numbers the workloads are made of (hidden states, lm_head weight,
 * sampled tokens, completion lengths, rewards) and rounds fp32 to the 16-bit
 * storage types.  Both the CPU oracle and the GPU path consume its output.
 *
 * Counter-based generator: value (seed, stream, i) is the i-th output of a
 * splitmix64 sequence whose starting state is itself a splitmix64 hash of
 * (seed, stream).  Every element can be produced independently, so the fill
 * loops parallelise without changing a single bit of the result.
 *
 * Normals use the cosine branch of Box-Muller on two consecutive uniforms
 * (indices 2i and 2i+1).  Uniforms lie in (0, 1], so log(u) is finite.
 */
#include <stdint.h>
#include <math.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* i-th output of the splitmix64 sequence that starts at state s0 */
static inline uint64_t splitmix_at(uint64_t s0, uint64_t i) {
    return mix64(s0 + (i + 1) * GOLDEN);
}

uint64_t synth_stream_state(uint64_t seed, uint64_t stream) {
    return splitmix_at(mix64(seed), stream);
}

uint64_t synth_u64(uint64_t seed, uint64_t stream, uint64_t i) {
    return splitmix_at(synth_stream_state(seed, stream), i);
}

static inline double unit_open0(uint64_t x) {           /* (0, 1] */
    return (double)((x >> 11) + 1) * (1.0 / 9007199254740992.0);
}

static inline double normal_at(uint64_t s0, uint64_t i) {
    double u1 = unit_open0(splitmix_at(s0, 2 * i));
    double u2 = unit_open0(splitmix_at(s0, 2 * i + 1));
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

/* out[i] = base[i] + sigma * N_(offset+i)   (base may be NULL -> 0) */
void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                      float sigma, const float* base, float* out) {
    uint64_t s0 = synth_stream_state(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float v = (float)(sigma * normal_at(s0, offset + (uint64_t)i));
        out[i] = base ? base[i] + v : v;
    }
}

/* integers uniform in [lo, hi] (inclusive), by 64x64->128 multiply-high */
void synth_uniform_int(uint64_t seed, uint64_t stream, int64_t n, int64_t lo, int64_t hi,
                       int32_t* out) {
    uint64_t s0 = synth_stream_state(seed, stream);
    uint64_t span = (uint64_t)(hi - lo) + 1;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint64_t x = splitmix_at(s0, (uint64_t)i);
        unsigned __int128 prod = (unsigned __int128)x * span;
        out[i] = (int32_t)(lo + (int64_t)(uint64_t)(prod >> 64));
    }
}

/* Bernoulli(1/2) from the top bit */
void synth_bits(uint64_t seed, uint64_t stream, int64_t n, int32_t* out) {
    uint64_t s0 = synth_stream_state(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)(splitmix_at(s0, (uint64_t)i) >> 63);
}

/* Fisher-Yates permutation of 0..n-1 driven by stream `stream` */
void synth_permutation(uint64_t seed, uint64_t stream, int32_t n, int32_t* out) {
    uint64_t s0 = synth_stream_state(seed, stream);
    for (int32_t i = 0; i < n; ++i) out[i] = i;
    for (int32_t i = n - 1; i > 0; --i) {
        uint64_t x = splitmix_at(s0, (uint64_t)(n - 1 - i));
        unsigned __int128 prod = (unsigned __int128)x * (uint64_t)(i + 1);
        int32_t j = (int32_t)(uint64_t)(prod >> 64);
        int32_t t = out[i]; out[i] = out[j]; out[j] = t;
    }
}

/* fp32 -> bf16 bit pattern, round to nearest even (finite inputs) */
void synth_to_bf16(const float* in, int64_t n, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u;
        memcpy(&u, &in[i], 4);
        u += 0x7FFFu + ((u >> 16) & 1u);
        out[i] = (uint16_t)(u >> 16);
    }
}

/* fp32 -> IEEE binary16 bit pattern, round to nearest even, overflow -> inf */
void synth_to_f16(const float* in, int64_t n, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u;
        memcpy(&u, &in[i], 4);
        uint32_t sign = (u >> 16) & 0x8000u;
        uint32_t ax = u & 0x7FFFFFFFu;
        uint16_t h;
        if (ax >= 0x7F800000u) {                         /* inf / nan */
            h = (uint16_t)(sign | 0x7C00u | (ax > 0x7F800000u ? 0x200u : 0u));
        } else if (ax >= 0x477FF000u) {                  /* rounds to >= 65520 -> inf */
            h = (uint16_t)(sign | 0x7C00u);
        } else if (ax >= 0x38800000u) {                  /* normal half */
            uint32_t m = ax + 0xFFFu + ((ax >> 13) & 1u);
            h = (uint16_t)(sign | ((m - 0x38000000u) >> 13));
        } else {                                         /* subnormal half or zero */
            int e = (int)(ax >> 23);
            if (e < 102) {
                h = (uint16_t)sign;                      /* below half of the smallest subnormal */
            } else {
                uint32_t mant = (ax & 0x7FFFFFu) | 0x800000u;
                int shift = 126 - e;                     /* so that result = mant >> shift */
                uint32_t q = mant >> shift;
                uint32_t rem = mant & ((1u << shift) - 1u);
                uint32_t half = 1u << (shift - 1);
                if (rem > half || (rem == half && (q & 1u))) q += 1u;
                h = (uint16_t)(sign | q);
            }
        }
        out[i] = h;
    }
}

/* fp32 -> OCP FP8 E4M3 bit pattern of x / scale: round to nearest even,
 * saturating to +-448 (the format has no infinities; 0x7F / 0xFF are NaN). */
static uint8_t f32_to_e4m3(float xf) {
    double x = (double)xf;
    uint8_t sign = 0;
    if (x < 0) { sign = 0x80; x = -x; }
    if (x >= 448.0) return (uint8_t)(sign | 0x7E);
    if (x < ldexp(1.0, -10)) {                            /* below half the smallest subnormal */
        return sign;
    }
    int e;
    double m = frexp(x, &e);                              /* x = m * 2^e, m in [0.5, 1) */
    int exp_unbiased = e - 1;                             /* x = 1.f * 2^(e-1) */
    uint32_t code;
    if (exp_unbiased < -6) {                              /* subnormal: units of 2^-9 */
        double q = x / ldexp(1.0, -9);
        double fl = floor(q);
        double r = q - fl;
        uint32_t n = (uint32_t)fl;
        if (r > 0.5 || (r == 0.5 && (n & 1u))) n += 1;
        code = n;                                         /* n == 8 rolls into the smallest normal */
    } else {
        double frac = m * 2.0 - 1.0;                      /* in [0, 1) */
        double q = frac * 8.0;
        double fl = floor(q);
        double r = q - fl;
        uint32_t mant = (uint32_t)fl;
        if (r > 0.5 || (r == 0.5 && (mant & 1u))) mant += 1;
        uint32_t be = (uint32_t)(exp_unbiased + 7);
        if (mant == 8) { mant = 0; be += 1; }
        code = (be << 3) | mant;
        if (code > 0x7E) code = 0x7E;
    }
    return (uint8_t)(sign | code);
}

void synth_to_e4m3(const float* in, int64_t n, float scale, uint8_t* out) {
    const float inv = 1.0f / scale;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_e4m3(in[i] * inv);
}

/* fp32 -> OCP FP8 E5M2 bit pattern: 5 exponent bits (bias 15), 2 mantissa
 * bits; round to nearest even, saturating to +-57344 (the format's infinities
 * 0x7C / 0xFC and NaNs are never produced from finite inputs). */
static uint8_t f32_to_e5m2(float xf) {
    double x = (double)xf;
    uint8_t sign = 0;
    if (x < 0) { sign = 0x80; x = -x; }
    if (x >= 57344.0) return (uint8_t)(sign | 0x7B);
    if (x < ldexp(1.0, -17)) return sign;                 /* below half the smallest subnormal */
    int e;
    double m = frexp(x, &e);
    int exp_unbiased = e - 1;
    uint32_t code;
    if (exp_unbiased < -14) {                             /* subnormal: units of 2^-16 */
        double q = x / ldexp(1.0, -16);
        double fl = floor(q);
        double r = q - fl;
        uint32_t n = (uint32_t)fl;
        if (r > 0.5 || (r == 0.5 && (n & 1u))) n += 1;
        code = n;                                         /* n == 4 is the smallest normal's code */
    } else {
        double q = (m * 2.0 - 1.0) * 4.0;
        double fl = floor(q);
        double r = q - fl;
        uint32_t mant = (uint32_t)fl;
        if (r > 0.5 || (r == 0.5 && (mant & 1u))) mant += 1;
        uint32_t be = (uint32_t)(exp_unbiased + 15);
        if (mant == 4) { mant = 0; be += 1; }
        code = (be << 2) | mant;
        if (code > 0x7B) code = 0x7B;
    }
    return (uint8_t)(sign | code);
}

void synth_to_e5m2(const float* in, int64_t n, float scale, uint8_t* out) {
    const float inv = 1.0f / scale;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_e5m2(in[i] * inv);
}
