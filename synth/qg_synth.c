/*
 * Seeded synthetic inputs shared by the CPU oracle and the CUDA path.
 *
 * This file holds no arithmetic of the decode step itself: it only draws
 * random numbers and writes them out as f32 values, token ids or raw GGUF
 * k-quant block bytes.  Both sides receive the same bytes.
 *
 * Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014), used counter-based: value i of the stream
 * with seed s is mix(s + (i + 1) * 0x9E3779B97F4A7C15).  Any element can be
 * computed on its own, so the big tensors are filled in parallel and the
 * result does not depend on the thread count.
 *
 * Normals: Marsaglia's polar method (Marsaglia and Bray, 1964) with a natural
 * logarithm written here from the atanh series, so that only +, -, *, / and
 * sqrt are used.  Built with -ffp-contract=off, the output is bit-identical on
 * x86-64 and AArch64.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t sm64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_at(uint64_t seed, uint64_t i) {
    return sm64_mix(seed + (i + 1) * GOLDEN);
}

/* uniform double in [0, 1) from the top 53 bits */
static inline double u01(uint64_t x) { return (double)(x >> 11) * (1.0 / 9007199254740992.0); }

/* ln(s) for s > 0 using s = m * 2^e, m in [sqrt(1/2), sqrt(2)), and
 * ln(m) = 2 * atanh(z), z = (m - 1) / (m + 1), summed until the terms vanish. */
static double series_ln(double s) {
    uint64_t bits;
    memcpy(&bits, &s, 8);
    int e = (int)((bits >> 52) & 0x7FF) - 1023;
    bits = (bits & 0x000FFFFFFFFFFFFFULL) | 0x3FF0000000000000ULL; /* m in [1, 2) */
    double m;
    memcpy(&m, &bits, 8);
    if (m > 1.4142135623730951) { m = m * 0.5; e += 1; }
    double z = (m - 1.0) / (m + 1.0);
    double z2 = z * z, term = z, sum = 0.0;
    for (int k = 1; k < 60; k += 2) {
        double t = term / (double)k;
        double ns = sum + t;
        if (ns == sum) break;
        sum = ns;
        term = term * z2;
    }
    return (double)e * 0.69314718055994530942 + 2.0 * sum;
}

/* Normal j of stream `seed`: pair p = j/2 tries up to 32 (v1, v2) draws from
 * counters [64p, 64p + 64); both members of an accepted pair are used. */
static double normal_at(uint64_t seed, uint64_t j) {
    uint64_t p = j >> 1;
    for (int a = 0; a < 32; a++) {
        double v1 = 2.0 * u01(stream_at(seed, 64 * p + 2 * a)) - 1.0;
        double v2 = 2.0 * u01(stream_at(seed, 64 * p + 2 * a + 1)) - 1.0;
        double s = v1 * v1 + v2 * v2;
        if (s > 0.0 && s < 1.0) {
            double f = sqrt(-2.0 * series_ln(s) / s);
            return (j & 1) ? v2 * f : v1 * f;
        }
    }
    return 0.0;
}

/* IEEE binary16 bits of a finite non-negative float below 65504, round to
 * nearest even (only used for the block scales drawn in [0, dmax)). */
static uint16_t f32_to_f16_bits(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u;
    int32_t exp = (int32_t)((x >> 23) & 0xFF) - 127 + 15;
    uint32_t mant = x & 0x7FFFFFu;
    if (((x >> 23) & 0xFF) == 0) return (uint16_t)sign; /* zero / f32 subnormal */
    if (exp >= 31) return (uint16_t)(sign | 0x7BFFu);    /* clamp to max finite */
    if (exp <= 0) {                                      /* f16 subnormal */
        if (exp < -10) return (uint16_t)sign;
        mant |= 0x800000u;
        uint32_t shift = (uint32_t)(14 - exp);
        uint32_t q = mant >> shift;
        uint32_t rem = mant & ((1u << shift) - 1u), half = 1u << (shift - 1);
        if (rem > half || (rem == half && (q & 1u))) q++;
        return (uint16_t)(sign | q);
    }
    uint32_t q = ((uint32_t)exp << 10) | (mant >> 13);
    uint32_t rem = mant & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (q & 1u))) q++;
    return (uint16_t)(sign | q);
}

uint64_t qs_fnv1a64(const char* s) {
    uint64_t h = 0xCBF29CE484222325ULL;
    for (; *s; ++s) { h ^= (uint8_t)*s; h *= 0x100000001B3ULL; }
    return h;
}

/* Per-tensor sub-seed: SplitMix64 applied to master XOR FNV-1a(name). */
uint64_t qs_subseed(uint64_t master, const char* name) {
    return sm64_mix(master ^ qs_fnv1a64(name));
}

uint64_t qs_u64(uint64_t seed, uint64_t i) { return stream_at(seed, i); }
double qs_normal_f64(uint64_t seed, uint64_t j) { return normal_at(seed, j); }
double qs_ln(double s) { return series_ln(s); }
uint16_t qs_f16_bits(float f) { return f32_to_f16_bits(f); }

void qs_normal_f32(uint64_t seed, float mu, float sigma, float* out, int64_t n) {
    #pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; j++)
        out[j] = (float)((double)mu + (double)sigma * normal_at(seed, (uint64_t)j));
}

void qs_uniform_f32(uint64_t seed, float lo, float hi, float* out, int64_t n) {
    #pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; j++) {
        double u = u01(stream_at(seed, (uint64_t)j));
        out[j] = (float)((double)lo + ((double)hi - (double)lo) * u);
    }
}

void qs_bytes(uint64_t seed, uint8_t* out, int64_t n) {
    int64_t nw = n / 8;
    #pragma omp parallel for schedule(static)
    for (int64_t w = 0; w < nw; w++) {
        uint64_t v = stream_at(seed, (uint64_t)w);
        memcpy(out + 8 * w, &v, 8);
    }
    if (n % 8) {
        uint64_t v = stream_at(seed, (uint64_t)nw);
        memcpy(out + 8 * nw, &v, (size_t)(n % 8));
    }
}

/* Token ids uniform in [0, vocab). */
void qs_tokens(uint64_t seed, uint32_t vocab, uint32_t* out, int64_t n) {
    for (int64_t j = 0; j < n; j++) out[j] = (uint32_t)(stream_at(seed, (uint64_t)j) % vocab);
}

/*
 * Random Q4_K super-blocks (144 bytes each): fp16 d and dmin drawn uniform in
 * [0, dmax), then 140 uniform random bytes for the 12 packed scale/min bytes
 * and the 128 quant bytes.  The 12 bytes hold exactly eight 6-bit scales and
 * eight 6-bit mins with every bit used once, so uniform bytes give uniform
 * independent 6-bit scales and mins; the quant nibbles are uniform in 0..15.
 */
void qs_q4k_blocks(uint64_t seed, float dmax, uint8_t* out, int64_t nblocks) {
    #pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nblocks; b++) {
        uint64_t base = (uint64_t)b * 20;
        uint8_t* blk = out + 144 * b;
        float d = (float)((double)dmax * u01(stream_at(seed, base + 0)));
        float dm = (float)((double)dmax * u01(stream_at(seed, base + 1)));
        uint16_t hd = f32_to_f16_bits(d), hm = f32_to_f16_bits(dm);
        blk[0] = (uint8_t)(hd & 0xFF); blk[1] = (uint8_t)(hd >> 8);
        blk[2] = (uint8_t)(hm & 0xFF); blk[3] = (uint8_t)(hm >> 8);
        for (int w = 0; w < 18; w++) {
            uint64_t v = stream_at(seed, base + 2 + (uint64_t)w);
            int off = 4 + 8 * w;
            int len = (off + 8 <= 144) ? 8 : 144 - off;
            memcpy(blk + off, &v, (size_t)len);
        }
    }
}

/*
 * Random Q6_K super-blocks (210 bytes each): 128 low-nibble bytes, 64
 * high-2-bit bytes and 16 int8 scales, all uniform random bytes (so every
 * 6-bit quant is uniform in 0..63 and every scale uniform in -128..127), then
 * the fp16 d drawn uniform in [0, dmax).
 */
void qs_q6k_blocks(uint64_t seed, float dmax, uint8_t* out, int64_t nblocks) {
    #pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nblocks; b++) {
        uint64_t base = (uint64_t)b * 27;
        uint8_t* blk = out + 210 * b;
        for (int w = 0; w < 26; w++) {
            uint64_t v = stream_at(seed, base + (uint64_t)w);
            memcpy(blk + 8 * w, &v, 8);
        }
        float d = (float)((double)dmax * u01(stream_at(seed, base + 26)));
        uint16_t hd = f32_to_f16_bits(d);
        blk[208] = (uint8_t)(hd & 0xFF); blk[209] = (uint8_t)(hd >> 8);
    }
}
