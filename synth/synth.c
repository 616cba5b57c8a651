/*
 * Seeded synthetic inputs shared by the oracle and the CUDA path.
 *
 * This file holds none of the verify method's arithmetic: it only draws
 * numbers.  Every element is a pure function of (seed, tensor_id, index), so
 * any slice of any tensor can be regenerated independently and in parallel.
 *
 *   word(seed, t, i)  = splitmix64(key(seed, t) + i)          (64-bit counter RNG)
 *   key(seed, t)      = splitmix64(seed ^ splitmix64(t ^ 0xA5A5...))
 *   normal(seed,t,i)  = Box-Muller (cos branch) on two 53-bit uniforms drawn from
 *                       word(seed, t, 2i) and word(seed, t, 2i+1), in double
 *
 * splitmix64 is Steele, Lea and Flood's SplitMix generator (OOPSLA 2014) with
 * Vigna's published finaliser constants.  bf16 values are produced from the
 * double sample by round-to-nearest-even on the bit pattern of the float
 * nearest to it (an input quantiser, not a storage point of the method).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t sm64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t key_of(uint64_t seed, uint64_t tensor_id) {
    return sm64(seed ^ sm64(tensor_id ^ 0xA5A5A5A5A5A5A5A5ull));
}

/* uniform in (0, 1]: never zero, so log() is finite */
static inline double u01_open0(uint64_t w) {
    return ((double)(w >> 11) + 1.0) * (1.0 / 9007199254740992.0);
}
/* uniform in [0, 1) */
static inline double u01(uint64_t w) {
    return (double)(w >> 11) * (1.0 / 9007199254740992.0);
}

static inline double normal_at(uint64_t key, uint64_t i) {
    double u1 = u01_open0(sm64(key + 2 * i));
    double u2 = u01(sm64(key + 2 * i + 1));
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

/* float -> bf16 bit pattern, round to nearest even; NaN kept quiet. */
static inline uint16_t to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

void synth_normal_f64(uint64_t seed, uint64_t tensor_id, double mean, double sigma,
                      double* out, int64_t n) {
    uint64_t key = key_of(seed, tensor_id);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = mean + sigma * normal_at(key, (uint64_t)i);
}

void synth_normal_f32(uint64_t seed, uint64_t tensor_id, double mean, double sigma,
                      float* out, int64_t n) {
    uint64_t key = key_of(seed, tensor_id);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (float)(mean + sigma * normal_at(key, (uint64_t)i));
}

void synth_normal_bf16(uint64_t seed, uint64_t tensor_id, double mean, double sigma,
                       uint16_t* out, int64_t n) {
    uint64_t key = key_of(seed, tensor_id);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = to_bf16((float)(mean + sigma * normal_at(key, (uint64_t)i)));
}

/* integers uniform in [lo, hi) (modulo bias below 2^-40 for the ranges used) */
void synth_uniform_i32(uint64_t seed, uint64_t tensor_id, int32_t lo, int32_t hi,
                       int32_t* out, int64_t n) {
    uint64_t key = key_of(seed, tensor_id);
    uint64_t span = (uint64_t)((int64_t)hi - (int64_t)lo);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = lo + (int32_t)(sm64(key + (uint64_t)i) % span);
}

/* raw 64-bit words, for tests of the generator itself */
void synth_words(uint64_t seed, uint64_t tensor_id, uint64_t* out, int64_t n) {
    uint64_t key = key_of(seed, tensor_id);
    for (int64_t i = 0; i < n; ++i) out[i] = sm64(key + (uint64_t)i);
}
