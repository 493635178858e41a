/*
 * Seeded, counter-based synthetic input generator.
 *
 * Holds no arithmetic of the selective scan itself: it only turns
 * (seed, tensor id, element index) into pseudo-random numbers, so that
 * any element of any tensor can be regenerated on its own (a single
 * (batch, channel) row of a 671M-element tensor costs only that row).
 *
 * Definitions:
 *   splitmix64(x): Steele, Lea & Flood, "Fast splittable pseudorandom
 *     number generators" (OOPSLA 2014), the 64-bit finaliser with the
 *     published constants.
 *   word(seed, tid, i) = splitmix64(key(seed, tid) + i),
 *     key(seed, tid)   = splitmix64(seed * 0x100000001B3 ^ splitmix64(tid + 1)).
 *   uniform(seed, tid, i) = ((word >> 11) + 0.5) * 2^-53, in (0, 1).
 *   normal(seed, tid, i)  = Box-Muller on uniforms 2i and 2i+1:
 *     sqrt(-2 ln U1) * cos(2 pi U2), computed in double, rounded to float.
 *   bf16 rounding: round-to-nearest-even of the float's top 16 bits.
 */
#include <stdint.h>
#include <math.h>

static inline uint64_t splitmix64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tid) {
    return splitmix64(seed * 0x100000001B3ull ^ splitmix64(tid + 1));
}

static inline double unit_open(uint64_t w) {
    return ((double)(w >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static inline double normal_at(uint64_t key, uint64_t i) {
    double u1 = unit_open(splitmix64(key + 2 * i));
    double u2 = unit_open(splitmix64(key + 2 * i + 1));
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925 * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    union { float f; uint32_t u; } v;
    v.f = f;
    uint32_t lsb = (v.u >> 16) & 1u;
    return (uint16_t)((v.u + 0x7FFFu + lsb) >> 16);
}

/* normal samples for element indices idx[0..count) (idx == NULL: start + k) */
void synth_normal_f32(uint64_t seed, uint64_t tid, const int64_t* idx, int64_t start,
                      int64_t count, float* out) {
    uint64_t key = stream_key(seed, tid);
    for (int64_t k = 0; k < count; ++k) {
        uint64_t i = (uint64_t)(idx ? idx[k] : start + k);
        out[k] = (float)normal_at(key, i);
    }
}

void synth_normal_bf16(uint64_t seed, uint64_t tid, const int64_t* idx, int64_t start,
                       int64_t count, uint16_t* out) {
    uint64_t key = stream_key(seed, tid);
    for (int64_t k = 0; k < count; ++k) {
        uint64_t i = (uint64_t)(idx ? idx[k] : start + k);
        out[k] = f32_to_bf16_rne((float)normal_at(key, i));
    }
}

/* uniform samples in (0, 1), double */
void synth_uniform_f64(uint64_t seed, uint64_t tid, int64_t start, int64_t count, double* out) {
    uint64_t key = stream_key(seed, tid);
    for (int64_t k = 0; k < count; ++k) out[k] = unit_open(splitmix64(key + (uint64_t)(start + k)));
}

void synth_f32_to_bf16(const float* in, int64_t count, uint16_t* out) {
    for (int64_t k = 0; k < count; ++k) out[k] = f32_to_bf16_rne(in[k]);
}
