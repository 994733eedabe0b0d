/* Seeded, counter-based generator of synthetic normal deviates.
 *
 * Input generation only: it holds none of the attention, cache or allocator
 * arithmetic.  Both the oracle side and the CUDA side of every test and
 * benchmark receive the same host arrays produced here.
 *
 * Definition (so the Python helpers can reproduce the integer parts):
 *   mix64(z)   = SplitMix64 finaliser: z ^= z>>30; z *= 0xBF58476D1CE4E5B9;
 *                z ^= z>>27; z *= 0x94D049BB133111EB; z ^= z>>31
 *   key(s, t)  = mix64(s + (t+1) * 0x9E3779B97F4A7C15)     stream t of seed s
 *   h(k, i)    = mix64(k + (i+1) * 0x9E3779B97F4A7C15)     i-th draw of a stream
 *   normal(k, i) = sqrt(-2 ln u1) * cos(2 pi u2),  Box-Muller in double, with
 *                u1 = ((h(k,2i) >> 11) + 1) * 2^-53   in (0, 1]
 *                u2 =  (h(k,2i+1) >> 11)    * 2^-53   in [0, 1)
 * The float result is that double rounded to nearest float.
 */
#include <math.h>
#include <stdint.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t synth_key(uint64_t seed, uint64_t stream) {
    return mix64(seed + (stream + 1) * GOLDEN);
}

static inline double normal_at(uint64_t key, uint64_t i) {
    const double two_m53 = 1.0 / 9007199254740992.0;
    uint64_t a = mix64(key + (2 * i + 1) * GOLDEN);
    uint64_t b = mix64(key + (2 * i + 2) * GOLDEN);
    double u1 = (double)((a >> 11) + 1) * two_m53;
    double u2 = (double)(b >> 11) * two_m53;
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

/* out[j] = (float) normal(key(seed, stream), offset + j), j < n */
void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset,
                      int64_t n, float* out) {
    const uint64_t k = synth_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) out[j] = (float)normal_at(k, offset + (uint64_t)j);
}

/* out[j] = normal(key(seed, stream), offset + j) in double, j < n */
void synth_normal_f64(uint64_t seed, uint64_t stream, uint64_t offset,
                      int64_t n, double* out) {
    const uint64_t k = synth_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) out[j] = normal_at(k, offset + (uint64_t)j);
}

/* out[j] = h(key(seed, stream), offset + j), raw 64-bit draws */
void synth_u64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
               uint64_t* out) {
    const uint64_t k = synth_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) out[j] = mix64(k + (offset + (uint64_t)j + 1) * GOLDEN);
}
