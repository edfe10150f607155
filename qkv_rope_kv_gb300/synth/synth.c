/*
 * Seeded synthetic inputs for the decode QKV stage.
 *
 * This file only MAKES inputs (weights, bias, hidden vectors, positions).  It
 * holds none of the stage's arithmetic: no matvec, no bias add, no rotation,
 * no cache store.  Both the CUDA path (through the benchmark and the tests)
 * and the CPU oracle consume its output; neither depends on the other.
 *
 * Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014; constants as in Vigna's public-domain
 * splitmix64.c), used counter-style: the n-th output (n >= 1) of a stream
 * started at state s is mix(s + n * GOLDEN), so any element can be produced
 * independently and in parallel.
 *
 * Normal deviates: Box-Muller (Box and Muller 1958) in double precision,
 * pair p of a stream draws u1 from output 2p+1 and u2 from output 2p+2;
 * element 2p takes r*cos(2*pi*u2), element 2p+1 takes r*sin(2*pi*u2).
 *
 * Stream keys: key(seed, tensor, layer, index) chains mix() over the four
 * fields, so every (tensor, layer, row or position) gets its own stream.
 * Weight matrices are keyed PER ROW (index = global row number in the
 * concatenated wq|wk|wv layout), so a separately generated wq, wk or wv is
 * bit-identical to the matching row block of the concatenated matrix.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define SYNTH_GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* n-th output (n >= 1) of SplitMix64 started at `state`. */
uint64_t synth_splitmix64(uint64_t state, uint64_t n) {
    return mix64(state + n * SYNTH_GOLDEN);
}

uint64_t synth_stream_key(uint64_t seed, uint32_t tensor, uint32_t layer, uint32_t index) {
    uint64_t k = mix64(seed + SYNTH_GOLDEN);
    k = mix64(k + SYNTH_GOLDEN * (1ULL + (uint64_t)tensor));
    k = mix64(k + SYNTH_GOLDEN * (1ULL + (uint64_t)layer));
    k = mix64(k + SYNTH_GOLDEN * (1ULL + (uint64_t)index));
    return k;
}

/* Standard normal element `i` of the stream with key `key`. */
static inline double normal_at(uint64_t key, uint64_t i) {
    const uint64_t p = i >> 1;
    const uint64_t a = mix64(key + (2 * p + 1) * SYNTH_GOLDEN);
    const uint64_t b = mix64(key + (2 * p + 2) * SYNTH_GOLDEN);
    const double u1 = ((double)(a >> 11) + 1.0) * 0x1.0p-53; /* (0, 1] */
    const double u2 = (double)(b >> 11) * 0x1.0p-53;         /* [0, 1) */
    const double r = sqrt(-2.0 * log(u1));
    const double t = 6.283185307179586476925286766559 * u2;
    return (i & 1) ? r * sin(t) : r * cos(t);
}

/* Round-to-nearest-even f32 -> bf16 bit pattern (input quantisation of the
 * synthetic weights; NaN never occurs for finite normal deviates). */
static inline uint16_t f32_to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

double synth_normal_at(uint64_t key, uint64_t i) { return normal_at(key, i); }

/* out[i] = (float)(sigma * N_i), i in [0, n), one stream (tensor, layer, index). */
void synth_normal_f32(uint64_t seed, uint32_t tensor, uint32_t layer, uint32_t index,
                      int64_t n, double sigma, float* out) {
    const uint64_t key = synth_stream_key(seed, tensor, layer, index);
    for (int64_t i = 0; i < n; ++i) out[i] = (float)(sigma * normal_at(key, (uint64_t)i));
}

/* Row-keyed matrix: out[(r - row0) * ncols + c] = (float)(sigma * N(row r, c)). */
void synth_rows_f32(uint64_t seed, uint32_t tensor, uint32_t layer, int64_t row0, int64_t nrows,
                    int64_t ncols, double sigma, float* out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrows; ++r) {
        const uint64_t key = synth_stream_key(seed, tensor, layer, (uint32_t)(row0 + r));
        float* o = out + r * ncols;
        for (int64_t c = 0; c < ncols; ++c) o[c] = (float)(sigma * normal_at(key, (uint64_t)c));
    }
}

/* Same values as synth_rows_f32, rounded once more to bf16 (RN-even). */
void synth_rows_bf16(uint64_t seed, uint32_t tensor, uint32_t layer, int64_t row0, int64_t nrows,
                     int64_t ncols, double sigma, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrows; ++r) {
        const uint64_t key = synth_stream_key(seed, tensor, layer, (uint32_t)(row0 + r));
        uint16_t* o = out + r * ncols;
        for (int64_t c = 0; c < ncols; ++c)
            o[c] = f32_to_bf16_bits((float)(sigma * normal_at(key, (uint64_t)c)));
    }
}

int synth_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
