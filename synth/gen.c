/*
 * Seeded, counter-based synthetic input generator.
 *
 * This file holds no attention arithmetic: it only draws the raw numbers
 * (latent rows, RoPE-key rows, absorbed queries, sequence lengths, page
 * permutations) that both the fp64 oracle and the CUDA path consume.
 *
 * Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014).  The i-th output of a
 * SplitMix64 sequence whose state starts at `key` is
 *     mix64(key + (i + 1) * 0x9E3779B97F4A7C15)
 * so any element can be drawn without drawing the ones before it.  Each
 * tensor of a workload owns one (seed, stream) key.
 *
 * Normals: Box-Muller on two consecutive draws (u1 in (0,1], u2 in [0,1));
 * element 2k takes the cosine branch, element 2k+1 the sine branch.
 */
#include <math.h>
#include <stdint.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t draw(uint64_t key, uint64_t i) {
    return mix64(key + (i + 1) * GOLDEN_GAMMA);
}

uint64_t synth_stream_key(uint64_t seed, uint64_t stream) {
    return mix64(mix64(seed) ^ (stream * 0xD1B54A32D192ED03ULL + 0x632BE59BD9B4E019ULL));
}

uint64_t synth_draw_u64(uint64_t seed, uint64_t stream, uint64_t i) {
    return draw(synth_stream_key(seed, stream), i);
}

static inline double normal_at(uint64_t key, uint64_t i) {
    const uint64_t k = i >> 1;
    const uint64_t h1 = draw(key, 2 * k), h2 = draw(key, 2 * k + 1);
    const double u1 = ((double)(h1 >> 11) + 1.0) * 0x1.0p-53; /* (0, 1] */
    const double u2 = (double)(h2 >> 11) * 0x1.0p-53;         /* [0, 1) */
    const double r = sqrt(-2.0 * log(u1));
    const double a = 6.283185307179586476925286766559 * u2;
    return (i & 1) ? r * sin(a) : r * cos(a);
}

/* Round a double to the nearest bfloat16 (ties to even); returns the bits. */
static inline uint16_t to_bf16_bits(double x) {
    if (x != x) return 0x7FC0;
    union { float f; uint32_t u; } v;
    const double ax = fabs(x);
    double r;
    if (ax == 0.0) {
        r = x;
    } else if (ax < 0x1.0p-126) { /* bf16 subnormal spacing is 2^-133 */
        r = nearbyint(x * 0x1.0p133) * 0x1.0p-133;
    } else {
        int e;
        const double m = frexp(x, &e);           /* |m| in [0.5, 1) */
        r = ldexp(nearbyint(m * 256.0) / 256.0, e); /* 8 significant bits */
        if (fabs(r) > 0x1.FEp127) r = (x > 0) ? INFINITY : -INFINITY;
    }
    v.f = (float)r; /* exact: r has at most 8 significant bits */
    return (uint16_t)(v.u >> 16);
}

void synth_normal_f64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                      double scale, double* out) {
    const uint64_t key = synth_stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) out[j] = scale * normal_at(key, offset + (uint64_t)j);
}

void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                      double scale, float* out) {
    const uint64_t key = synth_stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) out[j] = (float)(scale * normal_at(key, offset + (uint64_t)j));
}

void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                       double scale, uint16_t* out) {
    const uint64_t key = synth_stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) out[j] = to_bf16_bits(scale * normal_at(key, offset + (uint64_t)j));
}

/* Gathered variant: out row r (of `width` elements) is element range
 * [row_index[r] * width, +width) of the stream.  Used to draw the raw rows of
 * a subset of tokens (e.g. one sequence) of a larger workload. */
void synth_normal_rows_bf16(uint64_t seed, uint64_t stream, const int64_t* row_index,
                            int64_t rows, int64_t width, double scale, uint16_t* out) {
    const uint64_t key = synth_stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const uint64_t base = (uint64_t)row_index[r] * (uint64_t)width;
        for (int64_t k = 0; k < width; ++k)
            out[r * width + k] = to_bf16_bits(scale * normal_at(key, base + (uint64_t)k));
    }
}

/* Uniform integers in [lo, hi] by multiply-shift on the top 32 bits. */
void synth_uniform_int(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                       int64_t lo, int64_t hi, int32_t* out) {
    const uint64_t key = synth_stream_key(seed, stream);
    const uint64_t span = (uint64_t)(hi - lo + 1);
    for (int64_t j = 0; j < n; ++j) {
        const uint64_t h = draw(key, offset + (uint64_t)j) >> 32;
        out[j] = (int32_t)(lo + (int64_t)((h * span) >> 32));
    }
}

/* Fisher-Yates shuffle of 0..n-1 (Durstenfeld's in-place form). */
void synth_permutation(uint64_t seed, uint64_t stream, int64_t n, int32_t* out) {
    const uint64_t key = synth_stream_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
    uint64_t t = 0;
    for (int64_t i = n - 1; i > 0; --i) {
        const uint64_t h = draw(key, t++) >> 32;
        const int64_t j = (int64_t)((h * (uint64_t)(i + 1)) >> 32);
        const int32_t tmp = out[i];
        out[i] = out[j];
        out[j] = tmp;
    }
}
