/*
 * Seeded synthetic-input kernels shared by the test harness, the benchmark and
 * the oracle-side checks.  Nothing here computes any step of speculative
 * verification or scheduling: it only produces random numbers, logits and
 * bf16 encodings.  The composite recipes (which seed feeds which array) live in
 * specsynth/__init__.py.
 *
 * Generators, each written from its published definition:
 *   - SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 *     generators", OOPSLA 2014), used in counter form: output i of stream
 *     `seed` is mix64(seed + (i + 1) * 0x9E3779B97F4A7C15).
 *   - Box-Muller transform (Box & Muller 1958): normals 2k and 2k+1 come from
 *     uniforms 2k and 2k+1 of the same stream.
 *   - Gumbel-max sampling (Gumbel 1954): argmax_v (y_v + G_v) with
 *     G_v = -log(-log U_v) is a draw from the categorical softmax(y).
 *   - fp32 -> bf16 by round-to-nearest-even on the bit pattern.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static const uint64_t GOLDEN = 0x9E3779B97F4A7C15ULL;

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_at(uint64_t seed, uint64_t i) {
    return mix64(seed + (i + 1ULL) * GOLDEN);
}

/* 53-bit uniform in [0, 1). */
static inline double u53(uint64_t seed, uint64_t i) {
    return (double)(stream_at(seed, i) >> 11) * 0x1.0p-53;
}

/* 53-bit uniform strictly inside (0, 1). */
static inline double u53_open(uint64_t seed, uint64_t i) {
    return ((double)(stream_at(seed, i) >> 11) + 0.5) * 0x1.0p-53;
}

void synth_raw64(uint64_t seed, uint64_t start, uint64_t n, uint64_t* out) {
    for (uint64_t k = 0; k < n; ++k) out[k] = stream_at(seed, start + k);
}

void synth_uniform_f64(uint64_t seed, uint64_t start, uint64_t n, double* out) {
    for (uint64_t k = 0; k < n; ++k) out[k] = u53(seed, start + k);
}

/* 24-bit uniforms: exactly representable in fp32 and never equal to 1. */
void synth_uniform_f32(uint64_t seed, uint64_t start, uint64_t n, float* out) {
    for (uint64_t k = 0; k < n; ++k)
        out[k] = (float)((double)(stream_at(seed, start + k) >> 40) * 0x1.0p-24);
}

static inline double normal_at(uint64_t seed, uint64_t i) {
    const double two_pi = 6.283185307179586476925286766559;
    uint64_t pair = i >> 1;
    double u1 = 1.0 - u53(seed, 2 * pair); /* (0, 1] */
    double u2 = u53(seed, 2 * pair + 1);
    double r = sqrt(-2.0 * log(u1));
    return (i & 1) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
}

/* out[k] = out[k] * accumulate + mean + std * N_{start+k}  (accumulate is 0 or 1) */
void synth_normal_f64(uint64_t seed, uint64_t start, uint64_t n, double mean, double stdev,
                      int accumulate, double* out) {
    for (uint64_t k = 0; k < n; ++k) {
        double v = mean + stdev * normal_at(seed, start + k);
        out[k] = accumulate ? out[k] + v : v;
    }
}

/* Round fp64 to fp32 (nearest), then fp32 to bf16 by round-to-nearest-even. */
void synth_to_bf16(const double* x, uint64_t n, uint16_t* out) {
    for (uint64_t k = 0; k < n; ++k) {
        float f = (float)x[k];
        uint32_t u;
        memcpy(&u, &f, 4);
        if ((u & 0x7F800000u) == 0x7F800000u) { /* inf / nan: truncate, keep nan quiet */
            uint16_t h = (uint16_t)(u >> 16);
            if (u & 0x007FFFFFu) h |= 0x0040;
            out[k] = h;
            continue;
        }
        uint32_t lsb = (u >> 16) & 1u;
        u += 0x7FFFu + lsb;
        out[k] = (uint16_t)(u >> 16);
    }
}

void synth_bf16_to_f32(const uint16_t* b, uint64_t n, float* out) {
    for (uint64_t k = 0; k < n; ++k) {
        uint32_t u = (uint32_t)b[k] << 16;
        memcpy(&out[k], &u, 4);
    }
}

void synth_to_f32(const double* x, uint64_t n, float* out) {
    for (uint64_t k = 0; k < n; ++k) out[k] = (float)x[k];
}

/*
 * Gumbel-max draw per row: rows are fp32 logits [R, V]; row r uses stream
 * indices [ (start_row + r) * V, (start_row + r + 1) * V ).  Returns the
 * argmax of y_v * inv_t + G_v (lowest index on exact ties).
 */
void synth_gumbel_argmax(const float* logits, uint64_t R, uint64_t V, double inv_t,
                         uint64_t seed, uint64_t start_row, int32_t* out) {
    for (uint64_t r = 0; r < R; ++r) {
        const float* row = logits + r * V;
        uint64_t base = (start_row + r) * V;
        double best = -INFINITY;
        int32_t arg = 0;
        for (uint64_t v = 0; v < V; ++v) {
            double g = -log(-log(u53_open(seed, base + v)));
            double key = (double)row[v] * inv_t + g;
            if (key > best) { best = key; arg = (int32_t)v; }
        }
        out[r] = arg;
    }
}

/* Plain argmax per fp32 row (lowest index on ties); used by the greedy-draft recipe. */
void synth_row_argmax(const float* logits, uint64_t R, uint64_t V, int32_t* out) {
    for (uint64_t r = 0; r < R; ++r) {
        const float* row = logits + r * V;
        float best = row[0];
        int32_t arg = 0;
        for (uint64_t v = 1; v < V; ++v)
            if (row[v] > best) { best = row[v]; arg = (int32_t)v; }
        out[r] = arg;
    }
}
