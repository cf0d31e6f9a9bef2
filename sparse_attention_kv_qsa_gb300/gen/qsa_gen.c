/*
 * Seeded synthetic input generator for QSA block selection.
 *
 * Draws random numbers only; computes no block score and no selection. The
 * CUDA path and the CPU oracle both consume the buffers written here.
 *
 * PCG32 = the XSH-RR 64/32 generator of M. E. O'Neill, "PCG: A Family of
 * Simple Fast Space-Efficient Statistically Good Algorithms for Random Number
 * Generation" (2014): a 64-bit LCG with multiplier 6364136223846793005 and an
 * odd increment (2*stream+1), output = rotr32(((s >> 18) ^ s) >> 27, s >> 59)
 * of the state before the step.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

typedef struct { uint64_t state, inc; } pcg32_t;

static uint32_t pcg32_next(pcg32_t *g) {
    uint64_t old = g->state;
    g->state = old * 6364136223846793005ULL + g->inc;
    uint32_t xs = (uint32_t)(((old >> 18) ^ old) >> 27);
    uint32_t rot = (uint32_t)(old >> 59);
    return (xs >> rot) | (xs << ((32u - rot) & 31u));
}

static void pcg32_seed(pcg32_t *g, uint64_t seed, uint64_t stream) {
    g->state = 0;
    g->inc = (stream << 1) | 1u;
    pcg32_next(g);
    g->state += seed;
    pcg32_next(g);
}

/* uniform double in [0,1) from two outputs (27 + 26 = 53 random bits) */
static double u53(pcg32_t *g) {
    uint64_t a = pcg32_next(g) >> 5, b = pcg32_next(g) >> 6;
    return ((double)a * 67108864.0 + (double)b) / 9007199254740992.0;
}

static const double kTwoPi = 6.283185307179586476925286766559;

void qsa_gen_u32(uint64_t seed, uint64_t stream, size_t n, uint32_t *out) {
    pcg32_t g; pcg32_seed(&g, seed, stream);
    for (size_t i = 0; i < n; ++i) out[i] = pcg32_next(&g);
}

void qsa_gen_uniform_f64(uint64_t seed, uint64_t stream, size_t n, double *out) {
    pcg32_t g; pcg32_seed(&g, seed, stream);
    for (size_t i = 0; i < n; ++i) out[i] = u53(&g);
}

/* standard normals by Box-Muller; both members of each pair are used */
void qsa_gen_normal_f64(uint64_t seed, uint64_t stream, size_t n, double *out) {
    pcg32_t g; pcg32_seed(&g, seed, stream);
    for (size_t i = 0; i < n; i += 2) {
        double u1 = 1.0 - u53(&g), u2 = u53(&g);
        double r = sqrt(-2.0 * log(u1)), th = kTwoPi * u2;
        out[i] = r * cos(th);
        if (i + 1 < n) out[i + 1] = r * sin(th);
    }
}

void qsa_gen_normal_f32(uint64_t seed, uint64_t stream, size_t n, float *out) {
    pcg32_t g; pcg32_seed(&g, seed, stream);
    for (size_t i = 0; i < n; i += 2) {
        double u1 = 1.0 - u53(&g), u2 = u53(&g);
        double r = sqrt(-2.0 * log(u1)), th = kTwoPi * u2;
        out[i] = (float)(r * cos(th));
        if (i + 1 < n) out[i + 1] = (float)(r * sin(th));
    }
}

/*
 * Student-t with 3 degrees of freedom at unit variance: t3 = Z / sqrt(V/3)
 * (V ~ chi^2_3) has variance 3, so t3/sqrt(3) = Z / sqrt(V). Each value uses
 * two Box-Muller pairs (Z1,Z2), (Z3,Z4): Z = Z1, V = Z2^2 + Z3^2 + Z4^2.
 */
void qsa_gen_student_t3_f32(uint64_t seed, uint64_t stream, size_t n, float *out) {
    pcg32_t g; pcg32_seed(&g, seed, stream);
    for (size_t i = 0; i < n; ++i) {
        double a1 = 1.0 - u53(&g), a2 = u53(&g);
        double b1 = 1.0 - u53(&g), b2 = u53(&g);
        double ra = sqrt(-2.0 * log(a1)), ta = kTwoPi * a2;
        double rb = sqrt(-2.0 * log(b1)), tb = kTwoPi * b2;
        double z = ra * cos(ta), z2 = ra * sin(ta);
        double z3 = rb * cos(tb), z4 = rb * sin(tb);
        out[i] = (float)(z / sqrt(z2 * z2 + z3 * z3 + z4 * z4));
    }
}

/* int8 uniform on [-127, 127]: (x * 255) >> 32 maps a uint32 onto 0..254 */
void qsa_gen_int8_127(uint64_t seed, uint64_t stream, size_t n, int8_t *out) {
    pcg32_t g; pcg32_seed(&g, seed, stream);
    for (size_t i = 0; i < n; ++i)
        out[i] = (int8_t)((int)(((uint64_t)pcg32_next(&g) * 255u) >> 32) - 127);
}

/* integers uniform on [lo, hi] by the same multiply-shift map */
void qsa_gen_int_range_f32(uint64_t seed, uint64_t stream, size_t n, int lo, int hi, float *out) {
    pcg32_t g; pcg32_seed(&g, seed, stream);
    uint64_t span = (uint64_t)(hi - lo + 1);
    for (size_t i = 0; i < n; ++i)
        out[i] = (float)((int64_t)(((uint64_t)pcg32_next(&g) * span) >> 32) + lo);
}
