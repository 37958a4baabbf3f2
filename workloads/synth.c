/*
 * synth.c -- seeded synthetic bf16 tensors for the TACO workloads.
 *
 * Input generation only: nothing here computes any step of the compression
 * method.  Both the CUDA path and the CPU oracle take their inputs from this
 * file, which depends on neither.
 *
 * Each value is a pure function of (seed, stream, element index).  The random
 * bits come from SplitMix64 used as a counter-based generator (Steele, Lea and
 * Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014): the
 * published output function applied to key + (index + 1) * gamma, with
 * gamma = 0x9E3779B97F4A7C15 and a per-(seed, stream) key.  The top 53 bits
 * give a uniform double strictly inside (0, 1).  Values are drawn in double,
 * rounded to float (nearest even) and then to bf16 (nearest even).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL
#define STREAM_MUL 0xD1B54A32D192ED03ULL

static uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static uint64_t stream_key(uint64_t seed, uint64_t stream)
{
    return mix64(seed * GAMMA + stream * STREAM_MUL);
}

static double uniform_open(uint64_t key, uint64_t idx)
{
    uint64_t bits = mix64(key + (idx + 1u) * GAMMA) >> 11;
    return ((double)bits + 0.5) * 0x1p-53;
}

static uint16_t to_bf16(double x)
{
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

uint64_t synth_u64(uint64_t seed, uint64_t stream, uint64_t idx)
{
    return mix64(stream_key(seed, stream) + (idx + 1u) * GAMMA);
}

double synth_uniform(uint64_t seed, uint64_t stream, uint64_t idx)
{
    return uniform_open(stream_key(seed, stream), idx);
}

/* Laplace(0, b) bulk; with probability p_out an element is replaced by a
 * fair-signed U[lo, hi) outlier.  Streams: 0 bulk, 1 select, 2 sign, 3 size. */
void synth_laplace_outliers(uint64_t seed, int64_t first, int64_t n, double b, double p_out,
                            double lo, double hi, uint16_t *out)
{
    uint64_t k0 = stream_key(seed, 0), k1 = stream_key(seed, 1);
    uint64_t k2 = stream_key(seed, 2), k3 = stream_key(seed, 3);
    for (int64_t i = 0; i < n; i++) {
        uint64_t idx = (uint64_t)(first + i);
        double u = uniform_open(k0, idx) - 0.5;
        double x = (u < 0 ? 1.0 : -1.0) * b * log1p(-2.0 * fabs(u));
        if (uniform_open(k1, idx) < p_out) {
            double sign = uniform_open(k2, idx) < 0.5 ? -1.0 : 1.0;
            x = sign * (lo + (hi - lo) * uniform_open(k3, idx));
        }
        out[i] = to_bf16(x);
    }
}

/* Student-t(nu) * scale * m_c.  t = z0 / sqrt((z1^2 + ... + z_nu^2) / nu) from
 * Box-Muller normals (streams 0..3 for nu <= 3); m_c is log-uniform in
 * [m_lo, m_hi), drawn per column from stream 10. */
void synth_student_t_channels(uint64_t seed, int64_t first, int64_t n, int64_t hidden, double scale,
                              double m_lo, double m_hi, uint16_t *out)
{
    const double two_pi = 6.283185307179586;
    uint64_t k[4], kc = stream_key(seed, 10);
    for (int s = 0; s < 4; s++)
        k[s] = stream_key(seed, (uint64_t)s);
    double lm0 = log(m_lo), lm1 = log(m_hi);
    for (int64_t i = 0; i < n; i++) {
        uint64_t idx = (uint64_t)(first + i);
        double r0 = sqrt(-2.0 * log(uniform_open(k[0], idx)));
        double a0 = two_pi * uniform_open(k[1], idx);
        double r1 = sqrt(-2.0 * log(uniform_open(k[2], idx)));
        double a1 = two_pi * uniform_open(k[3], idx);
        double z0 = r0 * cos(a0), z1 = r0 * sin(a0);
        double z2 = r1 * cos(a1), z3 = r1 * sin(a1);
        double t = z0 / sqrt((z1 * z1 + z2 * z2 + z3 * z3) / 3.0);
        uint64_t col = idx % (uint64_t)hidden;
        double m = exp(lm0 + (lm1 - lm0) * uniform_open(kc, col));
        out[i] = to_bf16(t * scale * m);
    }
}

/* N(0, sd^2) bulk (Box-Muller, streams 0 and 1); with probability p_big the
 * value is multiplied by `big` (stream 2); with probability p_zero it is set
 * to exactly +0 (stream 3), which takes precedence. */
void synth_gaussian_sparse(uint64_t seed, int64_t first, int64_t n, double sd, double p_big,
                           double big, double p_zero, uint16_t *out)
{
    const double two_pi = 6.283185307179586;
    uint64_t k0 = stream_key(seed, 0), k1 = stream_key(seed, 1);
    uint64_t k2 = stream_key(seed, 2), k3 = stream_key(seed, 3);
    for (int64_t i = 0; i < n; i++) {
        uint64_t idx = (uint64_t)(first + i);
        double z = sqrt(-2.0 * log(uniform_open(k0, idx))) * cos(two_pi * uniform_open(k1, idx));
        double x = sd * z;
        if (uniform_open(k2, idx) < p_big)
            x *= big;
        if (uniform_open(k3, idx) < p_zero)
            x = 0.0;
        out[i] = to_bf16(x);
    }
}

/* Uniform integers in [-range, range] times 2^exp2 (no transcendental
 * function: identical on every host), used for fixtures. */
void synth_small_ints(uint64_t seed, int64_t first, int64_t n, int range, int exp2, uint16_t *out)
{
    uint64_t k0 = stream_key(seed, 0);
    for (int64_t i = 0; i < n; i++) {
        uint64_t bits = mix64(k0 + ((uint64_t)(first + i) + 1u) * GAMMA);
        int v = (int)(bits % (uint64_t)(2 * range + 1)) - range;
        out[i] = to_bf16(ldexp((double)v, exp2));
    }
}
