/*
 * taco_oracle.c -- CPU oracle for TACO's fused FP8 compression operator.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, single-threaded
 * restatement of the method in "TACO: Efficient Communication Compression of
 * Intermediate Tensors for Scalable Tensor-Parallel LLM Training".  Only the
 * test suite, the package smoke check and the CPU-baseline leg of the
 * benchmark load it.  The CUDA library never links, includes or calls it, and
 * it shares no code, header, table or constant generator with the CUDA path.
 *
 * Arithmetic: every step of Algorithm 1 is one IEEE-754 binary32 operation
 * rounded to nearest-even, in the order the paper writes the steps (the
 * paper's receiver converts with Cvt_FP32 and its sender converts a float
 * with NVIDIA's float->fp8 intrinsic, Eqs. (10)-(11), so the operator is an
 * FP32 computation).  The one exception is the block sum of squares of
 * Eq. (6): it is accumulated in binary64 (each square of a bf16 or fp32 value
 * is exact there) and rounded once to binary32.  Build with
 * -ffp-contract=off and without -ffast-math so that no product is fused into
 * a following add and subnormals are kept.
 *
 * Open points of the paper and the readings taken here:
 *   - tau (target energy, Eq. 7) = 1.0, read as a target RMS;
 *   - eps (Eq. 6) = 1e-30, inside the square root;
 *   - Q_max (Eq. 9) = 448, the largest finite OCP E4M3 (E4M3FN) value;
 *   - H_B is the Sylvester Hadamard matrix in natural order,
 *     (H_B)_{ij} = (-1)^popcount(i & j), applied by an in-place butterfly
 *     with strides 1, 2, 4, ..., B/2 (Section 4.2.2, FWHT);
 *   - 1/sqrt(B) is the binary32 rounding of the exact value;
 *   - Cvt_FP8 (Eq. 10) rounds to nearest, ties to even, saturating to +-448,
 *     keeping the sign of zero and the subnormal grid;
 *   - an all-zero block (max|Z| = 0) stores s = 0 and all codes 0x00;
 *   - the packed record of block k sits at byte k*(B+8): B E4M3 codes in
 *     element order, then alpha_k, then s_k, both little-endian binary32
 *     (Section 4.4.2, metadata stored right after the codes);
 *   - the shard reduction decodes each shard to binary32 (no bf16 rounding),
 *     sums the shards left to right in shard order, and compresses the sum
 *     once from binary32 (Section 4.4.2, two-shot AllReduce: a compressed
 *     all-to-all exchange, then one reduction per owner).
 *
 * Ablation variants and code formats (the "_ex" entry points; the plain
 * entry points are ASH + DS with E4M3):
 *   - ASH + DS (the method), standard Hadamard + DS (alpha = 1, Section
 *     5.3.1 "standard Hadamard transform"), DS only (alpha = 1 and no
 *     rotation, Section 5.2.2 "Dual-Scale quantization in isolation") and
 *     ASH only (no post-rotation scale: s = 1 and the rotated value is cast
 *     directly, Section 5.2.2 "ASH alone");
 *   - codes E4M3 (Q_max 448), E5M2 (Q_max 57344, the largest finite OCP
 *     E5M2 value; Section 5.3.2 format ablation) rounded to nearest even and
 *     saturated to +-Q_max like E4M3, and INT8 (Q_max 127, Section 2's
 *     round(x / Delta) with Delta = max|x| / 127, ties to even, clamped to
 *     +-127; the INT8 fallback of Section 6 is ASH + DS with these codes);
 *   - the record layout stays [B codes | alpha | s], with alpha = 1 where the
 *     variant has no adaptive scale and s = 1 where it has no post-rotation
 *     scale; decoding is always q * s, then the inverse rotation if the
 *     variant rotates, then the division by alpha.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_TAU 1.0f
#define ORACLE_EPS 1e-30f
#define ORACLE_QMAX 448.0f
#define ORACLE_MAX_BLOCK 512

/* Variants and code formats of the "_ex" entry points. */
enum { VARIANT_ASH_DS = 0, VARIANT_HADAMARD_DS = 1, VARIANT_DS_ONLY = 2, VARIANT_ASH_ONLY = 3 };
enum { CODE_E4M3 = 0, CODE_E5M2 = 1, CODE_INT8 = 2 };

enum {
    ORACLE_OK = 0,
    ORACLE_ERR_BLOCK = -1,  /* B not a power of two in [2, 512] */
    ORACLE_ERR_SHAPE = -2,  /* n < 0 or n not a multiple of B */
    ORACLE_ERR_SHARDS = -3, /* P < 1 */
    ORACLE_ERR_SCHEME = -4, /* unknown variant or code format */
};

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

/* bfloat16 -> binary32 is exact: the bf16 bits are the high half. */
static float bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static float f32_from_bits(uint32_t u)
{
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Exact value of the bf16 bit pattern h, as a double (the pattern 0x7F80
 * with the sign is taken as 2^128, the first value past the largest finite
 * bf16, which is what round-to-nearest compares against). */
static double bf16_value_for_rounding(uint32_t h)
{
    if ((h & 0x7fffu) == 0x7f80u)
        return (h & 0x8000u) ? -ldexp(1.0, 128) : ldexp(1.0, 128);
    return (double)bf16_to_f32((uint16_t)h);
}

/* binary32 -> bfloat16, round to nearest, ties to even.  The two candidates
 * are the bf16 values that bracket f (truncation toward zero, and the next
 * pattern away from zero); the nearer one wins, a tie goes to the candidate
 * whose last mantissa bit is 0.  Differences are exact in binary64. */
static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) /* NaN: keep it a quiet NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    if ((u & 0x7fffffffu) == 0x7f800000u) /* infinity */
        return (uint16_t)(u >> 16);
    uint32_t toward_zero = u >> 16;
    if ((u & 0xffffu) == 0)
        return (uint16_t)toward_zero;
    uint32_t away = toward_zero + 1u;
    double x = fabs((double)f);
    double d_lo = x - fabs(bf16_value_for_rounding(toward_zero));
    double d_hi = fabs(bf16_value_for_rounding(away)) - x;
    if (d_lo < d_hi)
        return (uint16_t)toward_zero;
    if (d_hi < d_lo)
        return (uint16_t)away;
    return (uint16_t)(((toward_zero & 1u) == 0) ? toward_zero : away);
}

/* Magnitude of the E4M3 pattern whose low seven bits are c7 (0..126):
 * exponent field E = c7 >> 3 (bias 7), mantissa M = c7 & 7 (Eq. 4).
 * E = 0 is the subnormal range, 2^-6 * M/8. */
static double e4m3_magnitude(int c7)
{
    int E = c7 >> 3, M = c7 & 7;
    if (E == 0)
        return ldexp((double)M, -9);
    return ldexp(8.0 + (double)M, E - 10); /* 2^(E-7) * (1 + M/8) */
}

/* Cvt_FP32 of Eq. (11): the value of an E4M3 code.  0x7F / 0xFF are NaN. */
double taco_oracle_e4m3_value(uint8_t code)
{
    int c7 = code & 0x7f;
    if (c7 == 0x7f)
        return NAN;
    double v = e4m3_magnitude(c7);
    return (code & 0x80) ? -v : v;
}

/* Cvt_FP8 of Eq. (10): nearest E4M3 value, ties to the even code (even
 * mantissa), magnitudes at or above 448 saturate to 448, the sign is kept
 * (a negative value that rounds to zero gives 0x80). */
uint8_t taco_oracle_e4m3_encode(float u)
{
    if (isnan(u))
        return 0x7f;
    uint8_t sign = signbit(u) ? 0x80 : 0x00;
    double a = fabs((double)u);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7e);
    /* Largest lo with magnitude(lo) <= a; magnitude(126) = 448 > a. */
    int lo = 0, hi = 126;
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (e4m3_magnitude(mid) <= a)
            lo = mid;
        else
            hi = mid;
    }
    /* Compare 2a with lo + hi: both sides are exact in binary64. */
    double twice_mid = e4m3_magnitude(lo) + e4m3_magnitude(hi);
    double twice_a = 2.0 * a;
    int c;
    if (twice_a < twice_mid)
        c = lo;
    else if (twice_a > twice_mid)
        c = hi;
    else
        c = (lo % 2 == 0) ? lo : hi;
    return (uint8_t)(sign | c);
}

/* Magnitude of the E5M2 pattern whose low seven bits are c7 (0..123):
 * exponent field E = c7 >> 2 (bias 15), mantissa M = c7 & 3.  E = 0 is the
 * subnormal range, 2^-14 * M/4.  0x7C is infinity, 0x7D..0x7F NaN. */
static double e5m2_magnitude(int c7)
{
    int E = c7 >> 2, M = c7 & 3;
    if (E == 0)
        return ldexp((double)M, -16);
    return ldexp(4.0 + (double)M, E - 17); /* 2^(E-15) * (1 + M/4) */
}

double taco_oracle_e5m2_value(uint8_t code)
{
    int c7 = code & 0x7f;
    if (c7 == 0x7c)
        return (code & 0x80) ? -INFINITY : INFINITY;
    if (c7 > 0x7c)
        return NAN;
    double v = e5m2_magnitude(c7);
    return (code & 0x80) ? -v : v;
}

/* Nearest E5M2 value, ties to the even code, magnitudes at or above 57344
 * saturate to 57344, the sign of zero is kept. */
uint8_t taco_oracle_e5m2_encode(float u)
{
    if (isnan(u))
        return 0x7f;
    uint8_t sign = signbit(u) ? 0x80 : 0x00;
    double a = fabs((double)u);
    if (a >= 57344.0)
        return (uint8_t)(sign | 0x7b);
    int lo = 0, hi = 123; /* magnitude(123) = 57344 > a */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (e5m2_magnitude(mid) <= a)
            lo = mid;
        else
            hi = mid;
    }
    double twice_mid = e5m2_magnitude(lo) + e5m2_magnitude(hi);
    double twice_a = 2.0 * a;
    int c;
    if (twice_a < twice_mid)
        c = lo;
    else if (twice_a > twice_mid)
        c = hi;
    else
        c = (lo % 2 == 0) ? lo : hi;
    return (uint8_t)(sign | c);
}

/* round(u) to the nearest integer, ties to even, clamped to [-127, 127],
 * as a two's complement byte. */
uint8_t taco_oracle_int8_encode(float u)
{
    if (isnan(u))
        return 0;
    double a = (double)u;
    double f = floor(a);
    double d = a - f; /* exact: |a| < 2^24 or a is an integer */
    double r;
    if (d < 0.5)
        r = f;
    else if (d > 0.5)
        r = f + 1.0;
    else
        r = (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
    if (r > 127.0)
        r = 127.0;
    if (r < -127.0)
        r = -127.0;
    return (uint8_t)(int8_t)r;
}

double taco_oracle_int8_value(uint8_t code)
{
    return (double)(int8_t)code;
}

static int scheme_ok(int variant, int code)
{
    return variant >= VARIANT_ASH_DS && variant <= VARIANT_ASH_ONLY && code >= CODE_E4M3 && code <= CODE_INT8;
}

static float code_qmax(int code)
{
    return code == CODE_E4M3 ? ORACLE_QMAX : code == CODE_E5M2 ? 57344.0f : 127.0f;
}

static uint8_t code_encode(int code, float u)
{
    return code == CODE_E4M3 ? taco_oracle_e4m3_encode(u)
           : code == CODE_E5M2 ? taco_oracle_e5m2_encode(u)
                                : taco_oracle_int8_encode(u);
}

static double code_value(int code, uint8_t c)
{
    return code == CODE_E4M3 ? taco_oracle_e4m3_value(c)
           : code == CODE_E5M2 ? taco_oracle_e5m2_value(c)
                                : taco_oracle_int8_value(c);
}

/* ------------------------------------------------------------------ */
/* Hadamard rotation                                                   */
/* ------------------------------------------------------------------ */

/* Unnormalised in-place fast Walsh-Hadamard transform: v <- H_B v with
 * (H_B)_{ij} = (-1)^popcount(i & j).  Butterfly (a, b) -> (a + b, a - b)
 * at strides h = 1, 2, ..., B/2, each add rounded to binary32. */
void taco_oracle_fwht(float *v, int B)
{
    for (int h = 1; h < B; h *= 2)
        for (int i = 0; i < B; i += 2 * h)
            for (int j = i; j < i + h; j++) {
                float a = v[j], b = v[j + h];
                v[j] = a + b;
                v[j + h] = a - b;
            }
}

static float inv_sqrt_block(int B)
{
    return (float)(1.0 / sqrt((double)B));
}

static int block_ok(int B)
{
    return B >= 2 && B <= ORACLE_MAX_BLOCK && (B & (B - 1)) == 0;
}

/* ------------------------------------------------------------------ */
/* Sender: Algorithm 1 (its compression loop), Eqs. (5)-(10)          */
/* ------------------------------------------------------------------ */

static void compress_block(const float *G, int B, int variant, int code, uint8_t *rec)
{
    const int adaptive = variant == VARIANT_ASH_DS || variant == VARIANT_ASH_ONLY;
    const int rotate = variant != VARIANT_DS_ONLY;
    const int dual_scale = variant != VARIANT_ASH_ONLY;
    float alpha = 1.0f;
    float Z[ORACLE_MAX_BLOCK];
    if (adaptive) {
        /* Eq. (6): sigma_k = sqrt(mean_j G_kj^2 + eps). */
        double acc = 0.0;
        for (int j = 0; j < B; j++)
            acc += (double)G[j] * (double)G[j];
        float m = (float)(acc / (double)B);
        float sigma = sqrtf(m + ORACLE_EPS);

        /* Eq. (7): alpha_k = tau / sigma_k; G~_k = alpha_k * G_k. */
        alpha = ORACLE_TAU / sigma;
        for (int j = 0; j < B; j++)
            Z[j] = alpha * G[j];
    } else {
        for (int j = 0; j < B; j++)
            Z[j] = G[j];
    }

    /* Eq. (8): Z_k = (1/sqrt(B)) H_B G~_k. */
    if (rotate) {
        taco_oracle_fwht(Z, B);
        float r = inv_sqrt_block(B);
        for (int j = 0; j < B; j++)
            Z[j] = r * Z[j];
    }
    float zmax = 0.0f;
    for (int j = 0; j < B; j++)
        if (fabsf(Z[j]) > zmax)
            zmax = fabsf(Z[j]);

    /* Eq. (9): s_k = max|Z_k| / Q_max.  Eq. (10): q_k = Cvt(Z_k / s_k). */
    float s;
    if (!dual_scale) {
        s = 1.0f;
        for (int j = 0; j < B; j++)
            rec[j] = code_encode(code, Z[j]);
    } else if (zmax == 0.0f) {
        s = 0.0f;
        memset(rec, 0, (size_t)B);
    } else {
        s = zmax / code_qmax(code);
        for (int j = 0; j < B; j++)
            rec[j] = code_encode(code, Z[j] / s);
    }
    memcpy(rec + B, &alpha, 4);
    memcpy(rec + B + 4, &s, 4);
}

/* ------------------------------------------------------------------ */
/* Receiver: Algorithm 1 (its decompression loop), Eqs. (11)-(13)     */
/* ------------------------------------------------------------------ */

static void decompress_block(const uint8_t *rec, int B, int variant, int code, float *out)
{
    float alpha, s;
    memcpy(&alpha, rec + B, 4);
    memcpy(&s, rec + B + 4, 4);
    float Zh[ORACLE_MAX_BLOCK];
    for (int j = 0; j < B; j++) {
        float q = (float)code_value(code, rec[j]); /* Eq. (11) */
        Zh[j] = q * s;
    }
    if (variant != VARIANT_DS_ONLY) {
        taco_oracle_fwht(Zh, B); /* Eq. (12) */
        float r = inv_sqrt_block(B);
        for (int j = 0; j < B; j++)
            Zh[j] = r * Zh[j];
    }
    for (int j = 0; j < B; j++)
        out[j] = Zh[j] / alpha; /* Eq. (13) */
}

/* ------------------------------------------------------------------ */
/* Exported entry points                                               */
/* ------------------------------------------------------------------ */

int64_t taco_oracle_packed_bytes(int64_t n, int B)
{
    if (!block_ok(B) || n < 0 || n % B != 0)
        return -1;
    return n / B * (int64_t)(B + 8);
}

static int check_args(int64_t n, int B, int variant, int code)
{
    if (!block_ok(B))
        return ORACLE_ERR_BLOCK;
    if (n < 0 || n % B != 0)
        return ORACLE_ERR_SHAPE;
    if (!scheme_ok(variant, code))
        return ORACLE_ERR_SCHEME;
    return ORACLE_OK;
}

int taco_oracle_compress_bf16_ex(const uint16_t *x, int64_t n, int B, int variant, int code, uint8_t *packed)
{
    int st = check_args(n, B, variant, code);
    if (st != ORACLE_OK)
        return st;
    float G[ORACLE_MAX_BLOCK];
    for (int64_t k = 0; k < n / B; k++) {
        for (int j = 0; j < B; j++)
            G[j] = bf16_to_f32(x[k * B + j]);
        compress_block(G, B, variant, code, packed + k * (int64_t)(B + 8));
    }
    return ORACLE_OK;
}

int taco_oracle_compress_f32_ex(const float *x, int64_t n, int B, int variant, int code, uint8_t *packed)
{
    int st = check_args(n, B, variant, code);
    if (st != ORACLE_OK)
        return st;
    for (int64_t k = 0; k < n / B; k++)
        compress_block(x + k * B, B, variant, code, packed + k * (int64_t)(B + 8));
    return ORACLE_OK;
}

int taco_oracle_decompress_f32_ex(const uint8_t *packed, int64_t n, int B, int variant, int code, float *y)
{
    int st = check_args(n, B, variant, code);
    if (st != ORACLE_OK)
        return st;
    for (int64_t k = 0; k < n / B; k++)
        decompress_block(packed + k * (int64_t)(B + 8), B, variant, code, y + k * B);
    return ORACLE_OK;
}

/* Decompression to the tensor's own dtype: bf16, rounded to nearest even
 * from the binary32 G'_k. */
int taco_oracle_decompress_bf16_ex(const uint8_t *packed, int64_t n, int B, int variant, int code, uint16_t *y)
{
    int st = check_args(n, B, variant, code);
    if (st != ORACLE_OK)
        return st;
    float out[ORACLE_MAX_BLOCK];
    for (int64_t k = 0; k < n / B; k++) {
        decompress_block(packed + k * (int64_t)(B + 8), B, variant, code, out);
        for (int j = 0; j < B; j++)
            y[k * B + j] = f32_to_bf16_rne(out[j]);
    }
    return ORACLE_OK;
}

/* Receive side of the two-shot AllReduce (Section 4.4.2): the P compressed
 * shards of the same n elements are decoded to binary32, summed in shard
 * order, and the sum is compressed once, all with the same variant and code
 * format. */
int taco_oracle_reduce_shards_ex(const uint8_t *const *shards, int P, int64_t n, int B, int variant, int code,
                                 uint8_t *out)
{
    int st = check_args(n, B, variant, code);
    if (st != ORACLE_OK)
        return st;
    if (P < 1)
        return ORACLE_ERR_SHARDS;
    float S[ORACLE_MAX_BLOCK], t[ORACLE_MAX_BLOCK];
    for (int64_t k = 0; k < n / B; k++) {
        for (int j = 0; j < B; j++)
            S[j] = 0.0f;
        for (int p = 0; p < P; p++) {
            decompress_block(shards[p] + k * (int64_t)(B + 8), B, variant, code, t);
            for (int j = 0; j < B; j++)
                S[j] = S[j] + t[j];
        }
        compress_block(S, B, variant, code, out + k * (int64_t)(B + 8));
    }
    return ORACLE_OK;
}

/* The method itself: ASH + DS with E4M3 codes. */
int taco_oracle_compress_bf16(const uint16_t *x, int64_t n, int B, uint8_t *packed)
{
    return taco_oracle_compress_bf16_ex(x, n, B, VARIANT_ASH_DS, CODE_E4M3, packed);
}

int taco_oracle_compress_f32(const float *x, int64_t n, int B, uint8_t *packed)
{
    return taco_oracle_compress_f32_ex(x, n, B, VARIANT_ASH_DS, CODE_E4M3, packed);
}

int taco_oracle_decompress_f32(const uint8_t *packed, int64_t n, int B, float *y)
{
    return taco_oracle_decompress_f32_ex(packed, n, B, VARIANT_ASH_DS, CODE_E4M3, y);
}

int taco_oracle_decompress_bf16(const uint8_t *packed, int64_t n, int B, uint16_t *y)
{
    return taco_oracle_decompress_bf16_ex(packed, n, B, VARIANT_ASH_DS, CODE_E4M3, y);
}

int taco_oracle_reduce_shards(const uint8_t *const *shards, int P, int64_t n, int B, uint8_t *out)
{
    return taco_oracle_reduce_shards_ex(shards, P, n, B, VARIANT_ASH_DS, CODE_E4M3, out);
}

/* Array helpers for the tests. */
void taco_oracle_e4m3_encode_array(const float *u, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = taco_oracle_e4m3_encode(u[i]);
}

/* Encodes the binary32 bit patterns first, first+1, ..., first+count-1. */
void taco_oracle_e4m3_encode_bits(uint32_t first, int64_t count, uint8_t *out)
{
    for (int64_t i = 0; i < count; i++)
        out[i] = taco_oracle_e4m3_encode(f32_from_bits(first + (uint32_t)i));
}

void taco_oracle_e4m3_value_array(const uint8_t *codes, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = taco_oracle_e4m3_value(codes[i]);
}

void taco_oracle_bf16_round_array(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = f32_to_bf16_rne(x[i]);
}

void taco_oracle_fwht_rows(float *v, int64_t rows, int B)
{
    for (int64_t i = 0; i < rows; i++)
        taco_oracle_fwht(v + i * B, B);
}

void taco_oracle_code_encode_array(int code, const float *u, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = code_encode(code, u[i]);
}

/* Codes of the float32 values with bit patterns first, first + 1, ...
 * (modulo 2^32): every input of the conversion, for comparisons. */
void taco_oracle_code_encode_bits(int code, uint32_t first, int64_t count, uint8_t *out)
{
    for (int64_t i = 0; i < count; i++)
        out[i] = code_encode(code, f32_from_bits(first + (uint32_t)i));
}

void taco_oracle_code_value_array(int code, const uint8_t *codes, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = code_value(code, codes[i]);
}
