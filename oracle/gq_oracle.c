/*
 * gq_oracle.c -- CPU oracle for the Global-QSGD compress / aggregate / decompress path.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the plain, slow, single-threaded definition that the CUDA
 * library is checked against.  Only the test suite, the smoke check and the CPU-baseline leg of
 * bench.py load it; the product path never does.  It shares no code, header, table or constant
 * generator with the CUDA sources, and it includes none of them.
 *
 * Method: "Global-QSGD: Practical Floatless Quantization for Distributed Learning with Theoretical
 * Guarantees" (Xin, Canini, Richtarik, Horvath; arXiv 2305.18627), cited below as "Global-QSGD".
 * Random numbers: Philox4x32-10 from Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
 * Easy as 1, 2, 3" (SC'11), cited as "Philox (SC'11)".
 *
 * Precision.  The norm, the rounding probabilities and the dequantised mean are computed in fp64
 * (all exactly, except the norm's sum and square root and the final division of the mean).  The
 * one step carried in fp32 is the normalisation v = |x| / N: the quantiser works on fp32
 * gradients and an fp32 norm, and v is the correctly rounded fp32 quotient.
 *
 * Parity status (each function's pins live in tests/test_oracle_*.py):
 *   gqo_philox4x32_10      pinned: published known-answer vectors (tests/golden/)
 *   gqo_global_norm        pinned: closed forms, numpy.linalg.norm per axis, exact fsum
 *   gqo_level_split        pinned: exact expectation E[Q]=x, closed-form variance, fixed levels
 *   gqo_quantize           pinned: level split + Philox word, Monte-Carlo unbiasedness
 *   gqo_quantize_cols      the same arithmetic on a column window given alone: pinned equal to
 *                          gqo_quantize on the window of the whole matrix
 *   gqo_reduce_codes       pinned: hand-decoded codes, exact level values
 *   gqo_dequantize         pinned: hand examples, Monte-Carlo mean
 *   gqo_level_split_u16    pinned: the 16-bit-uniform mode's bias bound by brute force over
 *                          all 2^16 uniforms, Monte-Carlo mean, agreement with the exact split
 *   gqo_quantize_u16_cols  pinned: split + high half of the Philox word, ties H == F stay down
 *
 * Build: gcc -std=c99 -O2 -ffp-contract=off -fPIC -shared gq_oracle.c -lm
 * (-ffp-contract=off keeps every float operation a separately rounded IEEE operation on both
 * x86-64 and aarch64.)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Return codes (same meanings as the library's status values; defined here independently). */
#define GQO_OK 0
#define GQO_ERR_INVALID 1
#define GQO_ERR_UNSUPPORTED 2
#define GQO_ERR_NONFINITE 4

/* Element types of the gradient matrix. */
#define GQO_F32 0
#define GQO_BF16 1

/* Level grids: standard (linear) dithering Global-L_s and exponential dithering Global-E_s. */
#define GQO_LINEAR 0
#define GQO_EXP 1

/* Norm orders: 2 is the l2 norm, 0 stands for the l-infinity norm. */
#define GQO_INF 0

int gqo_abi_version(void) { return 1; }

/* ------------------------------------------------------------------------------------------ */
/* Philox4x32-10 (Philox (SC'11), the Philox-4x32 bijection with 10 rounds)                    */
/* ------------------------------------------------------------------------------------------ */

/* Full 64-bit product of two 32-bit words, split into high and low halves. */
static void mul_hi_lo(uint32_t a, uint32_t b, uint32_t *hi, uint32_t *lo)
{
    uint64_t prod = (uint64_t)a * (uint64_t)b;
    *hi = (uint32_t)(prod >> 32);
    *lo = (uint32_t)prod;
}

/*
 * One call of the Philox4x32-10 counter-based generator: four 32-bit counter words and two
 * 32-bit key words in, four 32-bit random words out.  Each round multiplies counter words 0 and
 * 2 by the two round multipliers, then forms the new counter from the high halves xor-ed with
 * the other two counter words and the round key, and the low halves.  The key advances by the
 * two Weyl increments between rounds.  The multipliers and increments are the ones the SC'11
 * paper gives for Philox-4x32 (the increments are the golden ratio and sqrt(3)-1 in 0.32 fixed
 * point).
 */
void gqo_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    const uint32_t mult0 = 0xD2511F53u, mult1 = 0xCD9E8D57u;
    const uint32_t weyl0 = 0x9E3779B9u, weyl1 = 0xBB67AE85u;
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    int round;
    for (round = 0; round < 10; ++round) {
        uint32_t hi0, lo0, hi1, lo1;
        if (round > 0) {
            k0 += weyl0;
            k1 += weyl1;
        }
        mul_hi_lo(mult0, c0, &hi0, &lo0);
        mul_hi_lo(mult1, c2, &hi1, &lo1);
        {
            uint32_t n0 = hi1 ^ c1 ^ k0;
            uint32_t n1 = lo1;
            uint32_t n2 = hi0 ^ c3 ^ k1;
            uint32_t n3 = lo0;
            c0 = n0;
            c1 = n1;
            c2 = n2;
            c3 = n3;
        }
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/* 16-bit half h (0..7) of a Philox output: the low half of word h/2 for even h, the high half
 * for odd h. */
static uint32_t half16(const uint32_t w[4], int h)
{
    uint32_t word = w[h >> 1];
    return (h & 1) ? (word >> 16) : (word & 0xFFFFu);
}

/*
 * The uniform 32-bit word r that decides the rounding of element (worker i, coordinate j) at
 * training step `step` under seed `seed`.  Global-QSGD leaves the source of randomness open; this
 * project fixes it as follows.  Key = (low 32 bits of seed, high 32 bits of seed).  The group of
 * eight coordinates j = 8t..8t+7 of worker i owns two counters,
 *     A = (t,         i, low 32 bits of step, high 32 bits of step)
 *     B = (2^31 + t,  i, low 32 bits of step, high 32 bits of step)
 * (t < 2^31 since d < 2^34).  The high 16 bits of r are half (j mod 8) of Philox(A) and the low
 * 16 bits are half (j mod 8) of Philox(B).  r is uniform on [0, 2^32) and independent across
 * elements.  (The split lets a caller decide "r < T" from the high half alone unless it equals
 * the high half of T, which happens with probability 2^-16.)
 */
uint32_t gqo_philox_word(uint64_t seed, uint64_t step, int64_t i, int64_t j)
{
    uint32_t ctr[4], key[2], a[4], b[4];
    int h = (int)(j & 7);
    ctr[0] = (uint32_t)((uint64_t)j >> 3);
    ctr[1] = (uint32_t)i;
    ctr[2] = (uint32_t)step;
    ctr[3] = (uint32_t)(step >> 32);
    key[0] = (uint32_t)seed;
    key[1] = (uint32_t)(seed >> 32);
    gqo_philox4x32_10(ctr, key, a);
    ctr[0] |= 0x80000000u;
    gqo_philox4x32_10(ctr, key, b);
    return (half16(a, h) << 16) | half16(b, h);
}

/* The words gqo_philox_word(seed, step, i, j) of worker i for the coordinates j = j0 .. j0 + w - 1,
 * into out[0 .. w - 1] (a loop over the definition above, for callers that need many words). */
int gqo_philox_words(uint64_t seed, uint64_t step, int64_t i, int64_t j0, int64_t w,
                     uint32_t *out)
{
    int64_t j;
    if (out == NULL || w < 0 || j0 < 0 || i < 0)
        return GQO_ERR_INVALID;
    for (j = 0; j < w; ++j)
        out[j] = gqo_philox_word(seed, step, i, j0 + j);
    return GQO_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* Input element access                                                                       */
/* ------------------------------------------------------------------------------------------ */

/* Element idx of the gradient buffer as an fp32 value.  bf16 is the high half of a binary32
 * word, so widening it is a 16-bit left shift of its bits. */
static float load_x(const void *x, int dtype, int64_t idx)
{
    if (dtype == GQO_F32)
        return ((const float *)x)[idx];
    {
        uint32_t bits = (uint32_t)((const uint16_t *)x)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return f;
    }
}

/* ------------------------------------------------------------------------------------------ */
/* Global norm ||x||_{q,p}                                                                     */
/* ------------------------------------------------------------------------------------------ */

/*
 * ||x||_{q,p} of the concatenated vector x = [x_1, ..., x_n] in R^{nd} (Global-QSGD, notation
 * paragraph of the preliminaries: the (sum over coordinates of ||.||_q^p)^(1/p) norm).  The
 * page's index ranges are garbled; the reading taken is: for every coordinate j, the q-norm over
 * the n workers of (x_1j, ..., x_nj); then the p-norm over j of those d numbers.  q and p are 2
 * or GQO_INF (0).  x is worker-major: element (i, j) is at i*d + j.
 *
 * Computed literally in fp64: the per-coordinate q-norm (sqrt of a sum of squares, or a max of
 * magnitudes), then the p-norm of those values.  Returns NaN if any element is NaN, +Inf if
 * any is infinite (and none is NaN), -1 for invalid arguments.
 */
double gqo_global_norm(const void *x, int dtype, int64_t n, int64_t d, int q, int p)
{
    int64_t i, j;
    int has_nan = 0, has_inf = 0;
    double outer = 0.0;
    if (x == NULL || n < 1 || d < 1 || (dtype != GQO_F32 && dtype != GQO_BF16))
        return -1.0;
    if ((q != 2 && q != GQO_INF) || (p != 2 && p != GQO_INF))
        return -1.0;
    for (j = 0; j < d; ++j) {
        double inner = 0.0; /* ||(x_1j, ..., x_nj)||_q */
        for (i = 0; i < n; ++i) {
            double v = (double)load_x(x, dtype, i * d + j);
            if (isnan(v)) {
                has_nan = 1;
                continue;
            }
            if (isinf(v)) {
                has_inf = 1;
                continue;
            }
            if (q == 2)
                inner += v * v;
            else if (fabs(v) > inner)
                inner = fabs(v);
        }
        if (q == 2)
            inner = sqrt(inner);
        if (p == 2)
            outer += inner * inner;
        else if (inner > outer)
            outer = inner;
    }
    if (has_nan)
        return NAN;
    if (has_inf)
        return INFINITY;
    return p == 2 ? sqrt(outer) : outer;
}

/* ------------------------------------------------------------------------------------------ */
/* Stochastic rounding onto the level grid                                                     */
/* ------------------------------------------------------------------------------------------ */

/*
 * Where |x| sits on the level grid.  Global-QSGD (Global-Q operator, formal definition) scales
 * each worker's vector by the global norm N and rounds v = |x|/N in [0, 1] at random to one of
 * the two adjacent levels lo <= v <= hi, up with probability (v - lo)/(hi - lo), which keeps the
 * result unbiased.  The grids (Global-QSGD, paragraph introducing the two forms of the
 * operator):
 *   Global-L_s (standard dithering):    levels m/s, m = 0..s (the page writes l_i = (s-i)/s);
 *   Global-E_s (exponential dithering): levels 0 and 2^-(s-k), k = 1..s.  The page writes
 *     "l_s = 0 and l_i = 2^-(s-i) for i in 1..s", which names l_s twice; the reading taken is
 *     the set {0, 2^-(s-1), ..., 1/2, 1} with level index k = 0 for the value 0.
 *
 * Output: *lo = index of the lower level (L: m with value m/s; E: k with value 0 for k = 0 and
 * 2^-(s-k) otherwise), *T = floor(P(up) * 2^32), so that "round up iff r < T" for a uniform
 * 32-bit word r rounds up with probability T / 2^32.  P(up) is computed exactly from v (every
 * step below is exact in fp64), so T is floor(P(up) * 2^32) exactly.
 *
 * v = fp32(|x| / N), clamped to 1: a norm handed in from outside that is smaller than |x|
 * saturates the element at the top level; a NaN element gets v = 0.  norm must be finite and
 * > 0.
 */
int gqo_level_split(float absx, float norm, int scheme, int s, int32_t *lo, uint32_t *T)
{
    float v;
    double f;
    if (!(norm > 0.0f) || isinf(norm) || s < 1 || lo == NULL || T == NULL)
        return GQO_ERR_INVALID;
    if (scheme == GQO_LINEAR) {
        if (s > 127)
            return GQO_ERR_UNSUPPORTED;
    } else if (scheme == GQO_EXP) {
        if (s > 62)
            return GQO_ERR_UNSUPPORTED;
    } else {
        return GQO_ERR_INVALID;
    }
    v = fabsf(absx) / norm; /* the one fp32 rounding */
    if (v > 1.0f)
        v = 1.0f;
    if (isnan(v))
        v = 0.0f; /* a NaN element under a finite norm contributes nothing */
    if (scheme == GQO_LINEAR) {
        double t = (double)v * (double)s; /* exact: 24-bit significand times a 7-bit integer */
        double m = floor(t);
        f = t - m; /* exact */
        *lo = (int32_t)m;
    } else {
        double smallest = ldexp(1.0, -(s - 1)); /* the lowest non-zero level 2^-(s-1) */
        if (v == 0.0f) {
            *lo = 0;
            f = 0.0;
        } else if ((double)v < smallest) {
            /* between the levels 0 and 2^-(s-1) */
            *lo = 0;
            f = (double)v / smallest; /* exact: division by a power of two */
        } else {
            /* between 2^e and 2^(e+1) with e = floor(log2 v), -(s-1) <= e <= 0 */
            int ex;
            frexp((double)v, &ex); /* v = mant * 2^ex with mant in [0.5, 1) */
            {
                int e = ex - 1;
                *lo = s + e; /* 2^e = 2^-(s - lo) */
                f = ldexp((double)v, -e) - 1.0; /* (v - 2^e) / (2^(e+1) - 2^e), exact */
            }
        }
    }
    *T = (uint32_t)floor(f * 4294967296.0); /* f * 2^32 is exact; f < 1 keeps T < 2^32 */
    return GQO_OK;
}

/*
 * Quantise coordinates j0 .. j0 + w - 1 of all n workers to signed integer codes, reading
 * x_ij at element i * ld + (j - j0) of xw (the window's columns, row stride ld).
 * Code c_ij = sign(x_ij) * k_ij where k_ij = lo + (r_ij < T_ij) is the level index chosen by
 * the stochastic rounding and r_ij = gqo_philox_word(seed, step, i, j): the random word is keyed
 * by the coordinate's index j in the whole vector.  The stored code is the signed level index
 * (Global-QSGD, theta example: one bit of sign and the remaining bits for the level).  codes is
 * n x w, worker-major, one int8 per element.
 *
 * norm is the fp32 global norm.  norm == 0 (all-zero input) gives all-zero codes and GQO_OK; a
 * non-finite norm gives all-zero codes and GQO_ERR_NONFINITE.
 */
int gqo_quantize_cols(const void *xw, int dtype, int64_t n, int64_t ld, int64_t j0, int64_t w,
                      float norm, int scheme, int s, uint64_t seed, uint64_t step, int8_t *codes)
{
    int64_t i, j;
    if (xw == NULL || codes == NULL || n < 1 || w < 0 || ld < w || j0 < 0)
        return GQO_ERR_INVALID;
    if (dtype != GQO_F32 && dtype != GQO_BF16)
        return GQO_ERR_INVALID;
    if (scheme != GQO_LINEAR && scheme != GQO_EXP)
        return GQO_ERR_INVALID;
    if (s < 1 || s > (scheme == GQO_LINEAR ? 127 : 62))
        return GQO_ERR_UNSUPPORTED;
    if (isnan(norm) || isinf(norm) || norm < 0.0f) {
        memset(codes, 0, (size_t)(n * w));
        return GQO_ERR_NONFINITE;
    }
    if (norm == 0.0f) {
        memset(codes, 0, (size_t)(n * w));
        return GQO_OK;
    }
    for (i = 0; i < n; ++i) {
        for (j = 0; j < w; ++j) {
            float xv = load_x(xw, dtype, i * ld + j);
            int32_t lo;
            uint32_t T, r;
            int32_t k;
            int rc = gqo_level_split(xv, norm, scheme, s, &lo, &T);
            if (rc != GQO_OK)
                return rc;
            r = gqo_philox_word(seed, step, i, j0 + j);
            k = lo + (r < T ? 1 : 0);
            codes[i * w + j] = (int8_t)(xv < 0.0f ? -k : k);
        }
    }
    return GQO_OK;
}

/*
 * Quantise the coordinate window [j0, j1) of the n x d matrix x (row-major): gqo_quantize_cols
 * on its columns j0 .. j1 - 1.
 */
int gqo_quantize(const void *x, int dtype, int64_t n, int64_t d, int64_t j0, int64_t j1,
                 float norm, int scheme, int s, uint64_t seed, uint64_t step, int8_t *codes)
{
    size_t esize = dtype == GQO_BF16 ? 2 : 4;
    if (x == NULL || codes == NULL || n < 1 || d < 1 || j0 < 0 || j1 > d || j0 > j1)
        return GQO_ERR_INVALID;
    return gqo_quantize_cols((const unsigned char *)x + (size_t)j0 * esize, dtype, n, d, j0,
                             j1 - j0, norm, scheme, s, seed, step, codes);
}

/* ------------------------------------------------------------------------------------------ */
/* The 16-bit-uniform rounding mode (an option)                                               */
/* ------------------------------------------------------------------------------------------ */

/*
 * Global-QSGD asks only for an unbiased random rounding between the two adjacent levels and fixes
 * no random source.  Besides the exact mode above this project offers a cheaper one, whose
 * decision uses a single 16-bit uniform per element, the high half H = r >> 16 of the element's
 * word (so one Philox call serves eight elements), and a 16-bit fraction F of the element's
 * position on the grid computed without a division:
 *
 *   Global-L_s: c1 = fp32(s / N) (one correctly rounded division for the whole matrix);
 *               P16 = |x| c1 2^16 rounded to the nearest integer, ties to the odd one (the
 *               product of two fp32 values is exact in fp64); P16 is clamped to s 2^16 (|x| > N
 *               saturates); lower level lo = P16 >> 16, F = P16 & 0xFFFF.
 *   Global-E_s: rcp = fp32(1 / N), w = min(fp32(|x| rcp), 1).  If w >= 2^-(s-1) (level 1 or
 *               more): lo = s + e with 2^e <= w < 2^(e+1), and F = the top 16 of w's 23 fraction
 *               bits (the rest truncated).  Else P16 = |x| rcp 2^(s-1) 2^16 rounded as for L
 *               (at most 2^16), lo = P16 >> 16, F = P16 & 0xFFFF.
 *
 * The element rounds up iff H < F, so P(up) = F / 2^16.  E[level] differs from the exact position
 * only through the 16-bit resolution of F and the rounding of c1 or rcp and w: by less than
 * 2^-16 + 2^-22 of the level spacing.  A NaN element gets code 0.  For a norm outside
 * [2^-100, 2^100] the decision is the exact mode's (gqo_level_split with the full word).
 *
 * Returns GQO_OK with (*lo, *F); 8 when the exact mode applies (norm out of range); errors as
 * gqo_level_split.
 */
#define GQO_USE_EXACT 8

/* Nearest integer to t >= 0, ties to the odd one. */
static double round_half_odd(double t)
{
    double f = floor(t), r = t - f;
    if (r > 0.5)
        return f + 1.0;
    if (r < 0.5)
        return f;
    return fmod(f, 2.0) == 1.0 ? f : f + 1.0;
}

int gqo_level_split_u16(float absx, float norm, int scheme, int s, int32_t *lo, uint32_t *F)
{
    float ax = fabsf(absx);
    if (!(norm > 0.0f) || isinf(norm) || s < 1 || lo == NULL || F == NULL)
        return GQO_ERR_INVALID;
    if ((scheme == GQO_LINEAR && s > 127) || (scheme == GQO_EXP && s > 62))
        return GQO_ERR_UNSUPPORTED;
    if (scheme != GQO_LINEAR && scheme != GQO_EXP)
        return GQO_ERR_INVALID;
    if (!(norm >= ldexpf(1.0f, -100) && norm <= ldexpf(1.0f, 100)))
        return GQO_USE_EXACT;
    if (isnan(ax)) {
        *lo = 0;
        *F = 0;
        return GQO_OK;
    }
    if (scheme == GQO_LINEAR) {
        float c1 = (float)s / norm;                     /* one fp32 rounding */
        double p16 = round_half_odd((double)ax * (double)c1 * 65536.0);
        if (p16 > (double)s * 65536.0)
            p16 = (double)s * 65536.0;
        *lo = (int32_t)(p16 / 65536.0);
        *F = (uint32_t)(p16 - (double)*lo * 65536.0);
    } else {
        float rcp = 1.0f / norm;                        /* one fp32 rounding */
        float w = ax * rcp;                             /* one fp32 rounding */
        if (w > 1.0f)
            w = 1.0f;
        if ((double)w >= ldexp(1.0, -(s - 1))) {
            int ex;
            uint32_t bits;
            frexp((double)w, &ex);                      /* w = mant 2^ex, mant in [0.5, 1) */
            memcpy(&bits, &w, sizeof bits);
            *lo = s + (ex - 1);
            *F = (bits & 0x7FFFFFu) >> 7;
        } else {
            double p16 = round_half_odd((double)ax * (double)rcp * ldexp(1.0, s - 1) * 65536.0);
            *lo = (int32_t)(p16 / 65536.0);
            *F = (uint32_t)(p16 - (double)*lo * 65536.0);
        }
    }
    return GQO_OK;
}

/* gqo_quantize_cols in the 16-bit-uniform mode: code = sign(x) (lo + (H < F)) with
 * H = gqo_philox_word(seed, step, i, j) >> 16; the exact mode's decision for norms outside
 * [2^-100, 2^100]. */
int gqo_quantize_u16_cols(const void *xw, int dtype, int64_t n, int64_t ld, int64_t j0,
                          int64_t w, float norm, int scheme, int s, uint64_t seed, uint64_t step,
                          int8_t *codes)
{
    int64_t i, j;
    if (xw == NULL || codes == NULL || n < 1 || w < 0 || ld < w || j0 < 0)
        return GQO_ERR_INVALID;
    if (dtype != GQO_F32 && dtype != GQO_BF16)
        return GQO_ERR_INVALID;
    if (scheme != GQO_LINEAR && scheme != GQO_EXP)
        return GQO_ERR_INVALID;
    if (s < 1 || s > (scheme == GQO_LINEAR ? 127 : 62))
        return GQO_ERR_UNSUPPORTED;
    if (isnan(norm) || isinf(norm) || norm < 0.0f) {
        memset(codes, 0, (size_t)(n * w));
        return GQO_ERR_NONFINITE;
    }
    if (norm == 0.0f) {
        memset(codes, 0, (size_t)(n * w));
        return GQO_OK;
    }
    for (i = 0; i < n; ++i) {
        for (j = 0; j < w; ++j) {
            float xe = load_x(xw, dtype, i * ld + j);
            uint32_t word = gqo_philox_word(seed, step, i, j0 + j);
            int32_t lo, lvl;
            uint32_t F;
            int rc = gqo_level_split_u16(xe, norm, scheme, s, &lo, &F);
            if (rc == GQO_USE_EXACT) {
                uint32_t T;
                rc = gqo_level_split(xe, norm, scheme, s, &lo, &T);
                if (rc != GQO_OK)
                    return rc;
                lvl = lo + (int32_t)(word < T);
            } else if (rc != GQO_OK) {
                return rc;
            } else {
                lvl = lo + (int32_t)((word >> 16) < F); /* H < F: up with probability F / 2^16 */
            }
            codes[i * w + j] = (int8_t)(xe < 0.0f ? -lvl : lvl);
        }
    }
    return GQO_OK;
}

/*
 * Sum the codes over the n workers: the reduction the allreduce performs.  For Global-L_s the
 * code is summed as it is (Global-QSGD, performance model: standard dithering reduces by the
 * native arithmetic sum).  For Global-E_s a code of level index k stands for the value
 * 2^-(s-k) = 2^(k-1) units of 2^-(s-1), so the sum adds sign * 2^(k-1) (0 for k = 0), which
 * keeps it an exact integer.  codes is n x w, worker-major; sums has w entries.
 */
int gqo_reduce_codes(const int8_t *codes, int scheme, int s, int64_t n, int64_t w,
                     int64_t *sums)
{
    int64_t i, j;
    if (codes == NULL || sums == NULL || n < 1 || w < 0)
        return GQO_ERR_INVALID;
    if (scheme != GQO_LINEAR && scheme != GQO_EXP)
        return GQO_ERR_INVALID;
    if (s < 1 || s > (scheme == GQO_LINEAR ? 127 : 62))
        return GQO_ERR_UNSUPPORTED;
    for (j = 0; j < w; ++j) {
        int64_t acc = 0;
        for (i = 0; i < n; ++i) {
            int c = codes[i * w + j];
            if (scheme == GQO_LINEAR) {
                acc += c;
            } else if (c != 0) {
                int k = c < 0 ? -c : c;
                int64_t units = (int64_t)1 << (k - 1);
                acc += c < 0 ? -units : units;
            }
        }
        sums[j] = acc;
    }
    return GQO_OK;
}

/*
 * Dequantise the code sums to the estimate of the mean gradient (1/n) sum_i Q(x_i), with
 * Q(x_i) = N * sign(x_i) * level (Global-QSGD, Global-Q operator; third step of the
 * communication hook).  One code unit is 1/s for Global-L_s and 2^-(s-1) for Global-E_s, so
 * out_j = N * S_j / (n * s) or N * S_j * 2^-(s-1) / n.  In fp64, N * S_j is exact while
 * |S_j| < 2^29 (a 24-bit significand times a 29-bit integer), the power-of-two scaling is exact,
 * and the division by n (or n * s) is the one rounding.
 */
int gqo_dequantize(const int64_t *sums, float norm, int scheme, int s, int64_t n, int64_t w,
                   double *out)
{
    int64_t j;
    if (sums == NULL || out == NULL || n < 1 || w < 0)
        return GQO_ERR_INVALID;
    if (scheme != GQO_LINEAR && scheme != GQO_EXP)
        return GQO_ERR_INVALID;
    if (s < 1 || s > (scheme == GQO_LINEAR ? 127 : 62))
        return GQO_ERR_UNSUPPORTED;
    if (isnan(norm) || isinf(norm)) {
        for (j = 0; j < w; ++j)
            out[j] = 0.0;
        return GQO_ERR_NONFINITE;
    }
    for (j = 0; j < w; ++j) {
        double num = (double)norm * (double)sums[j];
        if (scheme == GQO_LINEAR)
            out[j] = num / ((double)n * (double)s);
        else
            out[j] = ldexp(num, -(s - 1)) / (double)n;
    }
    return GQO_OK;
}

/*
 * The whole pipeline on the coordinate window [j0, j1): global norm over all d coordinates
 * (fp64), rounded once to the fp32 norm N that the quantiser uses; codes, code sums and the
 * dequantised mean for the window.  *norm64 receives the fp64 norm and *norm32 the fp32 one.
 * codes (n x w int8), sums (w int64) and out (w fp64) are written for the window.
 */
int gqo_allreduce_mean(const void *x, int dtype, int64_t n, int64_t d, int q, int p, int scheme,
                       int s, uint64_t seed, uint64_t step, int64_t j0, int64_t j1,
                       double *norm64, float *norm32, int8_t *codes, int64_t *sums, double *out)
{
    double nrm;
    float n32;
    int rc;
    int64_t w = j1 - j0;
    if (norm64 == NULL || norm32 == NULL || codes == NULL || sums == NULL || out == NULL)
        return GQO_ERR_INVALID;
    nrm = gqo_global_norm(x, dtype, n, d, q, p);
    if (nrm < 0.0)
        return GQO_ERR_INVALID;
    n32 = (float)nrm;
    *norm64 = nrm;
    *norm32 = n32;
    rc = gqo_quantize(x, dtype, n, d, j0, j1, n32, scheme, s, seed, step, codes);
    if (rc != GQO_OK && rc != GQO_ERR_NONFINITE)
        return rc;
    {
        int rc2 = gqo_reduce_codes(codes, scheme, s, n, w, sums);
        if (rc2 != GQO_OK)
            return rc2;
        rc2 = gqo_dequantize(sums, n32, scheme, s, n, w, out);
        if (rc2 != GQO_OK)
            return rc2;
    }
    return rc;
}

/* ------------------------------------------------------------------------------------------ */
/* Global-E allreduce with re-rounding at every hop                                           */
/* ------------------------------------------------------------------------------------------ */

/*
 * Global-QSGD's exponential dithering keeps the communicated data in the exponential code inside
 * the allreduce: every reduction step decodes two partial sums, adds them and rounds the result
 * at random back onto the grid, which adds variance ("extra variance due to stochastic rounding
 * during AllReduce", the theta worked example; the implementation paragraph's custom reduction
 * for exponential dithering; the performance model prefers the tree allreduce because it has
 * fewer such steps).  The pages do not spell the step out.  Reading taken: a partial sum is
 * kept in the same code, extended above level s (level index k stands for 2^(k-1) units of
 * 2^-(s-1), k = 0 for 0, any k up to 127); the sum t of two decoded values is an exact integer
 * number of units, and |t| > 0 is rounded between 2^e and 2^(e+1), e = floor(log2 |t|), up with
 * probability (|t| - 2^e) / 2^e (exact, so the step is unbiased); the sign of t is kept.
 */

/* Value of an extended Global-E code in units of 2^-(s-1). */
static int64_t exp_units(int c)
{
    int k = c < 0 ? -c : c;
    int64_t u;
    if (k == 0)
        return 0;
    u = (int64_t)1 << (k - 1);
    return c < 0 ? -u : u;
}

/* Where |t| units sit on the extended exponential grid: *lo = level index of 2^e (e + 1),
 * *T = floor(P(up) 2^32) with P(up) = (|t| - 2^e) / 2^e.  t = 0 gives lo = 0, T = 0. */
int gqo_exp_split_units(int64_t t, int32_t *lo, uint32_t *T)
{
    int e = 0;
    uint64_t a, frac;
    if (lo == NULL || T == NULL)
        return GQO_ERR_INVALID;
    a = (uint64_t)(t < 0 ? -t : t);
    if (a == 0) {
        *lo = 0;
        *T = 0;
        return GQO_OK;
    }
    while (e < 63 && (a >> (e + 1)) != 0)
        ++e;
    frac = a - ((uint64_t)1 << e); /* the distance above the lower level, < 2^e */
    *lo = e + 1;
    if (e <= 32)
        *T = (uint32_t)(frac << (32 - e)); /* exact: frac 2^(32 - e) < 2^32 */
    else
        *T = (uint32_t)(frac >> (e - 32));
    return GQO_OK;
}

/* Re-round t units with the random word of (seed, step, stream, j): the signed code. */
static int exp_reround(int64_t t, uint64_t seed, uint64_t step, int64_t stream_id, int64_t j)
{
    int32_t lo;
    uint32_t T;
    int k;
    gqo_exp_split_units(t, &lo, &T);
    k = lo + (gqo_philox_word(seed, step, stream_id, j) < T ? 1 : 0);
    return t < 0 ? -k : k;
}

/* Random-stream identifiers of the reduction steps (counter word 1; worker indices are below
 * 2^31): tree level l (1-based) combining into node m: 2^31 + l 2^24 + m; ring step h (1-based)
 * of chunk c: 2^31 + 2^30 + h 2^12 + c. */
int64_t gqo_exp_tree_stream(int l, int64_t m) { return (int64_t)0x80000000LL + ((int64_t)l << 24) + m; }
int64_t gqo_exp_ring_stream(int64_t h, int64_t c) { return (int64_t)0xC0000000LL + (h << 12) + c; }

/*
 * One reduction step on w coordinates (the custom reduction of the pages' Global-E allreduce):
 * out[j] = re-round(decode(a[j]) + decode(b[j])) with the random words of stream `stream_id` at
 * coordinates j0 + j.  Codes are signed level indices, |k| <= 62 on input.
 */
int gqo_exp_combine(const int8_t *a, const int8_t *b, int64_t w, int64_t j0, uint64_t seed,
                    uint64_t step, int64_t stream_id, int8_t *out)
{
    int64_t j;
    if (a == NULL || b == NULL || out == NULL || w < 0 || j0 < 0)
        return GQO_ERR_INVALID;
    for (j = 0; j < w; ++j)  /* 2^61 units at most per operand keeps every sum in int64 */
        if (a[j] > 62 || a[j] < -62 || b[j] > 62 || b[j] < -62)
            return GQO_ERR_UNSUPPORTED;
    for (j = 0; j < w; ++j) {
        int64_t t = exp_units(a[j]) + exp_units(b[j]);
        int c = exp_reround(t, seed, step, stream_id, j0 + j);
        if (c > 127 || c < -127)
            return GQO_ERR_UNSUPPORTED;
        out[j] = (int8_t)c;
    }
    return GQO_OK;
}

/*
 * Tree allreduce of n code rows (n x w, worker-major) with a re-rounding at every step (the
 * pages' tree: reduce recursively, then a recursive-doubling allgather that only copies).
 * Level l = 1, 2, ...: row i (a multiple of 2^l) takes re-round(row i + row i + 2^(l-1)) when
 * that partner exists, else it is kept.  root receives row 0 (w codes).  1 <= n <= 4096.
 */
int gqo_exp_tree_allreduce(const int8_t *codes, int64_t n, int64_t w, int64_t j0, uint64_t seed,
                           uint64_t step, int8_t *root)
{
    int64_t i, j;
    int l;
    int64_t *u;
    if (codes == NULL || root == NULL || n < 1 || n > 4096 || w < 0 || j0 < 0)
        return GQO_ERR_INVALID;
    u = (int64_t *)malloc(sizeof(int64_t) * (size_t)n);
    if (u == NULL)
        return GQO_ERR_INVALID;
    for (j = 0; j < w; ++j) {
        int8_t c0 = codes[j];
        for (i = 0; i < n; ++i)
            u[i] = exp_units(codes[i * w + j]);
        for (l = 1; ((int64_t)1 << (l - 1)) < n; ++l) {
            int64_t half = (int64_t)1 << (l - 1), stride = (int64_t)1 << l;
            for (i = 0; i + half < n; i += stride) {
                int c = exp_reround(u[i] + u[i + half], seed, step,
                                    gqo_exp_tree_stream(l, i >> l), j0 + j);
                u[i] = exp_units(c);
                if (c > 127 || c < -127) {
                    free(u);
                    return GQO_ERR_UNSUPPORTED;
                }
            }
        }
        /* the root's code: u[0] is a single level (or the untouched code when n = 1) */
        if (n == 1) {
            root[j] = c0;
        } else {
            int32_t lo;
            uint32_t T;
            gqo_exp_split_units(u[0], &lo, &T); /* exact level: T = 0 */
            root[j] = (int8_t)(u[0] < 0 ? -lo : lo);
        }
    }
    free(u);
    return GQO_OK;
}

/*
 * Ring allreduce of n code rows over d coordinates (the window [j0, j0 + w)): the coordinates
 * are split into n chunks of ceil(d / n) rounded up to a multiple of 16 (so that every chunk
 * starts on a group of 8 coordinates that share one Philox call; the last chunks may be short
 * or empty); chunk c is accumulated starting from worker c + 1 and
 * visits workers c + 2, ..., c (indices mod n), re-rounding after every step h = 1..n-1 (the
 * reduce-scatter; the allgather only copies).  root receives the reduced codes.
 */
int gqo_exp_ring_allreduce(const int8_t *codes, int64_t n, int64_t d, int64_t w, int64_t j0,
                           uint64_t seed, uint64_t step, int8_t *root)
{
    int64_t j, h, chunk;
    if (codes == NULL || root == NULL || n < 1 || n > 4096 || w < 0 || j0 < 0 || j0 + w > d)
        return GQO_ERR_INVALID;
    chunk = ((d + n - 1) / n + 15) / 16 * 16;
    for (j = 0; j < w; ++j) {
        int64_t c = (j0 + j) / chunk;
        int code = codes[((c + 1) % n) * w + j];
        for (h = 1; h < n; ++h) {
            int64_t t = exp_units(code) + exp_units(codes[((c + 1 + h) % n) * w + j]);
            code = exp_reround(t, seed, step, gqo_exp_ring_stream(h, c), j0 + j);
            if (code > 127 || code < -127)
                return GQO_ERR_UNSUPPORTED;
        }
        root[j] = (int8_t)code;
    }
    return GQO_OK;
}
