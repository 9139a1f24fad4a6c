/*
 * oracle.c -- plain, slow, single-threaded CPU oracle for the stateless
 * counter-based lowbias32 random fills.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file: only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA path; both are written independently from the definitions below.
 *
 * Every function is written as the plain definition, one element at a time,
 * in the order the sources state it.  Citations name the web page and the
 * section the definition comes from:
 *   [Phobos]  Phobos stdlib, "Random numbers" (sections hash32, uniform,
 *             randn, dropout; source std/random.ph).
 *   [Tandem-D] tandem-sycl, "Design" (sections Fills, Normals).
 *   [Tandem-P] tandem-cuda, "Performance" (section GPU, bounded fills).
 *   [PK]      perturbation-kernel, "Backends" (section "Why the GPU can be
 *             exact": Lemire's multiply-shift with rejection).
 * Readings the pages leave open are marked READING and are listed in the
 * design notes of the repository.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fexcess-precision=standard
 *        -fPIC -shared oracle.c -o liboracle.so -lm [-lquadmath on x86-64]
 * (no contraction of a*b+c into fma: every rounding below is the one written).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#if defined(__aarch64__)
/* long double is IEEE binary128 on aarch64 Linux. */
typedef long double quad;
#define Q_EXP expl
#define Q_LOG logl
#define Q_SQRT sqrtl
#define Q_ERFC erfcl
#define Q_ACOS acosl
#define Q_RINT rintl
#elif defined(__x86_64__)
#include <quadmath.h>
typedef __float128 quad;
#define Q_EXP expq
#define Q_LOG logq
#define Q_SQRT sqrtq
#define Q_ERFC erfcq
#define Q_ACOS acosq
#define Q_RINT rintq
#else
#error "the oracle needs a binary128 type (aarch64 long double or x86-64 __float128)"
#endif

/* ------------------------------------------------------------------------ */
/* hash32 = lowbias32 [Phobos, section hash32, std/random.ph:13]             */
/* ------------------------------------------------------------------------ */

/* _mix(x, s) = x ^ (x >>> s).  The page states the shifts are logical: an
 * arithmetic >> on the signed i32 has the bits it copies in masked off, which
 * is a logical shift of the 32-bit pattern.  READING: the body of _mix is not
 * printed; an xorshift by s is the reading the tile mean pins. */
static uint32_t mix(uint32_t x, unsigned s) { return x ^ (x >> s); }

/* Wrapping 32-bit multiplies by 2146121005 = 0x7FEB352D and by
 * -2073254261, whose two's-complement pattern is 0x846CA68B. */
uint32_t orc_hash32(uint32_t x)
{
    x = mix(x, 16);
    x = x * 2146121005u;
    x = mix(x, 15);
    x = x * (uint32_t)(-2073254261);
    x = mix(x, 16);
    return x;
}

/* The draw behind uniform(seed, counter): hash32(counter ^ hash32(seed))
 * [Phobos, section uniform, std/random.ph:21]. */
uint32_t orc_draw32(uint32_t seed, uint32_t counter)
{
    return orc_hash32(counter ^ orc_hash32(seed));
}

/* 64-bit draw: the 32-bit draw at counter 2c is the high word and the one at
 * 2c+1 the low word, counters wrapping mod 2^32 (as randn consumes 2c and
 * 2c+1 [Phobos, section randn]). */
uint64_t orc_draw64(uint32_t seed, uint32_t counter)
{
    uint32_t c2 = 2u * counter;
    return ((uint64_t)orc_draw32(seed, c2) << 32) | (uint64_t)orc_draw32(seed, c2 + 1u);
}

/* uniform(seed, c) = f32(draw & 8388607) * 1.1920928955078125e-7, the low 23
 * bits on a 2^-23 grid in [0, 1) [Phobos, section uniform].  The literal is
 * exactly 2^-23 and the product is exact. */
float orc_uniform_f32(uint32_t seed, uint32_t counter)
{
    return (float)(orc_draw32(seed, counter) & 8388607u) * 1.1920928955078125e-7f;
}

/* f64 uniform: the top 53 bits of the 64-bit draw times 2^-53 (exact). */
double orc_uniform_f64(uint32_t seed, uint32_t counter)
{
    return (double)(orc_draw64(seed, counter) >> 11) * 0x1p-53;
}

/* Narrow draws [Tandem-P, rows fill_u16, fill_f16_bits, fill_u8, fill_bool]:
 * element c is a byte, halfword or bit of the 32-bit draw at c >> 2, c >> 1
 * or c >> 5, least significant first.  READING: this layout. */
uint8_t orc_u8(uint32_t seed, uint32_t counter)
{
    return (uint8_t)(orc_draw32(seed, counter >> 2) >> (8u * (counter & 3u)));
}

uint16_t orc_u16(uint32_t seed, uint32_t counter)
{
    return (uint16_t)(orc_draw32(seed, counter >> 1) >> (16u * (counter & 1u)));
}

uint8_t orc_bool(uint32_t seed, uint32_t counter)
{
    return (uint8_t)((orc_draw32(seed, counter >> 5) >> (counter & 31u)) & 1u);
}

/* binary16 bits of m 2^-10, m the low 10 bits of the u16 element: zero, or
 * 2^(p-10) (1 + f) with p the position of m's leading one, biased exponent
 * p - 10 + 15, and the 10 bits of m below its leading one as the fraction.
 * READING: the f16 fill as a uniform on the 2^-10 grid. */
uint16_t orc_f16_bits(uint32_t seed, uint32_t counter)
{
    uint32_t m = orc_u16(seed, counter) & 0x3FFu;
    if (m == 0) return 0;
    unsigned p = 0;
    while ((m >> (p + 1)) != 0) ++p;
    uint32_t fraction = (m << (10u - p)) & 0x3FFu;
    return (uint16_t)(((p + 5u) << 10) | fraction);
}

/* ------------------------------------------------------------------------ */
/* Substreams for retries and ziggurat misses [Tandem-D, section Normals:     */
/* a draw that misses continues on split(g) of sub(PURPOSE) of the key, g the */
/* draw's global index].  READING, restated in hash32: the purpose key is     */
/* hash32(hash32(seed) ^ P), the element key hash32(g ^ purpose key) with g   */
/* the element's own counter, and the k-th word hash32(k ^ element key).      */
/* ------------------------------------------------------------------------ */

#define PURPOSE_BELOW32 0x42333220u  /* "B32 " */
#define PURPOSE_BELOW64 0x42363420u  /* "B64 " */
#define PURPOSE_NORMAL64 0x4E363420u /* "N64 " */

static uint32_t substream_key(uint32_t seed, uint32_t purpose, uint32_t g)
{
    uint32_t purpose_key = orc_hash32(orc_hash32(seed) ^ purpose);
    return orc_hash32(g ^ purpose_key);
}

static uint32_t substream32(uint32_t key, uint32_t k) { return orc_hash32(k ^ key); }

static uint64_t substream64(uint32_t key, uint32_t k)
{
    return ((uint64_t)substream32(key, 2u * k) << 32) | (uint64_t)substream32(key, 2u * k + 1u);
}

/* For the pins: the element keys of counters g[0..n) for one purpose (which
 * = 0 B32, 1 B64, 2 N64), and words k0 .. k0 + n - 1 of one element key. */
void orc_substream_keys(uint32_t seed, int which, const uint32_t *g, size_t n, uint32_t *out)
{
    const uint32_t purpose = which == 0 ? PURPOSE_BELOW32 : which == 1 ? PURPOSE_BELOW64 : PURPOSE_NORMAL64;
    for (size_t i = 0; i < n; ++i) out[i] = substream_key(seed, purpose, g[i]);
}

void orc_substream_words32(uint32_t key, uint32_t k0, size_t n, uint32_t *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = substream32(key, k0 + (uint32_t)i);
}

void orc_substream_words64(uint32_t key, uint32_t k0, size_t n, uint64_t *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = substream64(key, k0 + (uint32_t)i);
}

/* ------------------------------------------------------------------------ */
/* Bounded integers: Lemire's multiply-shift with rejection [PK; Tandem-P].  */
/* ------------------------------------------------------------------------ */

/* One step on a w-bit word x (1 <= w <= 64) for the bound b (1 <= b < 2^w):
 * the 2w-bit product x*b; its high w bits are the candidate value and it is
 * accepted when its low w bits are at least 2^w mod b (Lemire 2019, "Fast
 * Random Integer Generation in an Interval", exact threshold).  READING: the
 * exact threshold, not the conservative zone of the perturbation-kernel page;
 * both are exactly uniform. */
int orc_lemire_step(uint64_t x, uint64_t b, unsigned w, uint64_t *value)
{
    unsigned __int128 two_w = (unsigned __int128)1 << w;
    unsigned __int128 prod = (unsigned __int128)x * b;
    uint64_t low = (uint64_t)(prod % two_w);
    uint64_t threshold = (uint64_t)(two_w % b);
    *value = (uint64_t)(prod / two_w);
    return low >= threshold;
}

/* below32(b): the element's 32-bit draw, then the B32 substream's words. */
uint32_t orc_below32(uint32_t seed, uint32_t counter, uint32_t b)
{
    uint64_t v;
    if (b == 0) return 0; /* rejected by the API; never sampled */
    if (orc_lemire_step(orc_draw32(seed, counter), b, 32, &v)) return (uint32_t)v;
    uint32_t key = substream_key(seed, PURPOSE_BELOW32, counter);
    for (uint32_t k = 0;; ++k)
        if (orc_lemire_step(substream32(key, k), b, 32, &v)) return (uint32_t)v;
}

/* below64(b): the element's 64-bit draw, then the B64 substream's words. */
uint64_t orc_below64(uint32_t seed, uint32_t counter, uint64_t b)
{
    uint64_t v;
    if (b == 0) return 0;
    if (orc_lemire_step(orc_draw64(seed, counter), b, 64, &v)) return v;
    uint32_t key = substream_key(seed, PURPOSE_BELOW64, counter);
    for (uint32_t k = 0;; ++k)
        if (orc_lemire_step(substream64(key, k), b, 64, &v)) return v;
}

/* low + below(b), wrapped to the output type (two's complement)
 * [Tandem-P, rows "with a low bound into int32_t / int64_t"]. */
int32_t orc_range_i32(uint32_t seed, uint32_t counter, int32_t low, uint32_t b)
{
    return (int32_t)((uint32_t)low + orc_below32(seed, counter, b));
}

int64_t orc_range_i64_32(uint32_t seed, uint32_t counter, int64_t low, uint32_t b)
{
    return (int64_t)((uint64_t)low + (uint64_t)orc_below32(seed, counter, b));
}

int64_t orc_range_i64(uint32_t seed, uint32_t counter, int64_t low, uint64_t b)
{
    return (int64_t)((uint64_t)low + orc_below64(seed, counter, b));
}

/* ------------------------------------------------------------------------ */
/* randn [Phobos, section randn, std/random.ph:26]                           */
/* ------------------------------------------------------------------------ */

/* sqrt(-2 log(1 - u0)) * cos(6.283185307179586 u1) for the uniforms of the
 * 32-bit draws d0 and d1 (u = (d & 0x7FFFFF) 2^-23, section uniform),
 * evaluated in binary64 and returned unrounded to f32 (the reference value
 * the f32 path is held to). */
double orc_box_muller(uint32_t d0, uint32_t d1)
{
    double u0 = (double)(d0 & 0x7FFFFFu) * 0x1p-23;
    double u1 = (double)(d1 & 0x7FFFFFu) * 0x1p-23;
    return sqrt(-2.0 * log(1.0 - u0)) * cos(6.283185307179586 * u1);
}

/* randn(seed, c): the Box-Muller value of the draws at counters 2c and 2c+1
 * (their f32 uniforms are the uniforms above, exactly). */
double orc_randn(uint32_t seed, uint32_t counter)
{
    return orc_box_muller(orc_draw32(seed, 2u * counter), orc_draw32(seed, 2u * counter + 1u));
}

/* The sine branch of the same pair, sqrt(-2 log(1 - u0)) sin(2 pi u1) (the
 * second value of a Box-Muller pair [Tandem-D, section Normals]). */
double orc_box_muller_sin(uint32_t d0, uint32_t d1)
{
    double u0 = (double)(d0 & 0x7FFFFFu) * 0x1p-23;
    double u1 = (double)(d1 & 0x7FFFFFu) * 0x1p-23;
    return sqrt(-2.0 * log(1.0 - u0)) * sin(6.283185307179586 * u1);
}

/* out[i] = the cosine branch of (d0[i], d1[i]); out_sin[i], if out_sin is
 * not NULL, the sine branch. */
void orc_box_muller_fill(const uint32_t *d0, const uint32_t *d1, size_t n, double *out, double *out_sin)
{
    for (size_t i = 0; i < n; ++i) {
        out[i] = orc_box_muller(d0[i], d1[i]);
        if (out_sin) out_sin[i] = orc_box_muller_sin(d0[i], d1[i]);
    }
}

/* Paired Box-Muller (both branches of one uniform pair, as the tandem
 * pages draw pairs [Tandem-D, section Normals]): element c takes pair
 * q = c >> 1, the uniforms at 2q and 2q + 1, and the cosine branch for even
 * c (randn at counter q) or the sine branch for odd c.  READING: this
 * counter layout. */
double orc_randn_paired(uint32_t seed, uint32_t counter)
{
    uint32_t q = counter >> 1;
    double u0 = (double)orc_uniform_f32(seed, 2u * q);
    double u1 = (double)orc_uniform_f32(seed, 2u * q + 1u);
    double r = sqrt(-2.0 * log(1.0 - u0));
    return (counter & 1u) ? r * sin(6.283185307179586 * u1) : r * cos(6.283185307179586 * u1);
}

/* ------------------------------------------------------------------------ */
/* dropout [Phobos, section dropout, std/random.ph:30]                       */
/* ------------------------------------------------------------------------ */

/* where(uniform(seed, c) >= p, x / (1 - p), 0), all in f32 with IEEE
 * division; a tie u == p is kept. */
float orc_dropout(float x, float p, uint32_t seed, uint32_t counter)
{
    float u = orc_uniform_f32(seed, counter);
    float keep_scale_divisor = 1.0f - p;
    return (u >= p) ? x / keep_scale_divisor : 0.0f;
}

/* ------------------------------------------------------------------------ */
/* Deterministic binary64 exp and log for the ziggurat's slow path.          */
/* Both are fixed sequences of IEEE operations (+, -, *, /, fma, rint), so a */
/* second implementation that performs the same operations in the same order */
/* returns the same bits on any IEEE machine.                                */
/* ------------------------------------------------------------------------ */

/* ln 2 split for Cody & Waite's argument reduction (Cody & Waite 1980,
 * "Software Manual for the Elementary Functions"): the high part is ln 2
 * rounded to 32 significant bits, so k * high is exact for |k| < 2^21; the
 * low part is ln 2 - high rounded to binary64. */
static const double LN2_HIGH = 0x1.62e42ffp-1;
static const double LN2_LOW = -0x1.718432a1b0e26p-35;
static const double INV_LN2 = 0x1.71547652b82fep+0; /* 1/ln 2 rounded */
static const double SQRT2 = 0x1.6a09e667f3bcdp+0;   /* sqrt 2 rounded */

/* exp(t): k = rint(t / ln 2), r = t - k ln 2 by two fma, then the Taylor
 * polynomial of degree 13 in Horner form, then the exact scaling by 2^k.
 * Valid where the result is a normal number (the slow path needs t in
 * [-10, 0]). */
double orc_zexp(double t)
{
    double k = rint(t * INV_LN2);
    double r = fma(-k, LN2_HIGH, t);
    r = fma(-k, LN2_LOW, r);
    double p = 1.0 / 6227020800.0; /* 1/13! */
    p = fma(p, r, 1.0 / 479001600.0); /* 1/12! */
    p = fma(p, r, 1.0 / 39916800.0);  /* 1/11! */
    p = fma(p, r, 1.0 / 3628800.0);   /* 1/10! */
    p = fma(p, r, 1.0 / 362880.0);    /* 1/9! */
    p = fma(p, r, 1.0 / 40320.0);     /* 1/8! */
    p = fma(p, r, 1.0 / 5040.0);      /* 1/7! */
    p = fma(p, r, 1.0 / 720.0);       /* 1/6! */
    p = fma(p, r, 1.0 / 120.0);       /* 1/5! */
    p = fma(p, r, 1.0 / 24.0);        /* 1/4! */
    p = fma(p, r, 1.0 / 6.0);         /* 1/3! */
    p = fma(p, r, 0.5);               /* 1/2! */
    p = fma(p, r, 1.0);               /* 1/1! */
    p = fma(p, r, 1.0);               /* 1/0! */
    return ldexp(p, (int)k);
}

/* log(x) for normal positive x: x = 2^e m with m in (sqrt(1/2), sqrt 2],
 * s = (m - 1)/(m + 1), log m = 2 atanh s = 2 (s + s^3/3 + ... + s^23/23)
 * (Abramowitz & Stegun 4.1.27), then log x = e ln 2 + log m with the split
 * ln 2 above. */
double orc_zlog(double x)
{
    uint64_t bits;
    memcpy(&bits, &x, sizeof bits);
    int e = (int)(bits >> 52) - 1023;
    uint64_t mbits = (bits & 0x000FFFFFFFFFFFFFull) | 0x3FF0000000000000ull;
    double m;
    memcpy(&m, &mbits, sizeof m);
    if (m > SQRT2) {
        m = m * 0.5;
        e = e + 1;
    }
    double s = (m - 1.0) / (m + 1.0);
    double s2 = s * s;
    double p = 1.0 / 23.0;
    p = fma(p, s2, 1.0 / 21.0);
    p = fma(p, s2, 1.0 / 19.0);
    p = fma(p, s2, 1.0 / 17.0);
    p = fma(p, s2, 1.0 / 15.0);
    p = fma(p, s2, 1.0 / 13.0);
    p = fma(p, s2, 1.0 / 11.0);
    p = fma(p, s2, 1.0 / 9.0);
    p = fma(p, s2, 1.0 / 7.0);
    p = fma(p, s2, 1.0 / 5.0);
    p = fma(p, s2, 1.0 / 3.0);
    double two_s = s + s;
    double log_m = fma(two_s * s2, p, two_s);
    double de = (double)e;
    return fma(de, LN2_HIGH, fma(de, LN2_LOW, log_m));
}

/* ------------------------------------------------------------------------ */
/* Exponentials [Tandem-D, section Exponentials]: -ln(1 - u).  READING: the   */
/* f32 fill on the f32 uniform (its binary64 value here; the fill's own       */
/* binary32 log below), the f64 fill on the f64 uniform through this file's   */
/* own fixed-point logarithm (further below).                                */
/* ------------------------------------------------------------------------ */

double orc_exponential_f32(uint32_t seed, uint32_t counter)
{
    return -log(1.0 - (double)orc_uniform_f32(seed, counter));
}

/* The f32 exponential in binary32 arithmetic, this library's own logarithm
 * (the pages' two-float neg_log_f32 is not printed; their target, every draw
 * within 0.571 ulp, is kept).  READING: -ln(v) for v = 1 - u = V 2^-23 with
 * the integer V = 2^23 - m in [1, 2^23] (m the uniform's 23 bits), by a
 * table-driven reduction (Tang, "Table-driven implementation of the
 * logarithm function in IEEE floating-point arithmetic", 1990):
 *   V = 2^k M, M in [1, 2), E = 23 - k, so -ln v = E ln 2 - ln M;
 *   j = round((M - 1) 256) in [0, 256], inv_j = 1/(1 + j/256) rounded to 8
 *   significant bits, r = M inv_j - 1 (exact in binary32, |r| < 1.5 2^-8);
 *   -ln v = (E ln 2 + ln inv_j) - log1p(r),
 *   log1p(r) = r - r^2/2 + r^3/3 - r^4/4 + r^5/5 (Taylor; the next term is
 *   below 2^-37 of the result).
 * E ln 2 + ln inv_j is carried as hi + lo: ln 2 and ln inv_j are split into
 * a multiple of 2^-19 (hi) and the binary32 rounding of the rest (lo), so
 * E ln2_hi + hi_j is exact; hi - r is summed exactly (TwoSum, Knuth TAOCP
 * vol. 2, 4.2.2), its error, the lo terms and the Taylor tail added after,
 * and the result rounded once at the end.  Every operation below is one
 * IEEE binary32 operation (fmaf a single rounding). */
static float neglog_inv[257], neglog_hi[257], neglog_lo[257];
static float neglog_ln2_hi, neglog_ln2_lo;
static int neglog_ready;

/* x > 0 rounded to p significant bits, to nearest (ties to even) */
static double round_to_bits(double x, int p)
{
    int e;
    double m = frexp(x, &e); /* x = m 2^e, m in [0.5, 1) */
    return ldexp(nearbyint(ldexp(m, p)), e - p);
}

static void neglog_split(quad v, float *hi, float *lo)
{
    quad h = Q_RINT(v * 524288) / 524288; /* nearest multiple of 2^-19 */
    *hi = (float)h;                        /* exact: at most 20 bits */
    *lo = (float)(v - h);                  /* one rounding */
}

static void neglog_init(void)
{
    if (neglog_ready) return;
    for (int j = 0; j <= 256; ++j) {
        /* 1/(1 + j/256) = 256/(256 + j); binary64 then 8 bits rounds as the
         * exact value would: no 256/(256 + j) lies on an 8-bit midpoint */
        neglog_inv[j] = (float)round_to_bits(256.0 / (256.0 + j), 8);
        neglog_split(Q_LOG((quad)neglog_inv[j]), &neglog_hi[j], &neglog_lo[j]);
    }
    neglog_split(Q_LOG((quad)2), &neglog_ln2_hi, &neglog_ln2_lo);
    neglog_ready = 1;
}

void orc_neglog_table(float *inv, float *hi, float *lo, float *ln2)
{
    neglog_init();
    for (int j = 0; j <= 256; ++j) {
        inv[j] = neglog_inv[j];
        hi[j] = neglog_hi[j];
        lo[j] = neglog_lo[j];
    }
    ln2[0] = neglog_ln2_hi;
    ln2[1] = neglog_ln2_lo;
}

/* -ln(1 - m 2^-23) in binary32, m in [0, 2^23) */
float orc_neglog_f32(uint32_t m)
{
    neglog_init();
    uint32_t V = 8388608u - m;
    float x = (float)V; /* exact: V <= 2^23 */
    uint32_t bits;
    memcpy(&bits, &x, sizeof bits);
    int k = (int)(bits >> 23) - 127;
    uint32_t mant = bits & 8388607u;
    uint32_t mbits = mant | 0x3F800000u;
    float M;
    memcpy(&M, &mbits, sizeof M);
    uint32_t j = (mant + 16384u) >> 15; /* round((M - 1) 256) */
    float E = (float)(23 - k);
    float r = fmaf(M, neglog_inv[j], -1.0f);
    float t_hi = fmaf(E, neglog_ln2_hi, neglog_hi[j]);
    float t_lo = fmaf(E, neglog_ln2_lo, neglog_lo[j]);
    float s = t_hi - r;
    float bb = s - t_hi;
    float err = (t_hi - (s - bb)) + (-r - bb);
    float r2 = r * r;
    float p = fmaf(r, -0x1.99999ap-3f, 0.25f); /* 1/4 - r/5 */
    p = fmaf(r, p, -0x1.555556p-2f);           /* -1/3 + r/4 - r^2/5 */
    p = fmaf(r, p, 0.5f);                      /* 1/2 - r/3 + r^2/4 - r^3/5 */
    float c = fmaf(r2, p, err + t_lo); /* + the tail r^2 p = -log1p(r) - (-r), in one rounding */
    return s + c;
}

/* ------------------------------------------------------------------------ */
/* Precise f32 normal [Tandem-D, section Normals: the default float normal   */
/* agrees with other ports to 16 ulp + 1e-6; a precise f32 Box-Muller is a   */
/* build option].  READING: an opt-in fill with randn's definition (the      */
/* uniforms at 2c and 2c + 1, cosine branch) evaluated in binary32 to a few  */
/* ulp: z = sqrt(2 NL(u0)) cos(2 pi u1), NL the own -ln(1 - u) above, an     */
/* IEEE square root, and the own cos(2 pi u1) below.                          */
/* ------------------------------------------------------------------------ */

/* cos(2 pi m 2^-23): the quadrant q = m >> 21 and g = (m mod 2^21) 2^-23 in
 * [0, 1/4) are exact; cos(2 pi (q/4 + g)) is cos g, -sin g, -cos g or sin g
 * (in turns of 2 pi); above g = 1/8 the complement h = 1/4 - g (exact)
 * swaps sin and cos.  On x = k 2^-23 <= 1/8 the Taylor series of sin(2 pi x)
 * to x^9 and cos(2 pi x) to x^10 (truncation below 2^-28 relative), each
 * coefficient (2 pi)^n / n! rounded once to binary32, the leading ones (2 pi
 * and -(2 pi)^2/2) as hi + lo so that their rounding does not reach the
 * result. */
static float cp_s1_hi, cp_s1_lo, cp_s3, cp_s5, cp_s7, cp_s9;
static float cp_c2_hi, cp_c2_lo, cp_c4, cp_c6, cp_c8, cp_c10;
static int cp_ready;

static void cos2pi_init(void)
{
    if (cp_ready) return;
    quad tp = 2 * Q_ACOS((quad)-1); /* 2 pi */
    quad term[11];                   /* term[n] = (2 pi)^n / n! */
    term[0] = 1;
    for (int n = 1; n <= 10; ++n) term[n] = term[n - 1] * tp / n;
    cp_s1_hi = (float)term[1];
    cp_s1_lo = (float)(term[1] - cp_s1_hi);
    cp_s3 = (float)(-term[3]);
    cp_s5 = (float)term[5];
    cp_s7 = (float)(-term[7]);
    cp_s9 = (float)term[9];
    cp_c2_hi = (float)(-term[2]);
    cp_c2_lo = (float)(-term[2] - cp_c2_hi);
    cp_c4 = (float)term[4];
    cp_c6 = (float)(-term[6]);
    cp_c8 = (float)term[8];
    cp_c10 = (float)(-term[10]);
    cp_ready = 1;
}

void orc_cos2pi_coefficients(float *out) /* s1_hi s1_lo s3 s5 s7 s9 c2_hi c2_lo c4 c6 c8 c10 */
{
    cos2pi_init();
    const float v[12] = {cp_s1_hi, cp_s1_lo, cp_s3, cp_s5, cp_s7, cp_s9,
                         cp_c2_hi, cp_c2_lo, cp_c4, cp_c6, cp_c8, cp_c10};
    for (int i = 0; i < 12; ++i) out[i] = v[i];
}

float orc_cos2pi_grid(uint32_t m)
{
    cos2pi_init();
    uint32_t q = m >> 21;
    uint32_t f = m & 0x1FFFFFu;
    int swap = f > 0x100000u;
    uint32_t k = swap ? 0x200000u - f : f;
    float x = (float)k * 0x1p-23f; /* exact: k <= 2^20 */
    float x2 = x * x;
    float p = fmaf(x2, cp_s9, cp_s7);
    p = fmaf(x2, p, cp_s5);
    p = fmaf(x2, p, cp_s3);
    p = fmaf(x2, p, cp_s1_lo);
    float sin_x = fmaf(x, cp_s1_hi, x * p);
    float c = fmaf(x2, cp_c10, cp_c8);
    c = fmaf(x2, c, cp_c6);
    c = fmaf(x2, c, cp_c4);
    float t = x2 * fmaf(x2, c, cp_c2_lo);
    float cos_x = 1.0f + fmaf(x2, cp_c2_hi, t);
    float v = ((int)(q & 1u) ^ swap) ? sin_x : cos_x;
    return (q == 1u || q == 2u) ? -v : v;
}

/* randn(seed, counter) in binary32 to a few ulp */
float orc_randn_precise(uint32_t seed, uint32_t counter)
{
    float e = orc_neglog_f32(orc_draw32(seed, 2u * counter) & 8388607u);
    float r = sqrtf(e + e); /* 2 e exact; IEEE square root */
    return r * orc_cos2pi_grid(orc_draw32(seed, 2u * counter + 1u) & 8388607u);
}

/* The f32 exponential fill's value: -ln(1 - u) through orc_neglog_f32. */
float orc_exponential_f32_own(uint32_t seed, uint32_t counter)
{
    return orc_neglog_f32(orc_draw32(seed, counter) & 8388607u);
}

/* -ln(1 - m 2^-53) in binary64 by the library's own fixed-point logarithm,
 * integer arithmetic only (GB300's FP64 pipe is 1/64 of its FP32 rate).
 * READING (the pages' f64 logarithm is not printed; their exponentials need
 * only an own, reproducible log): with V = 2^53 - m (1 - u = V 2^-53 exactly),
 *   V = 2^k M, M in [1, 2), E = 53 - k, so -ln(1 - u) = E ln 2 - ln M;
 *   j = floor((M - 1) 2048), and I_j = 2^23/(2048 + j) rounded up to an
 *   integer (12 significant bits, I_j in [2049, 4096]): the reciprocal
 *   inv_j = I_j / 4096 >= 1/(1 + j/2048), so r = M inv_j - 1 is never negative
 *   and r < 1.5 2^-11 (Tang 1990's table reduction, one-sided).  With
 *   W = V 2^(62 - k) (M at scale 2^62), W I_j = (1 + r) 2^74, so W I_j modulo
 *   2^64 is r 2^74 exactly (r 2^74 < 1.5 2^63);
 *   log1p(r) = r S(r), S(r) = sum_k (-r)^(k-1) / k for k = 1 .. 6 (Taylor;
 *   the next term is below 2^-65 of the result), by Horner on a = r: every
 *   value S_k = 1/k - a S_(k+1) is positive.  Each product is floored to the
 *   scale of the value it feeds: S_5 and S_4 at 2^33 and S_3 at 2^64 take a
 *   floored to 2^-42 (a 32-bit number), S_2 at 2^64 and S_1 at 2^63 take a
 *   itself; a S_1 exact in 128 bits (scale 2^137);
 *   -ln(1 - u) = E ln 2 + ln inv_j - a S_1, with E ln 2 + ln inv_j at scale
 *   2^96 (ln 2 and ln inv_j each rounded once to the nearest multiple of
 *   2^-96) and a S_1 floored to it.
 *   For m <= 2^41 (u <= 2^-12, where E ln 2 + ln inv_j would cancel against
 *   log1p(r)) the value is the series itself: -ln(1 - u) = u S(-u) with the
 *   same Horner steps on a = u (every term added), a S_1 at scale 2^137;
 *   the positive fixed-point value rounded once to binary64, to nearest even.
 * Within 0.5007 ulp of the exact value on the inputs tried. */
#define NL64_BINS 2048
static int32_t nl64_i[NL64_BINS];
static __int128 nl64_lninv[NL64_BINS], nl64_ln2;
static uint64_t nl64_c[7]; /* 1/k at the scale of S_k: 2^63 (k = 1), 2^64 (k = 2, 3), 2^33 (k = 4 .. 6) */
static int nl64_ready;

static __int128 nl64_round96(quad v) { return (__int128)Q_RINT(v * (quad)79228162514264337593543950336.0); } /* 2^96 */

static void nl64_init(void)
{
    if (nl64_ready) return;
    for (int j = 0; j < NL64_BINS; ++j) {
        uint32_t d = 2048u + (uint32_t)j;
        nl64_i[j] = (int32_t)(((1u << 23) + d - 1u) / d); /* ceil(2^23 / (2048 + j)) */
        nl64_lninv[j] = nl64_round96(Q_LOG((quad)nl64_i[j] / 4096));
    }
    nl64_ln2 = nl64_round96(Q_LOG((quad)2));
    static const int scale[7] = {0, 63, 64, 64, 33, 33, 33}; /* of S_k */
    for (int k = 1; k <= 6; ++k) /* 1/k at 2^scale, to nearest (no k here gives a half) */
        nl64_c[k] = (uint64_t)((((unsigned __int128)1 << scale[k]) + (unsigned)k / 2) / (unsigned)k);
    nl64_ready = 1;
}

/* the positive integer y times 2^-scale, rounded to the nearest binary64 */
static double nl64_to_double(unsigned __int128 y, int scale)
{
    int n = 0;
    for (unsigned __int128 t = y; t; t >>= 1) ++n; /* bit length */
    uint64_t mant;
    int shift = n - 53;
    if (shift <= 0) {
        mant = (uint64_t)(y << -shift);
    } else {
        mant = (uint64_t)(y >> shift);
        unsigned __int128 rest = y - ((unsigned __int128)mant << shift);
        unsigned __int128 half = (unsigned __int128)1 << (shift - 1);
        if (rest > half || (rest == half && (mant & 1))) ++mant;
    }
    return ldexp((double)mant, shift - scale); /* mant <= 2^53: exact in binary64 */
}

/* a S_1 of the series above at scale 2^137 for a at scale 2^74; add = 1 takes
 * every Horner term with a plus sign (S(-a), for the small-u series), add = 0
 * with alternating signs (S(a)) */
static unsigned __int128 nl64_series(uint64_t a, int add)
{
    uint64_t a42 = a >> 32; /* a 2^42, floored; below 2^32 */
    uint64_t S = nl64_c[6]; /* S_6 at 2^33 */
    for (int t = 5; t >= 4; --t) {
        uint64_t p = (a42 * S) >> 42; /* floor(a S_(t+1)) at 2^33 */
        S = add ? nl64_c[t] + p : nl64_c[t] - p;
    }
    uint64_t p3 = (a42 * S) >> 11; /* floor(a S_4) at 2^64 */
    S = add ? nl64_c[3] + p3 : nl64_c[3] - p3;
    uint64_t p2 = (uint64_t)(((unsigned __int128)a * S) >> 74); /* floor(a S_3) at 2^64 */
    S = add ? nl64_c[2] + p2 : nl64_c[2] - p2;
    uint64_t p1 = (uint64_t)(((unsigned __int128)a * S) >> 75); /* floor(a S_2) at 2^63 */
    S = add ? nl64_c[1] + p1 : nl64_c[1] - p1;
    return (unsigned __int128)a * S; /* a S_1 at 2^137, exact */
}

double orc_neglog64(uint64_t m) /* m < 2^53 */
{
    nl64_init();
    if (m == 0) return 0.0;
    if (m <= (1ull << 41)) return nl64_to_double(nl64_series(m << 21, 1), 137); /* u 2^74 */
    uint64_t V = (1ull << 53) - m;
    int k = 63 - __builtin_clzll(V);
    int E = 53 - k;
    uint64_t W = V << (62 - k);                     /* M 2^62 */
    uint32_t j = (uint32_t)((W - (1ull << 62)) >> 51); /* floor((M - 1) 2048) */
    uint64_t a = W * (uint64_t)nl64_i[j];           /* (1 + r) 2^74 modulo 2^64: r 2^74 */
    unsigned __int128 Pm = nl64_series(a, 0);       /* log1p(r) 2^137 */
    __int128 T = (__int128)E * nl64_ln2 + nl64_lninv[j];
    __int128 y = T - (__int128)(Pm >> 41);
    return nl64_to_double((unsigned __int128)y, 96);
}

/* The f64 exponential fill: -ln(1 - u) on the f64 uniform u = (D64 >> 11)
 * 2^-53, through the fixed-point logarithm above. */
double orc_exponential_f64(uint32_t seed, uint32_t counter)
{
    return orc_neglog64(orc_draw64(seed, counter) >> 11);
}

void orc_neglog64_table(int32_t *inv4096, int64_t *lninv_hi, uint64_t *lninv_lo, int64_t *ln2, uint64_t *coef)
{
    nl64_init();
    for (int j = 0; j < NL64_BINS; ++j) {
        inv4096[j] = nl64_i[j];
        lninv_hi[j] = (int64_t)(nl64_lninv[j] >> 64);
        lninv_lo[j] = (uint64_t)nl64_lninv[j];
    }
    ln2[0] = (int64_t)(nl64_ln2 >> 64);
    ln2[1] = (int64_t)(uint64_t)nl64_ln2;
    for (int k = 0; k <= 6; ++k) coef[k] = nl64_c[k];
}

/* ------------------------------------------------------------------------ */
/* 1024-layer Marsaglia-Tsang ziggurat [Tandem-D, section Normals]           */
/* (Marsaglia & Tsang 2000, "The Ziggurat Method for Generating Random       */
/* Variables").                                                              */
/* ------------------------------------------------------------------------ */

#define ZIG_LAYERS 1024

static quad qf(quad x) { return Q_EXP(-x * x / 2); }

/* Tail area plus base rectangle for the rightmost edge r:
 * v = r f(r) + integral_r^inf f = r f(r) + sqrt(pi/2) erfc(r / sqrt 2). */
static quad zig_area(quad r)
{
    quad pi = Q_ACOS((quad)-1);
    return r * qf(r) + Q_SQRT(pi / 2) * Q_ERFC(r / Q_SQRT((quad)2));
}

/* Residual of the top layer for a trial r: build X[1] = r, X[j+1] =
 * f^-1(f(X[j]) + v/X[j]) up to X[N-1] and return f(X[N-1]) + v/X[N-1] - 1,
 * which is zero when the top layer (up to f(0) = 1) also has area v.  A layer
 * that would already pass f(0) means r is too small: return +1. */
static quad zig_residual(quad r, unsigned N)
{
    quad v = zig_area(r);
    quad x = r;
    for (unsigned j = 1; j + 1 < N; ++j) {
        quad y = qf(x) + v / x;
        if (y >= 1) return 1;
        x = Q_SQRT(-2 * Q_LOG(y));
    }
    return qf(x) + v / x - 1;
}

/* Table for N layers, each entry the binary128 value rounded once to binary64:
 * r the root of the residual (bisection to binary128 resolution), X[0] =
 * v/f(r), X[1] = r, X[j+1] as above, X[N] = 0, F[j] = f(X[j]), F[N] = 1.
 * X and F hold N+1 entries.  Returns 0, or -1 for N < 2. */
int orc_zig_table(unsigned N, double *X, double *F, double *r_out, double *v_out)
{
    if (N < 2) return -1;
    quad lo = 1, hi = 10;
    for (int it = 0; it < 200; ++it) {
        quad mid = (lo + hi) / 2;
        if (mid == lo || mid == hi) break;
        if (zig_residual(mid, N) > 0)
            lo = mid;
        else
            hi = mid;
    }
    quad r = (lo + hi) / 2;
    quad v = zig_area(r);
    quad x = r;
    X[0] = (double)(v / qf(r));
    F[0] = (double)qf(v / qf(r));
    X[1] = (double)r;
    F[1] = (double)qf(r);
    for (unsigned j = 1; j + 1 < N; ++j) {
        x = Q_SQRT(-2 * Q_LOG(qf(x) + v / x));
        X[j + 1] = (double)x;
        F[j + 1] = (double)qf(x);
    }
    X[N] = 0.0;
    F[N] = 1.0;
    if (r_out) *r_out = (double)r;
    if (v_out) *v_out = (double)v;
    return 0;
}

static double zig_X[ZIG_LAYERS + 1], zig_F[ZIG_LAYERS + 1];
static int zig_ready;

static void zig_init(void)
{
    if (!zig_ready) {
        orc_zig_table(ZIG_LAYERS, zig_X, zig_F, NULL, NULL);
        zig_ready = 1;
    }
}

/* Copy of the 1024-layer table the normals use (1025 entries each). */
void orc_zig1024(double *X, double *F)
{
    zig_init();
    memcpy(X, zig_X, sizeof zig_X);
    memcpy(F, zig_F, sizeof zig_F);
}

/* Fast-path test of one 64-bit draw w: layer j = the low 10 bits, sign bit
 * 10, magnitude x = (w >> 11) 2^-53 X[j] (one rounded multiply); the draw is
 * taken when x < X[j+1].  READING: this bit layout (10 + 1 + 53 = 64 bits). */
static int zig_fast(uint64_t w, double *x_out, unsigned *j_out, int *neg_out)
{
    unsigned j = (unsigned)(w & (ZIG_LAYERS - 1));
    int neg = (int)((w >> 10) & 1u);
    double x = ((double)(w >> 11) * 0x1p-53) * zig_X[j];
    *x_out = x;
    *j_out = j;
    *neg_out = neg;
    return x < zig_X[j + 1];
}

/* x[i] = the fast path's magnitude (w[i] >> 11) 2^-53 X[j] (one rounded
 * multiply, j = w[i] & 1023) of each 64-bit draw, fast or not. */
void orc_zig_candidates(const uint64_t *w, size_t n, double *x)
{
    unsigned j;
    int neg;
    zig_init();
    for (size_t i = 0; i < n; ++i) zig_fast(w[i], &x[i], &j, &neg);
}

/* 1 when the element's first draw takes the fast path, 0 when it misses. */
int orc_zig_first_draw_fast(uint32_t seed, uint32_t counter)
{
    double x;
    unsigned j;
    int neg;
    zig_init();
    return zig_fast(orc_draw64(seed, counter), &x, &j, &neg);
}

/* One standard normal per counter.  Element c takes the 64-bit draw at c; a
 * miss continues on the N64 substream of its own counter: the base layer's
 * miss samples the tail (Marsaglia 1964: a = -log(U1)/r, b = -log(U2), accept
 * when 2b >= a^2, value r + a, U in (0, 1]); another layer's miss takes the
 * wedge test y = F[j] + U (F[j+1] - F[j]) < exp(-x^2/2) and otherwise starts
 * over with a fresh 64-bit word.  READING: this order of substream words. */
double orc_normal_f64(uint32_t seed, uint32_t counter)
{
    zig_init();
    uint64_t w = orc_draw64(seed, counter);
    uint32_t key = substream_key(seed, PURPOSE_NORMAL64, counter);
    uint32_t k = 0;
    for (;;) {
        double x;
        unsigned j;
        int neg;
        if (zig_fast(w, &x, &j, &neg)) return neg ? -x : x;
        if (j == 0) {
            double r = zig_X[1];
            for (;;) {
                double u1 = (double)((substream64(key, k) >> 11) + 1) * 0x1p-53;
                double u2 = (double)((substream64(key, k + 1u) >> 11) + 1) * 0x1p-53;
                k += 2u;
                double a = -orc_zlog(u1) / r;
                double b = -orc_zlog(u2);
                if (b + b >= a * a) {
                    double z = r + a;
                    return neg ? -z : z;
                }
            }
        }
        double u = (double)(substream64(key, k) >> 11) * 0x1p-53;
        k += 1u;
        double y = zig_F[j] + u * (zig_F[j + 1] - zig_F[j]);
        double t = x * x;
        t = t * -0.5;
        if (y < orc_zexp(t)) return neg ? -x : x;
        w = substream64(key, k);
        k += 1u;
    }
}

/* ------------------------------------------------------------------------ */
/* Fills.  Element i of a fill takes the counter first + i mod 2^32; with a  */
/* non-NULL idx, output slot i holds element idx[i] of the fill instead      */
/* (sampled checks of large fills).                                          */
/* ------------------------------------------------------------------------ */

static uint32_t counter_of(uint32_t first, const uint64_t *idx, size_t i)
{
    return first + (uint32_t)(idx ? idx[i] : (uint64_t)i);
}

void orc_fill_u32(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, uint32_t *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_draw32(seed, counter_of(first, idx, i));
}

void orc_fill_u64(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, uint64_t *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_draw64(seed, counter_of(first, idx, i));
}

void orc_fill_f32(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, float *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_uniform_f32(seed, counter_of(first, idx, i));
}

void orc_fill_f64(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, double *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_uniform_f64(seed, counter_of(first, idx, i));
}

void orc_fill_u8(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, uint8_t *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_u8(seed, counter_of(first, idx, i));
}

void orc_fill_u16(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, uint16_t *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_u16(seed, counter_of(first, idx, i));
}

void orc_fill_bool(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, uint8_t *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_bool(seed, counter_of(first, idx, i));
}

void orc_fill_f16_bits(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, uint16_t *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_f16_bits(seed, counter_of(first, idx, i));
}

void orc_fill_u32_below(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, uint32_t b,
                        uint32_t *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_below32(seed, counter_of(first, idx, i), b);
}

void orc_fill_u64_below(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, uint64_t b,
                        uint64_t *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_below64(seed, counter_of(first, idx, i), b);
}

void orc_fill_i32_range(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, int32_t low,
                        uint32_t b, int32_t *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_range_i32(seed, counter_of(first, idx, i), low, b);
}

void orc_fill_i64_range32(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, int64_t low,
                          uint32_t b, int64_t *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_range_i64_32(seed, counter_of(first, idx, i), low, b);
}

void orc_fill_i64_range(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, int64_t low,
                        uint64_t b, int64_t *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_range_i64(seed, counter_of(first, idx, i), low, b);
}

void orc_fill_randn(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, double *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_randn(seed, counter_of(first, idx, i));
}

void orc_fill_randn_paired(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, double *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_randn_paired(seed, counter_of(first, idx, i));
}

void orc_fill_exponential_f32(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, double *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_exponential_f32(seed, counter_of(first, idx, i));
}

void orc_fill_exponential_f32_own(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, float *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_exponential_f32_own(seed, counter_of(first, idx, i));
}

void orc_fill_randn_precise(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, float *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_randn_precise(seed, counter_of(first, idx, i));
}

void orc_cos2pi_fill(const uint32_t *m, size_t n, float *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_cos2pi_grid(m[i]);
}

void orc_neglog_fill(const uint32_t *m, size_t n, float *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_neglog_f32(m[i]);
}

void orc_neglog64_fill(const uint64_t *m, size_t n, double *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_neglog64(m[i]);
}

void orc_fill_exponential_f64(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, double *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_exponential_f64(seed, counter_of(first, idx, i));
}

void orc_fill_normal_f64(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, double *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_normal_f64(seed, counter_of(first, idx, i));
}

/* x[i] is the input of output slot i (element idx[i] when idx is given). */
void orc_dropout_fill(const float *x, float p, uint32_t seed, uint32_t first, size_t n,
                      const uint64_t *idx, float *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_dropout(x[i], p, seed, counter_of(first, idx, i));
}

/* out[i] = 1 when the first draw of element i takes the ziggurat's fast path. */
void orc_fill_zig_fast(uint32_t seed, uint32_t first, size_t n, const uint64_t *idx, uint8_t *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = (uint8_t)orc_zig_first_draw_fast(seed, counter_of(first, idx, i));
}

void orc_zexp_fill(const double *t, size_t n, double *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_zexp(t[i]);
}

void orc_zlog_fill(const double *x, size_t n, double *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_zlog(x[i]);
}
