// rng_device.cuh -- device-side lowbias32 draws, for fusing random numbers
// into user kernels (a dropout in a GEMM epilogue, noise in an attention
// kernel) with no stored mask and no extra pass over memory.
//
// Every value is a pure function of (seed, counter), the same function the
// C ABI's fills compute (include/rng.h):
//   hash32 = lowbias32 (Phobos stdlib "Random numbers", section hash32);
//   draw32(k, c) = hash32(c ^ hash32(seed))             (section uniform);
//   uniform      = (draw32 & 0x7FFFFF) * 2^-23         (section uniform);
//   randn        = sqrt(-2 ln(1 - u(2c))) cos(2 pi u(2c + 1))  (section randn);
//   dropout      = uniform >= p ? x / (1 - p) : 0       (section dropout);
//   exponential  = -ln(1 - uniform), the own f32 logarithm neg_log_grid
//                  (tandem-sycl "Design", section Exponentials).
// A kernel that gives element e the counter first + e draws exactly what
// the corresponding fill writes: dropout() is bit-identical to
// rng_dropout_fwd, uniform() to rng_fill_f32, draw32() to rng_fill_u32;
// randn() is the value rng_fill_normal_f32 writes, randn_precise() the value
// rng_fill_normal_f32_precise writes.  The page's advice holds:
// use each element's flat index as its counter, and give different uses of
// one seed disjoint counters (randn reads the uniforms at 2c and 2c + 1).
//
// Keys are made once on the host (make_key, make_dropout) and passed to the
// kernel by value.  The header needs only <stdint.h>, nvcc and the generated
// table beside it (lowbias32_neglog_table.inc).  It also holds the page's
// dropout_rows tile kernel with its R autotuner.
#pragma once

#include <stdint.h>

namespace lowbias32 {

// ---- the hash -----------------------------------------------------------

// hash32 after its first xorshift: two multiply-xorshift rounds.
__host__ __device__ __forceinline__ uint32_t hash32_rounds(uint32_t x)
{
    x *= 0x7FEB352Du;  // 2146121005
    x ^= x >> 15;
    x *= 0x846CA68Bu;  // -2073254261 as a bit pattern
    x ^= x >> 16;
    return x;
}

// lowbias32: logical xorshifts by 16, 15, 16 around two wrapping multiplies.
__host__ __device__ __forceinline__ uint32_t hash32(uint32_t x) { return hash32_rounds(x ^ (x >> 16)); }

// A seed's key: hash32(seed) folded into hash32's first xorshift,
// (c ^ k) ^ ((c ^ k) >> 16) = c ^ (c >> 16) ^ (k ^ (k >> 16)).
struct Key {
    uint32_t folded;
};

__host__ __device__ __forceinline__ Key key_of_hash(uint32_t k) { return Key{k ^ (k >> 16)}; }
__host__ __device__ __forceinline__ Key make_key(uint32_t seed) { return key_of_hash(hash32(seed)); }

// ---- draws ----------------------------------------------------------------

// hash32(c ^ hash32(seed))
__host__ __device__ __forceinline__ uint32_t draw32(Key k, uint32_t c)
{
    return hash32_rounds(c ^ (c >> 16) ^ k.folded);
}

// The two words of the 64-bit draw at c: the draws at 2c (hi) and 2c + 1
// (lo), counters mod 2^32.  2c + 1 = 2c ^ 1 and bit 0 never reaches the
// shifted term, so the low word's first xorshift is the high word's ^ 1.
struct Words {
    uint32_t hi, lo;
};

__host__ __device__ __forceinline__ Words draw64_words(Key k, uint32_t c)
{
    const uint32_t a = c << 1;
    const uint32_t first = a ^ (a >> 16) ^ k.folded;
    return Words{hash32_rounds(first), hash32_rounds(first ^ 1u)};
}

__host__ __device__ __forceinline__ uint64_t draw64(Key k, uint32_t c)
{
    const Words w = draw64_words(k, c);
    return (static_cast<uint64_t>(w.hi) << 32) | w.lo;
}

// ---- uniforms ---------------------------------------------------------------

// (draw32 & 0x7FFFFF) * 2^-23, exactly: 0x3F800000 | m is 1 + m 2^-23 and
// subtracting 1 is exact.
__device__ __forceinline__ float uniform_of(uint32_t d)
{
    return __uint_as_float(0x3F800000u | (d & 0x7FFFFFu)) - 1.0f;
}

__device__ __forceinline__ float uniform(Key k, uint32_t c) { return uniform_of(draw32(k, c)); }

// ---- randn (Box-Muller, cosine branch) --------------------------------------

namespace detail {
__device__ __forceinline__ float lg2_approx(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float sqrt_approx(float x)
{
    float y;
    asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float cos_approx(float x)
{
    float y;
    asm("cos.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float sin_approx(float x)
{
    float y;
    asm("sin.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The last xorshift of hash32 fused with the uniform's mask: for y, hash32
// before its last xorshift (draw d = y ^ (y >> 16)), the bit pattern of
// 1 + (d & 0x7FFFFF) 2^-23.  Bits 0..22 of d are those of y ^ (y >> 16)
// (y >> 16 has no bits above 15), and the funnel shift places 0x3F80, the
// exponent of 1.0f, above y >> 16: one shift and one three-input logic op.
__device__ __forceinline__ uint32_t one_plus_uniform_bits(uint32_t y)
{
    return (y & 0x7FFFFFu) ^ __funnelshift_r(y, 0x3F80u, 16);
}

// hash32 from its first multiply's product p up to its last xorshift.
__device__ __forceinline__ uint32_t hash32_middle(uint32_t p)
{
    p ^= p >> 15;
    return p * 0x846CA68Bu;
}

constexpr float kTwoPi = 6.28318530717958647692f;
constexpr float kMinusTwoLn2 = -1.38629436f;

// -2 ln(1 - u0) from b0, the bit pattern of 1 + u0, given large = -2 ln 2
// log2(1 - u0) by the hardware log2 (1 - u0 = 2 - (1 + u0), exact).  For
// u0 >= 2^-7 (a grid index with a bit in 16..22) that is the value: the
// log2's absolute error, below 2^-22 on [1/2, 1], moves a radius of at least
// 0.125 by at most 1.4e-6.  Below, where a log2 near 1 has too little relative
// accuracy, (1 + u0)^2 - 1 = 2 u0 + u0^2 in one fma, the series of
// -2 ln(1 - u0) to second order: relative error below u0^2/3 + 2^-24, a
// radius error below 1.3e-6.  The fma is predicated on the test, so neither
// a select nor the second candidate costs an instruction where it is not
// taken.
__device__ __forceinline__ float radius_squared(uint32_t b0, float large)
{
    float s = large;
    asm("{\n\t.reg .pred p;\n\t.reg .b32 t;\n\t"
        "and.b32 t, %2, 0x7F0000;\n\t"
        "setp.eq.u32 p, t, 0;\n\t"
        "@p fma.rn.f32 %0, %1, %1, 0fBF800000;\n\t}"
        : "+f"(s)
        : "f"(__uint_as_float(b0)), "r"(b0));
    return s;
}

// The Box-Muller radius sqrt(-2 ln(1 - u0)) from b0, the bit pattern of 1 + u0.
__device__ __forceinline__ float box_muller_radius(uint32_t b0)
{
    const float large = __fmul_rn(lg2_approx(__fsub_rn(2.0f, __uint_as_float(b0))), kMinusTwoLn2);
    return sqrt_approx(radius_squared(b0, large));
}

// The angle 2 pi u1 in [0, 2 pi) from b1, the bit pattern of 1 + u1, as
// (1 + u1) 2 pi - 2 pi in one fused multiply-add (one rounding).  On this
// grid the hardware cosine and sine are within 2^-20.8 of the exact values
// over the whole turn, no worse than on [-pi, pi), so the angle needs no
// half-turn shift and the product no negation.
__device__ __forceinline__ float box_muller_angle(uint32_t b1)
{
    return __fmaf_rn(__uint_as_float(b1), kTwoPi, -kTwoPi);
}

// randn from the bit patterns of 1 + u0 and 1 + u1.
__device__ __forceinline__ float box_muller_bits(uint32_t b0, uint32_t b1)
{
    return __fmul_rn(box_muller_radius(b0), cos_approx(box_muller_angle(b1)));
}

#if defined(__CUDA_ARCH__) && __CUDA_ARCH__ >= 1000
// Two binary32 lanes in one 64-bit register; add, sub, mul and fma on .f32x2
// (sm_100 and later) round each lane like the scalar instruction, so the
// paired evaluation below returns box_muller_bits' values bit for bit.  A
// paired multiply whose result feeds a paired add may be contracted into one
// fma, unlike a scalar __fmul_rn: paired code here keeps such products scalar.
__device__ __forceinline__ unsigned long long f32x2_pack(float lo, float hi)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 f32x2_unpack(unsigned long long v)
{
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ unsigned long long f32x2_sub(unsigned long long a, unsigned long long b)
{
    unsigned long long d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long f32x2_add(unsigned long long a, unsigned long long b)
{
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long f32x2_mul(unsigned long long a, unsigned long long b)
{
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long f32x2_fma(unsigned long long a, unsigned long long b,
                                                        unsigned long long c)
{
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
#endif

// box_muller_bits for two elements (a and b), the steps other than the
// hardware log2, square root and cosine paired in f32x2 lanes where the
// target has them.
__device__ __forceinline__ float2 box_muller_bits_x2(uint32_t b0a, uint32_t b1a, uint32_t b0b, uint32_t b1b)
{
#if defined(__CUDA_ARCH__) && __CUDA_ARCH__ >= 1000
    const unsigned long long f0 = f32x2_pack(__uint_as_float(b0a), __uint_as_float(b0b));
    const float2 v = f32x2_unpack(f32x2_sub(f32x2_pack(2.0f, 2.0f), f0));
    const float2 large = f32x2_unpack(f32x2_mul(f32x2_pack(lg2_approx(v.x), lg2_approx(v.y)),
                                                f32x2_pack(kMinusTwoLn2, kMinusTwoLn2)));
    const float ra = sqrt_approx(radius_squared(b0a, large.x));
    const float rb = sqrt_approx(radius_squared(b0b, large.y));
    const float2 angle = f32x2_unpack(f32x2_fma(f32x2_pack(__uint_as_float(b1a), __uint_as_float(b1b)),
                                                f32x2_pack(kTwoPi, kTwoPi), f32x2_pack(-kTwoPi, -kTwoPi)));
    return f32x2_unpack(f32x2_mul(f32x2_pack(ra, rb), f32x2_pack(cos_approx(angle.x), cos_approx(angle.y))));
#else
    return make_float2(box_muller_bits(b0a, b1a), box_muller_bits(b0b, b1b));
#endif
}
}  // namespace detail

// The Box-Muller value of the 32-bit draws d0 (at 2c) and d1 (at 2c + 1):
// what randn gives for a counter whose draws these are.
__device__ __forceinline__ float randn_of_draws(uint32_t d0, uint32_t d1)
{
    return detail::box_muller_bits(0x3F800000u | (d0 & 0x7FFFFFu), 0x3F800000u | (d1 & 0x7FFFFFu));
}

// randn(seed, c) in f32, within 4e-6 (1 + |z|) of the exact value.  The
// draw at 2c + 1 starts from the draw at 2c's first xorshift ^ 1.
__device__ __forceinline__ float randn(Key k, uint32_t c)
{
    const uint32_t a = c << 1;
    const uint32_t x = a ^ (a >> 16) ^ k.folded;
    return detail::box_muller_bits(detail::one_plus_uniform_bits(detail::hash32_middle(x * 0x7FEB352Du)),
                                   detail::one_plus_uniform_bits(detail::hash32_middle((x ^ 1u) * 0x7FEB352Du)));
}

// Both Box-Muller branches of the draws d0 and d1: x = r cos(2 pi u1), the
// value randn_of_draws gives, and y = r sin(2 pi u1).
__device__ __forceinline__ float2 randn_pair_of_draws(uint32_t d0, uint32_t d1)
{
    const float r = detail::box_muller_radius(0x3F800000u | (d0 & 0x7FFFFFu));
    const float a = detail::box_muller_angle(0x3F800000u | (d1 & 0x7FFFFFu));
    return make_float2(__fmul_rn(r, detail::cos_approx(a)), __fmul_rn(r, detail::sin_approx(a)));
}

// Both Box-Muller branches of pair q (the uniforms at 2q and 2q + 1):
// x = r cos(2 pi u1), y = r sin(2 pi u1); x equals randn(k, q).  One
// 64-bit draw per two values.
__device__ __forceinline__ float2 randn_pair(Key k, uint32_t q)
{
    const Words w = draw64_words(k, q);
    return randn_pair_of_draws(w.hi, w.lo);
}

// The element with counter c of the paired normal fill: the cosine branch of
// pair c >> 1 for even c, its sine branch for odd c.
__device__ __forceinline__ float randn_paired(Key k, uint32_t c)
{
    const float2 v = randn_pair(k, c >> 1);
    return (c & 1u) ? v.y : v.x;
}

// ---- exponential ----------------------------------------------------------------

namespace detail {
#include "lowbias32_neglog_table.inc"
}  // namespace detail

// -ln(1 - m 2^-23) for a 23-bit m, in binary32 arithmetic: the library's own
// logarithm (tandem-sycl "Design", Exponentials: an own f32 logarithm, every
// draw within 0.571 ulp).  1 - m 2^-23 = V 2^-23 with the integer V = 2^23 - m;
// V = 2^k M, M in [1, 2), E = 23 - k; the bin j = round((M - 1) 256) gives
// inv_j (8 bits) and ln inv_j = hi_j + lo_j from a 4 KiB table, so
//   -ln(1 - u) = (E ln 2 + ln inv_j) - log1p(r),  r = M inv_j - 1 (exact),
// with E ln2_hi + hi_j exact, hi - r summed exactly (Fast2Sum), the error
// and the lo parts added, the Taylor tail r^2/2 - r^3/3 + r^4/4 - r^5/5 added
// to them in one fma, and one rounding at the end.  Within 0.5035 ulp of the exact value on all
// 2^23 inputs (correctly rounded on all but 82); m = 0 gives +0.  Every step
// is an explicit IEEE operation, so the result is the same bits on any
// IEEE machine that performs the same sequence.
namespace detail {
// The integer x in [0, 2^23] as binary32, exactly: 2^23 + x has x in its
// significand (x = 2^23 carries into the exponent: 2^24), and subtracting
// 2^23 is exact.  An ALU and an FMA-pipe operation instead of a conversion.
__device__ __forceinline__ float small_uint_to_float(uint32_t x)
{
    return __fsub_rn(__uint_as_float(0x4B000000u | x), 8388608.0f);
}
}  // namespace detail

// neg_log_grid with the table row j = round((M - 1) 256) fetched by load(j)
// (a copy of detail::kNegLogTable elsewhere, e.g. in shared memory): the same
// operations, so the same bits.
template <class Load>
__device__ __forceinline__ float neg_log_grid_by(uint32_t m, Load load)
{
    const uint32_t bits = __float_as_uint(detail::small_uint_to_float(0x800000u - m));  // V, exact
    const uint32_t mant = bits & 0x7FFFFFu;
    const float M = __uint_as_float(mant | 0x3F800000u);
    const float4 t = load((mant + 16384u) >> 15);  // {inv_j, hi_j, lo_j, 0}
    const float E = detail::small_uint_to_float(150u - (bits >> 23));      // 23 - k
    const float r = __fmaf_rn(M, t.x, -1.0f);
    const float t_hi = __fmaf_rn(E, detail::kNegLogLn2Hi, t.y);
    const float t_lo = __fmaf_rn(E, detail::kNegLogLn2Lo, t.z);
    // s = t_hi - r and its exact error -(r + bb) by Fast2Sum: |t_hi| >= |r|
    // or t_hi = 0 on every input (|t_hi| >= 0.0077 where nonzero, |r| <=
    // 0.0049), so the error equals TwoSum's; err + t_lo is formed as
    // t_lo - (r + bb), the same value
    const float s = __fsub_rn(t_hi, r);
    const float bb = __fsub_rn(s, t_hi);
    const float err_lo = __fsub_rn(t_lo, __fadd_rn(r, bb));
    float p = __fmaf_rn(r, -0x1.99999ap-3f, 0.25f);  // 1/4 - r/5
    p = __fmaf_rn(r, p, -0x1.555556p-2f);           // -1/3 + r/4 - r^2/5
    p = __fmaf_rn(r, p, 0.5f);                      // 1/2 - r/3 + r^2/4 - r^3/5
    return __fadd_rn(s, __fmaf_rn(__fmul_rn(r, r), p, err_lo));  // the tail r^2 p added in one rounding
}

__device__ __forceinline__ float neg_log_grid(uint32_t m)
{
    return neg_log_grid_by(m, [](uint32_t j) { return __ldg(&detail::kNegLogTable[j]); });
}

// -ln(1 - u) for u = uniform(k, c), by neg_log_grid; in [0, 23 ln 2].
__device__ __forceinline__ float exponential(Key k, uint32_t c) { return neg_log_grid(draw32(k, c) & 0x7FFFFFu); }

namespace detail {
// neg_log_grid of two inputs, its float steps paired in f32x2 lanes where the
// target has them (each lane rounded like the scalar step, so the values are
// neg_log_grid's bit for bit).
// neg_log_grid_x2 with the table rows fetched by load(j), as neg_log_grid_by.
template <class Load>
__device__ __forceinline__ float2 neg_log_grid_x2_by(uint32_t ma, uint32_t mb, Load load)
{
#if defined(__CUDA_ARCH__) && __CUDA_ARCH__ >= 1000
    const float2 V = f32x2_unpack(f32x2_sub(f32x2_pack(__uint_as_float(0x4B000000u | (0x800000u - ma)),
                                                       __uint_as_float(0x4B000000u | (0x800000u - mb))),
                                            f32x2_pack(8388608.0f, 8388608.0f)));
    const uint32_t bits_a = __float_as_uint(V.x), bits_b = __float_as_uint(V.y);
    const uint32_t mant_a = bits_a & 0x7FFFFFu, mant_b = bits_b & 0x7FFFFFu;
    const float4 ta = load((mant_a + 16384u) >> 15);
    const float4 tb = load((mant_b + 16384u) >> 15);
    const unsigned long long M = f32x2_pack(__uint_as_float(mant_a | 0x3F800000u), __uint_as_float(mant_b | 0x3F800000u));
    const unsigned long long E = f32x2_sub(f32x2_pack(__uint_as_float(0x4B000000u | (150u - (bits_a >> 23))),
                                                      __uint_as_float(0x4B000000u | (150u - (bits_b >> 23)))),
                                           f32x2_pack(8388608.0f, 8388608.0f));
    const unsigned long long r = f32x2_fma(M, f32x2_pack(ta.x, tb.x), f32x2_pack(-1.0f, -1.0f));
    const unsigned long long t_hi = f32x2_fma(E, f32x2_pack(kNegLogLn2Hi, kNegLogLn2Hi), f32x2_pack(ta.y, tb.y));
    const unsigned long long t_lo = f32x2_fma(E, f32x2_pack(kNegLogLn2Lo, kNegLogLn2Lo), f32x2_pack(ta.z, tb.z));
    const unsigned long long s = f32x2_sub(t_hi, r);
    const unsigned long long bb = f32x2_sub(s, t_hi);
    const unsigned long long err_lo = f32x2_sub(t_lo, f32x2_add(r, bb));  // Fast2Sum, as neg_log_grid_by
    unsigned long long p = f32x2_fma(r, f32x2_pack(-0x1.99999ap-3f, -0x1.99999ap-3f), f32x2_pack(0.25f, 0.25f));
    p = f32x2_fma(r, p, f32x2_pack(-0x1.555556p-2f, -0x1.555556p-2f));
    p = f32x2_fma(r, p, f32x2_pack(0.5f, 0.5f));
    return f32x2_unpack(f32x2_add(s, f32x2_fma(f32x2_mul(r, r), p, err_lo)));
#else
    return make_float2(neg_log_grid_by(ma, load), neg_log_grid_by(mb, load));
#endif
}

__device__ __forceinline__ float2 neg_log_grid_x2(uint32_t ma, uint32_t mb)
{
    return neg_log_grid_x2_by(ma, mb, [](uint32_t j) { return __ldg(&kNegLogTable[j]); });
}
}  // namespace detail

// ---- precise normal --------------------------------------------------------------

namespace detail {
#include "lowbias32_cos2pi.inc"
}  // namespace detail

// cos(2 pi m 2^-23) for a 23-bit m in binary32, the library's own: the
// quadrant q = m >> 21 and g = (m mod 2^21) 2^-23 in [0, 1/4) are exact, and
// cos(2 pi (q/4 + g)) is cos g, -sin g, -cos g or sin g (angles in turns);
// above g = 1/8 the complement 1/4 - g (exact) swaps sin and cos.  On x <= 1/8
// the Taylor series of sin(2 pi x) to x^9 and cos(2 pi x) to x^10 with
// binary32 coefficients, the leading ones hi + lo.  Within 0.90 ulp of the
// exact cosine on all 2^23 inputs; exact at the quarter turns.
__device__ __forceinline__ float cos2pi_grid(uint32_t m)
{
    const uint32_t q = m >> 21;
    const uint32_t f = m & 0x1FFFFFu;
    const bool swap = f > 0x100000u;
    const float x = __fmul_rn(detail::small_uint_to_float(swap ? 0x200000u - f : f), 0x1p-23f);  // exact
    const float x2 = __fmul_rn(x, x);
    float p = __fmaf_rn(x2, detail::kCos2PiS9, detail::kCos2PiS7);
    p = __fmaf_rn(x2, p, detail::kCos2PiS5);
    p = __fmaf_rn(x2, p, detail::kCos2PiS3);
    p = __fmaf_rn(x2, p, detail::kCos2PiS1Lo);
    const float sin_x = __fmaf_rn(x, detail::kCos2PiS1Hi, __fmul_rn(x, p));
    float c = __fmaf_rn(x2, detail::kCos2PiC10, detail::kCos2PiC8);
    c = __fmaf_rn(x2, c, detail::kCos2PiC6);
    c = __fmaf_rn(x2, c, detail::kCos2PiC4);
    const float t = __fmul_rn(x2, __fmaf_rn(x2, c, detail::kCos2PiC2Lo));
    const float cos_x = __fadd_rn(1.0f, __fmaf_rn(x2, detail::kCos2PiC2Hi, t));
    const float v = ((q & 1u) != 0u) != swap ? sin_x : cos_x;
    return (q == 1u || q == 2u) ? -v : v;
}

namespace detail {
// cos2pi_grid of two inputs, its float steps paired in f32x2 lanes where the
// target has them (the values are cos2pi_grid's bit for bit).
__device__ __forceinline__ float2 cos2pi_grid_x2(uint32_t ma, uint32_t mb)
{
#if defined(__CUDA_ARCH__) && __CUDA_ARCH__ >= 1000
    const uint32_t qa = ma >> 21, qb = mb >> 21;
    const uint32_t fa = ma & 0x1FFFFFu, fb = mb & 0x1FFFFFu;
    const bool swap_a = fa > 0x100000u, swap_b = fb > 0x100000u;
    const unsigned long long g = f32x2_sub(
        f32x2_pack(__uint_as_float(0x4B000000u | (swap_a ? 0x200000u - fa : fa)),
                   __uint_as_float(0x4B000000u | (swap_b ? 0x200000u - fb : fb))),
        f32x2_pack(8388608.0f, 8388608.0f));
    const unsigned long long x = f32x2_mul(g, f32x2_pack(0x1p-23f, 0x1p-23f));
    const unsigned long long x2 = f32x2_mul(x, x);
    unsigned long long p = f32x2_fma(x2, f32x2_pack(kCos2PiS9, kCos2PiS9), f32x2_pack(kCos2PiS7, kCos2PiS7));
    p = f32x2_fma(x2, p, f32x2_pack(kCos2PiS5, kCos2PiS5));
    p = f32x2_fma(x2, p, f32x2_pack(kCos2PiS3, kCos2PiS3));
    p = f32x2_fma(x2, p, f32x2_pack(kCos2PiS1Lo, kCos2PiS1Lo));
    const float2 sin_x = f32x2_unpack(f32x2_fma(x, f32x2_pack(kCos2PiS1Hi, kCos2PiS1Hi), f32x2_mul(x, p)));
    unsigned long long c = f32x2_fma(x2, f32x2_pack(kCos2PiC10, kCos2PiC10), f32x2_pack(kCos2PiC8, kCos2PiC8));
    c = f32x2_fma(x2, c, f32x2_pack(kCos2PiC6, kCos2PiC6));
    c = f32x2_fma(x2, c, f32x2_pack(kCos2PiC4, kCos2PiC4));
    const unsigned long long t = f32x2_mul(x2, f32x2_fma(x2, c, f32x2_pack(kCos2PiC2Lo, kCos2PiC2Lo)));
    const float2 cos_x = f32x2_unpack(f32x2_add(f32x2_pack(1.0f, 1.0f),
                                                f32x2_fma(x2, f32x2_pack(kCos2PiC2Hi, kCos2PiC2Hi), t)));
    const float va = ((qa & 1u) != 0u) != swap_a ? sin_x.x : cos_x.x;
    const float vb = ((qb & 1u) != 0u) != swap_b ? sin_x.y : cos_x.y;
    return make_float2((qa == 1u || qa == 2u) ? -va : va, (qb == 1u || qb == 2u) ? -vb : vb);
#else
    return make_float2(cos2pi_grid(ma), cos2pi_grid(mb));
#endif
}
}  // namespace detail

// randn's definition (the uniforms at 2c and 2c + 1, cosine branch) evaluated
// in binary32 to a few ulp: sqrt(2 neg_log_grid(u0)) cos2pi_grid(u1) with an
// IEEE square root; within 2.5 ulp of the exact value (tandem-sycl "Design",
// Normals: a precise f32 Box-Muller beside the default float normal).  Not
// the value randn() gives, which is held to 4e-6 (1 + |z|).
__device__ __forceinline__ float randn_precise(Key k, uint32_t c)
{
    const Words w = draw64_words(k, c);  // the draws at 2c and 2c + 1
    const float e = neg_log_grid(w.hi & 0x7FFFFFu);
    return __fmul_rn(__fsqrt_rn(__fadd_rn(e, e)), cos2pi_grid(w.lo & 0x7FFFFFu));
}

namespace detail {
// randn_precise of the draw pairs (a0, a1) and (b0, b1), the float steps
// paired in f32x2 lanes where the target has them (same values).
__device__ __forceinline__ float2 randn_precise_x2(uint32_t a0, uint32_t a1, uint32_t b0, uint32_t b1)
{
#if defined(__CUDA_ARCH__) && __CUDA_ARCH__ >= 1000
    const float2 e = neg_log_grid_x2(a0 & 0x7FFFFFu, b0 & 0x7FFFFFu);
    const float2 c = cos2pi_grid_x2(a1 & 0x7FFFFFu, b1 & 0x7FFFFFu);
    const float2 twice = f32x2_unpack(f32x2_add(f32x2_pack(e.x, e.y), f32x2_pack(e.x, e.y)));
    return f32x2_unpack(f32x2_mul(f32x2_pack(__fsqrt_rn(twice.x), __fsqrt_rn(twice.y)), f32x2_pack(c.x, c.y)));
#else
    const float ea = neg_log_grid(a0 & 0x7FFFFFu), eb = neg_log_grid(b0 & 0x7FFFFFu);
    return make_float2(__fmul_rn(__fsqrt_rn(__fadd_rn(ea, ea)), cos2pi_grid(a1 & 0x7FFFFFu)),
                       __fmul_rn(__fsqrt_rn(__fadd_rn(eb, eb)), cos2pi_grid(b1 & 0x7FFFFFu)));
#endif
}
}  // namespace detail

// ---- dropout ------------------------------------------------------------------

// Parameters of one dropout (seed, p): keep iff (draw32 & 0x7FFFFF) >=
// threshold = ceil(p 2^23) (uniform >= p, exactly), kept values x / divisor
// with divisor = 1 - p rounded to f32.
struct Dropout {
    Key key;
    uint32_t threshold;
    float divisor;
};

// Host side: p must lie in [0, 1).
inline Dropout make_dropout(uint32_t seed, float p)
{
    const double scaled = static_cast<double>(p) * 8388608.0;  // exact
    uint32_t t = static_cast<uint32_t>(scaled);
    if (static_cast<double>(t) < scaled) ++t;  // ceil
    return Dropout{make_key(seed), t, 1.0f - p};
}

__device__ __forceinline__ bool dropout_keep(const Dropout &d, uint32_t c)
{
    return (draw32(d.key, c) & 0x7FFFFFu) >= d.threshold;
}

// The element with counter c of dropout(x, p, seed, c): IEEE x / (1 - p) or +0.
__device__ __forceinline__ float dropout(const Dropout &d, float x, uint32_t c)
{
    return dropout_keep(d, c) ? __fdiv_rn(x, d.divisor) : 0.0f;
}

// ---- the dropout_rows tile kernel ---------------------------------------------

// Phobos "Random numbers", the dropout_rows listing: y = dropout(x) on a
// [rows, 256] f32 tensor, a block of 256 threads (one column each) per R
// rows, the counter of element (row, col) its flat index first + row 256 +
// col (mod 2^32), so every R gives exactly what rng_dropout_fwd gives for
// the flattened tensor.  Each thread loads its R elements before computing
// and storing them.  x == y is allowed (each element is read before it is
// written, by the same thread).
constexpr uint32_t kDropoutRowsCols = 256;

template <int R>
__global__ void __launch_bounds__(kDropoutRowsCols)
    dropout_rows_kernel(const float *x, float *y, uint32_t rows, Dropout d, uint32_t first)
{
    const uint32_t row0 = blockIdx.x * static_cast<uint32_t>(R);
    const uint32_t col = threadIdx.x;
    float v[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const size_t e = static_cast<size_t>(row0 + r) * kDropoutRowsCols + col;
        if (row0 + r < rows) v[r] = x[e];
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const size_t e = static_cast<size_t>(row0 + r) * kDropoutRowsCols + col;
        if (row0 + r < rows) y[e] = dropout(d, v[r], first + static_cast<uint32_t>(e));
    }
}

#ifdef __CUDACC__
// The candidate R (rows per block) the autotuner tries; the listing's own
// candidate list is the single value 16.
constexpr int kDropoutRowsCandidates[] = {1, 2, 4, 8, 16, 32};
constexpr int kDropoutRowsNumCandidates = 6;

// Launches dropout_rows_kernel<R> for a candidate R on stream s (rows <
// 2^32 / R); cudaErrorInvalidValue for an R outside the candidates.  (A
// function template only so that a translation unit that does not call it
// instantiates none of the kernels.)
template <class = void>
inline cudaError_t dropout_rows(const float *x, float *y, uint32_t rows, const Dropout &d, uint32_t first, int R,
                                cudaStream_t s = 0)
{
    if (rows == 0) return cudaSuccess;
    const uint32_t blocks = (rows + static_cast<uint32_t>(R) - 1u) / static_cast<uint32_t>(R);
    switch (R) {
    case 1: dropout_rows_kernel<1><<<blocks, kDropoutRowsCols, 0, s>>>(x, y, rows, d, first); break;
    case 2: dropout_rows_kernel<2><<<blocks, kDropoutRowsCols, 0, s>>>(x, y, rows, d, first); break;
    case 4: dropout_rows_kernel<4><<<blocks, kDropoutRowsCols, 0, s>>>(x, y, rows, d, first); break;
    case 8: dropout_rows_kernel<8><<<blocks, kDropoutRowsCols, 0, s>>>(x, y, rows, d, first); break;
    case 16: dropout_rows_kernel<16><<<blocks, kDropoutRowsCols, 0, s>>>(x, y, rows, d, first); break;
    case 32: dropout_rows_kernel<32><<<blocks, kDropoutRowsCols, 0, s>>>(x, y, rows, d, first); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// The listing's @autotune: times every candidate R on the caller's buffers
// (one untimed launch, then `reps` >= 1 launches between CUDA events on s,
// which is synchronised) and returns the R of the least mean time, or 0 on a
// CUDA error (then cudaGetLastError() or the returned launch status says
// which).  y is overwritten, with the same values whatever R.  ms, if not
// null, receives the mean milliseconds of each candidate, in the order of
// kDropoutRowsCandidates.
template <class = void>
inline int dropout_rows_autotune(const float *x, float *y, uint32_t rows, const Dropout &d, uint32_t first,
                                 cudaStream_t s = 0, int reps = 5, float *ms = nullptr)
{
    if (reps < 1) reps = 1;
    cudaEvent_t ev[2];
    if (cudaEventCreate(&ev[0]) != cudaSuccess) return 0;
    if (cudaEventCreate(&ev[1]) != cudaSuccess) {
        cudaEventDestroy(ev[0]);
        return 0;
    }
    int best = 0;
    float best_ms = 0.0f;
    bool ok = true;
    for (int k = 0; ok && k < kDropoutRowsNumCandidates; ++k) {
        const int R = kDropoutRowsCandidates[k];
        ok = dropout_rows(x, y, rows, d, first, R, s) == cudaSuccess && cudaEventRecord(ev[0], s) == cudaSuccess;
        for (int i = 0; ok && i < reps; ++i) ok = dropout_rows(x, y, rows, d, first, R, s) == cudaSuccess;
        float t = 0.0f;
        ok = ok && cudaEventRecord(ev[1], s) == cudaSuccess && cudaEventSynchronize(ev[1]) == cudaSuccess &&
             cudaEventElapsedTime(&t, ev[0], ev[1]) == cudaSuccess;
        t /= static_cast<float>(reps);
        if (ok && ms) ms[k] = t;
        if (ok && (best == 0 || t < best_ms)) {
            best = R;
            best_ms = t;
        }
    }
    cudaEventDestroy(ev[0]);
    cudaEventDestroy(ev[1]);
    return ok ? best : 0;
}
#endif  // __CUDACC__

}  // namespace lowbias32
