// f64_math.cuh -- the library's own binary64 functions, each a fixed
// sequence of exact integer or IEEE operations (+, -, *, /, fma with explicit
// rounding intrinsics), so that a second implementation performing the same
// operations returns the same bits on any IEEE machine: zexp and zlog for the
// ziggurat's slow path, and neglog64, the fixed-point -ln(1 - u) of the f64
// exponential fill.
#pragma once

#include <cstdint>

#include "zig_tables.inc"

namespace rngk {

// exp(t) for t in [-10, 0]: k = rint(t / ln 2) (the rounding done by adding
// and subtracting 1.5 2^52, which rounds to the nearest even integer exactly
// as rint does for |t / ln 2| < 2^51), r = t - k ln 2 by two fma (ln 2 =
// ln2_high + ln2_low, ln2_high with 32 significant bits), degree-13 Taylor
// polynomial in Horner form, exact scaling by 2^k on the exponent field.
__device__ __forceinline__ double zexp(double t)
{
    const double shifted = __dadd_rn(__dmul_rn(t, ZK_INV_LN2), 0x1.8p52);
    const int k = __double2loint(shifted);  // low word of 1.5 2^52 + k is k
    const double kd = __dsub_rn(shifted, 0x1.8p52);
    double r = __fma_rn(-kd, ZK_LN2_HIGH, t);
    r = __fma_rn(-kd, ZK_LN2_LOW, r);
    double p = ZK_INV_FACT_13;
    p = __fma_rn(p, r, ZK_INV_FACT_12);
    p = __fma_rn(p, r, ZK_INV_FACT_11);
    p = __fma_rn(p, r, ZK_INV_FACT_10);
    p = __fma_rn(p, r, ZK_INV_FACT_9);
    p = __fma_rn(p, r, ZK_INV_FACT_8);
    p = __fma_rn(p, r, ZK_INV_FACT_7);
    p = __fma_rn(p, r, ZK_INV_FACT_6);
    p = __fma_rn(p, r, ZK_INV_FACT_5);
    p = __fma_rn(p, r, ZK_INV_FACT_4);
    p = __fma_rn(p, r, ZK_INV_FACT_3);
    p = __fma_rn(p, r, ZK_INV_FACT_2);
    p = __fma_rn(p, r, ZK_INV_FACT_1);
    p = __fma_rn(p, r, ZK_INV_FACT_0);
    const uint64_t scale = static_cast<uint64_t>(static_cast<int64_t>(k)) << 52;  // k in [-15, 0]
    return __longlong_as_double(static_cast<long long>(static_cast<uint64_t>(__double_as_longlong(p)) + scale));
}

// log(x) for positive normal x: x = 2^e m with m in (sqrt(1/2), sqrt 2],
// s = (m - 1)/(m + 1), log m = 2 (s + s^3/3 + ... + s^23/23), then
// e ln2_high + (e ln2_low + log m).
__device__ __forceinline__ double zlog(double x)
{
    const uint64_t bits = static_cast<uint64_t>(__double_as_longlong(x));
    int e = static_cast<int>(bits >> 52) - 1023;
    double m = __longlong_as_double(static_cast<long long>((bits & 0x000FFFFFFFFFFFFFull) | 0x3FF0000000000000ull));
    if (m > ZK_SQRT2) {
        m = __dmul_rn(m, 0.5);
        e += 1;
    }
    const double s = __ddiv_rn(__dsub_rn(m, 1.0), __dadd_rn(m, 1.0));
    const double s2 = __dmul_rn(s, s);
    double p = ZK_INV_ODD_23;
    p = __fma_rn(p, s2, ZK_INV_ODD_21);
    p = __fma_rn(p, s2, ZK_INV_ODD_19);
    p = __fma_rn(p, s2, ZK_INV_ODD_17);
    p = __fma_rn(p, s2, ZK_INV_ODD_15);
    p = __fma_rn(p, s2, ZK_INV_ODD_13);
    p = __fma_rn(p, s2, ZK_INV_ODD_11);
    p = __fma_rn(p, s2, ZK_INV_ODD_9);
    p = __fma_rn(p, s2, ZK_INV_ODD_7);
    p = __fma_rn(p, s2, ZK_INV_ODD_5);
    p = __fma_rn(p, s2, ZK_INV_ODD_3);
    const double two_s = __dadd_rn(s, s);
    const double log_m = __fma_rn(__dmul_rn(two_s, s2), p, two_s);
    const double de = static_cast<double>(e);
    return __fma_rn(de, ZK_LN2_HIGH, __fma_rn(de, ZK_LN2_LOW, log_m));
}

// ---- the f64 exponential's fixed-point logarithm ----------------------------

#include "neglog64_table.inc"

// y 2^-scale for an integer 2^64 <= y < 2^128 (on both paths of neglog64 y is
// at least 2^84), rounded to the nearest binary64, ties to even.  y is shifted
// left until its leading one is bit 127 (z places); the high word H then holds
// the significand (bits 63 .. 11), the rounding bit (bit 10) and the top of
// the sticky bits, and whether any bit of the low word is set is folded into
// bit 0 of H, below the rounding bit, which keeps both the rounding and the
// tie decision.  One round-to-nearest conversion of that 64-bit integer (IEEE,
// on the otherwise idle FP64 pipe) rounds it to 53 bits; the exact power of
// two 2^(64 - z - scale) is then added to the exponent field.  The same result
// as rounding y 2^-scale directly; the conversion replaced seven ALU
// instructions of an integer rounding.  The small-u branch of neglog64 uses it
// (y up to 2^126); the main path, whose y is below 2^110, needs no shift.
__device__ __forceinline__ double fixed_to_double(unsigned __int128 y, int scale)
{
    const unsigned long long hi = static_cast<unsigned long long>(y >> 64);
    const unsigned long long lo = static_cast<unsigned long long>(y);
    const int z = __clzll(static_cast<long long>(hi));                // 0 .. 63: hi != 0
    const unsigned long long H = (hi << z) | ((lo >> 1) >> (63 - z));  // (hi:lo) << z, high word
    const unsigned long long L = lo << z;
    const double d = __ull2double_rn(H | static_cast<unsigned long long>(L != 0ull));  // in [2^63, 2^64]
    const long long adj = static_cast<long long>(64 - z - scale);
    return __longlong_as_double(static_cast<long long>(static_cast<unsigned long long>(__double_as_longlong(d)) +
                                                       (static_cast<unsigned long long>(adj) << 52)));
}

// a S_1 of log1p's series at scale 2^137 for a at scale 2^74: S = sum of
// (-a)^(k-1)/k to k = 6 by Horner, or with every term added (kAdd, the series
// of -ln(1 - u) in u), each product floored: S_5, S_4 in 32 bits at 2^33 from a
// at 2^42, S_3 at 2^64 from their 32 x 32 product, S_2 at 2^64 and S_1 at 2^63
// from a itself; a S_1 exact in 128 bits.
template <bool kAdd>
__device__ __forceinline__ unsigned __int128 neglog64_series(unsigned long long a)
{
    const unsigned a42 = static_cast<unsigned>(a >> 32);  // a 2^42, below 2^32
    unsigned p32 = __umulhi(a42, kNegLog64D6) >> 10;      // floor(a S 2^-42) at 2^33
    unsigned S32 = kAdd ? kNegLog64D5 + p32 : kNegLog64D5 - p32;
    p32 = __umulhi(a42, S32) >> 10;
    S32 = kAdd ? kNegLog64D4 + p32 : kNegLog64D4 - p32;
    unsigned long long p = (static_cast<unsigned long long>(a42) * S32) >> 11;  // at 2^64
    unsigned long long S = kAdd ? kNegLog64D3 + p : kNegLog64D3 - p;
    p = __umul64hi(a, S) >> 10;  // floor(a S 2^-74) at 2^64
    S = kAdd ? kNegLog64D2 + p : kNegLog64D2 - p;
    p = __umul64hi(a, S) >> 11;  // at 2^63
    S = kAdd ? kNegLog64D1 + p : kNegLog64D1 - p;
    return static_cast<unsigned __int128>(a) * S;
}

// -ln(1 - m 2^-53) for m < 2^53 in integer arithmetic only (tandem-sycl
// "Design", Exponentials: an own reproducible logarithm).  V = 2^53 - m = 2^k M,
// E = 53 - k; bin j = floor((M - 1) 2048) with I_j = 4096 inv_j, the reciprocal
// rounded up, so r = M inv_j - 1 is in [0, 1.5 2^-11); with W = M 2^62,
// W I_j = (1 + r) 2^74, so the 64-bit product is r 2^74 exactly.  log1p(r) =
// r S(r) by neglog64_series, all its Horner steps subtractions; -ln(1 - u) =
// E ln 2 + ln inv_j - r S at scale 2^96, rounded once to binary64 (by two
// exact conversions and one add on the FP64 pipe).  For m <=
// 2^41 (u <= 2^-12, about one draw in 4096), where that sum would cancel, the
// value is u S(-u) from the same series with every term added, at 2^137.
// Within 0.5007 ulp.
__device__ __forceinline__ double neglog64(unsigned long long m)
{
    if (m <= (1ull << 41)) {
        if (m == 0) return 0.0;
        return fixed_to_double(neglog64_series<true>(m << 21), 137);  // u 2^74
    }
    const unsigned long long V = (1ull << 53) - m;
    const int k = 63 - __clzll(static_cast<long long>(V));
    const int E = 53 - k;
    const unsigned long long W = V << (62 - k);  // M 2^62
    const unsigned j = static_cast<unsigned>((W - (1ull << 62)) >> 51);
    const ulonglong2 row = __ldg(&kNegLog64Table[j]);
    const unsigned inv = static_cast<unsigned>(row.y >> 48);
    const unsigned __int128 Pm = neglog64_series<false>(W * inv);  // log1p(r) 2^137
    const long long lninv_hi = static_cast<long long>(row.y << 16) >> 16;  // the signed 48-bit field
    // two's complement of lninv_hi 2^64 + low: the high word's 64-bit pattern above the low word
    const __int128 lninv = static_cast<__int128>(
        (static_cast<unsigned __int128>(static_cast<unsigned long long>(lninv_hi)) << 64) | row.x);
    const __int128 ln2 = static_cast<__int128>(
        (static_cast<unsigned __int128>(static_cast<unsigned long long>(kNegLog64Ln2Hi)) << 64) | kNegLog64Ln2Lo);
    const __int128 T = static_cast<__int128>(E) * ln2 + lninv;
    const unsigned __int128 y = static_cast<unsigned __int128>(T - static_cast<__int128>(Pm >> 41));
    // y 2^-96 with y in [2^84, 2^110), so y's high word is below 2^46: RN(y) =
    // RN(hi 2^53 + lo53) 2^11, lo53 the low word's top 53 bits with the sticky
    // bit of its low 11 bits at bit 0 (below the rounding position, bit 20 or
    // higher).  Both terms are exact binary64 values (two exact conversions),
    // their sum is rounded once, and the powers of two go to the exponent
    // field: three FP64-pipe operations instead of fixed_to_double's
    // normalising shifts (1.487 against 1.517 ms per 2^28 fill).
    const unsigned long long hi = static_cast<unsigned long long>(y >> 64);
    const unsigned long long lo = static_cast<unsigned long long>(y);
    const unsigned long long lo53 = (lo >> 11) | static_cast<unsigned long long>((lo & 0x7FFull) != 0ull);
    const double dh = __longlong_as_double(__double_as_longlong(__ull2double_rn(hi)) + (53ll << 52));  // hi 2^53
    const double d = __dadd_rn(dh, __ull2double_rn(lo53));
    return __longlong_as_double(__double_as_longlong(d) -
                                static_cast<long long>(static_cast<unsigned long long>(85) << 52));  // 2^(11 - 96)
}

}  // namespace rngk
