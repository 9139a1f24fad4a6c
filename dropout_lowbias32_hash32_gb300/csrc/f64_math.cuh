// f64_math.cuh -- the library's own binary64 exp and log: fixed sequences of
// IEEE operations (+, -, *, /, fma with explicit rounding intrinsics), so a
// second implementation performing the same operations in the same order
// returns the same bits on any IEEE machine.  Used by the ziggurat's slow
// path and by the f64 exponential fill.
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

}  // namespace rngk
