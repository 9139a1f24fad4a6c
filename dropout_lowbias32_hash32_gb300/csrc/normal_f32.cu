// normal_f32.cu -- randn: Box-Muller on the uniforms at counters 2c, 2c + 1.
//
// Phobos stdlib "Random numbers", section randn: z = sqrt(-2 log(1 - u0)) *
// cos(6.283185307179586 u1), u0 = uniform(seed, 2c), u1 = uniform(seed,
// 2c + 1); one value per counter (the cosine branch).
//
// Evaluation in f32, on the instruction budget of an HBM-speed fill:
//   1 - u0 = 2 - (1 + u0) from the pattern 0x3F800000 | m0, exact, in (0, 1];
//   L = ln(1 - u0): for u0 < 2^-5 the series -(u + u^2/2 + ... + u^5/5)
//   (Mercator series; relative error below 1e-7 there, where the radius is
//   small and an absolutely accurate log is not enough), otherwise
//   ln 2 * log2(1 - u0) from the hardware log2 (absolute error <= 2^-22 on
//   [1/2, 1], i.e. radius error <= 7e-7 for radii >= 1/4);
//   radius = sqrt(t), t = -2L, from the hardware square root (t is 0 or at
//   least 2^-22, never subnormal, so the flush-to-zero forms lose nothing);
//   cos(2 pi u1) = -cos(2 pi (u1 - 1/2)) with u1 - 1/2 = (1 + u1) - 3/2 exact,
//   so the hardware cosine runs on [-pi, pi), where its absolute error is
//   below 2^-21.4 (tandem-sycl "Design", section Normals: the angle shifted
//   by half a turn).
// Every value is within 4e-6 (1 + |z|) of the exact z.
#include "fill_kernel.cuh"
#include "hash32.cuh"

namespace rngk {
namespace {

// Hardware approximations (PTX .approx, flush-to-zero: no operand here is
// subnormal).
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

struct GenNormalF32 {
    using T = float;
    static constexpr uint32_t kVectorsPerStep = 2;
    uint32_t key;  // folded hash of the seed
    __device__ T operator()(uint32_t c) const
    {
        const Words h = draw64_words(key, c);  // the draws at 2c and 2c + 1
        const float one_plus_u0 = __uint_as_float(0x3F800000u | (h.hi & 0x7FFFFFu));
        const float u0 = one_plus_u0 - 1.0f;
        const float v = 2.0f - one_plus_u0;  // 1 - u0
        float series = __fmaf_rn(u0, 0.2f, 0.25f);
        series = __fmaf_rn(u0, series, 0.333333343f);
        series = __fmaf_rn(u0, series, 0.5f);
        series = __fmaf_rn(u0, series, 1.0f);
        const float minus_two_l_small = (2.0f * u0) * series;         // -2 ln(1 - u0), u0 small
        const float minus_two_l_large = -1.38629436f * lg2_approx(v);  // -2 ln 2 log2(1 - u0)
        const float t = (h.hi & 0x7C0000u) ? minus_two_l_large : minus_two_l_small;  // u0 >= 2^-5 ?
        const float u1_minus_half = __uint_as_float(0x3F800000u | (h.lo & 0x7FFFFFu)) - 1.5f;
        return -sqrt_approx(t) * cos_approx(u1_minus_half * 6.28318530717958647692f);
    }
};

}  // namespace

cudaError_t launch_fill_normal_f32(uint32_t key, uint32_t first, uint32_t n, float *out, cudaStream_t s)
{
    return launch_fill(GenNormalF32{key}, out, first, n, s);
}

}  // namespace rngk
