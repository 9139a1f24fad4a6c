// normal_f32.cu -- randn: Box-Muller on the uniforms at counters 2c, 2c + 1.
//
// Phobos stdlib "Random numbers", section randn: z = sqrt(-2 log(1 - u0)) *
// cos(6.283185307179586 u1), u0 = uniform(seed, 2c), u1 = uniform(seed,
// 2c + 1); one value per counter (the cosine branch).
//
// Evaluation in f32 (tandem-sycl "Design", section Normals, for the angle):
//   1 - u0 = 2 - (1 + u0) from the pattern 0x3F800000 | m0, exact, in (0, 1];
//   the logarithm is CUDA's logf, relative-accurate next to 1 where
//   1 - u0 = 1 - 2^-23 gives the smallest radii (an absolute-accurate fast
//   log would be off by ~1e-3 there);
//   cos(2 pi u1) = -cos(2 pi (u1 - 1/2)) with u1 - 1/2 = (1 + u1) - 3/2 exact,
//   so the fast cosine runs on [-pi, pi), where its absolute error is below
//   2^-21.4.
// The result is within 4e-6 (1 + |z|) of the exact z.
#include "fill_kernel.cuh"
#include "hash32.cuh"

namespace rngk {
namespace {

struct GenNormalF32 {
    using T = float;
    uint32_t key;
    __device__ T operator()(uint32_t c) const
    {
        const uint32_t a = (c << 1) ^ key;
        const uint32_t h0 = hash32(a);
        const uint32_t h1 = hash32(a ^ 1u);
        const float one_minus_u0 = 2.0f - __uint_as_float(0x3F800000u | (h0 & 0x7FFFFFu));
        const float u1_minus_half = __uint_as_float(0x3F800000u | (h1 & 0x7FFFFFu)) - 1.5f;
        const float radius = sqrtf(-2.0f * logf(one_minus_u0));
        return -radius * __cosf(u1_minus_half * 6.28318530717958647692f);
    }
};

}  // namespace

cudaError_t launch_fill_normal_f32(uint32_t key, uint32_t first, uint32_t n, float *out, cudaStream_t s)
{
    return launch_fill(GenNormalF32{key}, out, first, n, s);
}

}  // namespace rngk
