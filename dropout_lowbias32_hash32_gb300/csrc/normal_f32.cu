// normal_f32.cu -- randn: Box-Muller on the uniforms at counters 2c, 2c + 1.
//
// Phobos stdlib "Random numbers", section randn: z = sqrt(-2 log(1 - u0)) *
// cos(6.283185307179586 u1), u0 = uniform(seed, 2c), u1 = uniform(seed,
// 2c + 1); one value per counter (the cosine branch).
//
// Evaluated by lowbias32::randn (include/rng_device.cuh), in f32 on the
// instruction budget of an HBM-speed fill: 1 - u0 exact; -2 ln(1 - u0) as
// (1 + u0)^2 - 1 below u0 = 2^-7 and from the hardware log2 above; the
// hardware sqrt and cosine, the angle 2 pi u1 in one fma.  (tandem-sycl
// "Design", section Normals, shifts the angle by half a turn for its sincos;
// GB300's cosine is as accurate over the whole turn, so this one does not.)
// Every value is within 4e-6 (1 + |z|) of the exact z.
#include "fill_kernel.cuh"
#include "hash32.cuh"

namespace rngk {
namespace {

// A vector's four elements at c0 .. c0 + 3 read the draws at 2c0 .. 2c0 + 7.
// When c0 is a multiple of 4 (for every vector of a launch or for none:
// c0 = first + head + 4v), a = 2c0 is a multiple of 8, so the eight counters
// are a ^ i (i < 8) with one a >> 16, and their first xorshifts are
// x ^ i, x = a ^ (a >> 16) ^ key: one shift for the vector.  The first
// multiply of the odd draw follows from the even one's, (x ^ 1) M = x M +
// (x even ? M : -M), with the same sign for the vector's four pairs.  The
// host picks the aligned or the general generator for the launch (each is
// its own kernel); both return randn's values bit for bit (the same integer
// and IEEE operations).
template <bool kAligned>
struct GenNormalF32 {
    using T = float;
    static constexpr uint32_t kVectorsPerThread = 16;  // measured at 2^28: 1.7 % faster than 8, 0.6 % than 4
    // the aligned generator at 6 blocks per SM (256 threads): the compiler then
    // takes 40 registers instead of 34, the same 6 resident blocks, and the
    // 2^28 fill runs in 0.188 ms against 0.190; the general one would spill
    static constexpr int kMinBlocksPerSm = kAligned ? 6 : 0;
    static constexpr uint32_t kM1 = 0x7FEB352Du;
    uint32_t key;  // folded hash of the seed
    __device__ T operator()(uint32_t c) const { return lowbias32::randn(lowbias32::Key{key}, c); }
    __device__ Vec16<float> vec(uint32_t c0) const
    {
        namespace d = lowbias32::detail;
        uint32_t b0[4], b1[4];
        if constexpr (kAligned) {
            const uint32_t a = c0 << 1;
            const uint32_t x = a ^ (a >> 16) ^ key;
            const uint32_t odd_step = (x & 1u) ? 0u - kM1 : kM1;
#pragma unroll
            for (uint32_t j = 0; j < 4; ++j) {
                const uint32_t xj = x ^ (2u * j);
                b0[j] = d::one_plus_uniform_bits(d::hash32_middle(xj * kM1));
                b1[j] = d::one_plus_uniform_bits(d::hash32_middle(xj * kM1 + odd_step));
            }
        } else {
#pragma unroll
            for (uint32_t j = 0; j < 4; ++j) {
                const uint32_t a = (c0 + j) << 1;
                const uint32_t x = a ^ (a >> 16) ^ key;
                b0[j] = d::one_plus_uniform_bits(d::hash32_middle(x * kM1));
                b1[j] = d::one_plus_uniform_bits(d::hash32_middle((x ^ 1u) * kM1));
            }
        }
        const float2 p = d::box_muller_bits_x2(b0[0], b1[0], b0[1], b1[1]);
        const float2 q = d::box_muller_bits_x2(b0[2], b1[2], b0[3], b1[3]);
        Vec16<float> v;
        v.v[0] = p.x;
        v.v[1] = p.y;
        v.v[2] = q.x;
        v.v[3] = q.y;
        return v;
    }
};

// Paired normals: element c is the cosine branch of pair c >> 1 (even c)
// or its sine branch (odd c), pair q Box-Muller on the uniforms at 2q and
// 2q + 1; one 64-bit draw, one radius and one angle serve two elements.  A
// vector's four counters start at the same parity everywhere in a launch
// (c0 = first + head + 4v), so the branch below is uniform across the grid;
// an odd start needs three pairs per vector instead of two.
struct GenNormalF32Pairs {
    using T = float;
    static constexpr uint32_t kVectorsPerThread = 4;  // measured at 2^28: 0.8 % faster than 8, 7 % than 16
    uint32_t key;
    __device__ T operator()(uint32_t c) const { return lowbias32::randn_paired(lowbias32::Key{key}, c); }
    __device__ Vec16<float> vec(uint32_t c0) const
    {
        const lowbias32::Key k{key};
        Vec16<float> x;
        if ((c0 & 1u) == 0u) {
            const float2 a = lowbias32::randn_pair(k, c0 >> 1);
            const float2 b = lowbias32::randn_pair(k, (c0 + 2u) >> 1);
            x.v[0] = a.x;
            x.v[1] = a.y;
            x.v[2] = b.x;
            x.v[3] = b.y;
        } else {
            const float2 a = lowbias32::randn_pair(k, c0 >> 1);
            const float2 b = lowbias32::randn_pair(k, (c0 + 1u) >> 1);
            const float2 d = lowbias32::randn_pair(k, (c0 + 3u) >> 1);
            x.v[0] = a.y;
            x.v[1] = b.x;
            x.v[2] = b.y;
            x.v[3] = d.x;
        }
        return x;
    }
};

// The precise variant: randn's definition to a few ulp (lowbias32::randn_precise:
// the own binary32 -ln(1 - u0) and cos(2 pi u1), an IEEE square root), an
// opt-in fill with its own values (tandem-sycl "Design", Normals: a precise
// f32 Box-Muller as a build option).
struct GenNormalF32Precise {
    using T = float;
    static constexpr uint32_t kVectorsPerThread = 4;  // measured at 2^28: 1.3 % faster than 8, 14 % than 16
    uint32_t key;
    __device__ T operator()(uint32_t c) const { return lowbias32::randn_precise(lowbias32::Key{key}, c); }
    // a vector's four values, the float steps two at a time
    // (lowbias32::detail::randn_precise_x2: the same values)
    __device__ Vec16<float> vec(uint32_t c0) const
    {
        const lowbias32::Key k{key};
        const lowbias32::Words w0 = lowbias32::draw64_words(k, c0), w1 = lowbias32::draw64_words(k, c0 + 1u);
        const lowbias32::Words w2 = lowbias32::draw64_words(k, c0 + 2u), w3 = lowbias32::draw64_words(k, c0 + 3u);
        const float2 a = lowbias32::detail::randn_precise_x2(w0.hi, w0.lo, w1.hi, w1.lo);
        const float2 b = lowbias32::detail::randn_precise_x2(w2.hi, w2.lo, w3.hi, w3.lo);
        Vec16<float> v;
        v.v[0] = a.x;
        v.v[1] = a.y;
        v.v[2] = b.x;
        v.v[3] = b.y;
        return v;
    }
};

}  // namespace

cudaError_t launch_fill_normal_f32_precise(uint32_t key, uint32_t first, uint32_t n, float *out, cudaStream_t s)
{
    return launch_fill(GenNormalF32Precise{key}, out, first, n, s);
}

cudaError_t launch_fill_normal_f32_pairs(uint32_t key, uint32_t first, uint32_t n, float *out, cudaStream_t s)
{
    return launch_fill(GenNormalF32Pairs{key}, out, first, n, s);
}

cudaError_t launch_fill_normal_f32(uint32_t key, uint32_t first, uint32_t n, float *out, cudaStream_t s)
{
    // the body's vectors start at counters first + head + 4v
    if (((first + head_elems<float>(out, n)) & 3u) == 0u) return launch_fill(GenNormalF32<true>{key}, out, first, n, s);
    return launch_fill(GenNormalF32<false>{key}, out, first, n, s);
}

}  // namespace rngk
