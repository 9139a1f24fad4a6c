// normal_f32.cu -- randn: Box-Muller on the uniforms at counters 2c, 2c + 1.
//
// Phobos stdlib "Random numbers", section randn: z = sqrt(-2 log(1 - u0)) *
// cos(6.283185307179586 u1), u0 = uniform(seed, 2c), u1 = uniform(seed,
// 2c + 1); one value per counter (the cosine branch).
//
// Evaluated by lowbias32::randn (include/rng_device.cuh), in f32 on the
// instruction budget of an HBM-speed fill: 1 - u0 exact; ln(1 - u0) from the
// Mercator series below u0 = 2^-5 and the hardware log2 above; the hardware
// sqrt; cos(2 pi u1) = -cos(2 pi (u1 - 1/2)) so the hardware cosine runs on
// [-pi, pi) (tandem-sycl "Design", section Normals: the angle shifted by half
// a turn).  Every value is within 4e-6 (1 + |z|) of the exact z.
#include "fill_kernel.cuh"
#include "hash32.cuh"

namespace rngk {
namespace {

struct GenNormalF32 {
    using T = float;
    static constexpr uint32_t kVectorsPerThread = kHeavyVectorsPerThread;
    uint32_t key;  // folded hash of the seed
    __device__ T operator()(uint32_t c) const { return lowbias32::randn(lowbias32::Key{key}, c); }
};

// Paired normals: element c is the cosine branch of pair c >> 1 (even c)
// or its sine branch (odd c), pair q Box-Muller on the uniforms at 2q and
// 2q + 1; one 64-bit draw, one radius and one angle serve two elements.  A
// vector's four counters start at the same parity everywhere in a launch
// (c0 = first + head + 4v), so the branch below is uniform across the grid;
// an odd start needs three pairs per vector instead of two.
struct GenNormalF32Pairs {
    using T = float;
    static constexpr uint32_t kVectorsPerThread = kHeavyVectorsPerThread;
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
    static constexpr uint32_t kVectorsPerThread = kHeavyVectorsPerThread;
    uint32_t key;
    __device__ T operator()(uint32_t c) const { return lowbias32::randn_precise(lowbias32::Key{key}, c); }
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
    return launch_fill(GenNormalF32{key}, out, first, n, s);
}

}  // namespace rngk
