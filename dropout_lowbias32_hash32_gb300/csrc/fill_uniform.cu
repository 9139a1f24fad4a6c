// fill_uniform.cu -- u32, u64, f32 and f64 uniform fills.
//
// Phobos stdlib "Random numbers", section uniform: the f32 value is the
// draw's low 23 bits times 2^-23.  tandem-cuda "Performance", rows fill_u64
// and fill_f64: the 64-bit and double fills, here on the 64-bit draw (the
// draws at 2c and 2c + 1) and its top 53 bits times 2^-53.
#include "fill_kernel.cuh"
#include "hash32.cuh"

namespace rngk {
namespace {

struct GenU32 {
    using T = uint32_t;
    uint32_t key;
    __device__ T operator()(uint32_t c) const { return draw32(key, c); }
};

struct GenU64 {
    using T = uint64_t;
    uint32_t key;
    __device__ T operator()(uint32_t c) const { return draw64(key, c); }
};

// m * 2^-23 for the low 23 bits m: the pattern 0x3F800000 | m is the float
// 1 + m 2^-23, and subtracting 1 is exact (Sterbenz).
struct GenF32 {
    using T = float;
    uint32_t key;
    __device__ T operator()(uint32_t c) const
    {
        return __uint_as_float(0x3F800000u | (draw32(key, c) & 0x7FFFFFu)) - 1.0f;
    }
};

// m * 2^-53 for m < 2^53, exactly, from integer operations only (GB300's FP64
// pipe is far too narrow for an HBM-speed fill): normalise m so its leading
// one sits at bit 52, which becomes the implicit bit, and add the biased
// exponent 1022 - (clz(m) - 11) below it; the implicit bit carries into the
// exponent field.
__device__ __forceinline__ double scaled_u53_to_double(uint64_t m)
{
    const int lz = __clzll(m);
    const uint64_t bits = (static_cast<uint64_t>(1032 - lz) << 52) + (m << (lz - 11));
    return __longlong_as_double(m ? static_cast<long long>(bits) : 0ll);
}

struct GenF64 {
    using T = double;
    uint32_t key;
    __device__ T operator()(uint32_t c) const { return scaled_u53_to_double(draw64(key, c) >> 11); }
};

}  // namespace

cudaError_t launch_fill_u32(uint32_t key, uint32_t first, uint32_t n, uint32_t *out, cudaStream_t s)
{
    return launch_fill(GenU32{key}, out, first, n, s);
}

cudaError_t launch_fill_u64(uint32_t key, uint32_t first, uint32_t n, uint64_t *out, cudaStream_t s)
{
    return launch_fill(GenU64{key}, out, first, n, s);
}

cudaError_t launch_fill_f32(uint32_t key, uint32_t first, uint32_t n, float *out, cudaStream_t s)
{
    return launch_fill(GenF32{key}, out, first, n, s);
}

cudaError_t launch_fill_f64(uint32_t key, uint32_t first, uint32_t n, double *out, cudaStream_t s)
{
    return launch_fill(GenF64{key}, out, first, n, s);
}

}  // namespace rngk
