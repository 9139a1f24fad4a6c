// exponential.cu -- standard exponential fills: -ln(1 - u).
//
// tandem-sycl "Design", section Exponentials, and tandem-cuda
// "Performance", rows fill_exponential_f64 / _f32: exponentials by a
// logarithm of a uniform, f64 through the library's own logarithm and f32
// through an own binary32 logarithm within 0.571 ulp, both reproducible bit
// for bit.  Restated on hash32:
//   f32: e = -ln(1 - u), u = uniform(seed, c) on the 2^-23 grid, by
//        lowbias32::neg_log_grid of include/rng_device.cuh (a table-driven
//        binary32 logarithm, within 0.5035 ulp of the exact value on every
//        input); e in [0, 23 ln 2].
//   f64: e = -ln(1 - u), u = (D64 >> 11) 2^-53, by neglog64 of f64_math.cuh:
//        a fixed-point logarithm in 64- and 128-bit integer arithmetic
//        (GB300 retires 2 FP64 operations per SM and cycle, 1/64 of its FP32
//        rate), within 0.5015 ulp and reproducible bit for bit; e in
//        [0, 53 ln 2].
#include "f64_math.cuh"
#include "fill_kernel.cuh"
#include "hash32.cuh"

namespace rngk {
namespace {

struct GenExpF32 {
    using T = float;
    static constexpr uint32_t kVectorsPerThread = kHeavyVectorsPerThread;
    uint32_t key;
    __device__ T operator()(uint32_t c) const { return lowbias32::exponential(lowbias32::Key{key}, c); }
};

// -ln(1 - u) on the f64 uniform u = (D64 >> 11) 2^-53, by the fixed-point
// logarithm of f64_math.cuh (integer arithmetic only).
struct GenExpF64 {
    using T = double;
    static constexpr uint32_t kVectorsPerThread = 4;  // a long body: fewer copies of it than the default 8
    uint32_t key;
    __device__ T operator()(uint32_t c) const { return neglog64(draw64(key, c) >> 11); }
};

}  // namespace

cudaError_t launch_fill_exponential_f32(uint32_t key, uint32_t first, uint32_t n, float *out, cudaStream_t s)
{
    return launch_fill(GenExpF32{key}, out, first, n, s);
}

cudaError_t launch_fill_exponential_f64(uint32_t key, uint32_t first, uint32_t n, double *out, cudaStream_t s)
{
    return launch_fill(GenExpF64{key}, out, first, n, s);
}

}  // namespace rngk
