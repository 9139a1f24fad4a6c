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
//        input; here with its table in shared memory); e in [0, 23 ln 2].
//   f64: e = -ln(1 - u), u = (D64 >> 11) 2^-53, by neglog64 of f64_math.cuh:
//        a fixed-point logarithm in 32-, 64- and 128-bit integer arithmetic
//        (GB300 retires 2 FP64 operations per SM and cycle, 1/64 of its FP32
//        rate), within 0.5007 ulp and reproducible bit for bit; e in
//        [0, 53 ln 2].
#include "f64_math.cuh"
#include "fill_kernel.cuh"
#include "hash32.cuh"
#include "neglog_table_kernel.cuh"

namespace rngk {
namespace {

// -ln(1 - u) on the f64 uniform u = (D64 >> 11) 2^-53, by the fixed-point
// logarithm of f64_math.cuh (integer arithmetic only).
struct GenExpF64 {
    using T = double;
    static constexpr uint32_t kVectorsPerThread = 4;  // measured: 1.445 ms per 2^28 fill; 2 1.447, 6 1.450, 8 1.488
    uint32_t key;
    __device__ T operator()(uint32_t c) const { return neglog64(draw64(key, c) >> 11); }
};

// The f32 exponential: lowbias32::exponential's values, with the
// logarithm's table in shared memory (neglog_table_kernel.cuh) and its float
// steps two elements at a time (neg_log_grid_x2_by, f32x2 lanes, the same
// bits).  16 vectors per thread amortise the 32 KiB staging; the launch bound
// of 4 blocks per SM holds the registers at 64.  At 2^28 this takes 0.285 ms
// against 0.336 for the per-element form with an L1 table (shared table
// alone 0.330, pairs with 8 vectors 0.303).
struct GenExpF32 {
    using T = float;
    static constexpr uint32_t kVectorsPerThread = 16;
    static constexpr int kMinBlocksPerSm = 4;
    uint32_t key;
    template <class Load>
    __device__ T operator()(uint32_t c, Load load) const
    {
        return lowbias32::neg_log_grid_by(lowbias32::draw32(lowbias32::Key{key}, c) & 0x7FFFFFu, load);
    }
    template <class Load>
    __device__ Vec16<T> vec(uint32_t c, Load load) const
    {
        const lowbias32::Key k{key};
        const float2 a = lowbias32::detail::neg_log_grid_x2_by(lowbias32::draw32(k, c) & 0x7FFFFFu,
                                                                lowbias32::draw32(k, c + 1u) & 0x7FFFFFu, load);
        const float2 b = lowbias32::detail::neg_log_grid_x2_by(lowbias32::draw32(k, c + 2u) & 0x7FFFFFu,
                                                                lowbias32::draw32(k, c + 3u) & 0x7FFFFFu, load);
        Vec16<T> x;
        x.v[0] = a.x;
        x.v[1] = a.y;
        x.v[2] = b.x;
        x.v[3] = b.y;
        return x;
    }
};

}  // namespace

cudaError_t launch_fill_exponential_f32(uint32_t key, uint32_t first, uint32_t n, float *out, cudaStream_t s)
{
    return launch_neglog_table_fill(GenExpF32{key}, out, first, n, s);
}

cudaError_t launch_fill_exponential_f64(uint32_t key, uint32_t first, uint32_t n, double *out, cudaStream_t s)
{
    return launch_fill(GenExpF64{key}, out, first, n, s);
}

}  // namespace rngk
