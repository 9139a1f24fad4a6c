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
//   f64: e = 0 - zlog(1 - u), u = (D64 >> 11) 2^-53; 1 - u is exact and
//        zlog is the fixed IEEE sequence of f64_math.cuh, so the value is
//        reproducible bit for bit; e in [0, 53 ln 2].
// GB300 retires 2 FP64 operations per SM and cycle; the f64 logarithm
// (a division and a degree-11 series, about 26 FP64 operations) makes that
// fill FP64-bound at a small fraction of the HBM rate.
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

// (w >> 11) 2^-53 exactly, from integer operations (as the f64 uniform fill)
__device__ __forceinline__ double u53_exact(Words w)
{
    if (w.hi == 0) return __dmul_rn(__uint2double_rn(w.lo >> 11), 0x1p-53);
    const uint32_t lo = w.lo & ~0x7FFu;
    const uint32_t z = __clz(w.hi);
    const uint32_t a_hi = __funnelshift_l(lo, w.hi, z);
    const uint32_t a_lo = lo << z;
    const uint32_t sig_hi = a_hi >> 11;
    const uint32_t sig_lo = __funnelshift_r(a_lo, a_hi, 11);
    return __hiloint2double(static_cast<int>(sig_hi + ((1021u - z) << 20)), static_cast<int>(sig_lo));
}

struct GenExpF64 {
    using T = double;
    static constexpr uint32_t kVectorsPerThread = kHeavyVectorsPerThread;
    uint32_t key;
    __device__ T operator()(uint32_t c) const
    {
        const double v = __dsub_rn(1.0, u53_exact(draw64_words(key, c)));  // exact, in (0, 1]
        return __dsub_rn(0.0, zlog(v));
    }
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
