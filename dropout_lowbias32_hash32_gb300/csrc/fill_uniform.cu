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

// `key` is the folded hash of the seed (hash32.cuh).
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

// (w >> 11) * 2^-53 for the 64-bit draw w = hi:lo, exactly, from integer
// operations only (GB300's FP64 pipe is too narrow to convert every element
// of an HBM-speed fill).  Clear the 11 bits below m = w >> 11, normalise on the high word so
// m's leading one reaches bit 63, take the 53-bit significand (implicit bit
// at bit 52) and add the biased exponent 1021 - z below it; the implicit bit
// carries one into the exponent field, giving 2^(-1-z) (1.f).  The high word
// is zero for one draw in 2^32; such m < 2^21 go through an exact
// integer-to-double conversion.
__device__ __noinline__ double scaled_small_u53(uint32_t lo)
{
    return __dmul_rn(__uint2double_rn(lo >> 11), 0x1p-53);
}

// The normalising conversion alone; `small` is set when the high word is
// zero (then the value must come from scaled_small_u53).
__device__ __forceinline__ double scaled_u53_candidate(Words w, bool &small)
{
    small |= w.hi == 0;
    const uint32_t lo = w.lo & ~0x7FFu;
    const uint32_t z = __clz(w.hi);
    const uint32_t a_hi = __funnelshift_l(lo, w.hi, z);  // (hi:lo) << z, high word
    const uint32_t a_lo = lo << z;
    const uint32_t sig_hi = a_hi >> 11;  // bit 20: the implicit bit
    const uint32_t sig_lo = __funnelshift_r(a_lo, a_hi, 11);
    return __hiloint2double(static_cast<int>(sig_hi + ((1021u - z) << 20)), static_cast<int>(sig_lo));
}

// The same value with one FP64 instruction: t = 1 + (m mod 2^52) 2^-52 is
// assembled from the word's bits and, with b the top bit of m,
// fma(t, 1/2, b ? 0 : -1/2) = (m mod 2^52) 2^-53 + b/2 = m 2^-53, exact for
// every m (no small case).  The integer conversion keeps the ALU pipe busy
// while the FP64 pipe idles; sending one element of each pair through the
// fma balances them (2 DFMA per SM and cycle carry half the elements at the
// fill's speed; all of them would make the FP64 pipe the bound).
__device__ __forceinline__ double scaled_u53_fma(Words w)
{
    const uint32_t t_lo = __funnelshift_r(w.lo, w.hi, 11);
    const uint32_t t_hi = ((w.hi >> 11) & 0xFFFFFu) | 0x3FF00000u;
    const uint32_t c_hi = ~static_cast<uint32_t>(static_cast<int32_t>(w.hi) >> 31) & 0xBFE00000u;  // -1/2 or 0
    return __fma_rn(__hiloint2double(static_cast<int>(t_hi), static_cast<int>(t_lo)), 0.5,
                    __hiloint2double(static_cast<int>(c_hi), 0));
}

__device__ __forceinline__ double scaled_u53_to_double(Words w)
{
    bool small = false;
    const double x = scaled_u53_candidate(w, small);
    return __builtin_expect(small, 0) ? scaled_small_u53(w.lo) : x;
}

struct GenF64 {
    using T = double;
    // measured at 2^28 with half the conversions on the FP64 pipe: 0.279 ms
    // against 0.285 at 4 and 0.289 at 16 (73 registers: the DFMA's latency
    // wants the warps that 40 registers leave room for)
    static constexpr uint32_t kVectorsPerThread = 8;
    uint32_t key;
    __device__ T operator()(uint32_t c) const { return scaled_u53_to_double(draw64_words(key, c)); }
    // both elements of a 16-byte vector: the first by the fma, the second by
    // the integer conversion with its branch on a zero high word.  At 2^28,
    // 0.290 ms against 0.303 with both integer (1/4 of the elements by the
    // fma: 0.295; 3/8: 0.289; 5/8: 0.336, FP64-bound).
    __device__ Vec16<T> vec(uint32_t c0) const
    {
        const Words w0 = draw64_words(key, c0), w1 = draw64_words(key, c0 + 1u);
        bool small = false;
        Vec16<T> x;
        x.v[0] = scaled_u53_fma(w0);
        x.v[1] = scaled_u53_candidate(w1, small);
        if (__builtin_expect(small, 0)) x.v[1] = scaled_u53_to_double(w1);
        return x;
    }
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
