// fill_bounded.cu -- bounded integers by Lemire's multiply-shift with
// rejection, and the low-bound ranges built on them.
//
// perturbation-kernel "Backends", section "Why the GPU can be exact": the
// multiply-shift with rejection is pure integer arithmetic, exact anywhere.
// tandem-cuda "Performance", bounded rows: the bounded fills run at the fill
// speed because a rejection is rare and its retry runs out of line.
//
// For a w-bit word x and bound b the 2w-bit product x*b gives the candidate
// (its high word) and is accepted when its low word is at least 2^w mod b,
// computed once on the host (Lemire's exact threshold: every value in [0, b)
// is hit by exactly floor(2^w / b) words).  The rejected fraction is
// (2^w mod b) / 2^w, e.g. 296 / 2^32 for b = 1000.  A rejected element draws
// its retry words from its own substream (keyed by its counter), so the
// result stays a pure function of (seed, counter).
#include "fill_kernel.cuh"
#include "hash32.cuh"

namespace rngk {
namespace {

// Retries are bounded at 2^16 words; below the 1/2 worst-case rejection
// rate the cap is never reached (probability < 2^-65536).
constexpr uint32_t kMaxRetries = 1u << 16;

__device__ __noinline__ uint32_t below32_retry(uint32_t purpose_key, uint32_t c, uint32_t bound,
                                               uint32_t threshold)
{
    const uint32_t skey = substream_key(purpose_key, c);
    uint64_t m = 0;
    for (uint32_t k = 0; k < kMaxRetries; ++k) {
        m = static_cast<uint64_t>(substream32(skey, k)) * bound;
        if (static_cast<uint32_t>(m) >= threshold) break;
    }
    return static_cast<uint32_t>(m >> 32);
}

__device__ __forceinline__ uint32_t below32(const Below32Args &a, uint32_t c)
{
    const uint64_t m = static_cast<uint64_t>(draw32(a.key, c)) * a.bound;
    if (__builtin_expect(static_cast<uint32_t>(m) < a.threshold, 0))
        return below32_retry(a.purpose_key, c, a.bound, a.threshold);
    return static_cast<uint32_t>(m >> 32);
}

__device__ __noinline__ uint64_t below64_retry(uint32_t purpose_key, uint32_t c, uint64_t bound,
                                               uint64_t threshold)
{
    const uint32_t skey = substream_key(purpose_key, c);
    uint64_t hi = 0;
    for (uint32_t k = 0; k < kMaxRetries; ++k) {
        const uint64_t x = substream64(skey, k);
        hi = __umul64hi(x, bound);
        if (x * bound >= threshold) break;
    }
    return hi;
}

__device__ __forceinline__ uint64_t below64(const Below64Args &a, uint32_t c)
{
    const uint64_t x = draw64(a.key, c);
    const uint64_t lo = x * a.bound;
    if (__builtin_expect(lo < a.threshold, 0)) return below64_retry(a.purpose_key, c, a.bound, a.threshold);
    return __umul64hi(x, a.bound);
}

struct GenBelow32 {
    using T = uint32_t;
    static constexpr uint32_t kVectorsPerThread = kHeavyVectorsPerThread;
    Below32Args a;
    __device__ T operator()(uint32_t c) const { return below32(a, c); }
};

struct GenBelow64 {
    using T = uint64_t;
    static constexpr uint32_t kVectorsPerThread = kHeavyVectorsPerThread;
    Below64Args a;
    __device__ T operator()(uint32_t c) const { return below64(a, c); }
};

// low + below, wrapped in two's complement (unsigned addition, then the
// bit pattern reinterpreted).
struct GenI32Range {
    using T = int32_t;
    static constexpr uint32_t kVectorsPerThread = kHeavyVectorsPerThread;
    Below32Args a;
    int32_t low;
    __device__ T operator()(uint32_t c) const
    {
        return static_cast<int32_t>(static_cast<uint32_t>(low) + below32(a, c));
    }
};

struct GenI64Range32 {
    using T = int64_t;
    Below32Args a;
    int64_t low;
    __device__ T operator()(uint32_t c) const
    {
        return static_cast<int64_t>(static_cast<uint64_t>(low) + below32(a, c));
    }
};

struct GenI64Range {
    using T = int64_t;
    static constexpr uint32_t kVectorsPerThread = kHeavyVectorsPerThread;
    Below64Args a;
    int64_t low;
    __device__ T operator()(uint32_t c) const
    {
        return static_cast<int64_t>(static_cast<uint64_t>(low) + below64(a, c));
    }
};

}  // namespace

cudaError_t launch_fill_u32_below(const Below32Args &a, uint32_t first, uint32_t n, uint32_t *out,
                                  cudaStream_t s)
{
    return launch_fill(GenBelow32{a}, out, first, n, s);
}

cudaError_t launch_fill_u64_below(const Below64Args &a, uint32_t first, uint32_t n, uint64_t *out,
                                  cudaStream_t s)
{
    return launch_fill(GenBelow64{a}, out, first, n, s);
}

cudaError_t launch_fill_i32_range(const Below32Args &a, int32_t low, uint32_t first, uint32_t n,
                                  int32_t *out, cudaStream_t s)
{
    return launch_fill(GenI32Range{a, low}, out, first, n, s);
}

cudaError_t launch_fill_i64_range32(const Below32Args &a, int64_t low, uint32_t first, uint32_t n,
                                    int64_t *out, cudaStream_t s)
{
    return launch_fill(GenI64Range32{a, low}, out, first, n, s);
}

cudaError_t launch_fill_i64_range(const Below64Args &a, int64_t low, uint32_t first, uint32_t n,
                                  int64_t *out, cudaStream_t s)
{
    return launch_fill(GenI64Range{a, low}, out, first, n, s);
}

}  // namespace rngk
