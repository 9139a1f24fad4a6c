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

// The candidate for counter c without its rejection test's branch: the
// value if accepted, and `reject` set when the low word is below the
// threshold (then the element must take its retries).
__device__ __forceinline__ uint32_t below32_candidate(const Below32Args &a, uint32_t c, bool &reject)
{
    const uint64_t m = static_cast<uint64_t>(draw32(a.key, c)) * a.bound;
    reject |= static_cast<uint32_t>(m) < a.threshold;
    return static_cast<uint32_t>(m >> 32);
}

// A 16-byte vector of a bounded fill: every element's candidate and one
// branch on the OR of their rejection tests (rare: about 4 (2^w mod b) / 2^w
// per vector), whose slow path recomputes the vector element by element with
// retries.  The same values as the per-element function.
template <class Gen, class T = typename Gen::T>
__device__ __forceinline__ Vec16<T> bounded_vec(const Gen &gen, uint32_t c0)
{
    constexpr uint32_t kPer = Vec16<T>::kPer;
    Vec16<T> x;
    bool reject = false;
#pragma unroll
    for (uint32_t k = 0; k < kPer; ++k) x.v[k] = gen.candidate(c0 + k, reject);
    if (__builtin_expect(reject, 0)) {
#pragma unroll
        for (uint32_t k = 0; k < kPer; ++k) x.v[k] = gen(c0 + k);
    }
    return x;
}

struct GenBelow32 {
    using T = uint32_t;
    static constexpr uint32_t kVectorsPerThread = kHeavyVectorsPerThread;
    Below32Args a;
    __device__ T operator()(uint32_t c) const { return below32(a, c); }
    __device__ T candidate(uint32_t c, bool &reject) const { return below32_candidate(a, c, reject); }
    __device__ Vec16<T> vec(uint32_t c0) const { return bounded_vec(*this, c0); }
};

// The 64-bit generators' vector: both elements' draws at once (for an even
// first counter the four 32-bit draws share one first xorshift) and the
// candidates.  kMode 0: bound below 2^32, so x b = (x_hi b + (x_lo b >> 32))
// 2^32 + lo(x_lo b) by two 32 x 32 -> 64 multiply-adds, and the value (< b)
// is the high word of the second; kMode 1: a 64-bit bound whose threshold
// 2^64 mod b is below 2^32; kMode 2: a threshold of 64 bits (the 64-bit
// products by the compiler's 64 x 64 forms, which measured faster than an
// explicit chain of 32-bit multiply-adds).  With a threshold below 2^32 a
// rejection needs the product's low 64 bits to have a zero high word, so the
// vector's test is that word against zero (2^-32 of elements, exactly
// rechecked by the slow path) instead of a 64-bit compare.
// kEven and kMode are the same for every vector of a launch (the host picks
// the instantiation); every value equals below64's.
template <uint32_t kMode>
__device__ __forceinline__ uint64_t below64_candidate_words(Words x, uint64_t bound, uint64_t threshold, bool &reject)
{
    const uint32_t b_lo = static_cast<uint32_t>(bound), b_hi = static_cast<uint32_t>(bound >> 32);
    const uint64_t p0 = static_cast<uint64_t>(x.lo) * b_lo;
    if constexpr (kMode == 0) {
        const uint64_t p1 = static_cast<uint64_t>(x.hi) * b_lo + (p0 >> 32);
        reject |= static_cast<uint32_t>(p1) == 0u;
        return p1 >> 32;
    } else {
        (void)p0;
        const uint64_t xx = (static_cast<uint64_t>(x.hi) << 32) | x.lo;
        const uint64_t low = xx * bound;
        if constexpr (kMode == 1) {
            reject |= static_cast<uint32_t>(low >> 32) == 0u;
        } else {
            reject |= low < threshold;
        }
        return __umul64hi(xx, bound);
    }
}

// Mode of a 64-bit bound (see below64_candidate_words).
inline uint32_t below64_mode(const Below64Args &a)
{
    return (a.bound >> 32) == 0 ? 0u : ((a.threshold >> 32) == 0 ? 1u : 2u);
}

template <class Gen, bool kEven, uint32_t kMode>
__device__ __forceinline__ Vec16<typename Gen::T> bounded64_vec(const Gen &gen, uint32_t c0)
{
    Words w0, w1;
    if constexpr (kEven) {
        draw64_pair_words(gen.a.key, c0, w0, w1);
    } else {
        w0 = draw64_words(gen.a.key, c0);
        w1 = draw64_words(gen.a.key, c0 + 1u);
    }
    bool reject = false;
    Vec16<typename Gen::T> x;
    x.v[0] = gen.finish(below64_candidate_words<kMode>(w0, gen.a.bound, gen.a.threshold, reject));
    x.v[1] = gen.finish(below64_candidate_words<kMode>(w1, gen.a.bound, gen.a.threshold, reject));
    if (__builtin_expect(reject, 0)) {
        x.v[0] = gen(c0);
        x.v[1] = gen(c0 + 1u);
    }
    return x;
}

template <bool kEven, uint32_t kMode>
struct GenBelow64 {
    using T = uint64_t;
    static constexpr uint32_t kVectorsPerThread = kHeavyVectorsPerThread;
    Below64Args a;
    __device__ T operator()(uint32_t c) const { return below64(a, c); }
    __device__ T finish(uint64_t v) const { return v; }
    __device__ Vec16<T> vec(uint32_t c0) const { return bounded64_vec<GenBelow64, kEven, kMode>(*this, c0); }
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
    __device__ T candidate(uint32_t c, bool &reject) const
    {
        return static_cast<int32_t>(static_cast<uint32_t>(low) + below32_candidate(a, c, reject));
    }
    __device__ Vec16<T> vec(uint32_t c0) const { return bounded_vec(*this, c0); }
};

struct GenI64Range32 {
    using T = int64_t;
    Below32Args a;
    int64_t low;
    __device__ T operator()(uint32_t c) const
    {
        return static_cast<int64_t>(static_cast<uint64_t>(low) + below32(a, c));
    }
    __device__ T candidate(uint32_t c, bool &reject) const
    {
        return static_cast<int64_t>(static_cast<uint64_t>(low) + below32_candidate(a, c, reject));
    }
    __device__ Vec16<T> vec(uint32_t c0) const { return bounded_vec(*this, c0); }
};

template <bool kEven, uint32_t kMode>
struct GenI64Range {
    using T = int64_t;
    static constexpr uint32_t kVectorsPerThread = kHeavyVectorsPerThread;
    Below64Args a;
    int64_t low;
    __device__ T operator()(uint32_t c) const
    {
        return static_cast<int64_t>(static_cast<uint64_t>(low) + below64(a, c));
    }
    __device__ T finish(uint64_t v) const { return static_cast<int64_t>(static_cast<uint64_t>(low) + v); }
    __device__ Vec16<T> vec(uint32_t c0) const { return bounded64_vec<GenI64Range, kEven, kMode>(*this, c0); }
};

// Launch a 64-bit generator family G<kEven, kMode> for a's bound: the body's
// vectors start at counters first + head + 2v, even for all or for none.
template <template <bool, uint32_t> class G, class... Extra>
cudaError_t launch_below64_family(const Below64Args &a, uint32_t first, uint32_t n, typename G<true, 0>::T *out,
                                  cudaStream_t s, Extra... extra)
{
    const bool even = ((first + head_elems<typename G<true, 0>::T>(out, n)) & 1u) == 0u;
    switch (below64_mode(a) + (even ? 0u : 3u)) {
    case 0: return launch_fill(G<true, 0>{a, extra...}, out, first, n, s);
    case 1: return launch_fill(G<true, 1>{a, extra...}, out, first, n, s);
    case 2: return launch_fill(G<true, 2>{a, extra...}, out, first, n, s);
    case 3: return launch_fill(G<false, 0>{a, extra...}, out, first, n, s);
    case 4: return launch_fill(G<false, 1>{a, extra...}, out, first, n, s);
    default: return launch_fill(G<false, 2>{a, extra...}, out, first, n, s);
    }
}

}  // namespace

cudaError_t launch_fill_u32_below(const Below32Args &a, uint32_t first, uint32_t n, uint32_t *out,
                                  cudaStream_t s)
{
    return launch_fill(GenBelow32{a}, out, first, n, s);
}

cudaError_t launch_fill_u64_below(const Below64Args &a, uint32_t first, uint32_t n, uint64_t *out,
                                  cudaStream_t s)
{
    return launch_below64_family<GenBelow64>(a, first, n, out, s);
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
    return launch_below64_family<GenI64Range>(a, first, n, out, s, low);
}

}  // namespace rngk
