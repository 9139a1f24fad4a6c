// hash32.cuh -- the library kernels' draw helpers beyond the public device
// header (include/rng_device.cuh): adapters that take the seed's folded key
// as a plain 32-bit kernel argument, the substreams of bounded retries and
// ziggurat misses, the paired 64-bit draws of an even counter, and the
// multiply-adds that keep shifts off the ALU pipe.
#pragma once

#include <cstdint>

#include "rng_device.cuh"

namespace rngk {

using lowbias32::hash32;
using lowbias32::Words;

// The key k folded into the first xorshift of hash32(c ^ k).
__host__ __device__ __forceinline__ uint32_t fold_key(uint32_t k) { return lowbias32::key_of_hash(k).folded; }

// The 32-bit draw at counter c (kf: the folded hash of the seed).
__device__ __forceinline__ uint32_t draw32(uint32_t kf, uint32_t c) { return lowbias32::draw32(lowbias32::Key{kf}, c); }

// The draws at 2c (hi) and 2c + 1 (lo).
__device__ __forceinline__ Words draw64_words(uint32_t kf, uint32_t c)
{
    return lowbias32::draw64_words(lowbias32::Key{kf}, c);
}

__device__ __forceinline__ uint64_t draw64(uint32_t kf, uint32_t c) { return lowbias32::draw64(lowbias32::Key{kf}, c); }

// d = a b + c (low or high 32 bits of the product) as one multiply-add, on
// the FMA pipe.  A multiplier that is a kernel argument keeps the compiler
// from turning a product by a power of two back into a shift on the ALU pipe:
// mad_hi(x, 2^(32 - s), c) is (x >> s) + c.
__device__ __forceinline__ uint32_t mad_lo(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t mad_hi(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("mad.hi.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// The 64-bit draws at an even counter c and at c + 1: the 32-bit draws at
// 2c .. 2c + 3 differ only in their counter's low two bits, which never reach
// the first xorshift's shifted term, so all four share it (the draw at 2c + k
// starts from the one at 2c ^ k).
__device__ __forceinline__ void draw64_pair_words(uint32_t kf, uint32_t c, Words &a, Words &b)
{
    const uint32_t x = c << 1;
    const uint32_t f = x ^ (x >> 16) ^ kf;
    a = Words{lowbias32::hash32_rounds(f), lowbias32::hash32_rounds(f ^ 1u)};
    b = Words{lowbias32::hash32_rounds(f ^ 2u), lowbias32::hash32_rounds(f ^ 3u)};
}

// Substream of one element for retries and ziggurat misses: element key
// hash32(c ^ purpose_key) with purpose_key = hash32(hash32(seed) ^ P) from
// the host (passed folded); word k is hash32(k ^ element key).
__device__ __forceinline__ uint32_t substream_key(uint32_t purpose_kf, uint32_t c) { return draw32(purpose_kf, c); }

__device__ __forceinline__ uint32_t substream32(uint32_t skey, uint32_t k) { return hash32(k ^ skey); }

__device__ __forceinline__ uint64_t substream64(uint32_t skey, uint32_t k)
{
    return (static_cast<uint64_t>(hash32((k << 1) ^ skey)) << 32) | hash32(((k << 1) | 1u) ^ skey);
}

}  // namespace rngk
