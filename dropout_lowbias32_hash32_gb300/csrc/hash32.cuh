// hash32.cuh -- device side of the lowbias32 counter-based generator.
//
// Phobos stdlib, "Random numbers", section hash32: lowbias32 in wrapping
// 32-bit arithmetic, multipliers 2146121005 (0x7FEB352D) and -2073254261
// (0x846CA68B as a bit pattern), logical xorshifts by 16, 15 and 16.
// Section uniform: a value is hash32(counter ^ hash32(seed)).
//
// The seed's hash (the key) enters only through the first xorshift:
//   (c ^ k) ^ ((c ^ k) >> 16) = c ^ (c >> 16) ^ (k ^ (k >> 16)),
// so the host folds the key once, kf = k ^ (k >> 16), and each draw costs
// one shift and one three-input xor before the two multiply-xorshift rounds.
#pragma once

#include <cstdint>

namespace rngk {

// hash32 after its first xorshift.
__host__ __device__ __forceinline__ uint32_t hash32_rounds(uint32_t x)
{
    x *= 0x7FEB352Du;
    x ^= x >> 15;
    x *= 0x846CA68Bu;
    x ^= x >> 16;
    return x;
}

__host__ __device__ __forceinline__ uint32_t hash32(uint32_t x) { return hash32_rounds(x ^ (x >> 16)); }

// The key k folded into the first xorshift of hash32(c ^ k).
__host__ __device__ __forceinline__ uint32_t fold_key(uint32_t k) { return k ^ (k >> 16); }

// hash32(c ^ k) from the folded key kf.
__device__ __forceinline__ uint32_t hash32_keyed(uint32_t kf, uint32_t c) { return hash32_rounds(c ^ (c >> 16) ^ kf); }

// The 32-bit draw at counter c (kf: the folded hash of the seed).
__device__ __forceinline__ uint32_t draw32(uint32_t kf, uint32_t c) { return hash32_keyed(kf, c); }

// The two words of the 64-bit draw at counter c: the draws at 2c (high) and
// 2c + 1 (low).  2c + 1 = 2c ^ 1, and bit 0 does not reach the shifted term,
// so the low word's first xorshift is the high word's with bit 0 flipped.
struct Words {
    uint32_t hi, lo;
};

__device__ __forceinline__ Words draw64_words(uint32_t kf, uint32_t c)
{
    const uint32_t a = c << 1;
    const uint32_t first = a ^ (a >> 16) ^ kf;
    return Words{hash32_rounds(first), hash32_rounds(first ^ 1u)};
}

__device__ __forceinline__ uint64_t draw64(uint32_t kf, uint32_t c)
{
    const Words w = draw64_words(kf, c);
    return (static_cast<uint64_t>(w.hi) << 32) | w.lo;
}

// Substream of one element for retries and ziggurat misses: element key
// hash32(c ^ purpose_key) with purpose_key = hash32(hash32(seed) ^ P) from
// the host (passed folded); word k is hash32(k ^ element key).
__device__ __forceinline__ uint32_t substream_key(uint32_t purpose_kf, uint32_t c)
{
    return hash32_keyed(purpose_kf, c);
}

__device__ __forceinline__ uint32_t substream32(uint32_t skey, uint32_t k) { return hash32(k ^ skey); }

__device__ __forceinline__ uint64_t substream64(uint32_t skey, uint32_t k)
{
    return (static_cast<uint64_t>(hash32((k << 1) ^ skey)) << 32) | hash32(((k << 1) | 1u) ^ skey);
}

}  // namespace rngk
