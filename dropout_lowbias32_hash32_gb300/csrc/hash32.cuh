// hash32.cuh -- device side of the lowbias32 counter-based generator.
//
// Phobos stdlib, "Random numbers", section hash32: lowbias32 in wrapping
// 32-bit arithmetic, multipliers 2146121005 (0x7FEB352D) and -2073254261
// (0x846CA68B as a bit pattern), logical xorshifts by 16, 15 and 16.
// Section uniform: a value is hash32(counter ^ hash32(seed)); the seed's hash
// (the "key") is computed once on the host and passed to every kernel.
#pragma once

#include <cstdint>

namespace rngk {

__host__ __device__ __forceinline__ uint32_t hash32(uint32_t x)
{
    x ^= x >> 16;
    x *= 0x7FEB352Du;
    x ^= x >> 15;
    x *= 0x846CA68Bu;
    x ^= x >> 16;
    return x;
}

// The 32-bit draw at counter c under a seed whose hash is `key`.
__device__ __forceinline__ uint32_t draw32(uint32_t key, uint32_t c) { return hash32(c ^ key); }

// The 64-bit draw at counter c: draws at 2c (high word) and 2c + 1 (low word).
// 2c is even, so (2c + 1) ^ key == (2c ^ key) ^ 1.
__device__ __forceinline__ uint64_t draw64(uint32_t key, uint32_t c)
{
    const uint32_t a = (c << 1) ^ key;
    return (static_cast<uint64_t>(hash32(a)) << 32) | hash32(a ^ 1u);
}

// Substream of one element for retries and ziggurat misses: element key
// hash32(c ^ purpose_key) with purpose_key = hash32(hash32(seed) ^ P) from
// the host; word k is hash32(k ^ element key).
__device__ __forceinline__ uint32_t substream_key(uint32_t purpose_key, uint32_t c)
{
    return hash32(c ^ purpose_key);
}

__device__ __forceinline__ uint32_t substream32(uint32_t skey, uint32_t k) { return hash32(k ^ skey); }

__device__ __forceinline__ uint64_t substream64(uint32_t skey, uint32_t k)
{
    return (static_cast<uint64_t>(hash32((k << 1) ^ skey)) << 32) | hash32(((k << 1) | 1u) ^ skey);
}

}  // namespace rngk
