// fill_narrow.cu -- u8, u16, bool and f16 fills (narrow outputs).
//
// tandem-cuda "Performance", rows fill_u16, fill_f16_bits, fill_u8 and
// fill_bool (one byte per bit), restated on hash32: every element remains a
// pure function of (seed, its counter c), and one 32-bit draw serves several
// consecutive counters.
//   u8:   byte c & 3 of draw32(seed, c >> 2)      (bits 8(c & 3) .. +7)
//   u16:  halfword c & 1 of draw32(seed, c >> 1)  (bits 16(c & 1) .. +15)
//   bool: bit c & 31 of draw32(seed, c >> 5), stored as a byte 0 or 1
//   f16:  the u16 element's low 10 bits m as the binary16 value m 2^-10, a
//         uniform on the 2^-10 grid in [0, 1) (bits of the exact half)
// The word index wraps with the counter (c >> 2 is taken mod 2^30, etc.).
// A 16-byte vector is assembled from the few words it spans with funnel
// shifts, so the fills hash 1/4, 1/2 and 1/32 of a word per output.
#include <cuda_fp16.h>

#include "fill_kernel.cuh"
#include "hash32.cuh"

namespace rngk {
namespace {

struct GenU8 {
    using T = uint8_t;
    uint32_t key;
    __device__ T operator()(uint32_t c) const
    {
        return static_cast<uint8_t>(draw32(key, (c >> 2) & 0x3FFFFFFFu) >> (8u * (c & 3u)));
    }
    // 16 bytes at counters c0 .. c0 + 15 from the 4 or 5 words they span
    __device__ Vec16<uint8_t> vec(uint32_t c0) const
    {
        const uint32_t w0 = c0 >> 2, shift = 8u * (c0 & 3u);
        uint32_t w[5];
#pragma unroll
        for (uint32_t k = 0; k < 4; ++k) w[k] = draw32(key, (w0 + k) & 0x3FFFFFFFu);
        // the fifth word only for a start inside a word (the same for every
        // vector of a launch)
        w[4] = shift ? draw32(key, (w0 + 4u) & 0x3FFFFFFFu) : 0u;
        uint4 u;
        u.x = __funnelshift_r(w[0], w[1], shift);
        u.y = __funnelshift_r(w[1], w[2], shift);
        u.z = __funnelshift_r(w[2], w[3], shift);
        u.w = __funnelshift_r(w[3], w[4], shift);
        Vec16<uint8_t> x;
        memcpy(&x, &u, sizeof u);
        return x;
    }
};

__device__ __forceinline__ uint4 halfwords(uint32_t key, uint32_t c0)
{
    // 8 halfwords at counters c0 .. c0 + 7 from the 4 or 5 words they span
    const uint32_t w0 = c0 >> 1, shift = 16u * (c0 & 1u);
    uint32_t w[5];
#pragma unroll
    for (uint32_t k = 0; k < 4; ++k) w[k] = draw32(key, (w0 + k) & 0x7FFFFFFFu);
    w[4] = shift ? draw32(key, (w0 + 4u) & 0x7FFFFFFFu) : 0u;
    return make_uint4(__funnelshift_r(w[0], w[1], shift), __funnelshift_r(w[1], w[2], shift),
                      __funnelshift_r(w[2], w[3], shift), __funnelshift_r(w[3], w[4], shift));
}

struct GenU16 {
    using T = uint16_t;
    uint32_t key;
    __device__ T operator()(uint32_t c) const
    {
        return static_cast<uint16_t>(draw32(key, (c >> 1) & 0x7FFFFFFFu) >> (16u * (c & 1u)));
    }
    __device__ Vec16<uint16_t> vec(uint32_t c0) const
    {
        const uint4 u = halfwords(key, c0);
        Vec16<uint16_t> x;
        memcpy(&x, &u, sizeof u);
        return x;
    }
};

// m 2^-10 as binary16 bits: (1 + m 2^-10) - 1 in half arithmetic, exact
// (the operands are within a factor two); two lanes per instruction.
__device__ __forceinline__ uint32_t f16_pair(uint32_t two_halfwords)
{
    const uint32_t ones_plus = (two_halfwords & 0x03FF03FFu) | 0x3C003C00u;
    __half2 h;
    memcpy(&h, &ones_plus, sizeof h);
    const __half2 r = __hsub2(h, __floats2half2_rn(1.0f, 1.0f));
    uint32_t bits;
    memcpy(&bits, &r, sizeof bits);
    return bits;
}

struct GenF16 {
    using T = uint16_t;
    static constexpr uint32_t kVectorsPerThread = kHeavyVectorsPerThread;
    uint32_t key;
    __device__ T operator()(uint32_t c) const
    {
        const uint32_t h = draw32(key, (c >> 1) & 0x7FFFFFFFu) >> (16u * (c & 1u));
        return static_cast<uint16_t>(f16_pair(h & 0xFFFFu));
    }
    __device__ Vec16<uint16_t> vec(uint32_t c0) const
    {
        const uint4 u = halfwords(key, c0);
        const uint4 f = make_uint4(f16_pair(u.x), f16_pair(u.y), f16_pair(u.z), f16_pair(u.w));
        Vec16<uint16_t> x;
        memcpy(&x, &f, sizeof f);
        return x;
    }
};

// four bits (the low nibble of n) spread to the low bit of four bytes
__device__ __forceinline__ uint32_t spread_nibble(uint32_t n) { return ((n & 0xFu) * 0x00204081u) & 0x01010101u; }

struct GenBool {
    using T = uint8_t;
    uint32_t key;
    __device__ T operator()(uint32_t c) const
    {
        return static_cast<uint8_t>((draw32(key, (c >> 5) & 0x07FFFFFFu) >> (c & 31u)) & 1u);
    }
    // 16 bits starting at bit c0 & 31 of word c0 >> 5, spanning two words
    __device__ Vec16<uint8_t> vec(uint32_t c0) const
    {
        const uint32_t w0 = c0 >> 5;
        const uint32_t lo = draw32(key, w0 & 0x07FFFFFFu), hi = draw32(key, (w0 + 1u) & 0x07FFFFFFu);
        const uint32_t bits = __funnelshift_r(lo, hi, c0 & 31u);
        const uint4 u = make_uint4(spread_nibble(bits), spread_nibble(bits >> 4), spread_nibble(bits >> 8),
                                   spread_nibble(bits >> 12));
        Vec16<uint8_t> x;
        memcpy(&x, &u, sizeof u);
        return x;
    }
};

}  // namespace

cudaError_t launch_fill_u8(uint32_t key, uint32_t first, uint32_t n, uint8_t *out, cudaStream_t s)
{
    return launch_fill(GenU8{key}, out, first, n, s);
}

cudaError_t launch_fill_u16(uint32_t key, uint32_t first, uint32_t n, uint16_t *out, cudaStream_t s)
{
    return launch_fill(GenU16{key}, out, first, n, s);
}

cudaError_t launch_fill_f16(uint32_t key, uint32_t first, uint32_t n, uint16_t *out, cudaStream_t s)
{
    return launch_fill(GenF16{key}, out, first, n, s);
}

cudaError_t launch_fill_bool(uint32_t key, uint32_t first, uint32_t n, uint8_t *out, cudaStream_t s)
{
    return launch_fill(GenBool{key}, out, first, n, s);
}

}  // namespace rngk
