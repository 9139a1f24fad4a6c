// fill_kernel.cuh -- the streaming fill kernel shared by every counter fill.
//
// Element i of a piece holds gen(first + i).  The output is cut into a head
// of fewer than 16/sizeof(T) elements up to its first 16-byte boundary, a
// body of whole 16-byte vectors and a ragged tail.  Each thread of the body
// computes one vector's elements in registers and writes them with one
// 16-byte store, so the 32 lanes of a warp write 512 contiguous bytes (four
// full 128-byte lines) per store instruction whatever the element type and
// whatever the first counter: with a stateless hash each element's counter
// costs nothing, only the output address decides alignment.  The grid is a
// whole number of waves (resident blocks x SMs) striding over the body.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace rngk {

template <class T>
struct Vec16 {
    static constexpr uint32_t kPer = 16 / sizeof(T);
    T v[kPer];
};

// Streaming store of one 16-byte vector (evict-first: the output is written
// once and not re-read by this kernel).
template <class T>
__device__ __forceinline__ void store16(T *p, const Vec16<T> &x)
{
    uint4 u;
    static_assert(sizeof(u) == sizeof(x), "16-byte vector");
    memcpy(&u, &x, sizeof(u));
    __stcs(reinterpret_cast<uint4 *>(p), u);
}

// Vectors a thread computes per loop step: a generator may declare
// `static constexpr uint32_t kVectorsPerStep = 2` to keep twice the
// independent hash chains in flight (the bounded and 64-bit fills, whose
// multiplies have long latencies); the plain draws stay at one, which keeps
// each warp's stores of one step in consecutive lines.
template <class Gen, class = void>
struct VectorsPerStep {
    static constexpr uint32_t value = 1;
};
template <class Gen>
struct VectorsPerStep<Gen, decltype(void(Gen::kVectorsPerStep))> {
    static constexpr uint32_t value = Gen::kVectorsPerStep;
};

// A generator may also compute a whole 16-byte vector at once,
// `Vec16<T> vec(uint32_t c0) const` for the elements at c0 .. c0 + kPer - 1,
// when neighbouring elements share one draw (the paired normals, the narrow
// fills); the kernel then calls it for the body and the per-element
// operator() only for the peeled head and tail.
template <class Gen, class = void>
struct HasVec {
    static constexpr bool value = false;
};
template <class Gen>
struct HasVec<Gen, decltype(void(&Gen::vec))> {
    static constexpr bool value = true;
};

template <class Gen>
__device__ __forceinline__ Vec16<typename Gen::T> gen_vec(const Gen &gen, uint32_t c)
{
    if constexpr (HasVec<Gen>::value) {
        return gen.vec(c);
    } else {
        Vec16<typename Gen::T> x;
#pragma unroll
        for (uint32_t k = 0; k < Vec16<typename Gen::T>::kPer; ++k) x.v[k] = gen(c + k);
        return x;
    }
}

template <class Gen>
__global__ void __launch_bounds__(kFillThreads)
fill_kernel(Gen gen, typename Gen::T *__restrict__ out, uint32_t first, uint32_t head, uint32_t n_vec,
            uint32_t n)
{
    using T = typename Gen::T;
    constexpr uint32_t kPer = Vec16<T>::kPer;
    const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t stride = gridDim.x * blockDim.x;

    const uint32_t tail0 = head + n_vec * kPer;
    if (tid < head) out[tid] = gen(first + tid);
    if (tid < n - tail0) out[tail0 + tid] = gen(first + tail0 + tid);

    T *body = out + head;
    const uint32_t c0 = first + head;
    uint32_t v = tid;
    if (VectorsPerStep<Gen>::value == 2) {
        for (; v + stride < n_vec; v += 2u * stride) {
            const Vec16<T> x = gen_vec(gen, c0 + v * kPer);
            const Vec16<T> y = gen_vec(gen, c0 + (v + stride) * kPer);
            store16(body + v * kPer, x);
            store16(body + (v + stride) * kPer, y);
        }
    }
    for (; v < n_vec; v += stride) store16(body + v * kPer, gen_vec(gen, c0 + v * kPer));
}

// Launch one piece of n elements (n <= kChunk).
template <class Gen>
cudaError_t launch_fill(const Gen &gen, typename Gen::T *out, uint32_t first, uint32_t n, cudaStream_t s)
{
    using T = typename Gen::T;
    const uint32_t head = head_elems<T>(out, n);
    const uint32_t n_vec = (n - head) / Vec16<T>::kPer;
    fill_kernel<Gen><<<fill_blocks(n_vec), kFillThreads, 0, s>>>(gen, out, first, head, n_vec, n);
    note_launch();
    return cudaGetLastError();
}

}  // namespace rngk
