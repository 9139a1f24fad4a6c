// fill_kernel.cuh -- the streaming fill kernel shared by every counter fill.
//
// Element i of a piece holds gen(first + i).  The output is cut into a head
// of fewer than 16/sizeof(T) elements up to its first 16-byte boundary, a
// body of whole 16-byte vectors and a ragged tail.  Each thread of the body
// computes one vector's elements in registers and writes them with one
// 16-byte store, so the 32 lanes of a warp write 512 contiguous bytes (four
// full 128-byte lines) per store instruction whatever the element type and
// whatever the first counter: with a stateless hash each element's counter
// costs nothing, only the output address decides alignment.
//
// Block b owns the contiguous run of kFillThreads x kVpt vectors starting at
// vector b kFillThreads kVpt, thread t its vectors t, t + kFillThreads, ...;
// the grid covers the body once (no grid-stride loop).  On GB300 this shape
// writes at about 7.7 TB/s, where a persistent grid (8 blocks per SM)
// striding over the same output reaches about 6.5 TB/s.
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

// Vectors per thread: kFillVectorsPerThread independent vectors (and hash
// chains) per thread, unless a generator declares its own
// `static constexpr uint32_t kVectorsPerThread`.
template <class Gen, class = void>
struct VectorsPerThread {
    static constexpr uint32_t value = kFillVectorsPerThread;
};
template <class Gen>
struct VectorsPerThread<Gen, decltype(void(Gen::kVectorsPerThread))> {
    static constexpr uint32_t value = Gen::kVectorsPerThread;
};

// Blocks of a chunked kernel over n_vec vectors, vpt per thread (at least one
// block, which also peels the head and the tail).
inline unsigned chunk_blocks(uint32_t n_vec, uint32_t vpt)
{
    const uint32_t per_block = kFillThreads * vpt;
    const uint32_t need = n_vec / per_block + (n_vec % per_block != 0u);
    return need == 0 ? 1u : need;
}

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

// Blocks per SM a generator asks the compiler to fit, which sets its register
// budget (`static constexpr int kMinBlocksPerSm`; default 0, no hint).
template <class Gen, class = void>
struct MinBlocksPerSm {
    static constexpr int value = 0;
};
template <class Gen>
struct MinBlocksPerSm<Gen, decltype(void(Gen::kMinBlocksPerSm))> {
    static constexpr int value = Gen::kMinBlocksPerSm;
};

template <class Gen>
__global__ void __launch_bounds__(kFillThreads, MinBlocksPerSm<Gen>::value)
fill_kernel(Gen gen, typename Gen::T *__restrict__ out, uint32_t first, uint32_t head, uint32_t n_vec,
            uint32_t n)
{
    using T = typename Gen::T;
    constexpr uint32_t kPer = Vec16<T>::kPer;
    constexpr uint32_t kVpt = VectorsPerThread<Gen>::value;
    const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x;

    const uint32_t tail0 = head + n_vec * kPer;
    if (tid < head) out[tid] = gen(first + tid);
    if (tid < n - tail0) out[tail0 + tid] = gen(first + tail0 + tid);

    T *body = out + head;
    const uint32_t c0 = first + head;
    const uint32_t block0 = blockIdx.x * (kFillThreads * kVpt);
    const uint32_t v0 = block0 + threadIdx.x;
    // block0 <= n_vec for every block of chunk_blocks' grid, so no wrap
    if (n_vec - block0 >= kFillThreads * kVpt) {
        Vec16<T> x[kVpt];
#pragma unroll
        for (uint32_t j = 0; j < kVpt; ++j) x[j] = gen_vec(gen, c0 + (v0 + j * kFillThreads) * kPer);
#pragma unroll
        for (uint32_t j = 0; j < kVpt; ++j) store16(body + (v0 + j * kFillThreads) * kPer, x[j]);
    } else {
#pragma unroll
        for (uint32_t j = 0; j < kVpt; ++j) {
            const uint32_t v = v0 + j * kFillThreads;
            if (v < n_vec) store16(body + v * kPer, gen_vec(gen, c0 + v * kPer));
        }
    }
}

// Launch one piece of n elements (n <= kChunk).
template <class Gen>
cudaError_t launch_fill(const Gen &gen, typename Gen::T *out, uint32_t first, uint32_t n, cudaStream_t s)
{
    using T = typename Gen::T;
    const uint32_t head = head_elems<T>(out, n);
    const uint32_t n_vec = (n - head) / Vec16<T>::kPer;
    fill_kernel<Gen><<<chunk_blocks(n_vec, VectorsPerThread<Gen>::value), kFillThreads, 0, s>>>(gen, out, first, head, n_vec, n);
    note_launch();
    return cudaGetLastError();
}

}  // namespace rngk
