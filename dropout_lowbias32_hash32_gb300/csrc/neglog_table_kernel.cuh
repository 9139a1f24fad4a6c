// neglog_table_kernel.cuh -- the chunked fill kernel for generators that
// gather rows of the own binary32 logarithm's table
// (lowbias32::detail::kNegLogTable, 257 rows of 16 bytes), with that table
// staged in shared memory.
//
// Through L1 the 16-byte gather of 32 random rows of the 4 KiB table takes
// about one wavefront per distinct line (the f32 exponential kept L1 93 %
// busy).  Each block here stages kNegLogCopies copies of the rows, copy q in
// 16-byte bank group q (row j of copy q at index 8 j + q), and lane l reads
// copy l mod 8, so every quarter-warp phase of a gather hits 8 distinct bank
// groups: 4 wavefronts per warp.  The generator computes a vector with
// `gen.vec(c0, load)` and an element with `gen(c, load)`, load(j) returning
// row j; otherwise the launch shape, the head and tail peel and the stores
// are fill_kernel's (fill_kernel.cuh).
#pragma once

#include "fill_kernel.cuh"
#include "rng_device.cuh"

namespace rngk {

constexpr uint32_t kNegLogRows = 257;
constexpr uint32_t kNegLogCopies = 8;

// Gen::kVectorsPerThread vectors per thread (amortising the 32 KiB staging),
// Gen::kMinBlocksPerSm as the launch bound's register budget.
template <class Gen>
__global__ void __launch_bounds__(kFillThreads, Gen::kMinBlocksPerSm)
neglog_table_kernel(Gen gen, typename Gen::T *__restrict__ out, uint32_t first, uint32_t head, uint32_t n_vec,
                    uint32_t n)
{
    using T = typename Gen::T;
    constexpr uint32_t kPer = Vec16<T>::kPer;
    constexpr uint32_t kVpt = Gen::kVectorsPerThread;
    __shared__ float4 table[kNegLogRows * kNegLogCopies];
    for (uint32_t i = threadIdx.x; i < kNegLogRows * kNegLogCopies; i += kFillThreads)
        table[i] = __ldg(&lowbias32::detail::kNegLogTable[i / kNegLogCopies]);
    __syncthreads();
    const float4 *copy = table + (threadIdx.x & (kNegLogCopies - 1u));
    const auto load = [copy](uint32_t j) { return copy[j * kNegLogCopies]; };

    const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t tail0 = head + n_vec * kPer;
    if (tid < head) out[tid] = gen(first + tid, load);
    if (tid < n - tail0) out[tail0 + tid] = gen(first + tail0 + tid, load);
    T *body = out + head;
    const uint32_t c0 = first + head;
    const uint32_t block0 = blockIdx.x * (kFillThreads * kVpt);
    const uint32_t v0 = block0 + threadIdx.x;
    if (n_vec - block0 >= kFillThreads * kVpt) {
        Vec16<T> x[kVpt];
#pragma unroll
        for (uint32_t j = 0; j < kVpt; ++j) x[j] = gen.vec(c0 + (v0 + j * kFillThreads) * kPer, load);
#pragma unroll
        for (uint32_t j = 0; j < kVpt; ++j) store16(body + (v0 + j * kFillThreads) * kPer, x[j]);
    } else {
#pragma unroll
        for (uint32_t j = 0; j < kVpt; ++j) {
            const uint32_t v = v0 + j * kFillThreads;
            if (v < n_vec) store16(body + v * kPer, gen.vec(c0 + v * kPer, load));
        }
    }
}

template <class Gen>
cudaError_t launch_neglog_table_fill(const Gen &gen, typename Gen::T *out, uint32_t first, uint32_t n, cudaStream_t s)
{
    using T = typename Gen::T;
    const uint32_t head = head_elems<T>(out, n);
    const uint32_t n_vec = (n - head) / Vec16<T>::kPer;
    neglog_table_kernel<Gen><<<chunk_blocks(n_vec, Gen::kVectorsPerThread), kFillThreads, 0, s>>>(gen, out, first, head,
                                                                                                  n_vec, n);
    note_launch();
    return cudaGetLastError();
}

}  // namespace rngk
