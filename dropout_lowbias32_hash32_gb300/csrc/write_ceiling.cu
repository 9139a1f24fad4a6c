// write_ceiling.cu -- a measurement aid: the plainest 16-byte store kernel,
// in the same launch shape as the fills (block b owns the b-th run of
// kFillThreads x kFillVectorsPerThread vectors), writing no random numbers.
// Its bandwidth and cudaMemsetAsync's are the write ceiling the fills are
// compared with (rng_debug_write_ceiling).
#include "fill_kernel.cuh"

namespace rngk {
namespace {

__global__ void __launch_bounds__(kFillThreads) store_ceiling_kernel(uint4 *__restrict__ out, uint32_t n_vec)
{
    const uint32_t block0 = blockIdx.x * (kFillThreads * kFillVectorsPerThread);
#pragma unroll
    for (uint32_t j = 0; j < kFillVectorsPerThread; ++j) {
        const uint32_t v = block0 + j * kFillThreads + threadIdx.x;
        if (v < n_vec) __stcs(out + v, make_uint4(v, v, v, v));
    }
}

}  // namespace

cudaError_t launch_store_ceiling(uint4 *out, uint32_t n_vec, cudaStream_t s)
{
    store_ceiling_kernel<<<chunk_blocks(n_vec, kFillVectorsPerThread), kFillThreads, 0, s>>>(out, n_vec);
    note_launch();
    return cudaGetLastError();
}

}  // namespace rngk
