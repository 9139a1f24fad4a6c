// dropout.cu -- fused dropout forward and backward.
//
// Phobos stdlib "Random numbers", section dropout: where(uniform(seed, c) >=
// p, x / (1 - p), 0) with c the element's flat index; the backward pass
// redraws the same mask from the same seed and counters instead of storing
// it, so one kernel serves both directions.
//
// uniform(seed, c) >= p  <=>  (D32 & 0x7FFFFF) >= T with T = ceil(p 2^23):
// the uniform is exactly m 2^-23 and p 2^23 is exact in binary64, so the
// integer compare (threshold from the host) decides exactly as the f32
// compare.  The kept value is the IEEE quotient x / (1 - p) (__fdiv_rn) with
// 1 - p rounded to f32 on the host.  Dropped elements are +0.  The element
// function is lowbias32::dropout of include/rng_device.cuh.
//
// When x and y share their offset within 16 bytes, every thread moves one
// 16-byte vector in and one out (warps read and write 512 contiguous bytes);
// otherwise a scalar grid-stride kernel keeps both sides coalesced.  x == y
// (in place) is fine: each element is read before it is written by the same
// thread, so neither pointer is declared __restrict__.
#include "fill_kernel.cuh"
#include "hash32.cuh"

namespace rngk {
namespace {

__device__ __forceinline__ float drop(float x, uint32_t key, uint32_t threshold, float divisor, uint32_t c)
{
    return lowbias32::dropout(lowbias32::Dropout{lowbias32::Key{key}, threshold, divisor}, x, c);
}

__global__ void __launch_bounds__(kFillThreads)
dropout_vec_kernel(const float *x, float *y, uint32_t key, uint32_t threshold, float divisor, uint32_t first,
                   uint32_t head, uint32_t n_vec, uint32_t n)
{
    const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t stride = gridDim.x * blockDim.x;
    const uint32_t tail0 = head + n_vec * 4u;
    if (tid < head) y[tid] = drop(x[tid], key, threshold, divisor, first + tid);
    if (tid < n - tail0) y[tail0 + tid] = drop(x[tail0 + tid], key, threshold, divisor, first + tail0 + tid);

    const float4 *xv = reinterpret_cast<const float4 *>(x + head);
    float4 *yv = reinterpret_cast<float4 *>(y + head);
    const uint32_t c0 = first + head;
    for (uint32_t v = tid; v < n_vec; v += stride) {
        const float4 a = __ldcs(xv + v);
        const uint32_t c = c0 + 4u * v;
        float4 b;
        b.x = drop(a.x, key, threshold, divisor, c);
        b.y = drop(a.y, key, threshold, divisor, c + 1u);
        b.z = drop(a.z, key, threshold, divisor, c + 2u);
        b.w = drop(a.w, key, threshold, divisor, c + 3u);
        __stcs(yv + v, b);
    }
}

__global__ void __launch_bounds__(kFillThreads)
dropout_scalar_kernel(const float *x, float *y, uint32_t key, uint32_t threshold, float divisor,
                      uint32_t first, uint32_t n)
{
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        y[i] = drop(__ldcs(x + i), key, threshold, divisor, first + i);
}

}  // namespace

cudaError_t launch_dropout(const float *x, float *y, uint32_t key, uint32_t threshold, float divisor,
                           uint32_t first, uint32_t n, cudaStream_t s)
{
    const uintptr_t ax = reinterpret_cast<uintptr_t>(x), ay = reinterpret_cast<uintptr_t>(y);
    if ((ax & 15u) == (ay & 15u)) {
        const uint32_t head = head_elems<float>(y, n);
        const uint32_t n_vec = (n - head) / 4u;
        dropout_vec_kernel<<<fill_blocks(n_vec), kFillThreads, 0, s>>>(x, y, key, threshold, divisor, first,
                                                                       head, n_vec, n);
    } else {
        dropout_scalar_kernel<<<fill_blocks((n + 3u) / 4u), kFillThreads, 0, s>>>(x, y, key, threshold,
                                                                                  divisor, first, n);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace rngk
