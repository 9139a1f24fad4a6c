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
// When x and y share their offset within 32 bytes, a kernel of 32-byte
// accesses runs (below).  Otherwise, when they share it within 16 bytes,
// every thread moves kFillVectorsPerThread 16-byte vectors in and out (warps
// read and write 512 contiguous bytes per instruction; block b owns the b-th
// contiguous run of kFillThreads x kFillVectorsPerThread vectors, its loads
// issued before its stores); otherwise a scalar kernel of the same chunked
// shape keeps both sides coalesced.  x == y (in place) is fine: each element
// is read before it is written by the same thread, so neither pointer is
// declared __restrict__.
#include "fill_kernel.cuh"
#include "hash32.cuh"

namespace rngk {
namespace {

__device__ __forceinline__ float drop(float x, uint32_t key, uint32_t threshold, float divisor, uint32_t c)
{
    return lowbias32::dropout(lowbias32::Dropout{lowbias32::Key{key}, threshold, divisor}, x, c);
}

__device__ __forceinline__ float4 drop4(float4 a, uint32_t key, uint32_t threshold, float divisor, uint32_t c)
{
    return make_float4(drop(a.x, key, threshold, divisor, c), drop(a.y, key, threshold, divisor, c + 1u),
                       drop(a.z, key, threshold, divisor, c + 2u), drop(a.w, key, threshold, divisor, c + 3u));
}

constexpr uint32_t kVpt = kFillVectorsPerThread;
// elements per thread of the scalar kernel (the same bytes per block as the
// vector kernel)
constexpr uint32_t kEpt = 4u * kFillVectorsPerThread;

__global__ void __launch_bounds__(kFillThreads)
dropout_vec_kernel(const float *x, float *y, uint32_t key, uint32_t threshold, float divisor, uint32_t first,
                   uint32_t head, uint32_t n_vec, uint32_t n)
{
    const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t tail0 = head + n_vec * 4u;
    if (tid < head) y[tid] = drop(x[tid], key, threshold, divisor, first + tid);
    if (tid < n - tail0) y[tail0 + tid] = drop(x[tail0 + tid], key, threshold, divisor, first + tail0 + tid);

    const float4 *xv = reinterpret_cast<const float4 *>(x + head);
    float4 *yv = reinterpret_cast<float4 *>(y + head);
    const uint32_t c0 = first + head;
    const uint32_t block0 = blockIdx.x * (kFillThreads * kVpt);
    const uint32_t v0 = block0 + threadIdx.x;
    // block0 <= n_vec for every block of chunk_blocks' grid, so no wrap
    if (n_vec - block0 >= kFillThreads * kVpt) {
        float4 a[kVpt];
#pragma unroll
        for (uint32_t j = 0; j < kVpt; ++j) a[j] = __ldcs(xv + v0 + j * kFillThreads);
#pragma unroll
        for (uint32_t j = 0; j < kVpt; ++j) {
            const uint32_t v = v0 + j * kFillThreads;
            __stcs(yv + v, drop4(a[j], key, threshold, divisor, c0 + 4u * v));
        }
    } else {
#pragma unroll
        for (uint32_t j = 0; j < kVpt; ++j) {
            const uint32_t v = v0 + j * kFillThreads;
            if (v < n_vec) __stcs(yv + v, drop4(__ldcs(xv + v), key, threshold, divisor, c0 + 4u * v));
        }
    }
}

// When x and y share their offset within 32 bytes: 32-byte accesses
// (ld/st.global.v8.f32, sm_100 and later), one per thread, so a warp moves
// 1 KiB per instruction; block b owns the b-th run of kFillThreads 32-byte
// vectors.  About 1.3 % faster at 2^28 than the 16-byte kernel (one A/B on
// one GB300).  Head and tail (fewer than 8 elements each) are scalar.
__global__ void __launch_bounds__(kFillThreads)
dropout_v8_kernel(const float *x, float *y, uint32_t key, uint32_t threshold, float divisor, uint32_t first,
                  uint32_t head, uint32_t n_vec, uint32_t n)
{
    const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t tail0 = head + n_vec * 8u;
    if (tid < head) y[tid] = drop(x[tid], key, threshold, divisor, first + tid);
    if (tid < n - tail0) y[tail0 + tid] = drop(x[tail0 + tid], key, threshold, divisor, first + tail0 + tid);
    if (tid >= n_vec) return;
    const uint32_t e = head + 8u * tid;
    float a[8];
    asm volatile("ld.global.L1::no_allocate.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=f"(a[0]), "=f"(a[1]), "=f"(a[2]), "=f"(a[3]), "=f"(a[4]), "=f"(a[5]), "=f"(a[6]), "=f"(a[7])
                 : "l"(x + e));
    float o[8];
#pragma unroll
    for (uint32_t k = 0; k < 8; ++k) o[k] = drop(a[k], key, threshold, divisor, first + e + k);
    asm volatile("st.global.L1::no_allocate.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 :: "l"(y + e), "f"(o[0]), "f"(o[1]), "f"(o[2]), "f"(o[3]), "f"(o[4]), "f"(o[5]), "f"(o[6]), "f"(o[7])
                 : "memory");
}

__global__ void __launch_bounds__(kFillThreads)
dropout_scalar_kernel(const float *x, float *y, uint32_t key, uint32_t threshold, float divisor,
                      uint32_t first, uint32_t n)
{
    const uint32_t block0 = blockIdx.x * (kFillThreads * kEpt);
    const uint32_t i0 = block0 + threadIdx.x;
    // block0 <= n for every block of chunk_blocks' grid, so no wrap
    if (n - block0 >= kFillThreads * kEpt) {
        float a[kEpt];
#pragma unroll
        for (uint32_t j = 0; j < kEpt; ++j) a[j] = __ldcs(x + i0 + j * kFillThreads);
#pragma unroll
        for (uint32_t j = 0; j < kEpt; ++j) {
            const uint32_t i = i0 + j * kFillThreads;
            y[i] = drop(a[j], key, threshold, divisor, first + i);
        }
    } else {
#pragma unroll
        for (uint32_t j = 0; j < kEpt; ++j) {
            const uint32_t i = i0 + j * kFillThreads;
            if (i < n) y[i] = drop(__ldcs(x + i), key, threshold, divisor, first + i);
        }
    }
}

}  // namespace

cudaError_t launch_dropout(const float *x, float *y, uint32_t key, uint32_t threshold, float divisor,
                           uint32_t first, uint32_t n, cudaStream_t s)
{
    const uintptr_t ax = reinterpret_cast<uintptr_t>(x), ay = reinterpret_cast<uintptr_t>(y);
    if ((ax & 31u) == (ay & 31u)) {
        // elements before y's first 32-byte boundary (y is 4-byte aligned)
        const uint32_t h = static_cast<uint32_t>(((32u - (ay & 31u)) & 31u) / 4u);
        const uint32_t head = h < n ? h : n;
        const uint32_t n_vec = (n - head) / 8u;
        const uint32_t threads = n_vec > 8u ? n_vec : 8u;  // at least the head's and tail's 8 threads
        dropout_v8_kernel<<<(threads + kFillThreads - 1u) / kFillThreads, kFillThreads, 0, s>>>(
            x, y, key, threshold, divisor, first, head, n_vec, n);
    } else if ((ax & 15u) == (ay & 15u)) {
        const uint32_t head = head_elems<float>(y, n);
        const uint32_t n_vec = (n - head) / 4u;
        dropout_vec_kernel<<<chunk_blocks(n_vec, kVpt), kFillThreads, 0, s>>>(x, y, key, threshold, divisor, first,
                                                                       head, n_vec, n);
    } else {
        dropout_scalar_kernel<<<chunk_blocks(n, kEpt), kFillThreads, 0, s>>>(x, y, key, threshold, divisor,
                                                                              first, n);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace rngk
