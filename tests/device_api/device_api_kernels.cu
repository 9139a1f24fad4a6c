// Kernels written against the public device header only (as a user's fused
// kernel would be), exported with C launchers for the device API tests.
#include <cstdint>

#include "rng_device.cuh"

namespace {

__global__ void draw_kernel(uint32_t seed, uint32_t first, uint32_t n, uint32_t *d32, uint64_t *d64, float *u,
                            float *z)
{
    const lowbias32::Key k = lowbias32::make_key(seed);
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const uint32_t c = first + i;
        d32[i] = lowbias32::draw32(k, c);
        d64[i] = lowbias32::draw64(k, c);
        u[i] = lowbias32::uniform(k, c);
        z[i] = lowbias32::randn(k, c);
    }
}

// The Phobos page's dropout_rows: R rows of 256 columns per block, the
// counter of element (r, col) its flat index (r0 + r) * 256 + col.
template <int R>
__global__ void dropout_rows_kernel(const float *x, float *y, uint32_t rows, lowbias32::Dropout d)
{
    const uint32_t r0 = blockIdx.x * R;
    const uint32_t col = threadIdx.x;  // 256 threads, one column each
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const uint32_t row = r0 + r;
        if (row < rows) {
            const uint32_t c = row * 256u + col;
            y[c] = lowbias32::dropout(d, x[c], c);
        }
    }
}

}  // namespace

extern "C" int device_api_draws(uint32_t seed, uint32_t first, uint32_t n, uint32_t *d32, uint64_t *d64, float *u,
                                float *z)
{
    draw_kernel<<<256, 256>>>(seed, first, n, d32, d64, u, z);
    return static_cast<int>(cudaDeviceSynchronize());
}

extern "C" int device_api_dropout_rows(const float *x, float *y, uint32_t rows, uint32_t seed, float p)
{
    const lowbias32::Dropout d = lowbias32::make_dropout(seed, p);
    dropout_rows_kernel<16><<<(rows + 15u) / 16u, 256>>>(x, y, rows, d);
    return static_cast<int>(cudaDeviceSynchronize());
}

extern "C" uint32_t device_api_host_hash32(uint32_t x) { return lowbias32::hash32(x); }
