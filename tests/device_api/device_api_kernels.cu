// Kernels written against the public device header only (as a user's fused
// kernel would be), exported with C launchers for the device API tests.
#include <cstdint>

#include "rng_device.cuh"

namespace {

__global__ void draw_kernel(uint32_t seed, uint32_t first, uint32_t n, uint32_t *d32, uint64_t *d64, float *u,
                            float *z, float *ex, float *zp)
{
    const lowbias32::Key k = lowbias32::make_key(seed);
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const uint32_t c = first + i;
        d32[i] = lowbias32::draw32(k, c);
        d64[i] = lowbias32::draw64(k, c);
        u[i] = lowbias32::uniform(k, c);
        z[i] = lowbias32::randn(k, c);
        ex[i] = lowbias32::exponential(k, c);
        zp[i] = lowbias32::randn_precise(k, c);
    }
}

}  // namespace

extern "C" int device_api_draws(uint32_t seed, uint32_t first, uint32_t n, uint32_t *d32, uint64_t *d64, float *u,
                                float *z, float *ex, float *zp)
{
    draw_kernel<<<256, 256>>>(seed, first, n, d32, d64, u, z, ex, zp);
    return static_cast<int>(cudaDeviceSynchronize());
}

// The header's dropout_rows with rows-per-block R (one of
// lowbias32::kDropoutRowsCandidates), or with R = 0 the R its autotuner picks
// (written to *chosen, the candidates' mean times to ms[0..5]).
extern "C" int device_api_dropout_rows(const float *x, float *y, uint32_t rows, uint32_t seed, float p,
                                       uint32_t first, int R, int *chosen, float *ms)
{
    const lowbias32::Dropout d = lowbias32::make_dropout(seed, p);
    if (R == 0) {
        R = lowbias32::dropout_rows_autotune(x, y, rows, d, first, 0, 5, ms);
        if (R == 0) {
            const cudaError_t e = cudaGetLastError();
            return e != cudaSuccess ? static_cast<int>(e) : -1;
        }
    }
    if (chosen) *chosen = R;
    const cudaError_t e = lowbias32::dropout_rows(x, y, rows, d, first, R);
    if (e != cudaSuccess) return static_cast<int>(e);
    return static_cast<int>(cudaDeviceSynchronize());
}

// The header's own f32 logarithm on given 23-bit inputs: out[i] =
// -ln(1 - m[i] 2^-23) by lowbias32::neg_log_grid.
// With paired = 1, elements 2q and 2q + 1 go through the paired form
// (detail::neg_log_grid_x2, the fills' form); n must then be even.
__global__ void neglog_kernel(const uint32_t *m, float *out, uint32_t n, int paired)
{
    const uint32_t stride = gridDim.x * blockDim.x;
    if (paired) {
        for (uint32_t q = blockIdx.x * blockDim.x + threadIdx.x; q < n / 2u; q += stride) {
            const float2 v = lowbias32::detail::neg_log_grid_x2(m[2u * q] & 0x7FFFFFu, m[2u * q + 1u] & 0x7FFFFFu);
            out[2u * q] = v.x;
            out[2u * q + 1u] = v.y;
        }
        return;
    }
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        out[i] = lowbias32::neg_log_grid(m[i] & 0x7FFFFFu);
}

extern "C" int device_api_neglog(const uint32_t *m, float *out, uint32_t n, int paired)
{
    if (paired && (n & 1u)) return -1;
    neglog_kernel<<<1024, 256>>>(m, out, n, paired);
    return static_cast<int>(cudaDeviceSynchronize());
}

// The header's own cos(2 pi m 2^-23) on given 23-bit inputs (cos2pi_grid).
// With paired = 1, elements 2q and 2q + 1 go through detail::cos2pi_grid_x2.
__global__ void cos2pi_kernel(const uint32_t *m, float *out, uint32_t n, int paired)
{
    const uint32_t stride = gridDim.x * blockDim.x;
    if (paired) {
        for (uint32_t q = blockIdx.x * blockDim.x + threadIdx.x; q < n / 2u; q += stride) {
            const float2 v = lowbias32::detail::cos2pi_grid_x2(m[2u * q] & 0x7FFFFFu, m[2u * q + 1u] & 0x7FFFFFu);
            out[2u * q] = v.x;
            out[2u * q + 1u] = v.y;
        }
        return;
    }
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        out[i] = lowbias32::cos2pi_grid(m[i] & 0x7FFFFFu);
}

extern "C" int device_api_cos2pi(const uint32_t *m, float *out, uint32_t n, int paired)
{
    if (paired && (n & 1u)) return -1;
    cos2pi_kernel<<<1024, 256>>>(m, out, n, paired);
    return static_cast<int>(cudaDeviceSynchronize());
}

// randn of given draw pairs: out[i] = lowbias32::randn_of_draws(d0[i], d1[i]),
// (pair_x[i], pair_y[i]) = lowbias32::randn_pair_of_draws(d0[i], d1[i]).
__global__ void box_muller_kernel(const uint32_t *d0, const uint32_t *d1, float *out, float *pair_x, float *pair_y,
                                  uint32_t n)
{
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        out[i] = lowbias32::randn_of_draws(d0[i], d1[i]);
        const float2 p = lowbias32::randn_pair_of_draws(d0[i], d1[i]);
        pair_x[i] = p.x;
        pair_y[i] = p.y;
    }
}

extern "C" int device_api_box_muller(const uint32_t *d0, const uint32_t *d1, float *out, float *pair_x,
                                     float *pair_y, uint32_t n)
{
    box_muller_kernel<<<1024, 256>>>(d0, d1, out, pair_x, pair_y, n);
    return static_cast<int>(cudaDeviceSynchronize());
}

extern "C" uint32_t device_api_host_hash32(uint32_t x) { return lowbias32::hash32(x); }
