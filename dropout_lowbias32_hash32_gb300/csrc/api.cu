// api.cu -- the extern "C" entry points declared in include/rng.h: argument
// checks (before anything is enqueued), per-fill keys derived once on the
// host, and the split of long fills into pieces of at most 2^31 elements.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "hash32.cuh"
#include "internal.h"
#include "rng.h"

namespace rngk {

uint32_t host_hash32(uint32_t x) { return hash32(x); }

namespace {

std::atomic<uint64_t> g_launches{0};
thread_local char t_error[256] = "";

std::mutex g_sm_mu;
std::vector<unsigned> g_sm_counts;

rng_status fail(rng_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_error, sizeof t_error, fmt, ap);
    va_end(ap);
    return st;
}

rng_status cuda_fail(cudaError_t e, const char *what)
{
    if (e == cudaErrorMemoryAllocation) return fail(RNG_ENOMEM, "%s: %s", what, cudaGetErrorString(e));
    return fail(RNG_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

template <class T>
rng_status check_out(const T *p, size_t n, const char *name)
{
    if (n == 0) return RNG_OK;
    if (p == nullptr) return fail(RNG_EINVAL, "%s is NULL with n = %zu", name, n);
    if (reinterpret_cast<uintptr_t>(p) % sizeof(T) != 0)
        return fail(RNG_EINVAL, "%s is not aligned to its %zu-byte element", name, sizeof(T));
    if (n > (UINTPTR_MAX - reinterpret_cast<uintptr_t>(p)) / sizeof(T))
        return fail(RNG_EINVAL, "%s + %zu elements runs past the end of the address space", name, n);
    return RNG_OK;
}

// Runs f(offset, first counter, length) for consecutive pieces of at most
// kChunk elements.
template <class F>
rng_status for_pieces(size_t n, uint32_t first, const char *what, F &&f)
{
    for (size_t off = 0; off < n; off += kChunk) {
        const size_t len = n - off < kChunk ? n - off : kChunk;
        const cudaError_t e = f(off, static_cast<uint32_t>(first + static_cast<uint32_t>(off)),
                                static_cast<uint32_t>(len));
        if (e != cudaSuccess) return cuda_fail(e, what);
    }
    return RNG_OK;
}

template <class T, class Launch>
rng_status fill(const char *what, uint32_t first, size_t n, T *out, Launch &&launch)
{
    if (rng_status st = check_out(out, n, "out")) return st;
    t_error[0] = '\0';
    return for_pieces(n, first, what, [&](size_t off, uint32_t c, uint32_t len) { return launch(c, len, out + off); });
}

Below32Args below32_args(uint32_t seed, uint32_t bound)
{
    return Below32Args{seed_key(seed), purpose_key(seed, kPurposeBelow32), bound, (0u - bound) % bound};
}

Below64Args below64_args(uint32_t seed, uint64_t bound)
{
    return Below64Args{seed_key(seed), purpose_key(seed, kPurposeBelow64), bound, (0ull - bound) % bound};
}

rng_status dropout(const char *what, const float *x, float *y, float p, uint32_t seed, uint32_t first, size_t n,
                   void *stream)
{
    if (!(p >= 0.0f && p < 1.0f)) return fail(RNG_EINVAL, "%s: p = %g is outside [0, 1)", what, (double)p);
    if (rng_status st = check_out(x, n, "x")) return st;
    if (rng_status st = check_out(y, n, "y")) return st;
    if (n == 0) return RNG_OK;
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x), ya = reinterpret_cast<uintptr_t>(y);
    const uintptr_t bytes = n * sizeof(float);
    if (xa != ya && xa < ya + bytes && ya < xa + bytes)
        return fail(RNG_EINVAL, "%s: x and y overlap without being the same array", what);
    t_error[0] = '\0';
    // keep iff m 2^-23 >= p  <=>  m >= ceil(p 2^23), exact in binary64
    const uint32_t threshold = static_cast<uint32_t>(std::ceil(static_cast<double>(p) * 8388608.0));
    const float divisor = 1.0f - p;
    const uint32_t key = seed_key(seed);
    return for_pieces(n, first, what, [&](size_t off, uint32_t c, uint32_t len) {
        return launch_dropout(x + off, y + off, key, threshold, divisor, c, len, static_cast<cudaStream_t>(stream));
    });
}

}  // namespace

unsigned sm_count()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
    std::lock_guard<std::mutex> lock(g_sm_mu);
    if (g_sm_counts.size() <= static_cast<size_t>(dev)) g_sm_counts.resize(dev + 1, 0);
    if (!g_sm_counts[dev]) {
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        g_sm_counts[dev] = sms > 0 ? static_cast<unsigned>(sms) : 1u;
    }
    return g_sm_counts[dev];
}

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

unsigned fill_blocks(uint32_t n_vec)
{
    const unsigned wave = sm_count() * kFillBlocksPerSm;
    const unsigned need = (n_vec + kFillThreads - 1u) / kFillThreads;
    return need == 0 ? 1u : (need < wave ? need : wave);
}

}  // namespace rngk

using namespace rngk;

#define RNG_STREAM(s) static_cast<cudaStream_t>(s)

extern "C" {

rng_status rng_fill_u32(uint32_t seed, uint32_t first_counter, size_t n, uint32_t *out, void *stream)
{
    const uint32_t key = seed_key(seed);
    return fill("rng_fill_u32", first_counter, n, out, [&](uint32_t c, uint32_t len, uint32_t *o) {
        return launch_fill_u32(key, c, len, o, RNG_STREAM(stream));
    });
}

rng_status rng_fill_u64(uint32_t seed, uint32_t first_counter, size_t n, uint64_t *out, void *stream)
{
    const uint32_t key = seed_key(seed);
    return fill("rng_fill_u64", first_counter, n, out, [&](uint32_t c, uint32_t len, uint64_t *o) {
        return launch_fill_u64(key, c, len, o, RNG_STREAM(stream));
    });
}

rng_status rng_fill_f32(uint32_t seed, uint32_t first_counter, size_t n, float *out, void *stream)
{
    const uint32_t key = seed_key(seed);
    return fill("rng_fill_f32", first_counter, n, out, [&](uint32_t c, uint32_t len, float *o) {
        return launch_fill_f32(key, c, len, o, RNG_STREAM(stream));
    });
}

rng_status rng_fill_f64(uint32_t seed, uint32_t first_counter, size_t n, double *out, void *stream)
{
    const uint32_t key = seed_key(seed);
    return fill("rng_fill_f64", first_counter, n, out, [&](uint32_t c, uint32_t len, double *o) {
        return launch_fill_f64(key, c, len, o, RNG_STREAM(stream));
    });
}

rng_status rng_fill_u8(uint32_t seed, uint32_t first_counter, size_t n, uint8_t *out, void *stream)
{
    const uint32_t key = seed_key(seed);
    return fill("rng_fill_u8", first_counter, n, out, [&](uint32_t c, uint32_t len, uint8_t *o) {
        return launch_fill_u8(key, c, len, o, RNG_STREAM(stream));
    });
}

rng_status rng_fill_u16(uint32_t seed, uint32_t first_counter, size_t n, uint16_t *out, void *stream)
{
    const uint32_t key = seed_key(seed);
    return fill("rng_fill_u16", first_counter, n, out, [&](uint32_t c, uint32_t len, uint16_t *o) {
        return launch_fill_u16(key, c, len, o, RNG_STREAM(stream));
    });
}

rng_status rng_fill_f16(uint32_t seed, uint32_t first_counter, size_t n, uint16_t *out, void *stream)
{
    const uint32_t key = seed_key(seed);
    return fill("rng_fill_f16", first_counter, n, out, [&](uint32_t c, uint32_t len, uint16_t *o) {
        return launch_fill_f16(key, c, len, o, RNG_STREAM(stream));
    });
}

rng_status rng_fill_bool(uint32_t seed, uint32_t first_counter, size_t n, uint8_t *out, void *stream)
{
    const uint32_t key = seed_key(seed);
    return fill("rng_fill_bool", first_counter, n, out, [&](uint32_t c, uint32_t len, uint8_t *o) {
        return launch_fill_bool(key, c, len, o, RNG_STREAM(stream));
    });
}

rng_status rng_fill_u32_below(uint32_t seed, uint32_t first_counter, size_t n, uint32_t bound, uint32_t *out,
                              void *stream)
{
    if (bound == 0) return fail(RNG_EINVAL, "rng_fill_u32_below: bound is 0");
    const Below32Args a = below32_args(seed, bound);
    return fill("rng_fill_u32_below", first_counter, n, out, [&](uint32_t c, uint32_t len, uint32_t *o) {
        return launch_fill_u32_below(a, c, len, o, RNG_STREAM(stream));
    });
}

rng_status rng_fill_u64_below(uint32_t seed, uint32_t first_counter, size_t n, uint64_t bound, uint64_t *out,
                              void *stream)
{
    if (bound == 0) return fail(RNG_EINVAL, "rng_fill_u64_below: bound is 0");
    const Below64Args a = below64_args(seed, bound);
    return fill("rng_fill_u64_below", first_counter, n, out, [&](uint32_t c, uint32_t len, uint64_t *o) {
        return launch_fill_u64_below(a, c, len, o, RNG_STREAM(stream));
    });
}

rng_status rng_fill_i32_range(uint32_t seed, uint32_t first_counter, size_t n, int32_t low, uint32_t bound,
                              int32_t *out, void *stream)
{
    if (bound == 0) return fail(RNG_EINVAL, "rng_fill_i32_range: bound is 0");
    const Below32Args a = below32_args(seed, bound);
    return fill("rng_fill_i32_range", first_counter, n, out, [&](uint32_t c, uint32_t len, int32_t *o) {
        return launch_fill_i32_range(a, low, c, len, o, RNG_STREAM(stream));
    });
}

rng_status rng_fill_i64_range32(uint32_t seed, uint32_t first_counter, size_t n, int64_t low, uint32_t bound,
                                int64_t *out, void *stream)
{
    if (bound == 0) return fail(RNG_EINVAL, "rng_fill_i64_range32: bound is 0");
    const Below32Args a = below32_args(seed, bound);
    return fill("rng_fill_i64_range32", first_counter, n, out, [&](uint32_t c, uint32_t len, int64_t *o) {
        return launch_fill_i64_range32(a, low, c, len, o, RNG_STREAM(stream));
    });
}

rng_status rng_fill_i64_range(uint32_t seed, uint32_t first_counter, size_t n, int64_t low, uint64_t bound,
                              int64_t *out, void *stream)
{
    if (bound == 0) return fail(RNG_EINVAL, "rng_fill_i64_range: bound is 0");
    const Below64Args a = below64_args(seed, bound);
    return fill("rng_fill_i64_range", first_counter, n, out, [&](uint32_t c, uint32_t len, int64_t *o) {
        return launch_fill_i64_range(a, low, c, len, o, RNG_STREAM(stream));
    });
}

rng_status rng_fill_normal_f32(uint32_t seed, uint32_t first_counter, size_t n, float *out, void *stream)
{
    const uint32_t key = seed_key(seed);
    return fill("rng_fill_normal_f32", first_counter, n, out, [&](uint32_t c, uint32_t len, float *o) {
        return launch_fill_normal_f32(key, c, len, o, RNG_STREAM(stream));
    });
}

rng_status rng_fill_normal_f32_pairs(uint32_t seed, uint32_t first_counter, size_t n, float *out, void *stream)
{
    const uint32_t key = seed_key(seed);
    return fill("rng_fill_normal_f32_pairs", first_counter, n, out, [&](uint32_t c, uint32_t len, float *o) {
        return launch_fill_normal_f32_pairs(key, c, len, o, RNG_STREAM(stream));
    });
}

rng_status rng_fill_normal_f32_precise(uint32_t seed, uint32_t first_counter, size_t n, float *out, void *stream)
{
    const uint32_t key = seed_key(seed);
    return fill("rng_fill_normal_f32_precise", first_counter, n, out, [&](uint32_t c, uint32_t len, float *o) {
        return launch_fill_normal_f32_precise(key, c, len, o, RNG_STREAM(stream));
    });
}

rng_status rng_fill_exponential_f32(uint32_t seed, uint32_t first_counter, size_t n, float *out, void *stream)
{
    const uint32_t key = seed_key(seed);
    return fill("rng_fill_exponential_f32", first_counter, n, out, [&](uint32_t c, uint32_t len, float *o) {
        return launch_fill_exponential_f32(key, c, len, o, RNG_STREAM(stream));
    });
}

rng_status rng_fill_exponential_f64(uint32_t seed, uint32_t first_counter, size_t n, double *out, void *stream)
{
    const uint32_t key = seed_key(seed);
    return fill("rng_fill_exponential_f64", first_counter, n, out, [&](uint32_t c, uint32_t len, double *o) {
        return launch_fill_exponential_f64(key, c, len, o, RNG_STREAM(stream));
    });
}

rng_status rng_fill_normal_f64(uint32_t seed, uint32_t first_counter, size_t n, double *out, void *stream)
{
    return fill("rng_fill_normal_f64", first_counter, n, out, [&](uint32_t c, uint32_t len, double *o) {
        return launch_normal_f64(seed, c, len, o, RNG_STREAM(stream));
    });
}

rng_status rng_fill_normal_f64_noalloc(uint32_t seed, uint32_t first_counter, size_t n, double *out, void *stream)
{
    if (n > kNoAllocMaxElements)
        return fail(RNG_EINVAL, "rng_fill_normal_f64_noalloc: n = %zu exceeds its maximum of 2^28 elements", n);
    if (rng_status st = check_out(out, n, "out")) return st;
    if (n == 0) return RNG_OK;
    t_error[0] = '\0';
    const cudaError_t e = launch_normal_f64_noalloc(seed, first_counter, static_cast<uint32_t>(n), out,
                                                    RNG_STREAM(stream));
    return e == cudaSuccess ? RNG_OK : cuda_fail(e, "rng_fill_normal_f64_noalloc");
}

rng_status rng_dropout_fwd(const float *x, float *y, float p, uint32_t seed, uint32_t first_counter, size_t n,
                           void *stream)
{
    return dropout("rng_dropout_fwd", x, y, p, seed, first_counter, n, stream);
}

rng_status rng_dropout_bwd(const float *dy, float *dx, float p, uint32_t seed, uint32_t first_counter, size_t n,
                           void *stream)
{
    return dropout("rng_dropout_bwd", dy, dx, p, seed, first_counter, n, stream);
}

const char *rng_status_string(rng_status status)
{
    switch (status) {
    case RNG_OK: return "RNG_OK";
    case RNG_EINVAL: return "RNG_EINVAL: invalid argument";
    case RNG_ECUDA: return "RNG_ECUDA: CUDA runtime error";
    case RNG_ENOMEM: return "RNG_ENOMEM: device allocation failed";
    default: return "unknown rng_status";
    }
}

const char *rng_last_error(void) { return t_error; }

rng_status rng_debug_set_miss_capacity(size_t capacity)
{
    set_miss_capacity_override(capacity);
    return RNG_OK;
}

rng_status rng_debug_last_miss_count(uint64_t *count)
{
    if (count == nullptr) return fail(RNG_EINVAL, "rng_debug_last_miss_count: count is NULL");
    const cudaError_t e = last_miss_count(count);
    return e == cudaSuccess ? RNG_OK : cuda_fail(e, "rng_debug_last_miss_count");
}

uint64_t rng_debug_launch_count(void) { return g_launches.load(); }

rng_status rng_debug_eval_f64(int which, const double *in, double *out, size_t n, void *stream)
{
    if (which < 0 || which > 4) return fail(RNG_EINVAL, "rng_debug_eval_f64: which must be 0 .. 4");
    if (rng_status st = check_out(in, n, "in")) return st;
    if (rng_status st = check_out(out, n, "out")) return st;
    t_error[0] = '\0';
    return for_pieces(n, 0, "rng_debug_eval_f64", [&](size_t off, uint32_t, uint32_t len) {
        return launch_eval_f64(which, in + off, out + off, len, RNG_STREAM(stream));
    });
}

rng_status rng_debug_write_ceiling(int which, void *buf, size_t bytes, void *stream)
{
    if (which != 0 && which != 1) return fail(RNG_EINVAL, "rng_debug_write_ceiling: which must be 0 or 1");
    if (bytes == 0) return RNG_OK;
    if (buf == nullptr) return fail(RNG_EINVAL, "rng_debug_write_ceiling: buf is NULL with bytes = %zu", bytes);
    if (bytes > UINTPTR_MAX - reinterpret_cast<uintptr_t>(buf))
        return fail(RNG_EINVAL, "rng_debug_write_ceiling: buf + %zu bytes runs past the end of the address space",
                    bytes);
    t_error[0] = '\0';
    if (which == 0) {
        const cudaError_t e = cudaMemsetAsync(buf, 0x5A, bytes, RNG_STREAM(stream));
        return e == cudaSuccess ? RNG_OK : fail(RNG_ECUDA, "rng_debug_write_ceiling: %s", cudaGetErrorString(e));
    }
    if (reinterpret_cast<uintptr_t>(buf) % 16 != 0 || bytes % 16 != 0)
        return fail(RNG_EINVAL, "rng_debug_write_ceiling: the store kernel needs a 16-byte aligned buffer of "
                                "whole 16-byte vectors");
    uint4 *out = static_cast<uint4 *>(buf);
    return for_pieces(bytes / 16, 0, "rng_debug_write_ceiling", [&](size_t off, uint32_t, uint32_t len) {
        return launch_store_ceiling(out + off, len, RNG_STREAM(stream));
    });
}

}  // extern "C"
