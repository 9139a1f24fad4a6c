// internal.h -- declarations shared by the library's translation units
// (launchers, launch accounting, error messages).  Not part of the C ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace rngk {

// Threads per block of the streaming fill kernels.
constexpr unsigned kFillThreads = 256;
// 16-byte vectors each thread of a chunked fill writes (block b writes the
// b-th run of kFillThreads x kFillVectorsPerThread vectors).
constexpr unsigned kFillVectorsPerThread = 4;
// The same for generators of many instructions per element (bounded
// integers, f64 and f16 uniforms, normals, exponentials), which gain from
// more independent vectors in flight per thread.
constexpr unsigned kHeavyVectorsPerThread = 8;
// Resident blocks per SM of the grid-stride kernels (2048 threads / SM).
constexpr unsigned kFillBlocksPerSm = 8;
// Largest number of elements one launch covers; the C ABI splits longer
// fills into pieces of at most this size (a fill cut anywhere equals the
// whole fill, so the pieces are independent launches).
constexpr size_t kChunk = size_t(1) << 31;

// Streaming multiprocessor count of the current device (cached per device).
unsigned sm_count();

// Accounting of kernel launches (rng_debug_launch_count).
void note_launch();

// Grid of a grid-stride fill over n_vec 16-byte vectors.
unsigned fill_blocks(uint32_t n_vec);

// Seed-derived keys, computed once per fill on the host and passed to the
// kernels folded (k ^ (k >> 16), see hash32.cuh).
uint32_t host_hash32(uint32_t x);
inline uint32_t folded(uint32_t k) { return k ^ (k >> 16); }
inline uint32_t seed_key(uint32_t seed) { return folded(host_hash32(seed)); }
inline uint32_t purpose_key(uint32_t seed, uint32_t purpose) { return folded(host_hash32(host_hash32(seed) ^ purpose)); }

constexpr uint32_t kPurposeBelow32 = 0x42333220u;  // "B32 "
constexpr uint32_t kPurposeBelow64 = 0x42363420u;  // "B64 "
constexpr uint32_t kPurposeNormal64 = 0x4E363420u; // "N64 "

// Elements before out's first 16-byte boundary (at most n), for T-aligned out.
template <class T>
inline uint32_t head_elems(const void *out, uint32_t n)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(out);
    const uint32_t h = static_cast<uint32_t>(((16u - (a & 15u)) & 15u) / sizeof(T));
    return h < n ? h : n;
}

// Launchers: one piece of at most kChunk elements, out already validated.
cudaError_t launch_fill_u32(uint32_t key, uint32_t first, uint32_t n, uint32_t *out, cudaStream_t s);
cudaError_t launch_fill_u64(uint32_t key, uint32_t first, uint32_t n, uint64_t *out, cudaStream_t s);
cudaError_t launch_fill_f32(uint32_t key, uint32_t first, uint32_t n, float *out, cudaStream_t s);
cudaError_t launch_fill_f64(uint32_t key, uint32_t first, uint32_t n, double *out, cudaStream_t s);
cudaError_t launch_fill_u8(uint32_t key, uint32_t first, uint32_t n, uint8_t *out, cudaStream_t s);
cudaError_t launch_fill_u16(uint32_t key, uint32_t first, uint32_t n, uint16_t *out, cudaStream_t s);
cudaError_t launch_fill_f16(uint32_t key, uint32_t first, uint32_t n, uint16_t *out, cudaStream_t s);
cudaError_t launch_fill_bool(uint32_t key, uint32_t first, uint32_t n, uint8_t *out, cudaStream_t s);

struct Below32Args {
    uint32_t key, purpose_key, bound, threshold;
};
struct Below64Args {
    uint32_t key, purpose_key;
    uint64_t bound, threshold;
};
cudaError_t launch_fill_u32_below(const Below32Args &a, uint32_t first, uint32_t n, uint32_t *out,
                                  cudaStream_t s);
cudaError_t launch_fill_u64_below(const Below64Args &a, uint32_t first, uint32_t n, uint64_t *out,
                                  cudaStream_t s);
cudaError_t launch_fill_i32_range(const Below32Args &a, int32_t low, uint32_t first, uint32_t n,
                                  int32_t *out, cudaStream_t s);
cudaError_t launch_fill_i64_range32(const Below32Args &a, int64_t low, uint32_t first, uint32_t n,
                                    int64_t *out, cudaStream_t s);
cudaError_t launch_fill_i64_range(const Below64Args &a, int64_t low, uint32_t first, uint32_t n,
                                  int64_t *out, cudaStream_t s);

cudaError_t launch_fill_normal_f32(uint32_t key, uint32_t first, uint32_t n, float *out, cudaStream_t s);
cudaError_t launch_fill_normal_f32_pairs(uint32_t key, uint32_t first, uint32_t n, float *out, cudaStream_t s);
cudaError_t launch_fill_normal_f32_precise(uint32_t key, uint32_t first, uint32_t n, float *out, cudaStream_t s);
cudaError_t launch_fill_exponential_f32(uint32_t key, uint32_t first, uint32_t n, float *out, cudaStream_t s);
cudaError_t launch_fill_exponential_f64(uint32_t key, uint32_t first, uint32_t n, double *out, cudaStream_t s);

// Dropout of one piece: keep iff (D32 & 0x7FFFFF) >= threshold, y = x / divisor.
cudaError_t launch_dropout(const float *x, float *y, uint32_t key, uint32_t threshold, float divisor,
                           uint32_t first, uint32_t n, cudaStream_t s);

// normal_f64: table pass + miss pass of one piece (returns a cudaError_t, or
// cudaErrorMemoryAllocation when the miss list cannot be allocated).
cudaError_t launch_normal_f64(uint32_t seed, uint32_t first, uint32_t n, double *out, cudaStream_t s);
void set_miss_capacity_override(size_t cap);
cudaError_t last_miss_count(uint64_t *count);
cudaError_t launch_eval_f64(int which, const double *in, double *out, uint32_t n, cudaStream_t s);

// normal_f64 with the miss list in a static device array (no allocation);
// n must not exceed kNoAllocMaxElements.
constexpr size_t kNoAllocMaxElements = size_t(1) << 28;
cudaError_t launch_normal_f64_noalloc(uint32_t seed, uint32_t first, uint32_t n, double *out, cudaStream_t s);

// Plain 16-byte stores of n_vec vectors (the write-ceiling measurement).
cudaError_t launch_store_ceiling(uint4 *out, uint32_t n_vec, cudaStream_t s);

}  // namespace rngk
