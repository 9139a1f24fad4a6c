/*
 * rng.h -- C ABI of the GB300 (sm_103a) stateless counter-based random fills.
 *
 * Every output element is a pure function of (seed, counter): element i of a
 * fill takes the counter c_i = (first_counter + i) mod 2^32.  The generator is
 * the lowbias32 hash32 of the Phobos stdlib page "Random numbers" (section
 * hash32), in wrapping 32-bit arithmetic:
 *
 *   hash32(x)  = mix(mix(mix(x,16) * 0x7FEB352D, 15) * 0x846CA68B, 16),
 *                mix(x, s) = x ^ (x >> s) with a logical shift;
 *   D32(s, c)  = hash32(c ^ hash32(s))                  (section uniform);
 *   D64(s, c)  = D32(s, 2c) << 32 | D32(s, 2c + 1),      2c mod 2^32.
 *
 * Conventions shared by every call below.
 *   - Pointers are device pointers (cudaMalloc, torch CUDA tensors, managed
 *     memory) on the calling thread's current CUDA device.  The caller owns
 *     them; the library never allocates or frees an output.
 *   - Each output must be aligned to its element size.  No alignment beyond
 *     that is required: a start that is not 16-byte aligned is peeled off with
 *     scalar stores and the rest is written in whole 16-byte vectors.
 *   - `stream` is a cudaStream_t (NULL: the legacy default stream).  Calls are
 *     stream-ordered and asynchronous: they return once the work is enqueued.
 *   - n == 0 is a no-op that returns RNG_OK without touching any pointer.
 *     n may exceed 2^32; counters then wrap and values repeat with period
 *     2^32 (2^31 for the 64-bit and normal draws, which consume counters 2c
 *     and 2c + 1).
 *   - Errors.  RNG_EINVAL is returned before anything is enqueued: a NULL or
 *     misaligned pointer with n > 0, a pointer whose n elements would run
 *     past the end of the address space, a bound of 0, p outside [0, 1) or
 *     NaN, partially overlapping input and output.  RNG_ECUDA reports an error
 *     returned by the CUDA runtime while enqueuing (launch failure, invalid
 *     stream); faults of the device work itself surface at the caller's next
 *     synchronisation, as for any CUDA kernel.  RNG_ENOMEM reports a failed
 *     allocation of the library's own per-device ziggurat miss list.
 *     rng_last_error() gives a message for the calling thread's last error.
 *   - Every call is thread-safe, except that calls of
 *     rng_fill_normal_f64_noalloc whose work overlaps on the GPU race (see
 *     there).
 *   - The fills other than the two f64 normals keep no device state: their
 *     launches can be captured into a CUDA graph and replayed.
 *   - A fill cut at any element equals the whole fill: filling [a, b) with
 *     first_counter + a gives elements a..b-1 of the fill from first_counter.
 */
#ifndef LOWBIAS32_RNG_H
#define LOWBIAS32_RNG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int rng_status;
#define RNG_OK 0
#define RNG_EINVAL 1
#define RNG_ECUDA 2
#define RNG_ENOMEM 3

/* ---- uniform fills ------------------------------------------------------ */

/* out[i] = D32(seed, c_i).  Phobos "Random numbers", section uniform: the
 * hash of the counter keyed by the hashed seed. */
rng_status rng_fill_u32(uint32_t seed, uint32_t first_counter, size_t n, uint32_t *out,
                        void *stream);

/* out[i] = D64(seed, c_i): the draws at 2c_i (high word) and 2c_i + 1 (low
 * word), the counter pair randn consumes (Phobos "Random numbers", section
 * randn); tandem-cuda "Performance" row fill_u64 gives the fill. */
rng_status rng_fill_u64(uint32_t seed, uint32_t first_counter, size_t n, uint64_t *out,
                        void *stream);

/* out[i] = uniform(seed, c_i) = (D32 & 0x7FFFFF) * 2^-23, exactly: the low 23
 * bits on the 2^-23 grid in [0, 1) (Phobos "Random numbers", section uniform). */
rng_status rng_fill_f32(uint32_t seed, uint32_t first_counter, size_t n, float *out,
                        void *stream);

/* out[i] = (D64(seed, c_i) >> 11) * 2^-53, exactly: the top 53 bits on the
 * 2^-53 grid in [0, 1) (tandem-cuda "Performance", row fill_f64). */
rng_status rng_fill_f64(uint32_t seed, uint32_t first_counter, size_t n, double *out,
                        void *stream);

/* ---- narrow fills ----------------------------------------------------------- */
/* (tandem-cuda "Performance", rows fill_u16, fill_f16_bits, fill_u8 and
 * fill_bool, restated on hash32.)  Each element stays a pure function of its
 * counter; one 32-bit draw serves 4, 2 or 32 consecutive counters, the word
 * index wrapping with the counter. */

/* out[i] = byte (c_i & 3) of D32(seed, c_i >> 2), bits 8(c_i & 3) .. +7. */
rng_status rng_fill_u8(uint32_t seed, uint32_t first_counter, size_t n, uint8_t *out, void *stream);

/* out[i] = halfword (c_i & 1) of D32(seed, c_i >> 1), bits 16(c_i & 1) .. +15. */
rng_status rng_fill_u16(uint32_t seed, uint32_t first_counter, size_t n, uint16_t *out, void *stream);

/* out[i] = binary16 bits of m 2^-10, m the low 10 bits of the u16 element at
 * c_i: a uniform on the 2^-10 grid in [0, 1), exactly. */
rng_status rng_fill_f16(uint32_t seed, uint32_t first_counter, size_t n, uint16_t *out, void *stream);

/* out[i] = bit (c_i & 31) of D32(seed, c_i >> 5), one byte (0 or 1) per bit. */
rng_status rng_fill_bool(uint32_t seed, uint32_t first_counter, size_t n, uint8_t *out, void *stream);

/* ---- bounded integers: Lemire's multiply-shift with rejection ------------ */
/* (perturbation-kernel "Backends", section "Why the GPU can be exact";
 * tandem-cuda "Performance", bounded rows.)  For a w-bit word x the candidate
 * is floor(x * bound / 2^w); it is accepted when (x * bound) mod 2^w >=
 * 2^w mod bound (Lemire's exact threshold), which makes every value in
 * [0, bound) exactly equally likely.  A rejected element retries on its own
 * substream, keyed by its counter: the k-th retry word is hash32(k ^ K) with
 * K = hash32(c_i ^ hash32(hash32(seed) ^ P)), P = 0x42333220 ("B32 ") for
 * 32-bit and 0x42363420 ("B64 ") for 64-bit words, whose k-th word is
 * hash32(2k ^ K) << 32 | hash32((2k + 1) ^ K).  bound == 0 is RNG_EINVAL. */

/* out[i] = below32(bound) on the 32-bit draw D32(seed, c_i). */
rng_status rng_fill_u32_below(uint32_t seed, uint32_t first_counter, size_t n, uint32_t bound,
                              uint32_t *out, void *stream);

/* out[i] = below64(bound) on the 64-bit draw D64(seed, c_i). */
rng_status rng_fill_u64_below(uint32_t seed, uint32_t first_counter, size_t n, uint64_t bound,
                              uint64_t *out, void *stream);

/* out[i] = low + below32(bound), wrapped to int32 (two's complement)
 * (tandem-cuda "Performance", row "with a low bound into int32_t"). */
rng_status rng_fill_i32_range(uint32_t seed, uint32_t first_counter, size_t n, int32_t low,
                              uint32_t bound, int32_t *out, void *stream);

/* out[i] = low + below32(bound) into int64, wrapped (8-byte elements from
 * 32-bit draws; tandem-cuda "Performance", row "into int64_t"). */
rng_status rng_fill_i64_range32(uint32_t seed, uint32_t first_counter, size_t n, int64_t low,
                                uint32_t bound, int64_t *out, void *stream);

/* out[i] = low + below64(bound), wrapped to int64. */
rng_status rng_fill_i64_range(uint32_t seed, uint32_t first_counter, size_t n, int64_t low,
                              uint64_t bound, int64_t *out, void *stream);

/* ---- normals ------------------------------------------------------------- */

/* out[i] = randn(seed, c_i) = sqrt(-2 ln(1 - u0)) cos(2 pi u1) with u0 =
 * uniform(seed, 2c_i), u1 = uniform(seed, 2c_i + 1) (Phobos "Random
 * numbers", section randn): one value per counter, the cosine branch of
 * Box-Muller, |out| <= sqrt(46 ln 2) ~ 5.648.  Computed in f32: below u0 =
 * 2^-7 the series (1 + u0)^2 - 1 of -2 ln(1 - u0), above it the hardware
 * log2; the hardware square root; the hardware cosine on the angle 2 pi u1
 * in [0, 2 pi) (no half-turn shift as in tandem-sycl "Design", section
 * Normals: GB300's cosine is as accurate over the whole turn).  Each value is
 * within 4e-6 (1 + |z|) of the exact z. */
rng_status rng_fill_normal_f32(uint32_t seed, uint32_t first_counter, size_t n, float *out,
                               void *stream);

/* Paired Box-Muller: both branches of each uniform pair, one 64-bit draw
 * per two values (half the hashing of rng_fill_normal_f32).  With q = c_i >> 1,
 * u0 = uniform(seed, 2q), u1 = uniform(seed, 2q + 1), r = sqrt(-2 ln(1 - u0)):
 * out[i] = r cos(2 pi u1) for even c_i (= randn(seed, q)), r sin(2 pi u1) for
 * odd c_i.  The pages' randn keeps the cosine branch only (Phobos "Random
 * numbers", section randn); tandem-sycl "Design", section Normals, draws
 * Box-Muller pairs.  Same accuracy as rng_fill_normal_f32: within
 * 4e-6 (1 + |z|) of the exact value. */
rng_status rng_fill_normal_f32_pairs(uint32_t seed, uint32_t first_counter, size_t n, float *out,
                                     void *stream);

/* Precise f32 normal: randn's definition (u0 = uniform(seed, 2 c_i), u1 =
 * uniform(seed, 2 c_i + 1), z = sqrt(-2 ln(1 - u0)) cos(2 pi u1)) evaluated
 * in binary32 to a few ulp: the library's own -ln(1 - u0) (within 0.5035 ulp)
 * and cos(2 pi u1) (within 0.90 ulp), an IEEE square root, so out[i] is
 * within 2.5 ulp of the exact value and reproducible bit for bit.  An opt-in
 * variant with its own values: tandem-sycl "Design", section Normals, keeps a
 * precise f32 Box-Muller as a build option beside the default float normal.
 * rng_fill_normal_f32 is faster and within 4e-6 (1 + |z|). */
rng_status rng_fill_normal_f32_precise(uint32_t seed, uint32_t first_counter, size_t n, float *out,
                                       void *stream);

/* out[i] = standard normal from the 1024-layer Marsaglia-Tsang ziggurat on
 * the 64-bit draw D64(seed, c_i) (tandem-sycl "Design", section Normals).
 * Layer j = w & 1023, sign = bit 10, magnitude x = (w >> 11) 2^-53 X[j]
 * rounded once; x < X[j+1] is stored at once (99.57 % of elements).  The
 * rest (0.43 %) are appended to a device miss list and resolved by a second
 * kernel on the substream hash32(k ^ K), K = hash32(c_i ^ hash32(hash32(seed)
 * ^ 0x4E363420)) ("N64 "): the base layer samples the tail beyond r =
 * X[1] (Marsaglia 1964), the others take the wedge test against exp(-x^2/2)
 * and otherwise start over with a fresh 64-bit word.  Both exp and log of
 * that path are fixed IEEE operation sequences, so the result is bit-exact
 * and reproducible.  The layer tables are static device data of the library
 * (no allocation).  The miss list (4 bytes per expected miss plus slack) is
 * the one device allocation: made per device on first use, grown when a
 * longer fill needs more, and held until the process exits; fills on
 * different streams that share it are ordered through its last event.  If
 * the list overflows, the second kernel walks the whole fill again. */
rng_status rng_fill_normal_f64(uint32_t seed, uint32_t first_counter, size_t n, double *out,
                               void *stream);

/* Allocation-free variant of rng_fill_normal_f64, for callers that cannot
 * call cudaMalloc: code whose device memory is entirely owned by another
 * allocator (a framework's caching allocator that reserved the pool up front,
 * where a cudaMalloc of ours would fail or fragment it), and latency-critical
 * paths that cannot accept cudaMalloc's implicit device synchronisation.  The
 * pages have no counterpart: it exists for those callers only.
 *   - Same values as rng_fill_normal_f64, bit for bit.
 *   - The miss counter and list live in one static device array of the
 *     library (8 MiB + 256 bytes, present on every device that loads the
 *     library until the process exits); the call makes no device allocation.
 *   - n must not exceed 2^28 elements; larger n returns RNG_EINVAL.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *     The address is kept for the rest of the process: it assumes that the
 *     device's primary context is not reset (cudaDeviceReset) meanwhile.
 *   - Every call shares the array and clears its counter first: calls whose
 *     work overlaps on the GPU (other streams, other threads) race on it and
 *     give unspecified values.  Order them on one stream or with events.
 *   - Otherwise as rng_fill_normal_f64 (device pointers, stream-ordered). */
rng_status rng_fill_normal_f64_noalloc(uint32_t seed, uint32_t first_counter, size_t n, double *out,
                                       void *stream);

/* ---- exponentials (tandem-sycl "Design", section Exponentials) ------------ */

/* out[i] = -ln(1 - u), u = uniform(seed, c_i): 1 - u = V 2^-23 exact in
 * (0, 1], and the library's own table-driven binary32 logarithm of it
 * (neg_log_grid in include/rng_device.cuh: exact reduction by 8-bit
 * reciprocals, a TwoSum and a series to r^5, one final rounding), within
 * 0.5035 ulp of the exact value on every input and reproducible bit for bit;
 * in [0, 23 ln 2]. */
rng_status rng_fill_exponential_f32(uint32_t seed, uint32_t first_counter, size_t n, float *out,
                                    void *stream);

/* out[i] = -ln(1 - u), u = (D64(seed, c_i) >> 11) 2^-53, by neglog64: a
 * fixed-point logarithm in 32-, 64- and 128-bit integer arithmetic with no
 * FP64 arithmetic (one u64 -> f64 conversion rounds the result).  1 - u =
 * V 2^-53 with the integer V = 2^53 - m is reduced exactly by 2048 one-sided
 * reciprocals (r in [0, 1.5 2^-11)), log1p of the reduced argument is a
 * Horner series to r^5 in fixed point, the exponent and table terms are added
 * at scale 2^96, and the sum is rounded once to binary64; below u = 2^-12 the
 * value is the series in u itself.  Within 0.5007 ulp of -ln(1 - u),
 * reproducible bit for bit, in [0, 53 ln 2]; +0 at u = 0.  Bound by the
 * integer pipes on GB300. */
rng_status rng_fill_exponential_f64(uint32_t seed, uint32_t first_counter, size_t n, double *out,
                                    void *stream);

/* ---- dropout (Phobos "Random numbers", section dropout) ------------------- */

/* y[i] = uniform(seed, c_i) >= p ? x[i] / (1 - p) : +0, in f32 with IEEE
 * division; 1 - p is rounded to f32 first; a tie u == p is kept.  p must lie
 * in [0, 1).  x and y may be the same array (in place) but must not overlap
 * otherwise.  Reads 4 and writes 4 bytes per element. */
rng_status rng_dropout_fwd(const float *x, float *y, float p, uint32_t seed,
                           uint32_t first_counter, size_t n, void *stream);

/* dx[i] = the same mask applied to dy[i], redrawn from the same seed and
 * counters instead of stored (the page's backward pass): bit-for-bit the
 * forward computation on dy. */
rng_status rng_dropout_bwd(const float *dy, float *dx, float p, uint32_t seed,
                           uint32_t first_counter, size_t n, void *stream);

/* ---- status -------------------------------------------------------------- */

/* A static string naming the status code. */
const char *rng_status_string(rng_status status);

/* The calling thread's message for its last non-OK status (static storage
 * per thread; "" when none). */
const char *rng_last_error(void);

/* ---- test and measurement hooks ------------------------------------------ */

/* Caps the number of entries the ziggurat miss list may hold (0 forces every
 * normal_f64 fill through the whole-fill walk of the second kernel);
 * SIZE_MAX restores the default capacity.  Applies to later fills on every
 * device. */
rng_status rng_debug_set_miss_capacity(size_t capacity);

/* Number of entries the most recent normal_f64 fill's table pass listed on
 * the current device (of its last chunk of at most 2^31 elements; above the
 * capacity when the list overflowed): every draw that misses the fast path,
 * plus the few fast draws the table pass leaves to the second kernel (those
 * its integer product cannot round, about 1e-4 of the elements, and about
 * 1e-6 whose product shares X[j+1]'s high word).  Synchronises the device. */
rng_status rng_debug_last_miss_count(uint64_t *count);

/* Number of kernels this library has launched since it was loaded, over all
 * devices and threads. */
uint64_t rng_debug_launch_count(void);

/* Evaluates the library's own binary64 functions on the device, out[i] =
 * f(in[i]) for i < n (in and out device arrays of doubles): the normal_f64
 * slow path's exp (which = 0) or log (which = 1), or (which = 2) the f64
 * exponential's fixed-point -ln(1 - m 2^-53) with m the low 53 bits of
 * in[i]'s bit pattern.  which = 3 and 4 take in[i]'s bit pattern as a 64-bit
 * ziggurat draw w and return its fast-path magnitude RNE((w >> 11) 2^-53
 * X[w & 1023]): by the table pass's integer product (NaN for a draw it
 * defers to the miss pass) and by its fma.  For checking those functions on
 * chosen inputs; which outside 0 .. 4 is RNG_EINVAL. */
rng_status rng_debug_eval_f64(int which, const double *in, double *out, size_t n, void *stream);

/* A measurement aid with no counterpart on the pages: the write ceiling the
 * fills are compared with.  which = 0 enqueues cudaMemsetAsync(buf, 0x5A,
 * bytes); which = 1 launches the plainest 16-byte store kernel over buf, in
 * the launch shape of the fills (buf 16-byte aligned, bytes a multiple of
 * 16).  buf is a caller-owned device buffer whose contents are overwritten;
 * stream-ordered on stream.  RNG_EINVAL for another which, buf == NULL with
 * bytes > 0, buf + bytes past the end of the address space, or (which = 1) a
 * misaligned buf or size; bytes == 0 is a no-op. */
rng_status rng_debug_write_ceiling(int which, void *buf, size_t bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LOWBIAS32_RNG_H */
