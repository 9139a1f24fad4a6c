// normal_f64.cu -- f64 standard normals by a 1024-layer Marsaglia-Tsang
// ziggurat in two kernels: a table pass that writes every element and lists
// the misses, and a miss pass that resolves them.
//
// tandem-sycl "Design", section Normals: one 64-bit draw per element; 0.43 %
// of draws miss the fast path and continue on a substream keyed by the
// draw's global index, so a fill cut at any element equals the whole fill;
// the table pass queues a block's misses locally and appends them to a device
// list with one atomic add; the second kernel takes one miss per thread and,
// if the list overflowed, walks the whole fill again; the layer table lives in
// global memory (constant memory serialises lanes that read different
// layers); the fast path makes no calls.
//
// Draw w = D64(seed, c): layer j = w & 1023, sign = bit 10, m = w >> 11 (53
// bits); x = RNE((m 2^-53) X[j]); fast iff x < X[j+1].  GB300's FP64 pipe
// retires 2 fma per SM and cycle (1/64 of FP32), so the fast path spends
// exactly one FP64 instruction per element: t = 1 + (m mod 2^52) 2^-52 is
// assembled from the draw's bits, and fma(t, X[j]/2, b ? 0 : -X[j]/2) with
// b = bit 52 of m equals (m 2^-53) X[j] before its single rounding, so it
// returns the IEEE product bit for bit.
//
// Miss of layer 0: the tail beyond r = X[1] (Marsaglia 1964: a = -log(U1)/r,
// b = -log(U2), accept when 2b >= a^2, value r + a, U in (0, 1]).  Miss of
// layer j >= 1: the wedge test y = F[j] + U (F[j+1] - F[j]) < exp(-x^2/2);
// a rejected wedge starts over with the substream's next 64-bit word.  The
// substream words are taken in that order.  exp and log are this file's own
// fixed sequences of IEEE operations (Cody & Waite reduction + Taylor for
// exp; exponent split + atanh series for log), so the slow path returns the
// same bits on every IEEE machine.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <map>
#include <memory>
#include <mutex>

#include "fill_kernel.cuh"
#include "hash32.cuh"
#include "internal.h"
#include "zig_tables.inc"

namespace rngk {
namespace {

constexpr uint32_t kLayers = 1024;

// Layer table, global memory, read through the read-only path.
__device__ const double kZigX[kLayers + 1] = {ZIG_X_VALUES};
__device__ const double kZigF[kLayers + 1] = {ZIG_F_VALUES};
__device__ const double2 kZigHalfXNext[kLayers] = {ZIG_HALFX_XNEXT_VALUES};  // {X[j]/2, X[j+1]}

constexpr uint32_t kTableThreads = 256;
constexpr uint32_t kTableIters = 8;  // 16-byte vectors per thread and block
constexpr uint32_t kTableVecPerBlock = kTableThreads * kTableIters;  // 4096 elements
constexpr uint32_t kQueue = 1024;  // per-block miss queue (17.5 misses expected per block)
constexpr uint32_t kMissThreads = 128;
constexpr uint32_t kMaxRounds = 4096;  // rejection rounds of one miss (never reached)

// ---- fast path ------------------------------------------------------------

struct FastDraw {
    uint64_t bits;  // the signed fast-path value
    bool fast;
};

// Fast path of the 64-bit draw w = hi:lo (see the file comment).
__device__ __forceinline__ FastDraw zig_fast(Words w)
{
    const double2 e = __ldg(&kZigHalfXNext[w.lo & (kLayers - 1u)]);
    // t = 1 + (m mod 2^52) 2^-52, m = (hi:lo) >> 11
    const uint32_t t_lo = __funnelshift_r(w.lo, w.hi, 11);
    const uint32_t t_hi = ((w.hi >> 11) & 0xFFFFFu) | 0x3FF00000u;
    // addend 0 when bit 52 of m (bit 31 of hi) is set, else -X[j]/2
    const uint32_t keep = static_cast<uint32_t>(static_cast<int32_t>(w.hi) >> 31);
    const uint32_t c_hi = (static_cast<uint32_t>(__double2hiint(e.x)) ^ 0x80000000u) & ~keep;
    const uint32_t c_lo = static_cast<uint32_t>(__double2loint(e.x)) & ~keep;
    const double x = __fma_rn(__hiloint2double(static_cast<int>(t_hi), static_cast<int>(t_lo)), e.x,
                              __hiloint2double(static_cast<int>(c_hi), static_cast<int>(c_lo)));
    const uint64_t xb = static_cast<uint64_t>(__double_as_longlong(x));
    FastDraw d;
    // both values are non-negative, so their bit patterns order like them
    d.fast = xb < static_cast<uint64_t>(__double_as_longlong(e.y));
    d.bits = xb | (static_cast<uint64_t>(w.lo & 0x400u) << 53);  // bit 10 -> sign bit
    return d;
}

// ---- slow path --------------------------------------------------------------

// exp(t) for t in [-10, 0]: k = rint(t / ln 2), r = t - k ln 2 by two fma
// (ln 2 = ln2_high + ln2_low, ln2_high with 32 significant bits), degree-13
// Taylor polynomial in Horner form, exact scaling by 2^k.
__device__ __forceinline__ double zexp(double t)
{
    const double k = rint(__dmul_rn(t, ZK_INV_LN2));
    double r = __fma_rn(-k, ZK_LN2_HIGH, t);
    r = __fma_rn(-k, ZK_LN2_LOW, r);
    double p = ZK_INV_FACT_13;
    p = __fma_rn(p, r, ZK_INV_FACT_12);
    p = __fma_rn(p, r, ZK_INV_FACT_11);
    p = __fma_rn(p, r, ZK_INV_FACT_10);
    p = __fma_rn(p, r, ZK_INV_FACT_9);
    p = __fma_rn(p, r, ZK_INV_FACT_8);
    p = __fma_rn(p, r, ZK_INV_FACT_7);
    p = __fma_rn(p, r, ZK_INV_FACT_6);
    p = __fma_rn(p, r, ZK_INV_FACT_5);
    p = __fma_rn(p, r, ZK_INV_FACT_4);
    p = __fma_rn(p, r, ZK_INV_FACT_3);
    p = __fma_rn(p, r, ZK_INV_FACT_2);
    p = __fma_rn(p, r, ZK_INV_FACT_1);
    p = __fma_rn(p, r, ZK_INV_FACT_0);
    const double scale = __longlong_as_double(static_cast<long long>(1023 + static_cast<int>(k)) << 52);
    return __dmul_rn(p, scale);
}

// log(x) for positive normal x: x = 2^e m with m in (sqrt(1/2), sqrt 2],
// s = (m - 1)/(m + 1), log m = 2 (s + s^3/3 + ... + s^23/23), then
// e ln2_high + (e ln2_low + log m).
__device__ __forceinline__ double zlog(double x)
{
    const uint64_t bits = static_cast<uint64_t>(__double_as_longlong(x));
    int e = static_cast<int>(bits >> 52) - 1023;
    double m = __longlong_as_double(static_cast<long long>((bits & 0x000FFFFFFFFFFFFFull) | 0x3FF0000000000000ull));
    if (m > ZK_SQRT2) {
        m = __dmul_rn(m, 0.5);
        e += 1;
    }
    const double s = __ddiv_rn(__dsub_rn(m, 1.0), __dadd_rn(m, 1.0));
    const double s2 = __dmul_rn(s, s);
    double p = ZK_INV_ODD_23;
    p = __fma_rn(p, s2, ZK_INV_ODD_21);
    p = __fma_rn(p, s2, ZK_INV_ODD_19);
    p = __fma_rn(p, s2, ZK_INV_ODD_17);
    p = __fma_rn(p, s2, ZK_INV_ODD_15);
    p = __fma_rn(p, s2, ZK_INV_ODD_13);
    p = __fma_rn(p, s2, ZK_INV_ODD_11);
    p = __fma_rn(p, s2, ZK_INV_ODD_9);
    p = __fma_rn(p, s2, ZK_INV_ODD_7);
    p = __fma_rn(p, s2, ZK_INV_ODD_5);
    p = __fma_rn(p, s2, ZK_INV_ODD_3);
    const double two_s = __dadd_rn(s, s);
    const double log_m = __fma_rn(__dmul_rn(two_s, s2), p, two_s);
    const double de = static_cast<double>(e);
    return __fma_rn(de, ZK_LN2_HIGH, __fma_rn(de, ZK_LN2_LOW, log_m));
}

__device__ __forceinline__ double u53(uint64_t w) { return __dmul_rn(__ull2double_rn(w >> 11), 0x1p-53); }

// The value of element counter c whose first draw missed the fast path
// (also correct, if slower, for one that did not).
__device__ __noinline__ double zig_slow(uint32_t key, uint32_t normal_key, uint32_t c)
{
    uint64_t w = draw64(key, c);
    const uint32_t skey = substream_key(normal_key, c);
    uint32_t k = 0;
    for (uint32_t round = 0; round < kMaxRounds; ++round) {
        const uint32_t j = static_cast<uint32_t>(w) & (kLayers - 1u);
        const bool neg = (w >> 10) & 1u;
        const double x = __dmul_rn(u53(w), kZigX[j]);
        if (x < kZigX[j + 1]) return neg ? -x : x;
        if (j == 0) {
            const double r = kZigX[1];
            for (uint32_t t = 0; t < kMaxRounds; ++t) {
                const double u1 = __dmul_rn(__ull2double_rn((substream64(skey, k) >> 11) + 1u), 0x1p-53);
                const double u2 = __dmul_rn(__ull2double_rn((substream64(skey, k + 1u) >> 11) + 1u), 0x1p-53);
                k += 2u;
                const double a = __ddiv_rn(-zlog(u1), r);
                const double b = -zlog(u2);
                if (__dadd_rn(b, b) >= __dmul_rn(a, a)) {
                    const double z = __dadd_rn(r, a);
                    return neg ? -z : z;
                }
            }
            break;
        }
        const double u = u53(substream64(skey, k));
        k += 1u;
        const double y = __dadd_rn(kZigF[j], __dmul_rn(u, __dsub_rn(kZigF[j + 1], kZigF[j])));
        const double t = __dmul_rn(__dmul_rn(x, x), -0.5);
        if (y < zexp(t)) return neg ? -x : x;
        w = substream64(skey, k);
        k += 1u;
    }
    return __longlong_as_double(0x7FF8000000000000ll);
}

// ---- kernels -----------------------------------------------------------------

__global__ void __launch_bounds__(kTableThreads)
zig_table_pass(uint32_t key, uint32_t first, double *__restrict__ out, uint32_t head, uint32_t n_vec, uint32_t n,
               uint32_t *__restrict__ list, unsigned long long *__restrict__ count, unsigned long long capacity)
{
    __shared__ uint32_t queue[kQueue];
    __shared__ uint32_t queued;
    __shared__ unsigned long long base;
    if (threadIdx.x == 0) queued = 0;
    __syncthreads();
    const uint32_t lane = threadIdx.x & 31u;

    // warp-aggregated append of the lanes' misses to the block's queue
    auto push = [&](bool miss, uint32_t e) {
        const uint32_t ballot = __ballot_sync(0xFFFFFFFFu, miss);
        if (ballot) {
            uint32_t slot0 = 0;
            if (lane == 0) slot0 = atomicAdd(&queued, static_cast<uint32_t>(__popc(ballot)));
            slot0 = __shfl_sync(0xFFFFFFFFu, slot0, 0);
            if (miss) {
                const uint32_t slot = slot0 + __popc(ballot & ((1u << lane) - 1u));
                if (slot < kQueue) queue[slot] = e;
            }
        }
    };

    const uint32_t v_begin = blockIdx.x * kTableVecPerBlock;
#pragma unroll 2
    for (uint32_t it = 0; it < kTableIters; ++it) {
        const uint32_t v = v_begin + it * kTableThreads + threadIdx.x;
        const uint32_t e0 = head + 2u * v;
        bool miss0 = false, miss1 = false;
        if (v < n_vec) {
            const FastDraw a = zig_fast(draw64_words(key, first + e0));
            const FastDraw b = zig_fast(draw64_words(key, first + e0 + 1u));
            const uint4 u = make_uint4(static_cast<uint32_t>(a.bits), static_cast<uint32_t>(a.bits >> 32),
                                       static_cast<uint32_t>(b.bits), static_cast<uint32_t>(b.bits >> 32));
            __stcs(reinterpret_cast<uint4 *>(out + e0), u);
            miss0 = !a.fast;
            miss1 = !b.fast;
        }
        push(miss0, e0);
        push(miss1, e0 + 1u);
    }
    // the peeled head and tail (at most one element each), by warp 0 of block 0
    if (blockIdx.x == 0 && threadIdx.x < 32u) {
        const uint32_t tail0 = head + 2u * n_vec;
        uint32_t e = 0;
        bool here = false;
        if (threadIdx.x == 0 && head) {
            e = 0;
            here = true;
        } else if (threadIdx.x == 1 && tail0 < n) {
            e = tail0;
            here = true;
        }
        bool miss = false;
        if (here) {
            const FastDraw d = zig_fast(draw64_words(key, first + e));
            out[e] = __longlong_as_double(static_cast<long long>(d.bits));
            miss = !d.fast;
        }
        push(miss, e);
    }
    __syncthreads();
    const uint32_t total = queued;
    if (total == 0) return;
    // one atomic per block; a full queue forces the count past the capacity,
    // which sends the miss pass through the whole-fill walk
    if (threadIdx.x == 0)
        base = atomicAdd(count, total <= kQueue ? static_cast<unsigned long long>(total) : capacity + 1ull);
    __syncthreads();
    if (total <= kQueue) {
        for (uint32_t i = threadIdx.x; i < total; i += kTableThreads) {
            const unsigned long long slot = base + i;
            if (slot < capacity) list[slot] = queue[i];
        }
    }
}

__global__ void __launch_bounds__(kMissThreads)
zig_miss_pass(uint32_t key, uint32_t normal_key, uint32_t first, double *__restrict__ out, uint32_t n,
              const uint32_t *__restrict__ list, const unsigned long long *__restrict__ count,
              unsigned long long capacity)
{
    const unsigned long long misses = *count;
    const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t stride = gridDim.x * blockDim.x;
    if (misses <= capacity) {
        const uint32_t m = static_cast<uint32_t>(misses);
        for (uint32_t i = tid; i < m; i += stride) {
            const uint32_t e = list[i];
            out[e] = zig_slow(key, normal_key, first + e);
        }
    } else {
        for (uint32_t e = tid; e < n; e += stride)
            if (!zig_fast(draw64_words(key, first + e)).fast) out[e] = zig_slow(key, normal_key, first + e);
    }
}

__global__ void eval_f64_kernel(int which, const double *in, double *out, uint32_t n)
{
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        out[i] = which ? zlog(in[i]) : zexp(in[i]);
}

// ---- per-device resources -------------------------------------------------

// The miss list and its counter, allocated on first use and kept to the end
// of the process; fills sharing them are ordered through `last`.
struct ZigDevice {
    std::mutex mu;
    uint32_t *list = nullptr;
    unsigned long long *count = nullptr;
    size_t allocated = 0;
    cudaEvent_t last = nullptr;
    bool recorded = false;
};

std::mutex g_devices_mu;
std::map<int, std::unique_ptr<ZigDevice>> g_devices;
std::atomic<size_t> g_capacity_override{SIZE_MAX};

ZigDevice &device_state(int dev)
{
    std::lock_guard<std::mutex> lock(g_devices_mu);
    auto &slot = g_devices[dev];
    if (!slot) slot.reset(new ZigDevice);
    return *slot;
}

// Expected misses n p (p = 0.42766 %) plus 16 standard deviations and slack.
size_t default_capacity(uint32_t n)
{
    const double mean = static_cast<double>(n) * 0.0042766;
    return static_cast<size_t>(mean + 16.0 * std::sqrt(mean + 1.0) + 4096.0);
}

}  // namespace

void set_miss_capacity_override(size_t cap) { g_capacity_override.store(cap); }

cudaError_t launch_normal_f64(uint32_t seed, uint32_t first, uint32_t n, double *out, cudaStream_t s)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    ZigDevice &z = device_state(dev);
    std::lock_guard<std::mutex> lock(z.mu);

    const size_t want = default_capacity(n);
    if (!z.last && (err = cudaEventCreateWithFlags(&z.last, cudaEventDisableTiming)) != cudaSuccess) return err;
    if (!z.count && cudaMalloc(&z.count, sizeof(unsigned long long)) != cudaSuccess)
        return cudaErrorMemoryAllocation;
    if (z.allocated < want) {
        if (z.recorded && (err = cudaEventSynchronize(z.last)) != cudaSuccess) return err;
        if (z.list) cudaFree(z.list);
        z.list = nullptr;
        z.allocated = 0;
        if (cudaMalloc(&z.list, want * sizeof(uint32_t)) != cudaSuccess) return cudaErrorMemoryAllocation;
        z.allocated = want;
    }
    const size_t cap_override = g_capacity_override.load();
    const unsigned long long capacity = static_cast<unsigned long long>(want < cap_override ? want : cap_override);

    if (z.recorded && (err = cudaStreamWaitEvent(s, z.last, 0)) != cudaSuccess) return err;
    if ((err = cudaMemsetAsync(z.count, 0, sizeof(unsigned long long), s)) != cudaSuccess) return err;

    const uint32_t key = seed_key(seed);
    const uint32_t head = head_elems<double>(out, n);
    const uint32_t n_vec = (n - head) / 2u;
    const uint32_t blocks = n_vec ? (n_vec + kTableVecPerBlock - 1u) / kTableVecPerBlock : 1u;
    zig_table_pass<<<blocks, kTableThreads, 0, s>>>(key, first, out, head, n_vec, n, z.list, z.count, capacity);
    note_launch();

    const uint32_t max_blocks = sm_count() * 4u;
    const uint32_t want_blocks = (n + 8191u) / 8192u;
    const uint32_t miss_blocks = want_blocks < 1u ? 1u : (want_blocks > max_blocks ? max_blocks : want_blocks);
    zig_miss_pass<<<miss_blocks, kMissThreads, 0, s>>>(key, purpose_key(seed, kPurposeNormal64), first, out, n,
                                                       z.list, z.count, capacity);
    note_launch();
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if ((err = cudaEventRecord(z.last, s)) != cudaSuccess) return err;
    z.recorded = true;
    return cudaSuccess;
}

cudaError_t last_miss_count(uint64_t *count)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    ZigDevice &z = device_state(dev);
    std::lock_guard<std::mutex> lock(z.mu);
    if (!z.recorded) {
        *count = 0;
        return cudaSuccess;
    }
    if ((err = cudaEventSynchronize(z.last)) != cudaSuccess) return err;
    unsigned long long c = 0;
    err = cudaMemcpy(&c, z.count, sizeof c, cudaMemcpyDeviceToHost);
    *count = c;
    return err;
}

cudaError_t launch_eval_f64(int which, const double *in, double *out, uint32_t n, cudaStream_t s)
{
    eval_f64_kernel<<<fill_blocks((n + 3u) / 4u), kFillThreads, 0, s>>>(which, in, out, n);
    note_launch();
    return cudaGetLastError();
}

// ---- allocation-free variant (rng_fill_normal_f64_noalloc) ------------------
//
// For callers that cannot call cudaMalloc: the miss counter and the miss list
// live in this file-scope device array instead of the lazily allocated
// per-device list above.  Layout: the 64-bit miss counter in the first 256
// bytes, then kNoAllocListEntries 32-bit list entries (8 MiB + 256 bytes in
// all).  Every device that loads the library holds the array until the
// process exits, and every call shares it: two calls that overlap on the GPU
// race on it (their outputs are then unspecified).  The counter is cleared by
// each call before its table pass.

namespace {

constexpr size_t kNoAllocListEntries = size_t(1) << 21;
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[256 + kNoAllocListEntries * sizeof(uint32_t)];

// Device address of g_noalloc_scratch per device (host code cannot use the
// symbol itself: on the host it names a stand-in, not device memory).
std::atomic<unsigned char *> g_noalloc_addr[kNoAllocMaxDevices];
std::atomic<unsigned> g_noalloc_sms[kNoAllocMaxDevices];

}  // namespace

cudaError_t launch_normal_f64_noalloc(uint32_t seed, uint32_t first, uint32_t n, double *out, cudaStream_t s)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
    unsigned char *scratch = g_noalloc_addr[dev].load();
    if (scratch == nullptr) {
        // set-up on this device's first call, with the device current
        void *addr = nullptr;
        if ((err = cudaGetSymbolAddress(&addr, g_noalloc_scratch)) != cudaSuccess) return err;
        int sms = 0;
        if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
        g_noalloc_sms[dev].store(sms > 0 ? static_cast<unsigned>(sms) : 1u);
        scratch = static_cast<unsigned char *>(addr);
        g_noalloc_addr[dev].store(scratch);
    }
    unsigned long long *count = reinterpret_cast<unsigned long long *>(scratch);
    uint32_t *list = reinterpret_cast<uint32_t *>(scratch + 256);
    const size_t want = default_capacity(n);
    const unsigned long long capacity =
        static_cast<unsigned long long>(want < kNoAllocListEntries ? want : kNoAllocListEntries);

    if ((err = cudaMemsetAsync(count, 0, sizeof(unsigned long long), s)) != cudaSuccess) return err;
    const uint32_t key = seed_key(seed);
    const uint32_t head = head_elems<double>(out, n);
    const uint32_t n_vec = (n - head) / 2u;
    const uint32_t blocks = n_vec ? (n_vec + kTableVecPerBlock - 1u) / kTableVecPerBlock : 1u;
    zig_table_pass<<<blocks, kTableThreads, 0, s>>>(key, first, out, head, n_vec, n, list, count, capacity);
    note_launch();
    const uint32_t max_blocks = g_noalloc_sms[dev].load() * 4u;
    const uint32_t want_blocks = (n + 8191u) / 8192u;
    const uint32_t miss_blocks = want_blocks < 1u ? 1u : (want_blocks > max_blocks ? max_blocks : want_blocks);
    zig_miss_pass<<<miss_blocks, kMissThreads, 0, s>>>(key, purpose_key(seed, kPurposeNormal64), first, out, n,
                                                       list, count, capacity);
    note_launch();
    return cudaGetLastError();
}

}  // namespace rngk
