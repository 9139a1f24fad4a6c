// normal_f64.cu -- f64 standard normals by a 1024-layer Marsaglia-Tsang
// ziggurat in two kernels: a table pass that writes every element and lists
// the misses, and a miss pass that resolves them.
//
// tandem-sycl "Design", section Normals: one 64-bit draw per element; 0.43 %
// of draws miss the fast path and continue on a substream keyed by the
// draw's global index, so a fill cut at any element equals the whole fill;
// misses are queued locally and appended to a device list with one atomic
// add (here: per-warp queues in shared memory, flushed 32 entries at a time;
// the few fast draws the integer product cannot round join them);
// the second kernel takes one miss per thread and, if the list overflowed,
// walks the whole fill again; the layer table is not in constant memory,
// which serialises lanes that read different layers (here: the table pass
// reads 8 bank-staggered shared-memory replicas, the slow path global
// memory through L1); the fast path makes no calls.
//
// Misses of the base layer (1.3 % of misses) need two logarithms and a
// division, the others (wedges) one exponential: the table pass keeps them in
// two lists so that the miss pass runs each kind in dense warps instead of
// holding a warp of wedges for one tail lane.
//
// Draw w = D64(seed, c): layer j = w & 1023, sign = bit 10, m = w >> 11 (53
// bits); x = RNE((m 2^-53) X[j]); fast iff x < X[j+1].  GB300's FP64 pipe
// retires 2 fma per SM and cycle (1/64 of FP32), so the fast path spends at
// most one FP64 instruction per element: t = 1 + (m mod 2^52) 2^-52 is
// assembled from the draw's bits, and fma(t, X[j]/2, b ? 0 : -X[j]/2) with
// b = bit 52 of m equals (m 2^-53) X[j] before its single rounding, so it
// returns the IEEE product bit for bit.  One element in four takes the same
// product in exact integer arithmetic instead (scaled_by_u53_int), which
// moves work from the FP64 pipe to the ALU and FMA pipes.  The table pass
// computes -|x| (scaled_by_u53_neg: the fma's operands are built by
// multiply-adds on the FMA pipe rather than logic ops on the ALU pipe) and
// sets the draw's sign with one logic op.
//
// Miss of layer 0: the tail beyond r = X[1] (Marsaglia 1964: a = -log(U1)/r,
// b = -log(U2), accept when 2b >= a^2, value r + a, U in (0, 1]).  Miss of
// layer j >= 1: the wedge test y = F[j] + U (F[j+1] - F[j]) < exp(-x^2/2);
// a rejected wedge starts over with the substream's next 64-bit word.  The
// substream words are taken in that order.  exp and log are this file's own
// fixed sequences of IEEE operations (Cody & Waite reduction + Taylor for
// exp; exponent split + atanh series for log), so the slow path returns the
// same bits on every IEEE machine.  The miss pass stores each resolved value
// with its three sector neighbours (recomputed) as one 32-byte sector, since
// a lone 8-byte store into an output that has left L2 costs a
// read-modify-write of the sector in HBM.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <map>
#include <memory>
#include <mutex>
#include <type_traits>

#include "fill_kernel.cuh"
#include "hash32.cuh"
#include "internal.h"
#include "f64_math.cuh"
#include "zig_tables.inc"

namespace rngk {
namespace {

constexpr uint32_t kLayers = 1024;

// Layer table, global memory, read through the read-only path.
__device__ const double kZigX[kLayers + 1] = {ZIG_X_VALUES};
__device__ const double2 kZigHalfXNext[kLayers] = {ZIG_HALFX_XNEXT_VALUES};  // {X[j]/2, X[j+1]}
__device__ const double2 kZigFHalfDiff[kLayers] = {ZIG_F_HALFDIFF_VALUES};   // {F[j], (F[j+1]-F[j])/2}

// Table pass: one persistent block of 1024 threads per SM.  The block keeps
// kTableCopies copies of the {X[j]/2, X[j+1]} table in shared memory, copy q
// in 16-byte bank group q (entry j of copy q at index 8j + q); lane l reads
// copy l mod 8, so the eight lanes of each quarter-warp phase of a 16-byte
// gather hit eight different bank groups whatever their layers: 4 wavefronts
// per warp instead of one per distinct cache line from L1.
constexpr uint32_t kTableThreads = 1024;
constexpr uint32_t kTableCopies = 8;
constexpr uint32_t kTableWarps = kTableThreads / 32u;
// Each warp queues its misses (element index, bit 31 set for a base-layer
// miss) in shared memory and flushes them 32 at a time with one atomic per
// list; two pushes of up to 32 entries can follow a flush check.
constexpr uint32_t kWarpQueue = 96;
constexpr size_t kTableSmem =
    kLayers * kTableCopies * sizeof(uint4) + kTableWarps * kWarpQueue * sizeof(uint32_t);
constexpr uint32_t kMissThreads = 128;
constexpr uint32_t kMissBlocksPerSm = 12;  // 48 resident warps per SM (at most 42 registers)
constexpr uint32_t kMaxRounds = 4096;  // rejection rounds of one miss (never reached)

// Where the table pass lists its misses: counts[0] wedge misses, counts[1]
// base-layer (tail) misses; a count above its capacity means the list
// overflowed and the miss pass walks the whole fill.
struct MissList {
    unsigned long long *counts;
    uint32_t *wedge;
    uint32_t *tail;
    unsigned long long wedge_cap, tail_cap;
};

// ---- fast path ------------------------------------------------------------

// RNE((m 2^-53) v) for the 64-bit word w = hi:lo, m = w >> 11, from half_v =
// v/2 (v positive normal), in one fma: t = 1 + (m mod 2^52) 2^-52 is
// assembled from the word's bits; with b = bit 52 of m, t v/2 - (1 - b) v/2
// = (m 2^-53) v exactly, and the fma rounds that value once.
__device__ __forceinline__ double scaled_by_u53(Words w, double half_v)
{
    const uint32_t t_lo = __funnelshift_r(w.lo, w.hi, 11);
    const uint32_t t_hi = ((w.hi >> 11) & 0xFFFFFu) | 0x3FF00000u;
    const uint32_t keep = static_cast<uint32_t>(static_cast<int32_t>(w.hi) >> 31);  // all ones iff b
    const uint32_t c_hi = (static_cast<uint32_t>(__double2hiint(half_v)) ^ 0x80000000u) & ~keep;
    const uint32_t c_lo = static_cast<uint32_t>(__double2loint(half_v)) & ~keep;
    return __fma_rn(__hiloint2double(static_cast<int>(t_hi), static_cast<int>(t_lo)), half_v,
                    __hiloint2double(static_cast<int>(c_hi), static_cast<int>(c_lo)));
}

// The top 32 bits of v's 53-bit significand, its leading 1 at bit 31, from
// half_v = v/2 (v positive normal): the integer product's multiplier.
__host__ __device__ __forceinline__ uint32_t significand_hi(uint32_t half_v_hi, uint32_t half_v_lo)
{
    return ((half_v_hi << 11) | (half_v_lo >> 21)) | 0x80000000u;
}

// The same product with no FP64 instruction: RNE((m 2^-53) v) for m = w >> 11
// and v = 2 half_v, bit for bit what scaled_by_u53 returns.  m is normalised,
// n = (w with its low 11 bits cleared) << clz(hi) in [2^63, 2^64), and v's
// significand sits at the top of a 64-bit word (sig_hi from the table, the
// low word half_v's low word << 11; both have 53 significant bits).  The high
// 64 bits T of their 128-bit product hold the mantissa (T >> 11, or T >> 10
// when T's top bit is clear) and the first 10 or 11 discarded bits; r, those
// bits left-aligned, gives the rounding: below one half (r < 2^31) round
// down, above it round up.  At exactly one half in T the low 64 bits would
// decide a tie, and for hi = 0 (m < 2^32) the normalisation needs the low
// word; both return false (about 7e-4 of draws) and the element takes the
// miss pass, which recomputes it with the fma.  The exponent is v/2's, plus
// T's top bit, minus the normalising shift.
template <bool kNegative>
__device__ __forceinline__ bool scaled_by_u53_int(Words w, uint32_t v_hi, uint32_t v_lo, uint32_t sig_hi,
                                                  uint64_t &bits)
{
    const uint32_t z = __clz(w.hi);
    const uint32_t m_lo = w.lo & 0xFFFFF800u;
    const uint64_t n = (static_cast<uint64_t>(__funnelshift_l(m_lo, w.hi, z)) << 32) | (m_lo << z);
    const uint64_t sig = (static_cast<uint64_t>(sig_hi) << 32) | (v_lo << 11);
    const uint64_t T = __umul64hi(n, sig);
    const uint32_t t_hi = static_cast<uint32_t>(T >> 32), t_lo = static_cast<uint32_t>(T);
    const uint32_t top = t_hi >> 31;
    const uint32_t shift = 10u + top;
    const uint32_t r = t_lo << (22u - top);
    // biased exponent minus the mantissa's leading 1; with kNegative the sign
    // bit rides above it (0x800 - 1), so the result is -RNE(...)
    const uint32_t exponent = ((v_hi >> 20) + (kNegative ? 0x7FFu : 0xFFFFFFFFu) + top - z) << 20;
    bits = ((static_cast<uint64_t>((t_hi >> shift) + exponent) << 32) | __funnelshift_r(t_lo, t_hi, shift)) + (r >> 31);
    return (r != 0x80000000u) & (w.hi != 0u);
}

__device__ __forceinline__ bool scaled_by_u53_int(Words w, double half_v, uint64_t &bits)
{
    const uint32_t v_hi = static_cast<uint32_t>(__double2hiint(half_v));
    const uint32_t v_lo = static_cast<uint32_t>(__double2loint(half_v));
    return scaled_by_u53_int<false>(w, v_hi, v_lo, significand_hi(v_hi, v_lo), bits);
}

// Powers of two for mad_lo / mad_hi, passed to the table pass as an argument.
struct Pow2 {
    uint32_t p20, p21;
};

// -RNE((m 2^-53) v) for w = hi:lo, m = w >> 11, from half_v = v/2 (words
// v_hi, v_lo), in one fma: with t = 1 + (m mod 2^52) 2^-52 and b = bit 52 of
// m, fma(-t, v/2, (1 - b) v/2) = -(m 2^-53) v before its single rounding.
// keep = -b (all ones iff b); -t's high word is (hi >> 11) - b 2^20 +
// 0xBFF00000 (sign, exponent 1023, top 20 fraction bits) and (1 - b) v/2 is
// v/2 keep + v/2 word by word: multiply-adds, no logic op.
__device__ __forceinline__ double scaled_by_u53_neg(Words w, uint32_t v_hi, uint32_t v_lo, Pow2 p)
{
    const uint32_t t_lo = __funnelshift_r(w.lo, w.hi, 11);
    const uint32_t keep = static_cast<uint32_t>(static_cast<int32_t>(w.hi) >> 31);
    const uint32_t t_hi = mad_lo(keep, p.p20, mad_hi(w.hi, p.p21, 0xBFF00000u));
    const uint32_t c_hi = mad_lo(v_hi, keep, v_hi), c_lo = mad_lo(v_lo, keep, v_lo);
    return __fma_rn(__hiloint2double(static_cast<int>(t_hi), static_cast<int>(t_lo)),
                    __hiloint2double(static_cast<int>(v_hi), static_cast<int>(v_lo)),
                    __hiloint2double(static_cast<int>(c_hi), static_cast<int>(c_lo)));
}

struct FastDraw {
    uint64_t bits;  // the signed fast-path value
    bool fast;
    bool base;      // the draw's layer is 0 (a miss goes to the tail)
};

__device__ __forceinline__ FastDraw zig_fast(Words w)
{
    const uint32_t j = w.lo & (kLayers - 1u);
    const double2 e = __ldg(&kZigHalfXNext[j]);
    const uint64_t xb = static_cast<uint64_t>(__double_as_longlong(scaled_by_u53(w, e.x)));
    FastDraw d;
    // both values are non-negative, so their bit patterns order like them
    d.fast = xb < static_cast<uint64_t>(__double_as_longlong(e.y));
    d.bits = xb | (static_cast<uint64_t>(w.lo & 0x400u) << 53);  // bit 10 -> sign bit
    d.base = j == 0;
    return d;
}

// zig_fast with the product by the integer form where it decides (the fma
// where it defers): the same values, with no FP64 instruction in the
// common case.
__device__ __forceinline__ double scaled_by_u53_any(Words w, double half_v);
__device__ __forceinline__ FastDraw zig_fast_int(Words w)
{
    const uint32_t j = w.lo & (kLayers - 1u);
    const double2 e = __ldg(&kZigHalfXNext[j]);
    const uint64_t xb = static_cast<uint64_t>(__double_as_longlong(scaled_by_u53_any(w, e.x)));
    FastDraw d;
    d.fast = xb < static_cast<uint64_t>(__double_as_longlong(e.y));
    d.bits = xb | (static_cast<uint64_t>(w.lo & 0x400u) << 53);
    d.base = j == 0;
    return d;
}

// ---- slow path --------------------------------------------------------------

// ((w >> 11) + 1) 2^-53, in (0, 1]
__device__ __forceinline__ double u53_open(Words w)
{
    const uint64_t m = ((static_cast<uint64_t>(w.hi) << 32 | w.lo) >> 11) + 1u;
    return __dmul_rn(__ull2double_rn(m), 0x1p-53);
}

// The value of element counter c whose first draw missed the fast path
// (also correct, if slower, for one that did not).  skf is the element's
// substream key, folded: its 64-bit word k is draw64_words(skf, k).
// The wedge test y < zexp(-x^2/2), y = F[j] + U (F[j+1] - F[j]) with U the
// wedge word's (w >> 11) 2^-53, is decided in binary32 where that is safe:
// +1 (accept) or -1 (reject) when y lies outside exp(-x^2/2) (1 -+ 2^-16),
// else 0 (take the exact test).  GB300 converts binary64 on its narrow FP64
// pipe, so the binary32 operands are built from bits: x, F[j] and
// (F[j+1] - F[j])/2 as binary32 truncations (relative error below 2^-23
// each), U as the word's top 23 bits (1 + U32 from the bits, minus 1, exact;
// U - U32 < 2^-23).  Then -x^2/2 carries at most 3 2^-23 + 2^-24 of
// |x^2/2| <= 8.2 and __expf its documented 2 + 1.173 |t| ulp.  y32 =
// fma(U32, 2 D32, F32) is within 2^-23 F + 2^-22 (F[j+1] - F[j]) + 2^-24 y
// of y, and (F[j+1] - F[j]) / F[j] <= 1.06 over the layers (largest at
// j = 1), so within 2^-21 y.  With the margin's product the estimate is
// within 5.5e-6 (2^-17.4) of the exact comparison, inside the margin of
// 1.5e-5 (2^-16).  zexp is within 2 ulp of binary64 exp, so a screened
// decision is the exact one and the values stay those of the exact test.
// Candidates inside the margin (about one in 10^3) build the binary64 y and
// take the exact test; the screened path spends no FP64 instruction.
__device__ __forceinline__ float float_rz_of_positive(double d)
{
    // a normal binary64 in binary32's range, truncated: the 11-bit exponent
    // and the top 23 mantissa bits sit in bits 23..33 and 0..22 of the word
    // shifted right by 29; rebias the exponent by 1023 - 127 modulo 2^32
    const uint32_t w = __funnelshift_r(static_cast<uint32_t>(__double2loint(d)),
                                       static_cast<uint32_t>(__double2hiint(d)), 29);
    return __uint_as_float(w - (896u << 23));
}

__device__ __forceinline__ int wedge_screen(double x, double2 f, Words u)
{
    const float x32 = float_rz_of_positive(x);
    const float e32 = __expf(__fmul_rn(__fmul_rn(x32, x32), -0.5f));
    const float u32 = __fsub_rn(__uint_as_float(0x3F800000u | (u.hi >> 9)), 1.0f);
    const float y32 = __fmaf_rn(u32, __fmul_rn(float_rz_of_positive(f.y), 2.0f), float_rz_of_positive(f.x));
    if (y32 < __fmul_rn(e32, 1.0f - 0x1p-16f)) return 1;
    if (y32 > __fmul_rn(e32, 1.0f + 0x1p-16f)) return -1;
    return 0;
}

// The fast path's product of draw w with v = 2 half_v, by the integer form
// where it decides and the fma where it defers.
__device__ __forceinline__ double scaled_by_u53_any(Words w, double half_v)
{
    uint64_t bits;
    if (scaled_by_u53_int(w, half_v, bits)) return __longlong_as_double(static_cast<long long>(bits));
    return scaled_by_u53(w, half_v);
}

// x with its sign bit set when neg, by an integer operation (a negation of a
// double may otherwise take GB300's narrow FP64 pipe)
__device__ __forceinline__ double with_sign(double x, bool neg)
{
    return __longlong_as_double(__double_as_longlong(x) | (static_cast<long long>(neg) << 63));
}

__device__ __noinline__ double zig_slow(uint32_t key, uint32_t normal_key, uint32_t c)
{
    Words w = draw64_words(key, c);
    const uint32_t skf = fold_key(substream_key(normal_key, c));
    uint32_t k = 0;
    for (uint32_t round = 0; round < kMaxRounds; ++round) {
        const uint32_t j = w.lo & (kLayers - 1u);
        const bool neg = w.lo & 0x400u;
        const double2 e = __ldg(&kZigHalfXNext[j]);
        const double x = scaled_by_u53_any(w, e.x);
        if (__double_as_longlong(x) < __double_as_longlong(e.y)) return with_sign(x, neg);
        if (j == 0) {
            const double r = kZigX[1];
            for (uint32_t t = 0; t < kMaxRounds; ++t) {
                const double u1 = u53_open(draw64_words(skf, k));
                const double u2 = u53_open(draw64_words(skf, k + 1u));
                k += 2u;
                const double a = __ddiv_rn(-zlog(u1), r);
                const double b = -zlog(u2);
                if (__dadd_rn(b, b) >= __dmul_rn(a, a)) {
                    const double z = __dadd_rn(r, a);
                    return with_sign(z, neg);
                }
            }
            break;
        }
        const double2 f = __ldg(&kZigFHalfDiff[j]);
        const Words u = draw64_words(skf, k);
        k += 1u;
        const int screen = wedge_screen(x, f, u);
        if (screen > 0) return with_sign(x, neg);
        if (screen == 0) {
            const double y = __dadd_rn(f.x, scaled_by_u53(u, f.y));
            if (y < zexp(__dmul_rn(__dmul_rn(x, x), -0.5))) return with_sign(x, neg);
        }
        w = draw64_words(skf, k);
        k += 1u;
    }
    return __longlong_as_double(0x7FF8000000000000ll);
}

// ---- kernels -----------------------------------------------------------------

// Write element e's resolved value v.  The table pass has written the whole
// output and its lines have long left L2, so a lone 8-byte store makes L2 read
// the rest of its 32-byte sector back from HBM (a read-modify-write at a
// random address for every miss; that, not the slow path, set the miss
// pass's time).  So the other three elements of e's sector are recomputed by
// the fast path (the integer product, which leaves the FP64 pipe to the slow
// path; the fma where it defers), whose values equal the table pass's, and
// the four are stored as one 32-byte sector.  If a neighbour also missed (about 1.3 % of
// sectors) or the sector runs past either end of the fill, only e is stored:
// the neighbour's own thread writes its value.
__device__ __forceinline__ void store_resolved(double *__restrict__ out, uint32_t n, uint32_t key, uint32_t first,
                                               uint32_t e, double v)
{
    const uint32_t pos = static_cast<uint32_t>((reinterpret_cast<uintptr_t>(out + e) >> 3) & 3u);
    if (e >= pos && e - pos + 3u < n) {
        const uint32_t s0 = e - pos;
        unsigned long long b[4];
        bool all = true;
#pragma unroll
        for (uint32_t k = 0; k < 4u; ++k) {
            if (k == pos) {
                b[k] = static_cast<unsigned long long>(__double_as_longlong(v));
            } else {
                const FastDraw d = zig_fast_int(draw64_words(key, first + s0 + k));
                b[k] = d.bits;
                all = all && d.fast;
            }
        }
        if (all) {
            asm volatile("st.global.v4.b64 [%0], {%1, %2, %3, %4};" ::"l"(out + s0), "l"(b[0]), "l"(b[1]), "l"(b[2]),
                         "l"(b[3])
                         : "memory");
            return;
        }
    }
    out[e] = v;
}

// Flush the first `cnt` (<= 32) entries of a warp's queue to the global
// lists (one atomic per list), then move the rest of the queue down.
__device__ __forceinline__ void warp_queue_flush(uint32_t *q, uint32_t &qn, uint32_t cnt, const MissList &ml)
{
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t below = (1u << lane) - 1u;
    __syncwarp();
    const bool have = lane < cnt;
    const uint32_t e = have ? q[lane] : 0u;
    const bool tail = have && (e >> 31);
    const uint32_t tails = __ballot_sync(0xFFFFFFFFu, tail);
    const uint32_t wedges = __ballot_sync(0xFFFFFFFFu, have && !tail);
    unsigned long long wbase = 0, tbase = 0;
    if (lane == 0) {
        if (wedges) wbase = atomicAdd(&ml.counts[0], static_cast<unsigned long long>(__popc(wedges)));
        if (tails) tbase = atomicAdd(&ml.counts[1], static_cast<unsigned long long>(__popc(tails)));
    }
    wbase = __shfl_sync(0xFFFFFFFFu, wbase, 0);
    tbase = __shfl_sync(0xFFFFFFFFu, tbase, 0);
    if (tail) {
        const unsigned long long slot = tbase + __popc(tails & below);
        if (slot < ml.tail_cap) ml.tail[slot] = e & 0x7FFFFFFFu;
    } else if (have) {
        const unsigned long long slot = wbase + __popc(wedges & below);
        if (slot < ml.wedge_cap) ml.wedge[slot] = e;
    }
    const uint32_t rest = qn - cnt;
    const uint32_t r0 = lane < rest ? q[cnt + lane] : 0u;
    const uint32_t r1 = lane + 32u < rest ? q[cnt + 32u + lane] : 0u;
    __syncwarp();
    if (lane < rest) q[lane] = r0;
    if (lane + 32u < rest) q[32u + lane] = r1;
    __syncwarp();
    qn = rest;
}

// The table pass's shared-memory entry of layer j, 16 bytes: X[j]/2 (low,
// high word; the fma's multiplier), the high word of -X[j+1] (the fast test
// on -x) and significand_hi of X[j] (the integer product's multiplier).
__device__ __forceinline__ uint4 table_entry(uint32_t j)
{
    const double2 e = __ldg(&kZigHalfXNext[j]);
    const uint32_t lo = static_cast<uint32_t>(__double2loint(e.x)), hi = static_cast<uint32_t>(__double2hiint(e.x));
    return make_uint4(lo, hi, static_cast<uint32_t>(__double2hiint(e.y)) | 0x80000000u, significand_hi(hi, lo));
}

// Elements taking the integer product: bit k of kIntMask for the second
// element of step k of each group of four steps, bit 4 + k for the first.
// GB300 retires 2 DFMA per SM and cycle; with one product in four on the
// integer pipes the FP64, ALU and FMA pipes are about equally loaded (one in
// eight left the FP64 pipe 85 % busy, three in eight moved the load onto the
// ALU pipe and ran slower).
constexpr uint32_t kIntMask = 0x05u;  // steps 0 and 2, second element: one product in four

// Fast path with the layer table in shared memory (this lane's copy), by the
// fma (integer = false) or the integer product (a draw it cannot decide is a
// miss).  Both give y = -|x|.  The test compares high words only: y and
// -X[j+1] are negative, so as unsigned words a smaller high word of y means
// |x| < X[j+1]; an equal one (about 1e-6 of draws) is sent to the miss pass,
// whose full test decides it.  y is -|x| except where x = 0 (m = 0: the
// fma's exact zero sum is +0), so the value takes |y| with the draw's sign
// (bit 10) as its sign bit: one three-input logic op.
template <bool kInteger>
__device__ __forceinline__ FastDraw zig_fast_shared(Words w, const uint4 *my_copy, Pow2 p)
{
    const uint32_t j = w.lo & (kLayers - 1u);
    const uint4 t = my_copy[j * kTableCopies];
    uint64_t yb;
    bool exact = true;
    if constexpr (kInteger) {
        exact = scaled_by_u53_int<true>(w, t.y, t.x, t.w, yb);
    } else {
        yb = static_cast<uint64_t>(__double_as_longlong(scaled_by_u53_neg(w, t.y, t.x, p)));
    }
    FastDraw d;
    const uint32_t y_hi = static_cast<uint32_t>(yb >> 32);
    d.fast = exact & (y_hi < t.z);
    const uint32_t sign = w.lo << 21;  // bit 10 at bit 31
    d.bits = (static_cast<uint64_t>((y_hi & 0x7FFFFFFFu) | (sign & 0x80000000u)) << 32) | static_cast<uint32_t>(yb);
    d.base = j == 0;
    return d;
}



// kEven: the first counter of every vector is even, so the four 32-bit draws
// of a vector's two elements share one first xorshift (draw64_pair_words).
template <bool kEven>
__global__ void __launch_bounds__(kTableThreads, 1)
zig_table_pass(uint32_t key, uint32_t first, double *__restrict__ out, uint32_t head, uint32_t n_vec, uint32_t n,
               MissList ml, Pow2 p)
{
    extern __shared__ __align__(16) unsigned char smem[];
    uint4 *table = reinterpret_cast<uint4 *>(smem);
    uint32_t *queues = reinterpret_cast<uint32_t *>(smem + kLayers * kTableCopies * sizeof(uint4));
    for (uint32_t i = threadIdx.x; i < kLayers * kTableCopies; i += kTableThreads) table[i] = table_entry(i / kTableCopies);
    __syncthreads();

    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t below = (1u << lane) - 1u;
    uint32_t *q = queues + (threadIdx.x >> 5) * kWarpQueue;
    uint32_t qn = 0;  // warp-uniform
    const uint4 *my_copy = table + (lane & (kTableCopies - 1u));

    auto push = [&](bool miss, bool base, uint32_t e) {
        const uint32_t ballot = __ballot_sync(0xFFFFFFFFu, miss);
        if (miss) q[qn + __popc(ballot & below)] = e | (static_cast<uint32_t>(base) << 31);
        qn += __popc(ballot);
    };
    // One 16-byte vector (two elements) per lane and step: draws, products
    // and the streaming store.  int_a / int_b (constant at each call) select
    // the integer product for the first / second element.  Returns the
    // step's miss and base-layer flags: bits 0, 1 (first, second element
    // missed) and 2, 3 (their layer is 0).
    auto compute = [&](uint32_t v, auto int_a, auto int_b) -> uint32_t {
        const uint32_t e0 = head + 2u * v;
        Words wa, wb;
        if constexpr (kEven) {
            draw64_pair_words(key, first + e0, wa, wb);
        } else {
            wa = draw64_words(key, first + e0);
            wb = draw64_words(key, first + e0 + 1u);
        }
        const FastDraw a = zig_fast_shared<decltype(int_a)::value>(wa, my_copy, p);
        const FastDraw b = zig_fast_shared<decltype(int_b)::value>(wb, my_copy, p);
        const uint4 u = make_uint4(static_cast<uint32_t>(a.bits), static_cast<uint32_t>(a.bits >> 32),
                                   static_cast<uint32_t>(b.bits), static_cast<uint32_t>(b.bits >> 32));
        __stcs(reinterpret_cast<uint4 *>(out + e0), u);
        return static_cast<uint32_t>(!a.fast) | (static_cast<uint32_t>(!b.fast) << 1) |
               (static_cast<uint32_t>(a.base) << 2) | (static_cast<uint32_t>(b.base) << 3);
    };
    // Misses are rare (a warp step of 64 elements has one with probability
    // 0.24), so the queue is touched only when the warp's vote finds one.
    auto record = [&](uint32_t v, uint32_t flags) {
        if (__any_sync(0xFFFFFFFFu, (flags & 3u) != 0u)) {
            const uint32_t e0 = head + 2u * v;
            push((flags & 1u) != 0u, (flags & 4u) != 0u, e0);
            push((flags & 2u) != 0u, (flags & 8u) != 0u, e0 + 1u);
            while (qn >= 32u) warp_queue_flush(q, qn, 32u, ml);
        }
    };
    using FMA = std::false_type;
    auto I = [](auto bit) { return std::integral_constant<bool, ((kIntMask >> decltype(bit)::value) & 1u) != 0>{}; };

    // warp-uniform stride over 16-byte vectors: each warp stores 512
    // contiguous bytes per step; whole warps four steps at a time, then
    // whole warps, then the ragged end.  A group of four steps computes and
    // stores all eight elements before it votes on any miss, so that their
    // products (GB300's FP64 pipe has a long latency) overlap instead of
    // each step's vote waiting for its own (2 % of the fill); kIntMask picks
    // the group's integer products.
    const uint32_t stride = gridDim.x * kTableThreads;
    uint32_t vb = blockIdx.x * kTableThreads + (threadIdx.x & ~31u);
    for (; vb + 3u * stride + 32u <= n_vec; vb += 4u * stride) {
        const uint32_t f0 = compute(vb + lane, I(std::integral_constant<int, 4>{}), I(std::integral_constant<int, 0>{}));
        const uint32_t f1 =
            compute(vb + stride + lane, I(std::integral_constant<int, 5>{}), I(std::integral_constant<int, 1>{}));
        const uint32_t f2 =
            compute(vb + 2u * stride + lane, I(std::integral_constant<int, 6>{}), I(std::integral_constant<int, 2>{}));
        const uint32_t f3 =
            compute(vb + 3u * stride + lane, I(std::integral_constant<int, 7>{}), I(std::integral_constant<int, 3>{}));
        record(vb + lane, f0);
        record(vb + stride + lane, f1);
        record(vb + 2u * stride + lane, f2);
        record(vb + 3u * stride + lane, f3);
    }
    for (; vb + 32u <= n_vec; vb += stride) record(vb + lane, compute(vb + lane, FMA{}, FMA{}));
    for (; vb < n_vec; vb += stride) {
        const bool valid = vb + lane < n_vec;
        record(vb + lane, valid ? compute(vb + lane, FMA{}, FMA{}) : 0u);
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
        FastDraw d{};
        if (here) {
            d = zig_fast_shared<false>(draw64_words(key, first + e), my_copy, p);
            out[e] = __longlong_as_double(static_cast<long long>(d.bits));
        }
        push(here && !d.fast, d.base, e);
        while (qn >= 32u) warp_queue_flush(q, qn, 32u, ml);
    }
    if (qn) warp_queue_flush(q, qn, qn, ml);
}

__global__ void __launch_bounds__(kMissThreads, kMissBlocksPerSm)
zig_miss_pass(uint32_t key, uint32_t normal_key, uint32_t first, double *__restrict__ out, uint32_t n,
              MissList ml)
{
    const unsigned long long nw = ml.counts[0], nt = ml.counts[1];
    const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t stride = gridDim.x * blockDim.x;
    if (nw <= ml.wedge_cap && nt <= ml.tail_cap) {
        // each list entry's index is loaded one entry ahead, so that its L2
        // latency overlaps the current entry's work
        uint32_t i = tid;
        uint32_t e = i < nw ? ml.wedge[i] : 0u;
        for (; i < nw; i += stride) {
            const uint32_t next = i + stride < nw ? ml.wedge[i + stride] : 0u;
            store_resolved(out, n, key, first, e, zig_slow(key, normal_key, first + e));
            e = next;
        }
        for (i = tid; i < nt; i += stride) {
            const uint32_t t = ml.tail[i];
            store_resolved(out, n, key, first, t, zig_slow(key, normal_key, first + t));
        }
    } else {
        // the list overflowed: every element is written again, since the
        // table pass leaves a deferred draw's value to this pass
        for (uint32_t e = tid; e < n; e += stride) {
            const FastDraw d = zig_fast(draw64_words(key, first + e));
            out[e] = d.fast ? __longlong_as_double(static_cast<long long>(d.bits)) : zig_slow(key, normal_key, first + e);
        }
    }
}

// The fast path's magnitude RNE((m 2^-53) X[j]) of the 64-bit draw w (j = w &
// 1023, m = w >> 11): by the integer product (NaN where it defers the draw)
// or by the fma.
__device__ double zig_candidate(unsigned long long w, bool integer)
{
    // the table pass's forms (they return -|x|, or +0), from its table
    // entry, with the sign bit cleared
    const Words words{static_cast<uint32_t>(w >> 32), static_cast<uint32_t>(w)};
    const uint4 t = table_entry(words.lo & (kLayers - 1u));
    uint64_t bits;
    if (!integer)
        bits = static_cast<uint64_t>(__double_as_longlong(scaled_by_u53_neg(words, t.y, t.x, Pow2{1u << 20, 1u << 21})));
    else if (!scaled_by_u53_int<true>(words, t.y, t.x, t.w, bits))
        return __longlong_as_double(0x7FF8000000000000ll);
    return __longlong_as_double(static_cast<long long>(bits & 0x7FFFFFFFFFFFFFFFull));
}

__global__ void eval_f64_kernel(int which, const double *in, double *out, uint32_t n)
{
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    {
        const unsigned long long bits = static_cast<unsigned long long>(__double_as_longlong(in[i]));
        out[i] = which == 4   ? zig_candidate(bits, false)
                 : which == 3 ? zig_candidate(bits, true)
                 : which == 2 ? neglog64(bits & 0x1FFFFFFFFFFFFFull)
                 : which      ? zlog(in[i])
                              : zexp(in[i]);
    }
}

// Expected entries of n elements plus 16 standard deviations and slack: the
// misses (p = 0.42766 %, of which the base layer's 5.36e-5) and the draws the
// integer product defers (about 7.3e-4 of the kIntMask elements, at most
// 8e-4 of them, in their layer's list).
size_t wedge_capacity(uint32_t n)
{
    const double int_fraction = __builtin_popcount(kIntMask) / 8.0;
    const double mean = static_cast<double>(n) * (0.0042766 + 8e-4 * int_fraction);
    return static_cast<size_t>(mean + 16.0 * std::sqrt(mean + 1.0) + 4096.0);
}

size_t tail_capacity(uint32_t n)
{
    const double mean = static_cast<double>(n) * (5.36e-5 + 1e-7);
    return static_cast<size_t>(mean + 16.0 * std::sqrt(mean + 1.0) + 1024.0);
}

constexpr int kMaxDevices = 64;
std::atomic<bool> g_table_smem_set[kMaxDevices];  // dynamic shared memory limit raised on the device

// Table pass + miss pass of one piece into the lists of `ml` (counts cleared
// here first).
cudaError_t enqueue_ziggurat(uint32_t seed, uint32_t first, uint32_t n, double *out, const MissList &ml,
                             unsigned sms, cudaStream_t s)
{
    cudaError_t err = cudaMemsetAsync(ml.counts, 0, 2 * sizeof(unsigned long long), s);
    if (err != cudaSuccess) return err;
    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!g_table_smem_set[dev].load()) {
        err = cudaFuncSetAttribute(zig_table_pass<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(kTableSmem));
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(zig_table_pass<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kTableSmem));
        if (err != cudaSuccess) return err;
        g_table_smem_set[dev].store(true);
    }
    const uint32_t key = seed_key(seed);
    const uint32_t head = head_elems<double>(out, n);
    const uint32_t n_vec = (n - head) / 2u;
    const uint32_t want = (n_vec + kTableThreads - 1u) / kTableThreads;
    const uint32_t blocks = want < 1u ? 1u : (want < sms ? want : sms);
    // element head + 2v has counter first + head + 2v: even for every vector
    // iff first + head is
    const Pow2 p{1u << 20, 1u << 21};
    if (((first + head) & 1u) == 0u)
        zig_table_pass<true><<<blocks, kTableThreads, kTableSmem, s>>>(key, first, out, head, n_vec, n, ml, p);
    else
        zig_table_pass<false><<<blocks, kTableThreads, kTableSmem, s>>>(key, first, out, head, n_vec, n, ml, p);
    note_launch();
    const uint32_t max_blocks = sms * kMissBlocksPerSm;
    const uint32_t want_blocks = (n + 4095u) / 4096u;
    const uint32_t walk_blocks = want_blocks < 1u ? 1u : (want_blocks > max_blocks ? max_blocks : want_blocks);
    // about one list entry per thread (a thread's entries are resolved one
    // after another, each a chain of dependent loads and hashes), and at
    // least the grid that walks the whole fill if the lists overflow
    const unsigned long long list_blocks = (ml.wedge_cap + ml.tail_cap + kMissThreads - 1u) / kMissThreads;
    const uint32_t miss_blocks = list_blocks > walk_blocks ? static_cast<uint32_t>(list_blocks) : walk_blocks;
    zig_miss_pass<<<miss_blocks, kMissThreads, 0, s>>>(key, purpose_key(seed, kPurposeNormal64), first, out, n, ml);
    note_launch();
    return cudaGetLastError();
}

// ---- per-device resources -------------------------------------------------

// The miss lists and their counters, allocated on first use (grown when a
// longer fill needs more) and kept to the end of the process; fills sharing
// them are ordered through `last`.
struct ZigDevice {
    std::mutex mu;
    unsigned char *buffer = nullptr;  // counters (256 bytes), wedge list, tail list
    size_t wedge_alloc = 0, tail_alloc = 0;
    unsigned long long *counts = nullptr;
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

}  // namespace

void set_miss_capacity_override(size_t cap) { g_capacity_override.store(cap); }

cudaError_t launch_normal_f64(uint32_t seed, uint32_t first, uint32_t n, double *out, cudaStream_t s)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    ZigDevice &z = device_state(dev);
    std::lock_guard<std::mutex> lock(z.mu);

    const size_t want_w = wedge_capacity(n), want_t = tail_capacity(n);
    if (!z.last && (err = cudaEventCreateWithFlags(&z.last, cudaEventDisableTiming)) != cudaSuccess) return err;
    if (z.wedge_alloc < want_w || z.tail_alloc < want_t) {
        if (z.recorded && (err = cudaEventSynchronize(z.last)) != cudaSuccess) return err;
        const size_t w = want_w > z.wedge_alloc ? want_w : z.wedge_alloc;
        const size_t t = want_t > z.tail_alloc ? want_t : z.tail_alloc;
        if (z.buffer) cudaFree(z.buffer);
        z.buffer = nullptr;
        z.wedge_alloc = z.tail_alloc = 0;
        if (cudaMalloc(&z.buffer, 256 + (w + t) * sizeof(uint32_t)) != cudaSuccess) {
            cudaGetLastError();  // an allocation failure is not sticky: clear it
            return cudaErrorMemoryAllocation;
        }
        z.wedge_alloc = w;
        z.tail_alloc = t;
        z.counts = reinterpret_cast<unsigned long long *>(z.buffer);
    }
    const size_t cap = g_capacity_override.load();
    MissList ml;
    ml.counts = z.counts;
    ml.wedge = reinterpret_cast<uint32_t *>(z.buffer + 256);
    ml.tail = ml.wedge + z.wedge_alloc;
    ml.wedge_cap = static_cast<unsigned long long>(want_w < cap ? want_w : cap);
    ml.tail_cap = static_cast<unsigned long long>(want_t < cap ? want_t : cap);

    if (z.recorded && (err = cudaStreamWaitEvent(s, z.last, 0)) != cudaSuccess) return err;
    if ((err = enqueue_ziggurat(seed, first, n, out, ml, sm_count(), s)) != cudaSuccess) return err;
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
    unsigned long long c[2] = {0, 0};
    err = cudaMemcpy(c, z.counts, sizeof c, cudaMemcpyDeviceToHost);
    *count = c[0] + c[1];
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
// For callers that cannot call cudaMalloc: the miss counters and lists live
// in this file-scope device array instead of the lazily allocated per-device
// buffer above.  Layout: the two 64-bit miss counters in the first 256 bytes,
// then kNoAllocWedgeEntries wedge entries and kNoAllocTailEntries tail
// entries of 32 bits (8 MiB + 256 bytes in all).  Every device that loads the
// library holds the array until the process exits, and every call shares it:
// two calls that overlap on the GPU race on it (their outputs are then
// unspecified).  The counters are cleared by each call before its table pass.

namespace {

constexpr size_t kNoAllocTailEntries = size_t(1) << 16;
constexpr size_t kNoAllocWedgeEntries = (size_t(1) << 21) - kNoAllocTailEntries;
constexpr int kNoAllocMaxDevices = kMaxDevices;

static __device__ __align__(256) unsigned char
    g_noalloc_scratch[256 + (kNoAllocWedgeEntries + kNoAllocTailEntries) * sizeof(uint32_t)];

// Device address of g_noalloc_scratch per device (host code cannot use the
// symbol itself: on the host it names a stand-in, not device memory).  Looked
// up once per device and kept, like g_table_smem_set: both would be stale
// after a cudaDeviceReset of the primary context, which the library does not
// expect of its callers.
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
    MissList ml;
    ml.counts = reinterpret_cast<unsigned long long *>(scratch);
    ml.wedge = reinterpret_cast<uint32_t *>(scratch + 256);
    ml.tail = ml.wedge + kNoAllocWedgeEntries;
    const size_t want_w = wedge_capacity(n), want_t = tail_capacity(n);
    ml.wedge_cap = static_cast<unsigned long long>(want_w < kNoAllocWedgeEntries ? want_w : kNoAllocWedgeEntries);
    ml.tail_cap = static_cast<unsigned long long>(want_t < kNoAllocTailEntries ? want_t : kNoAllocTailEntries);
    return enqueue_ziggurat(seed, first, n, out, ml, g_noalloc_sms[dev].load(), s);
}

}  // namespace rngk
