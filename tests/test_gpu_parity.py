"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bit-exact for every integer, uniform, bounded, dropout and f64-normal fill;
within |err| <= 4e-6 (1 + |z|) for the f32 Box-Muller normal.  Sizes span
several tiles and waves of each kernel plus ragged tails; every fill runs at
the unaligned starts and the counter wrap, with its output at a 16-byte
boundary and one element past it."""
import math

import numpy as np
import pytest

from dropout_lowbias32_hash32_gb300 import workloads

pytestmark = pytest.mark.gpu

U32 = 1 << 32
FIRSTS = (0, 1, 3, U32 - 5)
# 3 waves of the u32 fill (152 SMs x 8 blocks x 256 threads x 4 elements) + a ragged tail
BIG = 3 * 152 * 8 * 256 * 4 + 13
# around the vector width, around one block's run of every generator (256
# threads x 4, 8 or 16 vectors x 16/sizeof(T) elements: 2048 .. 32768) and
# around 2^16 (the pages' small-fill cutoff; this library has none)
SMALL = (1, 2, 3, 5, 15, 16, 17, 31, 33, 1000, 2047, 2048, 2049, 4095, 4096, 4097, 8191, 8192, 8193,
         16383, 16384, 16385, 32767, 32768, 32769, 65535, 65536, 65537)


@pytest.fixture(scope="module")
def torch():
    import torch
    assert torch.cuda.is_available(), "these tests need the GB300"
    return torch


@pytest.fixture(scope="module")
def rng(torch):
    import dropout_lowbias32_hash32_gb300 as rng
    return rng


def _out(torch, dtype, n, offset):
    return torch.empty(n + offset, dtype=dtype, device="cuda")[offset:]


def _bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a).view(np.uint8)


def _host(t):
    return t.cpu().numpy()


def _assert_equal(name, got, want, any_nan=False):
    if any_nan:
        # IEEE 754 leaves the payload of a NaN result open: compare NaN-ness
        # there and bits everywhere else
        nan_g, nan_w = np.isnan(got), np.isnan(want)
        assert np.array_equal(nan_g, nan_w), f"{name}: NaN positions differ"
        got, want = got[~nan_g], want[~nan_w]
    if not np.array_equal(_bits(got), _bits(want)):
        g, w = got.view(np.uint8).reshape(got.size, -1), want.view(np.uint8).reshape(want.size, -1)
        bad = np.nonzero(np.any(g != w, axis=1))[0]
        raise AssertionError(f"{name}: {bad.size} of {got.size} elements differ, first {bad[:8]}: "
                             f"got {got[bad[:4]]} want {want[bad[:4]]}")


# name -> (gpu call(out, first), torch dtype, oracle call(first, n), numpy view dtype)
def fills(rng, torch, orc):
    t = torch
    return {
        "u32": (lambda o, f: rng.rng_fill_u32(0x9E3779B9, f, o), t.int32,
                lambda f, n: orc.fill_u32(0x9E3779B9, f, n).view(np.int32)),
        "u64": (lambda o, f: rng.rng_fill_u64(0x9E3779B9, f, o), t.int64,
                lambda f, n: orc.fill_u64(0x9E3779B9, f, n).view(np.int64)),
        "f32": (lambda o, f: rng.rng_fill_f32(0x9E3779B9, f, o), t.float32,
                lambda f, n: orc.fill_f32(0x9E3779B9, f, n)),
        "f64": (lambda o, f: rng.rng_fill_f64(0x9E3779B9, f, o), t.float64,
                lambda f, n: orc.fill_f64(0x9E3779B9, f, n)),
        "u32_below_1000": (lambda o, f: rng.rng_fill_u32_below(1, f, 1000, o), t.int32,
                           lambda f, n: orc.fill_u32_below(1, f, 1000, n).view(np.int32)),
        "u32_below_2^32-2": (lambda o, f: rng.rng_fill_u32_below(2, f, U32 - 2, o), t.int32,
                             lambda f, n: orc.fill_u32_below(2, f, U32 - 2, n).view(np.int32)),
        "u32_below_2^31+1": (lambda o, f: rng.rng_fill_u32_below(3, f, (1 << 31) + 1, o), t.int32,
                             lambda f, n: orc.fill_u32_below(3, f, (1 << 31) + 1, n).view(np.int32)),
        "u64_below_1000": (lambda o, f: rng.rng_fill_u64_below(3, f, 1000, o), t.int64,
                           lambda f, n: orc.fill_u64_below(3, f, 1000, n).view(np.int64)),
        "u64_below_2^64-2": (lambda o, f: rng.rng_fill_u64_below(4, f, (1 << 64) - 2, o), t.int64,
                             lambda f, n: orc.fill_u64_below(4, f, (1 << 64) - 2, n).view(np.int64)),
        "u64_below_2^63+1": (lambda o, f: rng.rng_fill_u64_below(1, f, (1 << 63) + 1, o), t.int64,
                             lambda f, n: orc.fill_u64_below(1, f, (1 << 63) + 1, n).view(np.int64)),
        "i32_range": (lambda o, f: rng.rng_fill_i32_range(1, f, -500, 1000, o), t.int32,
                      lambda f, n: orc.fill_i32_range(1, f, -500, 1000, n)),
        "i32_range_wrap": (lambda o, f: rng.rng_fill_i32_range(2, f, (1 << 31) - 10, 1000, o), t.int32,
                           lambda f, n: orc.fill_i32_range(2, f, (1 << 31) - 10, 1000, n)),
        "i64_range32": (lambda o, f: rng.rng_fill_i64_range32(3, f, -500, 1000, o), t.int64,
                        lambda f, n: orc.fill_i64_range32(3, f, -500, 1000, n)),
        "i64_range": (lambda o, f: rng.rng_fill_i64_range(4, f, -500, 1000, o), t.int64,
                      lambda f, n: orc.fill_i64_range(4, f, -500, 1000, n)),
        "normal_f64": (lambda o, f: rng.rng_fill_normal_f64(7, f, o), t.float64,
                       lambda f, n: orc.fill_normal_f64(7, f, n)),
        "normal_f32_precise": (lambda o, f: rng.rng_fill_normal_f32_precise(7, f, o), t.float32,
                               lambda f, n: orc.fill_randn_precise(7, f, n)),
        "exponential_f32": (lambda o, f: rng.rng_fill_exponential_f32(13, f, o), t.float32,
                            lambda f, n: orc.fill_exponential_f32_own(13, f, n)),
        "exponential_f64": (lambda o, f: rng.rng_fill_exponential_f64(13, f, o), t.float64,
                            lambda f, n: orc.fill_exponential_f64(13, f, n)),
        "u8": (lambda o, f: rng.rng_fill_u8(0x9E3779B9, f, o), t.uint8,
               lambda f, n: orc.fill_u8(0x9E3779B9, f, n)),
        "u16": (lambda o, f: rng.rng_fill_u16(0x9E3779B9, f, o), t.int16,
                lambda f, n: orc.fill_u16(0x9E3779B9, f, n).view(np.int16)),
        "f16": (lambda o, f: rng.rng_fill_f16(0x9E3779B9, f, o), t.int16,
                lambda f, n: orc.fill_f16_bits(0x9E3779B9, f, n).view(np.int16)),
        "bool": (lambda o, f: rng.rng_fill_bool(0x9E3779B9, f, o), t.uint8,
                 lambda f, n: orc.fill_bool(0x9E3779B9, f, n)),
    }


FILL_NAMES = ["u32", "u64", "f32", "f64", "u32_below_1000", "u32_below_2^32-2", "u32_below_2^31+1",
              "u64_below_1000", "u64_below_2^64-2", "u64_below_2^63+1", "i32_range", "i32_range_wrap",
              "i64_range32", "i64_range", "normal_f64", "u8", "u16", "f16", "bool", "exponential_f32",
              "exponential_f64", "normal_f32_precise"]


@pytest.mark.parametrize("name", FILL_NAMES)
def test_fill_bit_exact_small_and_unaligned(rng, torch, orc, name):
    gpu, dtype, ref = fills(rng, torch, orc)[name]
    for first in FIRSTS:
        for offset in (0, 1):
            for n in SMALL:
                out = gpu(_out(torch, dtype, n, offset), first)
                _assert_equal(f"{name} first={first} offset={offset} n={n}", _host(out), ref(first, n))


@pytest.mark.parametrize("name", FILL_NAMES)
def test_fill_bit_exact_several_waves(rng, torch, orc, name):
    gpu, dtype, ref = fills(rng, torch, orc)[name]
    for first, offset in ((0, 0), (3, 1), (U32 - 5, 0)):
        out = gpu(_out(torch, dtype, BIG, offset), first)
        _assert_equal(f"{name} first={first} offset={offset} n={BIG}", _host(out), ref(first, BIG))


@pytest.mark.parametrize("name", FILL_NAMES)
def test_fill_of_length_zero_writes_nothing(rng, torch, orc, name):
    gpu, dtype, _ = fills(rng, torch, orc)[name]
    guard = torch.full((4,), 7, dtype=dtype, device="cuda")
    gpu(guard[2:2], 0)
    torch.cuda.synchronize()
    assert bool((guard == 7).all())


@pytest.mark.parametrize("name", FILL_NAMES)
def test_fill_leaves_neighbours_untouched(rng, torch, orc, name):
    gpu, dtype, ref = fills(rng, torch, orc)[name]
    for n, offset in ((37, 3), (4099, 1), (4096, 2)):
        buf = torch.full((n + offset + 5,), 7, dtype=dtype, device="cuda")
        gpu(buf[offset:offset + n], 11)
        host = _host(buf)
        assert np.all(host[:offset] == 7) and np.all(host[offset + n:] == 7)
        _assert_equal(name, host[offset:offset + n], ref(11, n))


def test_normal_f32_within_tolerance(rng, torch, orc):
    """|z_gpu - z| <= 4e-6 (1 + |z|) against the oracle's binary64 value."""
    for first, n, offset in ((0, 1 << 22, 0), (1, 4099, 1), (3, 65537, 0), (U32 - 5, BIG, 1)):
        z = _host(rng.rng_fill_normal_f32(7, first, _out(torch, torch.float32, n, offset))).astype(np.float64)
        ref = orc.fill_randn(7, first, n)
        err = np.abs(z - ref) / (1 + np.abs(ref))
        assert err.max() <= 4e-6, (first, n, err.max(), np.argmax(err))


def test_normal_f32_extreme_radius(rng, torch, orc):
    """Counters whose first uniform is the largest grid value 1 - 2^-23 (the
    radius sqrt(46 ln 2)) and those where it is 0 (radius 0)."""
    d = orc.fill_u32(7, 0, 1 << 26)[::2] & 0x7FFFFF
    for target in ((1 << 23) - 1, 0, 1):
        cs = np.nonzero(d == target)[0]
        assert cs.size
        out = torch.empty(1, dtype=torch.float32, device="cuda")
        for c in cs[:4]:
            z = float(_host(rng.rng_fill_normal_f32(7, int(c), out))[0])
            ref = orc.randn(7, int(c))
            assert abs(z - ref) <= 4e-6 * (1 + abs(ref))


def test_normal_f32_pairs_within_tolerance(rng, torch, orc):
    """Paired Box-Muller at every start parity, across the counter wrap and
    with every output offset: within 4e-6 (1 + |z|) of the oracle, and its
    even elements equal to rng_fill_normal_f32's values at counter c / 2."""
    for first in (0, 1, 2, 3, U32 - 5, U32 - 2, U32 - 1):
        for offset in (0, 1, 2, 3):
            for n in (1, 2, 3, 5, 17, 4099, 65537):
                z = _host(rng.rng_fill_normal_f32_pairs(7, first, _out(torch, torch.float32, n, offset)))
                ref = orc.fill_randn_paired(7, first, n)
                err = np.abs(z.astype(np.float64) - ref) / (1 + np.abs(ref))
                assert err.max() <= 4e-6, (first, offset, n, err.max())
    n = BIG
    for first in (0, 1):
        z = _host(rng.rng_fill_normal_f32_pairs(7, first, _out(torch, torch.float32, n, 0)))
        ref = orc.fill_randn_paired(7, first, n)
        assert np.max(np.abs(z.astype(np.float64) - ref) / (1 + np.abs(ref))) <= 4e-6
    pairs = _host(rng.rng_fill_normal_f32_pairs(9, 0, _out(torch, torch.float32, 20000, 0)))
    cos_branch = _host(rng.rng_fill_normal_f32(9, 0, _out(torch, torch.float32, 10000, 0)))
    assert np.array_equal(pairs[0::2].view(np.uint32), cos_branch.view(np.uint32))


def test_exponential_f32_large_and_within_the_bound(rng, torch, orc):
    """The f32 exponential fill, bit-exact against the oracle's own-log value at
    a size of several waves, and within 0.5035 ulp of -ln(1 - u) in binary64
    (at u = 0 exactly +0)."""
    for first, n, offset in ((0, 1 << 22, 0), (U32 - 5, BIG, 3)):
        e = _host(rng.rng_fill_exponential_f32(13, first, _out(torch, torch.float32, n, offset)))
        assert np.array_equal(e.view(np.uint32), orc.fill_exponential_f32_own(13, first, n).view(np.uint32))
        ref = orc.fill_exponential_f32(13, first, n)
        ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
        nz = ref > 0
        assert np.all(np.abs(e[nz].astype(np.float64) - ref[nz]) <= 0.5035 * ulp[nz])
        assert np.all(e[~nz] == 0) and not np.any(np.signbit(e))


@pytest.mark.parametrize("p", [0.1, 0.5, 0.0, 0.999, 2.0 ** -30])
def test_dropout_bit_exact(rng, torch, orc, p):
    for n, first in ((BIG, 0), (4099, U32 - 5), (1, 3), (17, 1)):
        x = workloads.dropout_x(n)
        dy = workloads.dropout_dy(n)
        for offset in (0, 1):
            xg = _out(torch, torch.float32, n, offset)
            xg.copy_(torch.from_numpy(x))
            y = rng.rng_dropout_fwd(xg, _out(torch, torch.float32, n, offset), p, 42, first)
            _assert_equal(f"fwd p={p} n={n} offset={offset}", _host(y), orc.dropout(x, p, 42, first))
            dyg = _out(torch, torch.float32, n, 1 - offset)
            dyg.copy_(torch.from_numpy(dy))
            dx = rng.rng_dropout_bwd(dyg, _out(torch, torch.float32, n, offset), p, 42, first)
            _assert_equal(f"bwd p={p} n={n}", _host(dx), orc.dropout(dy, p, 42, first))
            # the backward pass drops exactly the elements the forward pass dropped
            both = (x != 0) & (dy != 0)
            assert np.array_equal((_host(y) != 0)[both], (_host(dx) != 0)[both])


def test_dropout_special_values_and_in_place(rng, torch, orc):
    sp = workloads.special_floats()
    x = np.tile(sp, 700)
    for p in (0.1, 0.5):
        want = orc.dropout(x, p, 42, 9)
        xg = torch.from_numpy(x).cuda()
        _assert_equal("special", _host(rng.rng_dropout_fwd(xg, torch.empty_like(xg), p, 42, 9)), want,
                      any_nan=True)
        rng.rng_dropout_fwd(xg, xg, p, 42, 9)  # in place
        _assert_equal("in place", _host(xg), want, any_nan=True)


def test_dropout_mixed_alignment_takes_the_scalar_path(rng, torch, orc):
    n = 100003
    x = workloads.dropout_x(n)
    xg = _out(torch, torch.float32, n, 1)
    xg.copy_(torch.from_numpy(x))
    for offset in (0, 2, 3):
        y = rng.rng_dropout_fwd(xg, _out(torch, torch.float32, n, offset), 0.5, 42, 5)
        _assert_equal(f"mixed offset {offset}", _host(y), orc.dropout(x, 0.5, 42, 5))


def test_dropout_every_alignment(rng, torch, orc):
    """Every offset of x within 32 bytes, with y at the same offset (32-byte
    kernel), 16 bytes away (16-byte kernel) and 4 bytes away (scalar kernel),
    and in place: every element equals the oracle's."""
    n = 100003
    x = workloads.dropout_x(n + 8)
    for ox in range(8):
        xs = x[ox:ox + n]
        want = orc.dropout(xs, 0.3, 42, 7)
        buf = torch.empty(n + 16, dtype=torch.float32, device="cuda")  # 256-byte aligned
        buf[:n + 8].copy_(torch.from_numpy(x))
        xg = buf[ox:ox + n]
        for oy in (ox, (ox + 4) % 8, (ox + 1) % 8):
            y = rng.rng_dropout_fwd(xg, _out(torch, torch.float32, n, oy), 0.3, 42, 7)
            _assert_equal(f"x offset {ox}, y offset {oy}", _host(y), want)
        rng.rng_dropout_fwd(xg, xg, 0.3, 42, 7)
        _assert_equal(f"in place at offset {ox}", _host(xg), want)


def test_slow_path_exp_log_bit_exact(rng, torch, orc):
    """The ziggurat slow path's own exp and log, layer by layer."""
    g = np.random.default_rng(4)
    t = np.concatenate([g.uniform(-10, 0, 1 << 20), -np.linspace(0, 10, 4097), [0.0, -0.0]])
    out = torch.empty(t.size, dtype=torch.float64, device="cuda")
    _assert_equal("zexp", _host(rng.rng_debug_eval_f64(0, torch.from_numpy(t).cuda(), out)), orc.zexp_array(t))
    x = np.concatenate([g.uniform(0, 1, 1 << 20), 2.0 ** -g.uniform(0, 53, 1 << 18),
                        1 - g.integers(1, 1 << 20, 4096) * 2.0 ** -53, [2.0 ** -53, 0.5, 1.0]])
    x = x[x > 0]
    out = torch.empty(x.size, dtype=torch.float64, device="cuda")
    _assert_equal("zlog", _host(rng.rng_debug_eval_f64(1, torch.from_numpy(x).cuda(), out)), orc.zlog_array(x))


def test_f64_fixed_point_log_on_chosen_inputs(rng, torch, orc):
    """The f64 exponential's fixed-point log on the device, on the oracle pin's
    inputs (every table bin edge at the two largest exponents, edge values and
    random inputs of every bit length) and 2^20 more, bit for bit."""
    import pins
    g = np.random.default_rng(6)
    m = np.concatenate([pins._neglog64_sample(), g.integers(0, 1 << 53, 1 << 20, dtype=np.uint64)])
    out = torch.empty(m.size, dtype=torch.float64, device="cuda")
    got = _host(rng.rng_debug_eval_f64(2, torch.from_numpy(m.view(np.float64)).cuda(), out))
    _assert_equal("neglog64", got, orc.neglog64_array(m))


def test_normal_f64_miss_list_overflow_walks_the_fill(rng, torch, orc):
    """A list too short for the misses (capacity 0 and 5) sends the second
    kernel through the whole fill: the values must not change."""
    n = 65537
    want = orc.fill_normal_f64(7, 3, n)
    try:
        for cap in (0, 5, 300):
            rng.rng_debug_set_miss_capacity(cap)
            out = rng.rng_fill_normal_f64(7, 3, _out(torch, torch.float64, n, 1))
            _assert_equal(f"capacity {cap}", _host(out), want)
            assert rng.rng_debug_last_miss_count() > cap
    finally:
        rng.rng_debug_set_miss_capacity(None)
    out = rng.rng_fill_normal_f64(7, 3, _out(torch, torch.float64, n, 0))
    _assert_equal("default capacity", _host(out), want)


# The share of the table pass's elements that take the exact integer product
# instead of the fma (its kIntMask: this many of every eight).
INT_PRODUCT_FRACTION = 2 / 8


def deferred_bounds(n):
    """Bounds on the fast draws the table pass defers to the second kernel:
    INT_PRODUCT_FRACTION of the elements take the integer product, which
    defers a draw when the 10 or 11 discarded bits it sees are exactly one
    half (probability 2^-10 or 2^-11), within 5 standard deviations."""
    lo, hi = n * INT_PRODUCT_FRACTION * 2.0 ** -11, n * INT_PRODUCT_FRACTION * 2.0 ** -10
    return lo - 5 * math.sqrt(lo), hi + 5 * math.sqrt(hi) + 1e-5 * n


def test_normal_f64_miss_count(rng, torch, orc):
    """The oracle's fast path misses 0.42766 % of the elements (tandem-sycl
    'Design', Normals: 0.43 %); the table pass lists those and the few fast
    draws it defers."""
    n = 1 << 24
    rng.rng_fill_normal_f64(7, 0, torch.empty(n, dtype=torch.float64, device="cuda"))
    got = rng.rng_debug_last_miss_count()
    want = int(n - orc.fill_zig_fast(7, 0, n).astype(np.int64).sum())
    lo, hi = deferred_bounds(n)
    assert lo < got - want < hi, (got, want)
    p = 0.0042766
    assert abs(want - p * n) < 5 * math.sqrt(p * n)


@pytest.mark.parametrize("name", ["u32", "u64_below_1000", "i64_range", "normal_f64", "exponential_f32", "u8",
                                  "normal_f32_precise"])
def test_resume_from_a_counter(rng, torch, orc, name):
    """Checkpoint and resume: a stream position is (seed, next counter), so a
    fill done in pieces, each started at first_counter + its offset, equals
    the fill done at once (the ziggurat's misses included)."""
    gpu, dtype, _ = fills(rng, torch, orc)[name]
    n, first = 1 << 20, U32 - 70000  # the counters wrap inside the fill
    whole = _host(gpu(_out(torch, dtype, n, 0), first))
    cuts = [0, 12345, 12346, 500001, n]
    parts = [_host(gpu(_out(torch, dtype, b - a, a % 3), (first + a) % U32)) for a, b in zip(cuts, cuts[1:])]
    assert np.array_equal(_bits(np.concatenate(parts)), _bits(whole))


@pytest.mark.parametrize("world", [2, 3, 8])
def test_ranks_counter_ranges_concatenate_to_the_fill(rng, torch, orc, world):
    """The multi-process split (sharding.py) simulated on one GPU: each rank's
    slice, filled independently from its own first counter, concatenates in
    rank order to the single-process fill (no rank waits on another)."""
    from dropout_lowbias32_hash32_gb300 import sharding
    n, first = 1000003, U32 - 12345
    for name in ("u64_below_1000", "normal_f64", "exponential_f64", "u8"):
        gpu, dtype, _ = fills(rng, torch, orc)[name]
        whole = _host(gpu(_out(torch, dtype, n, 0), first))
        parts = []
        for rank in range(world):
            off, length = sharding.shard(n, rank, world)
            parts.append(_host(gpu(_out(torch, dtype, length, 0), sharding.first_counter(first, off))))
        assert np.array_equal(_bits(np.concatenate(parts)), _bits(whole)), (name, world)


def _near_half_draws(X, gen, count):
    """64-bit ziggurat draws whose product m X[j] (m = w >> 11) lies exactly on,
    just above or just below the midpoint between two binary64 values: m
    solves m M = 2^(s-1) + delta (mod 2^s) for X[j]'s significand M, s the
    number of discarded bits, so the rounding is decided by delta alone."""
    out = []
    while len(out) < count:
        j = int(gen.integers(0, 1024))
        lead = int(gen.integers(33, 53))           # m's top bit (w's is lead + 11, so hi != 0)
        m_lo, e = math.frexp(float(X[j]))
        M = int(m_lo * (1 << 53))
        t = (M & -M).bit_length() - 1               # M = M' 2^t
        Mo = M >> t
        delta = [0, 1 << t, -(1 << t), 1 << (t + 20), -(1 << (t + 20))][len(out) % 5]
        for s_bits in (lead, lead + 1):
            mod = 1 << (s_bits - t)
            target = (1 << (s_bits - 1)) + delta
            if target % (1 << t):
                continue
            m0 = ((target >> t) * pow(Mo, -1, mod)) % mod
            k_lo = -(-((1 << lead) - m0) // mod)
            k_hi = ((1 << (lead + 1)) - 1 - m0) // mod
            if k_lo > k_hi:
                continue
            m = m0 + mod * int(gen.integers(k_lo, k_hi + 1))
            if (m * M).bit_length() - 53 != s_bits:
                continue
            out.append((m << 11) | (int(gen.integers(0, 2)) << 10) | j)
            break
    return np.array(out, dtype=np.uint64)


def test_ziggurat_integer_product(rng, torch, orc):
    """The table pass's integer product against the oracle's rounded product
    (and the fma form against both): equal bit for bit, or NaN where it defers
    the draw, and it defers only where hi = 0 or the product's discarded part
    starts with exactly one half at T's resolution (10 or 11 bits).  Random
    draws, every layer, every count of leading zeros, and constructed draws
    on, just above and just below a rounding midpoint."""
    from fractions import Fraction
    X, _ = orc.zig1024()
    gen = np.random.default_rng(11)
    w = gen.integers(0, 1 << 63, 1 << 18, dtype=np.uint64) * np.uint64(2) + gen.integers(0, 2, 1 << 18, dtype=np.uint64)
    w[:1024] = (w[:1024] & ~np.uint64(1023)) | np.arange(1024, dtype=np.uint64)
    w[1024:1088] >>= np.arange(64, dtype=np.uint64)
    w = np.concatenate([w, _near_half_draws(X, gen, 2000), np.array([0, 2047, (1 << 32) - 1, 1 << 32, (1 << 64) - 1],
                                                                       dtype=np.uint64)])
    ref = orc.zig_candidates(w)
    inp = torch.from_numpy(w.view(np.float64)).cuda()
    fma = _host(rng.rng_debug_eval_f64(4, inp, torch.empty_like(inp)))
    integer = _host(rng.rng_debug_eval_f64(3, inp, torch.empty_like(inp)))
    assert np.array_equal(fma.view(np.uint64), ref.view(np.uint64))
    deferred = np.isnan(integer)
    assert np.array_equal(integer[~deferred].view(np.uint64), ref[~deferred].view(np.uint64))
    for wi in w[deferred].tolist():
        if wi >> 32 == 0:
            continue
        exact = Fraction(wi >> 11, 1 << 53) * Fraction(float(X[wi & 1023]))
        _, e = math.frexp(float(exact))
        frac = exact * Fraction(2) ** (53 - e)
        frac -= math.floor(frac)
        assert Fraction(1, 2) <= frac < Fraction(1, 2) + Fraction(1, 1 << 10), hex(wi)
    # the constructed midpoints: an exact tie or just above it defers, just below it does not
    near = w[(1 << 18):(1 << 18) + 2000]
    kinds = np.arange(near.size) % 5
    near_int = integer[(1 << 18):(1 << 18) + 2000]
    assert np.all(np.isnan(near_int[(kinds == 0) | (kinds == 1)]))
    assert not np.any(np.isnan(near_int[(kinds == 2) | (kinds == 4)]))
    assert deferred[:1 << 18].mean() < 2e-3  # random draws: about 7.3e-4


def test_normal_f64_unrolled_table_pass(rng, torch, orc):
    """A fill long enough for the table pass's four-step loop (one product in
    eight by the integer form), with a one-element head (output 8 bytes off a
    16-byte boundary), a ragged tail and counters that wrap: every element
    equals the oracle's."""
    n = (1 << 22) + 5
    first = U32 - 3
    out = rng.rng_fill_normal_f64(7, first, _out(torch, torch.float64, n, 1))
    _assert_equal("normal_f64 2^22 + 5", _host(out), orc.fill_normal_f64(7, first, n))


def test_normal_f64_streams_share_the_miss_list(rng, torch, orc):
    """Fills on two streams use the same per-device miss list in turn."""
    n = 1 << 20
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for k in range(6):
        s = s1 if k % 2 == 0 else s2
        o = torch.empty(n, dtype=torch.float64, device="cuda")
        o.record_stream(s)
        with torch.cuda.stream(s):
            rng.rng_fill_normal_f64(7, k * n, o)
        outs.append(o)
    torch.cuda.synchronize()
    for k, o in enumerate(outs):
        _assert_equal(f"stream fill {k}", _host(o), orc.fill_normal_f64(7, k * n, n))


def test_normal_f64_from_concurrent_host_threads(rng, torch, orc):
    """Four host threads, each on its own stream, fill concurrently (the C
    calls release the GIL); sizes grow so that the shared miss list is
    reallocated while other threads' fills are queued.  Every output equals
    the oracle's."""
    import threading
    sizes = [1 << 16, 1 << 20, 3 << 20, 1 << 22]
    results, errors = {}, []

    def work(t):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for k, n in enumerate(sizes[t:] + sizes[:t]):
                    o = torch.empty(n, dtype=torch.float64, device="cuda")
                    rng.rng_fill_normal_f64(100 + t, k * 977, o)
                    results[(t, k)] = (n, o)
            s.synchronize()
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for (t, k), (n, o) in sorted(results.items()):
        _assert_equal(f"thread {t} fill {k}", _host(o), orc.fill_normal_f64(100 + t, k * 977, n))


def test_launch_counts(rng, torch):
    o32 = torch.empty(1 << 16, dtype=torch.float32, device="cuda")
    o64 = torch.empty(1 << 16, dtype=torch.float64, device="cuda")
    before = rng.rng_debug_launch_count()
    rng.rng_fill_f32(1, 0, o32)
    rng.rng_fill_normal_f32(1, 0, o32)
    rng.rng_dropout_fwd(o32, o32, 0.5, 1, 0)
    assert rng.rng_debug_launch_count() - before == 3
    before = rng.rng_debug_launch_count()
    rng.rng_fill_normal_f64(1, 0, o64)
    assert rng.rng_debug_launch_count() - before == 2


def test_zero_high_word_of_the_64_bit_draw(rng, torch, orc):
    """hash32(0) = 0, so draw32(seed, c) = 0 exactly at c = hash32(seed): for a
    seed with even hash32(seed) the 64-bit draw at c = hash32(seed) / 2 (and
    c + 2^31) has a zero high word, the one case in 2^32 the f64 conversions
    take out of line.  Checked at both elements of a 16-byte vector (the f64
    fill converts the first by an fma, the second by integer operations with
    a branch for this case), in the peeled head and in the tail."""
    seeds = [s for s in range(1, 64) if orc.hash32(s) % 2 == 0][:3]
    assert seeds
    for seed in seeds:
        for c in (orc.hash32(seed) >> 1, (orc.hash32(seed) >> 1) + (1 << 31)):
            assert orc.fill_u64(seed, c, 1)[0] >> 32 == 0
            # (first, offset): c at index 6 (a vector's first element), 1 (its
            # second), 0 behind an 8-byte offset (the head), 4 behind it (a
            # second element) and 63 behind it (the tail)
            for first, offset in ((c - 6, 0), (c - 1, 0), (c, 1), (c - 4, 1), (c - 63, 1)):
                first &= U32 - 1
                got = _host(rng.rng_fill_f64(seed, first, _out(torch, torch.float64, 64, offset)))
                assert np.array_equal(got.view(np.uint64), orc.fill_f64(seed, first, 64).view(np.uint64))
                assert got[(c - first) % U32] < 2.0 ** -32
                got = _host(rng.rng_fill_exponential_f64(seed, first, _out(torch, torch.float64, 64, offset)))
                assert np.array_equal(got.view(np.uint64), orc.fill_exponential_f64(seed, first, 64).view(np.uint64))


@pytest.mark.gpu
def test_write_ceiling_hook_writes_what_it_states(rng, torch):
    """The measurement aid behind bench.py's write ceiling: the store kernel
    writes vector index v to each word of 16-byte vector v, memset 0x5A bytes."""
    n_vec = 3 * 1024 + 17  # several blocks' runs and a ragged last run
    buf = torch.empty(n_vec * 4, dtype=torch.int32, device="cuda")
    before = rng.rng_debug_launch_count()
    rng.rng_debug_write_ceiling(1, buf)
    assert rng.rng_debug_launch_count() - before == 1
    got = _host(buf).view(np.uint32).reshape(n_vec, 4)
    assert np.array_equal(got, np.repeat(np.arange(n_vec, dtype=np.uint32)[:, None], 4, axis=1))
    rng.rng_debug_write_ceiling(0, buf)
    assert np.all(_host(buf).view(np.uint8) == 0x5A)


def test_fill_longer_than_one_piece(rng, torch, orc):
    """n > 2^31 is split into pieces of 2^31 elements; the seam is invisible
    (a fill, the ziggurat with its miss lists, and dropout with its input)."""
    n = (1 << 31) + 1000
    out = rng.rng_fill_u32(5, U32 - 7, torch.empty(n, dtype=torch.int32, device="cuda"))
    idx = np.concatenate([np.arange(0, 64), np.arange((1 << 31) - 64, (1 << 31) + 64), np.arange(n - 64, n),
                          np.random.default_rng(1).integers(0, n, 1 << 16)])
    got = _host(out[torch.from_numpy(idx).cuda()])
    _assert_equal("u32 > 2^31", got, orc.fill_u32(5, U32 - 7, idx=idx).view(np.int32))
    del out
    out = rng.rng_fill_normal_f64(7, 1, torch.empty(n, dtype=torch.float64, device="cuda"))
    got = _host(out[torch.from_numpy(idx).cuda()])
    _assert_equal("normal_f64 > 2^31", got, orc.fill_normal_f64(7, 1, idx=idx))
    del out
    torch.cuda.empty_cache()
    # dropout reads its input piece by piece: x[i] = (i mod 1001) - 500, counters from first = 11
    x = (torch.arange(n, device="cuda", dtype=torch.int64) % 1001 - 500).to(torch.float32)
    y = rng.rng_dropout_fwd(x, torch.empty_like(x), 0.3, 42, 11)
    got = _host(y[torch.from_numpy(idx).cuda()])
    xs = ((idx % 1001) - 500).astype(np.float32)
    _assert_equal("dropout > 2^31", got, orc.dropout(xs, 0.3, 42, 11, idx=idx))
    del x, y
    torch.cuda.empty_cache()


def test_bad_arguments_raise(rng, torch):
    o = torch.empty(8, dtype=torch.float32, device="cuda")
    with pytest.raises(rng.RngError):
        rng.rng_dropout_fwd(o, o, 1.0, 1, 0)
    with pytest.raises(rng.RngError):
        rng.rng_fill_u32_below(1, 0, 0, torch.empty(8, dtype=torch.int32, device="cuda"))
    with pytest.raises(rng.RngError):
        rng.rng_dropout_fwd(o[:6], o[2:8], 0.5, 1, 0)
    with pytest.raises(TypeError):
        rng.rng_fill_u32(1, 0, torch.empty(8, dtype=torch.int32))


def test_degenerate_bounds(rng, torch, orc):
    """bound 1 gives zeros; the largest bounds (2^32 - 1, 2^64 - 1) reject
    almost nothing and still match the oracle bit for bit."""
    n = 70001
    out32 = torch.empty(n, dtype=torch.int32, device="cuda")
    out64 = torch.empty(n, dtype=torch.int64, device="cuda")
    assert not bool(rng.rng_fill_u32_below(1, 5, 1, out32).any())
    assert not bool(rng.rng_fill_u64_below(1, 5, 1, out64).any())
    for b in (2, U32 - 1):
        _assert_equal(f"u32_below {b}", _host(rng.rng_fill_u32_below(6, U32 - 3, b, out32)),
                      orc.fill_u32_below(6, U32 - 3, b, n).view(np.int32))
    for b in (2, (1 << 64) - 1, 1 << 63):
        _assert_equal(f"u64_below {b}", _host(rng.rng_fill_u64_below(6, U32 - 3, b, out64)),
                      orc.fill_u64_below(6, U32 - 3, b, n).view(np.int64))
    lo = -(1 << 63)
    _assert_equal("i64_range extremes", _host(rng.rng_fill_i64_range(6, 1, lo, (1 << 64) - 1, out64)),
                  orc.fill_i64_range(6, 1, lo, (1 << 64) - 1, n))


def test_dropout_largest_p_drops_everything(rng, torch, orc):
    p = float(np.nextafter(np.float32(1), np.float32(0)))  # 1 - 2^-24
    x = workloads.dropout_x(4099)
    y = rng.rng_dropout_fwd(torch.from_numpy(x).cuda(), torch.empty(4099, device="cuda"), p, 42, 0)
    assert np.all(_host(y).view(np.uint32) == 0)
    _assert_equal("p max", _host(y), orc.dropout(x, p, 42, 0))


def test_fill_longer_than_the_counter_period(rng, torch, orc):
    """n > 2^32 elements: counters wrap inside one call, so element i + 2^32
    repeats element i (u8 fill: 4 GiB)."""
    n = (1 << 32) + 1000
    out = rng.rng_fill_u8(5, 7, torch.empty(n, dtype=torch.uint8, device="cuda"))
    head = _host(out[:1000])
    assert np.array_equal(_host(out[1 << 32:]), head)
    idx = np.concatenate([np.arange(1000), np.random.default_rng(3).integers(0, n, 1 << 16)])
    _assert_equal("u8 > 2^32", _host(out[torch.from_numpy(idx).cuda()]), orc.fill_u8(5, 7, idx=idx))
    del out
    torch.cuda.empty_cache()
