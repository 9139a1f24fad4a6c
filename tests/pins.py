"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each pin takes an ``oracle.Oracle`` and raises AssertionError when the facts
do not hold.  ``test_oracle_pins.py`` runs every pin on the oracle;
``test_oracle_mutations.py`` plants plausible mistakes in copies of the
oracle and checks that a pin fails on each.  The facts come from the pages
(worked examples under tests/golden/, each cited there), from closed forms and
from exhaustive or brute-force enumeration on small cases.
"""
from __future__ import annotations

import math

import numpy as np
from scipy import special, stats

from helpers import golden

U32 = 1 << 32
U64 = 1 << 64


def _ulps(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.abs(a - b) / np.spacing(np.maximum(np.abs(a), np.abs(b)))


# ---------------------------------------------------------------- hash32 ---
def pin_tile_mean(orc):
    """Phobos 'Random numbers' tile figure: seed 1, counters (r + iota(0)) * 32
    + iota(1) over an 8 x 32 tile, mean 0.513, every value k * 2^-23 in [0, 1)."""
    g = golden("phobos_uniform_tile.txt")
    rows, cols, seed = int(g["rows"]), int(g["cols"]), int(g["seed"])
    c = (np.arange(rows)[:, None] * cols + np.arange(cols)[None, :]).ravel()
    u = orc.fill_f32(seed, 0, idx=c).astype(np.float64)
    assert round(float(u.mean()), 3) == float(g["mean_3dp"]), u.mean()
    scaled = u * 2.0 ** -int(g["grid_log2"])
    assert np.all(scaled == np.floor(scaled)) and np.all((u >= 0) & (u < 1))


def pin_uniform_grid(orc):
    """Every uniform is a multiple of 2^-23 in [0, 1); 2^24 consecutive counters
    give 2^24 distinct draws (a bijection of the counter), and the uniform is
    the draw's low 23 bits.  (No chi-square here: hash32 of consecutive
    counters has a small but detectable bias in 1024-bin histograms at 2^24
    draws, a property of the method itself.)"""
    seed = 0x9E3779B9
    u = orc.fill_f32(seed, 0, 1 << 24).astype(np.float64)
    k = u * 2.0 ** 23
    assert np.all(k == np.floor(k)) and k.min() >= 0 and k.max() < 2 ** 23
    d = orc.fill_u32(seed, 0, 1 << 24)
    assert np.array_equal(d & 0x7FFFFF, k.astype(np.uint32))
    d.sort()
    assert np.all(np.diff(d) != 0)


def pin_hash_bijective(orc):
    """lowbias32 is a bijection of the 32-bit words (odd multipliers and
    xorshifts are invertible): undo each step with its inverse and recover the
    counter; the seed enters only as the XOR key hash32(seed)."""
    rng = np.random.default_rng(5)
    c = rng.integers(0, U32, 1 << 18, dtype=np.uint64)
    seed = 0x12345678
    y = orc.fill_u32(seed, 0, idx=c).astype(np.uint64)
    m1, m2 = 2146121005, (-2073254261) % U32
    inv1, inv2 = pow(m1, -1, U32), pow(m2, -1, U32)
    x = y ^ (y >> 16)
    x = (x * inv2) & 0xFFFFFFFF
    x = x ^ (x >> 15) ^ (x >> 30)
    x = (x * inv1) & 0xFFFFFFFF
    x = x ^ (x >> 16)
    assert np.array_equal(x ^ orc.hash32(seed), c)


# --------------------------------------------------------- 64-bit draws ----
def pin_draw64_words(orc):
    """The 64-bit draw holds the 32-bit draw at 2c in its high word and the one
    at 2c + 1 in its low word, 2c wrapping mod 2^32; the f64 uniform is its top
    53 bits times 2^-53, exactly."""
    seed = 0x9E3779B9
    c = np.array([0, 1, 3, (1 << 31) - 1, 1 << 31, (1 << 31) + 5, U32 - 5, U32 - 1], np.uint64)
    d64 = orc.fill_u64(seed, 0, idx=c)
    hi = orc.fill_u32(seed, 0, idx=(2 * c) % U32).astype(np.uint64)
    lo = orc.fill_u32(seed, 0, idx=(2 * c + 1) % U32).astype(np.uint64)
    assert np.array_equal(d64, (hi << np.uint64(32)) | lo)
    f = orc.fill_f64(seed, 0, idx=c)
    assert np.array_equal(f * 2.0 ** 53, (d64 >> np.uint64(11)).astype(np.float64))
    assert np.all((f >= 0) & (f < 1))


def pin_narrow_fills(orc):
    """The narrow fills carve the pinned 32-bit draws: four u8 (two u16)
    elements at counters 4w .. 4w + 3 (2w, 2w + 1) are draw32(seed, w) in
    little-endian order, and 32 bool elements at 32w .. 32w + 31 are its
    bits, least significant first; the f16 element is numpy's binary16 of
    (u16 & 0x3FF) 2^-10, a multiple of 2^-10 in [0, 1); bools are fair."""
    seed, words = 0x9E3779B9, 4096
    w = orc.fill_u32(seed, 0, words)
    assert np.array_equal(orc.fill_u8(seed, 0, 4 * words).view("<u4"), w)
    assert np.array_equal(orc.fill_u16(seed, 0, 2 * words).view("<u4"), w)
    bits = orc.fill_bool(seed, 0, 32 * words).reshape(words, 32).astype(np.uint64)
    assert np.array_equal((bits << np.arange(32, dtype=np.uint64)).sum(axis=1).astype(np.uint32), w)
    u16 = orc.fill_u16(seed, 5, 1 << 16)
    f16 = orc.fill_f16_bits(seed, 5, 1 << 16)
    expect = ((u16 & 0x3FF).astype(np.float64) * 2.0 ** -10).astype(np.float16)
    assert np.array_equal(f16, expect.view(np.uint16))
    vals = f16.view(np.float16).astype(np.float64)
    assert vals.min() >= 0 and vals.max() < 1 and np.all(vals * 1024 == np.floor(vals * 1024))
    b = orc.fill_bool(seed, 3, 1 << 20)
    assert abs(b.mean() - 0.5) < 5 * 0.5 / math.sqrt(b.size)


# ------------------------------------------------------- bounded integers --
def pin_lemire_exhaustive_8bit(orc):
    """Over every 8-bit word and every bound 1..255, the multiply-shift with
    its rejection threshold gives each value in [0, b) exactly floor(256/b)
    times and rejects exactly 256 mod b words: the same histogram as brute-force
    rejection (accept x < b * floor(256/b), return x mod b)."""
    w = 8
    for b in range(1, 256):
        hist = np.zeros(b, np.int64)
        rejected = 0
        for x in range(1 << w):
            ok, v = orc.lemire_step(x, b, w)
            if ok:
                assert v < b
                hist[v] += 1
            else:
                rejected += 1
        brute = np.bincount([x % b for x in range(1 << w) if x < b * ((1 << w) // b)], minlength=b)
        assert np.array_equal(hist, brute), b
        assert rejected == (1 << w) % b, b


def pin_lemire_exhaustive_16bit(orc):
    """As above on 16-bit words for bounds that cover tiny, odd, power-of-two
    and near-maximal ranges."""
    w = 16
    for b in (1, 3, 7, 1000, 4096, 32769, 65535):
        hist = np.zeros(b, np.int64)
        rejected = 0
        for x in range(1 << w):
            ok, v = orc.lemire_step(x, b, w)
            if ok:
                hist[v] += 1
            else:
                rejected += 1
        assert hist.min() == hist.max() == (1 << w) // b, b
        assert rejected == (1 << w) % b, b


def pin_lemire_wide_words(orc):
    """On 32- and 64-bit words the step is floor(x b / 2^w), accepted iff
    (x b) mod 2^w >= 2^w mod b, evaluated here with exact Python integers."""
    rng = np.random.default_rng(9)
    for w in (32, 64):
        for _ in range(2000):
            x = int(rng.integers(0, 1 << 62)) * 4 + int(rng.integers(0, 4))
            x %= 1 << w
            b = int(rng.integers(1, 1 << 62)) % (1 << w) or 1
            ok, v = orc.lemire_step(x, b, w)
            assert v == (x * b) >> w
            assert ok == (((x * b) % (1 << w)) >= ((1 << w) % b))


def _chi2_uniform(values: np.ndarray, b: int, bins: int = 64) -> float:
    idx = (values.astype(object) * bins // b).astype(np.int64) if b >= U32 else (
        values.astype(np.uint64) * np.uint64(bins) // np.uint64(b)).astype(np.int64)
    obs = np.bincount(idx, minlength=bins).astype(np.float64)
    lo = np.array([(k * b + bins - 1) // bins for k in range(bins + 1)], dtype=object)
    exp = np.array([float(lo[k + 1] - lo[k]) / b for k in range(bins)]) * values.size
    return stats.chisquare(obs, exp).pvalue


def pin_below_distributions(orc):
    """below32 / below64 values lie in [0, b) and are uniform, including bounds
    where about half of all words are rejected (b = 2^31 + 1, 2^63 + 1), so the
    substream retries carry half of the values."""
    n = 1 << 17
    for b in (1000, (1 << 31) + 1, U32 - 2):
        v = orc.fill_u32_below(1, 0, b, n)
        assert int(v.max()) < b
        assert _chi2_uniform(v, b) > 1e-4, b
    for b in (1000, (1 << 63) + 1, U64 - 2):
        v = orc.fill_u64_below(2, 0, b, n)
        assert int(v.max()) < b
        if b < U32:
            assert _chi2_uniform(v, b) > 1e-4, b
        else:
            hi = (v.astype(object) * 64 // b).astype(np.int64)
            assert stats.chisquare(np.bincount(hi, minlength=64)).pvalue > 1e-4, b
    assert not np.any(orc.fill_u32_below(3, 0, 1, 4096))
    # First words rejected at about (2^31 - 1) / 2^32 for b = 2^31 + 1
    b = (1 << 31) + 1
    d = orc.fill_u32(4, 0, 1 << 15)
    rejected = sum(not orc.lemire_step(int(x), b, 32)[0] for x in d)
    p = ((1 << 31) - 1) / U32
    assert abs(rejected / d.size - p) < 5 * math.sqrt(p * (1 - p) / d.size)


def pin_ranges_wrap(orc):
    """low + below(b) wraps in two's complement into int32 / int64."""
    n = 4096
    low32 = (1 << 31) - 10
    base = orc.fill_u32_below(3, 7, 1000, n).astype(np.int64)
    r32 = orc.fill_i32_range(3, 7, low32, 1000, n).astype(np.int64)
    assert np.array_equal(r32, (low32 + base + (1 << 31)) % U32 - (1 << 31))
    assert np.array_equal(orc.fill_i64_range32(3, 7, -500, 1000, n), base - 500)
    b64 = orc.fill_u64_below(3, 7, 1000, n).astype(np.int64)
    assert np.array_equal(orc.fill_i64_range(3, 7, -500, 1000, n), b64 - 500)


# ------------------------------------------------------------------ randn --
_HASH_INV = (pow(2146121005, -1, U32), pow((-2073254261) % U32, -1, U32))


def _unhash32(y: np.ndarray) -> np.ndarray:
    """hash32^-1 of 32-bit words (uint64 array): the xorshifts and the odd
    multipliers undone in reverse order (see pin_hash_bijective)."""
    inv1, inv2 = (np.uint64(v) for v in _HASH_INV)
    x = y ^ (y >> np.uint64(16))
    x = (x * inv2) & np.uint64(0xFFFFFFFF)
    x = x ^ (x >> np.uint64(15)) ^ (x >> np.uint64(30))
    x = (x * inv1) & np.uint64(0xFFFFFFFF)
    return x ^ (x >> np.uint64(16))


def _counters_with_low23(orc, seed: int, word: int, targets):
    """Counters c whose uniform at 2c + word has the given 23-bit grid index.
    hash32 is a bijection, so they are constructed: for the 512 draws D = h
    2^23 + t, the counter k = hash32^-1(D) ^ hash32(seed), and those of k's
    parity are 2c + word (about 256 per target).  The oracle's draws at them
    are checked to carry the target."""
    key = np.uint64(orc.hash32(seed))
    out = {}
    for t in targets:
        d = (np.arange(512, dtype=np.uint64) << np.uint64(23)) | np.uint64(t)
        ks = _unhash32(d) ^ key
        ks = ks[(ks & np.uint64(1)) == np.uint64(word)]
        assert np.all((orc.fill_u32(seed, 0, idx=ks) & 0x7FFFFF) == t), (seed, word, t)
        out[t] = np.sort(ks >> np.uint64(1)).astype(np.int64)
    return out


def pin_randn_special_angles(orc):
    """Closed forms of the Box-Muller value at the angles where cos is exact:
    u1 = 0 gives +r, u1 = 1/2 gives -r, u1 = 1/4 and 3/4 give |z| < 1e-15 r,
    with r = sqrt(-2 ln(1 - u0)); u0 = 0 gives z = 0."""
    seed = 7
    hits = _counters_with_low23(orc, seed, 1, (0, 1 << 21, 1 << 22, 3 << 21))
    for t, cs in hits.items():
        assert cs.size, t
        u0 = orc.fill_f32(seed, 0, idx=(2 * cs) % U32).astype(np.float64)
        r = np.sqrt(-2.0 * np.log1p(-u0))
        z = orc.fill_randn(seed, 0, idx=cs)
        if t == 0:
            assert np.allclose(z, r, rtol=1e-15, atol=0)
        elif t == 1 << 22:
            assert np.allclose(z, -r, rtol=1e-15, atol=0)
        else:
            assert np.all(np.abs(z) <= 1e-15 * r + 1e-300)
    zero = _counters_with_low23(orc, seed, 0, (0,))[0]
    assert zero.size and np.all(orc.fill_randn(seed, 0, idx=zero) == 0)


def pin_box_muller_closed_forms(orc):
    """The Box-Muller value of a draw pair (section randn on the uniforms of
    section uniform): u0 = 1/2 gives r = sqrt(2 ln 2), u1 = 0 and 1/2 give +r
    and -r, u1 = 1/4 gives |z| < 1e-15; u0 = 0 gives 0; only the low 23 bits
    of each draw count; randn(seed, c) is the pair (draw32(2c), draw32(2c+1)).
    The sine branch at the quarter turns, and as the paired fill's odd
    elements."""
    r = np.sqrt(2.0 * np.log(2.0))
    hi = np.uint32(0xFF800000)
    d0 = np.array([1 << 22, 1 << 22, 1 << 22, 0, (1 << 22) | hi, 0x5A5A5A | hi], dtype=np.uint32)
    d1 = np.array([0, 1 << 22, 1 << 21, 12345, hi, 0x3C3C3C], dtype=np.uint32)
    z = orc.box_muller_array(d0, d1)
    assert abs(z[0] - r) <= 1e-15 * r and abs(z[1] + r) <= 1e-15 * r and abs(z[2]) <= 1e-15 * r
    assert z[3] == 0 and z[4] == z[0]
    assert z[5] == orc.box_muller_array([0x5A5A5A], [0x3C3C3C])[0]
    seed = 99
    w = orc.fill_u32(seed, 0, 2000)
    assert np.array_equal(orc.box_muller_array(w[0::2], w[1::2]), orc.fill_randn(seed, 0, 1000))
    # the sine branch: u1 = 1/4 gives +r, u1 = 3/4 gives -r, u1 = 0 gives 0;
    # it is the odd element of the paired fill
    _, y = orc.box_muller_array(d0[:3], np.array([1 << 21, 3 << 21, 0], dtype=np.uint32), sine=True)
    assert abs(y[0] - r) <= 1e-15 * r and abs(y[1] + r) <= 1e-15 * r and y[2] == 0
    x, y = orc.box_muller_array(w[0::2], w[1::2], sine=True)
    paired = orc.fill_randn_paired(seed, 0, 2000)
    assert np.array_equal(x, paired[0::2]) and np.array_equal(y, paired[1::2])


def pin_randn_tail_end(orc):
    """Phobos 'Random numbers', randn: the 2^-23 grid ends the tails near 5.6,
    i.e. |z| <= sqrt(-2 ln 2^-23); the largest radius is reached at u0 = 1 - 2^-23."""
    g = golden("phobos_randn_tail.txt")
    bound = math.sqrt(-2.0 * math.log(2.0 ** int(g["grid_log2"])))
    assert round(bound, 1) == float(g["tail_end_1dp"])
    z = orc.fill_randn(11, 0, 1 << 22)
    assert np.abs(z).max() <= bound * (1 + 1e-15)
    top = _counters_with_low23(orc, 11, 0, ((1 << 23) - 1,))[(1 << 23) - 1]
    assert top.size
    u1 = orc.fill_f32(11, 0, idx=(2 * top + 1) % U32).astype(np.float64)
    assert np.allclose(orc.fill_randn(11, 0, idx=top), bound * np.cos(2 * np.pi * u1), rtol=1e-13, atol=1e-13)


def _normal_stats(z: np.ndarray):
    n = z.size
    assert abs(z.mean()) < 5 / math.sqrt(n), z.mean()
    assert abs(z.var() - 1) < 5 * math.sqrt(2 / n), z.var()
    assert abs(stats.skew(z)) < 5 * math.sqrt(6 / n)
    assert abs(stats.kurtosis(z)) < 5 * math.sqrt(24 / n)
    edges = stats.norm.ppf(np.linspace(0, 1, 201))
    obs = np.histogram(z, bins=edges)[0]
    assert stats.chisquare(obs).pvalue > 1e-3


def pin_randn_distribution(orc):
    """Moments and a 200-bin equiprobable chi-square of 2^22 randn values."""
    _normal_stats(orc.fill_randn(3, 0, 1 << 22))


def pin_randn_paired(orc):
    """Paired Box-Muller: the even element of pair q is randn(seed, q); both
    elements share one radius, x^2 + y^2 = -2 ln(1 - u0) (cos^2 + sin^2 = 1),
    and their angle is 2 pi u1: atan2(y, x) = 2 pi u1 (mod 2 pi); at u1 = 1/4
    the odd element is +r and the even one 0.  Moments, a 200-bin chi-square
    and no correlation between the two branches."""
    n = 1 << 20
    z = orc.fill_randn_paired(5, 0, 2 * n)
    x, y = z[0::2], z[1::2]
    assert np.array_equal(x, orc.fill_randn(5, 0, n))
    u0 = orc.fill_f32(5, 0, idx=2 * np.arange(n)).astype(np.float64)
    u1 = orc.fill_f32(5, 0, idx=2 * np.arange(n) + 1).astype(np.float64)
    assert np.allclose(x * x + y * y, -2.0 * np.log1p(-u0), rtol=1e-12, atol=1e-15)
    r = np.hypot(x, y)
    big = r > 1e-3
    ang = np.mod(np.arctan2(y[big], x[big]), 2 * np.pi)
    diff = np.abs(ang - 2 * np.pi * u1[big])
    assert np.all(np.minimum(diff, 2 * np.pi - diff) < 1e-9)
    quarter = _counters_with_low23(orc, 5, 1, (1 << 21,))[1 << 21]
    assert quarter.size
    zq = orc.fill_randn_paired(5, 0, idx=2 * quarter + 1)
    rq = np.sqrt(-2.0 * np.log1p(-orc.fill_f32(5, 0, idx=2 * quarter).astype(np.float64)))
    assert np.allclose(zq, rq, rtol=1e-14, atol=0)
    _normal_stats(y)
    assert abs(np.corrcoef(x, y)[0, 1]) < 5 / math.sqrt(n)


def pin_exponentials(orc):
    """-ln(1 - u): at u = 0 the value is +0 and at the top of the 2^-23 grid
    23 ln 2; the f64 fill is within 2 ulp of numpy's -log1p(-u) on the exact
    f64 uniform; both have mean 1, variance 1 and pass a 200-bin chi-square
    against 1 - exp(-x)."""
    n = 1 << 21
    u = orc.fill_f32(13, 0, n).astype(np.float64)
    e = orc.fill_exponential_f32(13, 0, n)
    assert np.allclose(e, -np.log1p(-u), rtol=1e-15, atol=0)
    hits = _counters_with_low23(orc, 7, 0, (0, (1 << 23) - 1))
    c0, ctop = 2 * hits[0][:4], 2 * hits[(1 << 23) - 1][:4]
    assert c0.size and ctop.size
    assert np.all(orc.fill_exponential_f32(7, 0, idx=c0) == 0)
    assert np.allclose(orc.fill_exponential_f32(7, 0, idx=ctop), 23 * math.log(2), rtol=1e-15)
    u64 = orc.fill_f64(13, 0, n)
    e64 = orc.fill_exponential_f64(13, 0, n)
    ref = -np.log1p(-u64)
    nz = ref > 0
    assert _ulps(e64[nz], ref[nz]).max() <= 2
    assert np.all(e64[~nz] == 0) and not np.any(np.signbit(e64))
    edges = np.append(-np.log1p(-np.linspace(0, 1, 201)[:-1]), np.inf)
    for x in (e, e64):
        assert abs(x.mean() - 1) < 5 / math.sqrt(n) and abs(x.var() - 1) < 5 * math.sqrt(8 / n)
        assert stats.chisquare(np.histogram(x, bins=edges)[0]).pvalue > 1e-3


_NEGLOG_CACHE = {}


def _neglog_all(orc):
    """The own f32 log on every 23-bit input, with the binary64 -ln(1 - u)
    (numpy's log of the exact binary64 value 1 - u: within 2^-52 relative)."""
    if orc.path not in _NEGLOG_CACHE:
        _NEGLOG_CACHE.clear()
        m = np.arange(1 << 23, dtype=np.uint32)
        ref = -np.log((8388608.0 - m) * 2.0 ** -23)
        _NEGLOG_CACHE[orc.path] = (m, orc.neglog_array(m), ref)
    return _NEGLOG_CACHE[orc.path]


def pin_neglog_f32_exhaustive(orc):
    """The f32 exponential's own log against the exact -ln(1 - u) on all 2^23
    inputs (tandem-cuda "Performance" and tandem-sycl "Design", Exponentials:
    every draw within 0.571 ulp).  Measured: within 0.5027 ulp (0.5044 without
    the r^5 Taylor term), and the correctly rounded binary32 value on all but
    82 inputs, where the exact value lies within 0.003 ulp of a rounding
    boundary; u = 0 gives +0 and the top of the grid 23 ln 2 rounded."""
    m, e, ref = _neglog_all(orc)
    nz = ref > 0
    ulp = np.spacing(ref[nz].astype(np.float32)).astype(np.float64)
    err = np.abs(e[nz].astype(np.float64) - ref[nz]) / ulp
    assert err.max() <= 0.5035
    assert np.count_nonzero(e != ref.astype(np.float32)) <= 120
    assert e[0] == 0 and not np.signbit(e[0])
    assert e[-1] == np.float32(23 * math.log(2))
    assert np.all(np.diff(e) >= 0)  # monotone in u


def pin_neglog_f32_maps_back(orc):
    """1 - exp(-e) maps every value back to its own draw's grid point (the
    property the pages' 0.571 ulp bound is for): round(2^23 (1 - exp(-e))) = m."""
    m, e, _ = _neglog_all(orc)
    back = np.rint(-np.expm1(-e.astype(np.float64)) * 8388608.0)
    assert np.array_equal(back.astype(np.int64), m.astype(np.int64))


def pin_neglog_f32_table(orc):
    """The own log's table against its definition: inv_j is 256/(256 + j)
    rounded to 8 significant bits (exact rationals), hi_j the nearest multiple
    of 2^-19 to ln inv_j and hi_j + lo_j = ln inv_j within 2^-43; ln2_hi and
    ln2_lo likewise for ln 2;
    and for every 24-bit M in [1, 2) with its bin j, M inv_j - 1 is exact in
    binary32 (the reduction step rounds nothing)."""
    from fractions import Fraction
    inv, hi, lo, ln2 = orc.neglog_table()
    for j in range(257):
        x = Fraction(256, 256 + j)
        e = x.numerator.bit_length() - x.denominator.bit_length()  # 2^e <= x < 2^(e+1) or 2^(e-1) <= ...
        if Fraction(2) ** e > x:
            e -= 1
        scaled = x / Fraction(2) ** (e - 7)  # in [128, 256)
        q, rem = divmod(scaled.numerator, scaled.denominator)
        if 2 * rem > scaled.denominator or (2 * rem == scaled.denominator and q % 2):
            q += 1
        assert Fraction(float(inv[j])) == q * Fraction(2) ** (e - 7), j
        for h, l, v in ((hi[j], lo[j], math.log(float(inv[j]))), (ln2[0], ln2[1], math.log(2))):
            scaled = v * 2 ** 19  # binary64 is enough: no value lies near a tie
            assert abs(scaled - math.floor(scaled) - 0.5) > 1e-6
            assert float(h) == round(scaled) / 2 ** 19  # the nearest multiple of 2^-19
            assert abs(float(h) + float(l) - v) <= 2.0 ** -43
    mant = np.arange(1 << 23, dtype=np.int64)
    j = (mant + 16384) >> 15
    num = (8388608 + mant) * (inv.astype(np.float64)[j] * 512).astype(np.int64) - (1 << 32)  # r 2^32
    odd = num.copy()
    nzr = odd != 0
    while True:
        even = nzr & (odd % 2 == 0)
        if not even.any():
            break
        odd[even] //= 2
    assert np.all(np.abs(odd) < (1 << 24))
    assert np.abs(num).max() < 1.5 * 2.0 ** -8 * 2 ** 32


def pin_exponential_f32_fill(orc):
    """The f32 exponential fill is the own log of the draw's 23 bits, within
    0.505 ulp of -log(1 - u) in binary64 on the same counters."""
    n = 1 << 20
    e = orc.fill_exponential_f32_own(13, 7, n).astype(np.float64)
    ref = orc.fill_exponential_f32(13, 7, n)
    nz = ref > 0
    assert np.all(e[~nz] == 0)
    assert (np.abs(e[nz] - ref[nz]) / np.spacing(ref[nz].astype(np.float32))).max() <= 0.505


def _cos2pi_reference(m):
    """cos(2 pi m 2^-23) in binary64 after the same exact reduction (quadrant
    and g in turns), so that its relative error stays near 2^-52 also next
    to the zeros of the cosine."""
    q = m >> 21
    g = (m & 0x1FFFFF).astype(np.float64) * 2.0 ** -23
    base = np.where(q % 2 == 0, np.cos(2 * np.pi * g), np.sin(2 * np.pi * g))
    return np.where((q == 1) | (q == 2), -base, base)


def pin_cos2pi_exhaustive(orc):
    """The precise normal's own cos(2 pi u) on all 2^23 grid angles: within
    0.95 ulp of the binary64 cosine (measured 0.90), exact at u = 0, 1/4, 1/2
    and 3/4, and symmetric, cos(2 pi u) = cos(2 pi (1 - u)) bit for bit
    wherever both sides reduce alike (all but the octant boundaries)."""
    m = np.arange(1 << 23, dtype=np.uint32)
    c = orc.cos2pi_array(m)
    ref = _cos2pi_reference(m)
    assert np.max(np.abs(ref - np.cos(2 * np.pi * m.astype(np.float64) * 2.0 ** -23))) < 1e-15
    nz = ref != 0
    ulp = np.spacing(np.abs(ref[nz]).astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(c[nz].astype(np.float64) - ref[nz]) / ulp) <= 0.95
    assert c[0] == 1 and c[1 << 22] == -1 and c[1 << 21] == 0 and c[3 << 21] == 0
    mm = m[1:]
    f = mm & 0x1FFFFF
    ok = (f != 0) & (f != 0x100000)
    assert np.array_equal(c[mm[ok]].view(np.uint32), c[((1 << 23) - mm[ok])].view(np.uint32))


def pin_cos2pi_coefficients(orc):
    """The Taylor coefficients (2 pi)^n / n! with the series' signs, each the
    binary32 rounding of the value (within half an ulp), and the hi + lo pairs
    of 2 pi and -(2 pi)^2/2 within 2^-44 relative."""
    k = orc.cos2pi_coefficients().astype(np.float64)
    tp = 2 * math.pi
    exact = {2: -tp ** 3 / 6, 3: tp ** 5 / 120, 4: -tp ** 7 / 5040, 5: tp ** 9 / 362880,
             8: tp ** 4 / 24, 9: -tp ** 6 / 720, 10: tp ** 8 / 40320, 11: -tp ** 10 / 3628800}
    for i, v in exact.items():
        assert abs(k[i] - v) <= 0.5000001 * float(np.spacing(np.float32(abs(v)))), i
    assert abs(k[0] + k[1] - tp) <= 2.0 ** -44 * tp and k[0] == np.float32(tp)
    assert abs(k[6] + k[7] + tp * tp / 2) <= 2.0 ** -44 * tp * tp / 2 and k[6] == np.float32(-tp * tp / 2)


def pin_randn_precise(orc):
    """The precise f32 normal against randn's binary64 value on the same
    counters: within 2.5 ulp (measured 2.40; the fast f32 path is held to
    4e-6 (1 + |z|)), zero where u0 = 0, and normal moments."""
    n = 1 << 22
    z = orc.fill_randn_precise(7, 0, n).astype(np.float64)
    ref = orc.fill_randn(7, 0, n)
    nz = ref != 0
    ulp = np.spacing(np.abs(ref[nz]).astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(z[nz] - ref[nz]) / ulp) <= 2.5
    assert np.all(z[~nz] == 0)
    _normal_stats(z)


def _neglog64_sample():
    """53-bit inputs: edge values, both sides of the small-u boundary m = 2^41,
    every bin edge of the log's table at the two largest exponents, and random
    values of every bit length."""
    g = np.random.default_rng(9)
    ms = [0, 1, 2, 3, (1 << 52) - 1, 1 << 52, (1 << 52) + 1, (1 << 53) - 2, (1 << 53) - 1]
    ms += [(1 << 41) + d for d in range(-3, 4)]
    for k in (52, 51):  # V = 2^53 - m in [2^k, 2^(k+1)): bin j starts at M = 1 + j/2048
        for j in range(1, 2048):
            edge = (1 << 53) - ((j << k) >> 11) - (1 << k)
            ms += [edge + d for d in (-1, 0, 1) if 0 <= edge + d < 1 << 53]
    bits = g.integers(1, 54, 1 << 18)
    ms += [int(x) >> (64 - int(b)) for x, b in zip(g.integers(0, 1 << 63, 1 << 18, dtype=np.uint64) << np.uint64(1),
                                                 bits)]
    return np.unique(np.array(ms, dtype=np.uint64))


def pin_neglog64_accuracy(orc):
    """The f64 exponential's own fixed-point log against -log1p(-u) in x87
    extended precision (64-bit significand; on x86-64 numpy's longdouble):
    within 0.501 ulp on the sample (measured 0.5005, part of it the
    reference's own error), and against mpmath at 50 digits on a subset: within
    0.5006 ulp (measured 0.50005).  +0 at m = 0, monotone in m, 53 ln 2 at the top."""
    ms = _neglog64_sample()
    y = orc.neglog64_array(ms)
    assert y[0] == 0 and not np.signbit(y[0])
    assert np.all(np.diff(y) >= 0)
    assert y[-1] == np.float64(53 * math.log(2)) or abs(y[-1] - 53 * math.log(2)) <= np.spacing(53 * math.log(2))
    if np.finfo(np.longdouble).nmant >= 63:
        u = ms.astype(np.longdouble) / np.longdouble(2) ** 53
        ref = -np.log1p(-u)
        nz = ref > 0
        err = np.abs(y[nz].astype(np.longdouble) - ref[nz]) / np.spacing(ref[nz].astype(np.float64))
        assert float(err.max()) <= 0.501
    import mpmath as mp
    mp.mp.dps = 50
    sub = ms[:: max(1, ms.size // 3000)]
    ys = orc.neglog64_array(sub)
    worst = 0.0
    for m, v in zip(sub, ys):
        if m == 0:
            continue
        ref = -mp.log1p(-mp.mpf(int(m)) / 2 ** 53)
        worst = max(worst, float(abs(mp.mpf(float(v)) - ref) / (mp.mpf(2) ** (math.frexp(float(ref))[1] - 53))))
    assert worst <= 0.5006


def pin_neglog64_powers_of_two(orc):
    """Where 1 - u is a power of two, 2^-k for m = 2^53 - 2^(53 - k), the
    reduction is exact (M = 1, r = 0) and -ln(1 - u) = k ln 2: the fixed-point
    log must return k ln 2 correctly rounded (mpmath, 50 digits) for every k
    in 1 .. 53, and their one-ulp neighbours in m must straddle it."""
    import mpmath as mp
    mp.mp.dps = 50
    ms = np.array([(1 << 53) - (1 << (53 - k)) for k in range(1, 54)], dtype=np.uint64)
    y = orc.neglog64_array(ms)
    for k, v in zip(range(1, 54), y):
        assert v == float(k * mp.log(2)), k
    below = orc.neglog64_array(ms - np.uint64(1))
    above = orc.neglog64_array(np.minimum(ms + np.uint64(1), np.uint64((1 << 53) - 1)))
    assert np.all(below <= y) and np.all(above[:-1] >= y[:-1])


def pin_neglog64_table(orc):
    """The fixed-point log's constants against their definitions: I_j =
    2^23/(2048 + j) rounded up to an integer (exact rationals), so that inv_j =
    I_j / 4096 is the smallest multiple of 2^-12 at or above 1/(1 + j/2048)
    and r = M inv_j - 1 lies in [0, 1.5 2^-11) on the whole bin [1 + j/2048,
    1 + (j + 1)/2048); ln(I_j / 4096) and ln 2 each the nearest integer
    multiple of 2^-96 (mpmath, 60 digits); the Horner constants 1/k at the
    scale of S_k: 2^63 for k = 1, 2^64 for k = 2, 3 and 2^33 for k = 4 .. 6."""
    import mpmath as mp
    from fractions import Fraction
    mp.mp.dps = 60
    inv, lninv, ln2, coef = orc.neglog64_table()
    assert len(inv) == len(lninv) == 2048
    for j in range(2048):
        q = -((-(1 << 23)) // (2048 + j))  # ceil(2^23 / (2048 + j))
        assert inv[j] == q and 2049 <= q <= 4096, j
        lo, hi = Fraction(2048 + j, 2048), Fraction(2049 + j, 2048)  # the bin of M
        assert lo * Fraction(q, 4096) - 1 >= 0 and hi * Fraction(q, 4096) - 1 < Fraction(3, 2 ** 12), j
        assert lninv[j] == int(mp.nint(mp.log(mp.mpf(inv[j]) / 4096) * mp.mpf(2) ** 96)), j
    assert inv[0] == 4096 and lninv[0] == 0 and inv[2047] == 2049
    assert ln2 == int(mp.nint(mp.log(2) * mp.mpf(2) ** 96))
    for k, scale in zip(range(1, 7), (63, 64, 64, 33, 33, 33)):
        assert coef[k] == int(mp.nint(mp.mpf(2) ** scale / k)), k


def pin_exponential_f64_fill(orc):
    """The f64 exponential fill is the fixed-point log of the draw's top 53
    bits: within 0.501 ulp of -log1p(-u) in extended precision on the same
    counters, with mean 1 and variance 1."""
    n = 1 << 20
    e = orc.fill_exponential_f64(13, 7, n)
    u64 = orc.fill_u64(13, 7, n) >> np.uint64(11)
    assert np.array_equal(e.view(np.uint64), orc.neglog64_array(u64).view(np.uint64))
    if np.finfo(np.longdouble).nmant >= 63:
        ref = -np.log1p(-(u64.astype(np.longdouble) / np.longdouble(2) ** 53))
        nz = ref > 0
        assert float((np.abs(e[nz].astype(np.longdouble) - ref[nz]) / np.spacing(ref[nz].astype(np.float64))).max()) <= 0.501
    assert abs(e.mean() - 1) < 5 / math.sqrt(n) and abs(e.var() - 1) < 5 * math.sqrt(8 / n)


# ---------------------------------------------------------------- dropout --
def pin_dropout(orc):
    """Phobos 'Random numbers', dropout: where(uniform >= p, x / (1 - p), 0)
    in f32.  Checked against numpy's IEEE f32 division and compare: the mask is
    uniform >= p (a tie is kept), the kept value is x / (1 - p), dropped
    elements are +0, the backward pass (same seed and counters) drops the same
    elements, p = 0 returns x, and the kept fraction is 1 - ceil(p 2^23) / 2^23."""
    rng = np.random.default_rng(1)
    n = 1 << 20
    x = rng.uniform(-1, 1, n).astype(np.float32)
    for p in (0.1, 0.5, 0.0, 0.999):
        p32 = np.float32(p)
        y = orc.dropout(x, p32, 42, 5)
        u = orc.fill_f32(42, 5, n)
        keep = u >= p32
        assert np.array_equal(y[keep].view(np.uint32), (x[keep] / (np.float32(1) - p32)).view(np.uint32))
        assert np.all(y[~keep].view(np.uint32) == 0)
        dy = rng.standard_normal(n).astype(np.float32)
        assert np.array_equal(orc.dropout(dy, p32, 42, 5) != 0, keep & (dy != 0))
        T = math.ceil(float(p32) * 2 ** 23)
        q = 1 - T / 2 ** 23
        assert abs(keep.mean() - q) <= 5 * math.sqrt(q * (1 - q) / n) + 1e-12
    assert np.array_equal(orc.dropout(x, 0.0, 42, 5).view(np.uint32), x.view(np.uint32))
    # a tie u == p is kept
    ties = np.nonzero(orc.fill_f32(42, 0, 1 << 25) == np.float32(0.5))[0]
    assert ties.size
    ones = np.ones(ties.size, np.float32)
    assert np.all(orc.dropout(ones, 0.5, 42, 0, idx=ties) == 2.0)
    # a dropped NaN is +0
    nan = np.full(n, np.nan, np.float32)
    y = orc.dropout(nan, 0.5, 42, 5)
    assert np.all((y.view(np.uint32) == 0) | np.isnan(y))


# ------------------------------------------------------------- exp / log ---
def pin_zexp_zlog(orc):
    """The slow path's own exp and log lie within 2 ulp of the C library's on
    dense samples of their domains, and are exact at the anchors."""
    rng = np.random.default_rng(3)
    t = np.concatenate([rng.uniform(-10, 0, 1 << 20), -np.linspace(0, 10, 4097)])
    assert _ulps(orc.zexp_array(t), np.exp(t)).max() <= 2
    x = np.concatenate([rng.uniform(0, 1, 1 << 20), 2.0 ** -rng.uniform(0, 53, 1 << 18),
                        1 - rng.integers(1, 1 << 20, 4096) * 2.0 ** -53, [2.0 ** -53, 0.5, 1.0]])
    x = x[x > 0]
    ref = np.log(x)
    got = orc.zlog_array(x)
    nz = ref != 0
    assert _ulps(got[nz], ref[nz]).max() <= 2
    assert orc.zlog(1.0) == 0 and orc.zexp(0.0) == 1.0


# --------------------------------------------------------------- ziggurat --
def pin_zig_table_published(orc):
    """Marsaglia & Tsang (2000): the 128-layer normal table has r =
    3.442619855899 and v = 9.91256303526217e-3; the same generator makes the
    1024-layer table."""
    g = golden("marsaglia_tsang_n128.txt")
    X, F, r, v = orc.zig_table(int(g["layers"]))
    assert abs(r - float(g["r"])) < 1e-11
    # the printed v agrees with the exact area to 11 significant digits
    assert abs(v / float(g["v"]) - 1) < 1e-11
    assert X[1] == r


def pin_zig_table_invariants(orc):
    """1024 layers of equal area v (the base strip's v = X[0] f(r)); X falls to
    X[1024] = 0, F = exp(-X^2/2) rises to F[1024] = 1."""
    X, F = orc.zig1024()
    _, _, r, v = orc.zig_table(1024)
    assert X[1] == r and X[1024] == 0 and F[1024] == 1
    assert np.all(np.diff(X) < 0) and np.all(np.diff(F) > 0)
    assert np.allclose(F, np.exp(-X * X / 2), rtol=1e-14, atol=0)
    assert abs(X[0] * F[1] / v - 1) < 1e-15
    area = X[1:1024] * (F[2:] - F[1:1024])
    assert np.max(np.abs(area / v - 1)) < 1e-12
    tail = math.sqrt(math.pi / 2) * special.erfc(r / math.sqrt(2))
    assert abs((r * F[1] + tail) / v - 1) < 1e-14


def pin_zig_candidate_rounding(orc):
    """The fast path's magnitude is the correctly rounded product of the
    53-bit draw and X[j] (Fraction -> float rounds to nearest even): random
    draws over every layer, draws with many leading zeros, and m = 2^53 - 1."""
    from fractions import Fraction
    X, _ = orc.zig1024()
    gen = np.random.default_rng(5)
    w = gen.integers(0, 1 << 63, 4000, dtype=np.uint64) * np.uint64(2) + gen.integers(0, 2, 4000, dtype=np.uint64)
    w[:1024] = (w[:1024] & ~np.uint64(1023)) | np.arange(1024, dtype=np.uint64)
    w[1024:1088] >>= np.arange(64, dtype=np.uint64)
    w[1088] = np.uint64((1 << 64) - 1)
    x = orc.zig_candidates(w)
    for wi, xi in zip(w.tolist(), x.tolist()):
        exact = Fraction(wi >> 11, 1 << 53) * Fraction(float(X[wi & 1023]))
        assert xi == float(exact), (hex(wi), xi, float(exact))


def pin_zig_miss_rate(orc):
    """tandem-sycl 'Design', Normals: 0.43 % of draws miss the fast path.  The
    table's miss probability mean(1 - X[j+1]/X[j]) rounds to it, and the
    measured first-draw miss fraction agrees within 5 sigma."""
    g = golden("tandem_ziggurat_miss.txt")
    X, _ = orc.zig1024()
    assert X.size - 1 == int(g["layers"])
    p = float(np.mean(1 - X[1:] / X[:-1]))
    assert round(100 * p, 2) == float(g["miss_percent_2dp"])
    n = 1 << 22
    fast = orc.fill_zig_fast(7, 0, n)
    miss = 1 - fast.mean()
    assert abs(miss - p) < 5 * math.sqrt(p * (1 - p) / n), (miss, p)


def pin_normal_f64_distribution(orc):
    """Moments, a 200-bin chi-square, the tail count P(|Z| > r) = erfc(r/sqrt 2)
    and the shape of the tail beyond r (Kolmogorov-Smirnov against the normal
    conditioned on |Z| > r) for 2^22 ziggurat normals."""
    n = 1 << 22
    z = orc.fill_normal_f64(7, 0, n)
    _normal_stats(z)
    X, _ = orc.zig1024()
    r = X[1]
    p = special.erfc(r / math.sqrt(2))
    tail = np.abs(z[np.abs(z) > r])
    assert abs(tail.size - p * n) < 5 * math.sqrt(p * n), tail.size
    cdf = lambda t: 1 - special.erfc(t / math.sqrt(2)) / special.erfc(r / math.sqrt(2))
    assert stats.kstest(tail, cdf).pvalue > 1e-3
    # the misses on their own (wedges and tail) are normal values too
    fast = orc.fill_zig_fast(7, 0, n).astype(bool)
    zm = z[~fast]
    assert zm.size > 10000
    assert abs(np.mean(zm)) < 5 * np.std(zm) / math.sqrt(zm.size)


def pin_zig_wedge_acceptance(orc):
    """The wedge test accepts a first-draw miss in layer j >= 1 with probability
    (integral of f over [X[j+1], X[j]] - F[j] (X[j] - X[j+1])) / wedge area, the
    area under the curve inside the layer's rectangle beyond X[j+1] (computed
    here with erf).  The measured acceptance over 2^22 elements agrees within
    5 sigma; fast-path elements return the draw's own magnitude and sign."""
    n = 1 << 22
    X, F = orc.zig1024()
    w = orc.fill_u64(7, 0, n)
    j = (w & np.uint64(1023)).astype(np.int64)
    neg = ((w >> np.uint64(10)) & np.uint64(1)).astype(bool)
    x = ((w >> np.uint64(11)).astype(np.float64) * 2.0 ** -53) * X[j]
    fast = x < X[j + 1]
    assert np.array_equal(fast, orc.fill_zig_fast(7, 0, n).astype(bool))
    z = orc.fill_normal_f64(7, 0, n)
    assert np.array_equal(np.abs(z[fast]), x[fast])
    assert np.array_equal(np.signbit(z[fast]), neg[fast])
    wedge = ~fast & (j >= 1)
    accepted = (np.abs(z[wedge]) == x[wedge]) & (np.signbit(z[wedge]) == neg[wedge])
    k = np.arange(1, 1024)
    a, b = X[k + 1], X[k]
    integ = math.sqrt(math.pi / 2) * (special.erf(b / math.sqrt(2)) - special.erf(a / math.sqrt(2)))
    p_acc = (integ - F[k] * (b - a)) / ((b - a) * (F[k + 1] - F[k]))
    per_layer = np.zeros(1024)
    per_layer[1:] = p_acc
    expected = per_layer[j[wedge]].mean()
    sigma = math.sqrt(expected * (1 - expected) / wedge.sum())
    assert abs(accepted.mean() - expected) < 5 * sigma, (accepted.mean(), expected)


# ------------------------------------------------------------ substreams --
def _first_words32(orc, keys) -> np.ndarray:
    return np.array([orc.substream_words32(int(k), 1)[0] for k in keys], dtype=np.uint32)


def _corr(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.corrcoef(a.astype(np.float64), b.astype(np.float64))[0, 1])


def pin_substream_purposes(orc):
    """A draw that is rejected or misses continues on a substream of its own
    purpose and its own counter (tandem-sycl "Design", Normals: split(g) of
    sub(PURPOSE) of the key, g the draw's global index).  For one seed the
    bounded-32, bounded-64 and normal-64 purposes give different element keys
    at the same counter, different counters give different keys, and the
    substreams' first words are uncorrelated with one another and with the
    main stream's draws at and next to the element's own counter (equal only
    at the 2^-32 chance rate)."""
    n = 1 << 13
    c0 = 12345
    counters = np.arange(c0, c0 + n, dtype=np.uint32)
    bound = 5 / math.sqrt(n)
    for seed in (1, 7, 0x9E3779B9):
        keys = {p: orc.substream_keys(seed, p, counters) for p in orc.PURPOSES}
        for p in orc.PURPOSES:
            assert np.unique(keys[p]).size == n, (seed, p)  # one key per counter
        words = {p: _first_words32(orc, keys[p]) for p in orc.PURPOSES}
        main = orc.fill_u32(seed, c0 - 2, n + 4)
        for i, p in enumerate(orc.PURPOSES):
            for q in orc.PURPOSES[i + 1:]:
                assert np.count_nonzero(keys[p] == keys[q]) <= 1, (seed, p, q)
                assert np.count_nonzero(words[p] == words[q]) <= 1, (seed, p, q)
                assert abs(_corr(words[p], words[q])) < bound, (seed, p, q)
            for shift in range(5):  # main-stream draws at c - 2 .. c + 2
                near = main[shift:shift + n]
                assert np.count_nonzero(words[p] == near) <= 1, (seed, p, shift)
                assert abs(_corr(words[p], near)) < bound, (seed, p, shift)


def pin_substream_is_the_generator(orc):
    """A substream is the generator itself keyed by the element key K: its
    32-bit word k is the draw at counter k of the seed s with hash32(s) = K,
    and its 64-bit word k the 64-bit draw at counter k, whose high word is the
    draw at 2k (the main stream's pinned word order), with the same counter
    wrap."""
    keys = [0, 1, 0xFFFFFFFF]
    for p in orc.PURPOSES:
        keys += [int(k) for k in orc.substream_keys(3, p, np.array([0, 77, U32 - 1], np.uint32))]
    seeds = _unhash32(np.array(keys, dtype=np.uint64))
    for key, s in zip(keys, (int(v) for v in seeds)):
        assert orc.hash32(s) == key
        assert np.array_equal(orc.substream_words32(key, 300), orc.fill_u32(s, 0, 300)), key
        assert np.array_equal(orc.substream_words64(key, 300), orc.fill_u64(s, 0, 300)), key
        assert np.array_equal(orc.substream_words32(key, 8, U32 - 4), orc.fill_u32(s, U32 - 4, 8)), key
        k0 = (1 << 31) - 4  # the 64-bit words' counters 2k wrap here
        assert np.array_equal(orc.substream_words64(key, 8, k0), orc.fill_u64(s, k0, 8)), key


def _lemire_first(words, b: int, w: int):
    """The first word of `words` that the exact-threshold Lemire step accepts,
    and its value (brute-force integer arithmetic)."""
    t = (1 << w) % b
    for x in words:
        prod = int(x) * b
        if prod % (1 << w) >= t:
            return prod >> w
    return None


def pin_retries_take_substream_words_in_order(orc):
    """An element whose own draw the Lemire step rejects returns the first
    accepted value among its substream's words 0, 1, 2, ... (bounds 2^31 + 1
    and 2^63 + 1, where about half of all draws are rejected), and the retried
    values are independent of the rejected first draw (8 x 8 contingency
    table, chi-square)."""
    for w, b, purpose, draws, fill, words in (
            (32, (1 << 31) + 1, "B32", orc.fill_u32, orc.fill_u32_below, orc.substream_words32),
            (64, (1 << 63) + 1, "B64", orc.fill_u64, orc.fill_u64_below, orc.substream_words64)):
        seed, c0, n = 5, 100, 2048
        d = draws(seed, c0, n)
        v = fill(seed, c0, b, n)
        keys = orc.substream_keys(seed, purpose, np.arange(c0, c0 + n, dtype=np.uint32))
        rejected = 0
        for i in range(n):
            first = _lemire_first([d[i]], b, w)
            if first is not None:
                assert int(v[i]) == first, (w, i)
                continue
            rejected += 1
            assert int(v[i]) == _lemire_first(words(int(keys[i]), 64), b, w), (w, i)
        assert rejected > n // 3, (w, rejected)
        # independence of the retried value from the rejected first draw
        n = 1 << 16
        d = draws(seed, 0, n)
        v = fill(seed, 0, b, n)
        top = w - 3
        d_obj = d.astype(object)
        rej = np.array([(int(x) * b) % (1 << w) < (1 << w) % b for x in d_obj])
        first_bin = (d[rej] >> np.uint64(top) if w == 64 else d[rej] >> np.uint32(top)).astype(np.int64)
        value_bin = (v[rej].astype(object) * 8 // b).astype(np.int64)
        table = np.zeros((8, 8))
        np.add.at(table, (first_bin, value_bin), 1)
        table = table[table.sum(axis=1) > 0]
        assert stats.chi2_contingency(table)[1] > 1e-4, w


# ---------------------------------------------------------- slice invariant -
def pin_slice_invariant(orc):
    """A fill cut at any element equals the whole fill (tandem-sycl 'Design',
    Normals), for every fill, across the 2^32 counter wrap; a sampled fill
    (idx) equals the dense one."""
    rng = np.random.default_rng(2)
    n = 3000
    fills = [
        lambda f, m, idx=None: orc.fill_u8(9, f, m, idx),
        lambda f, m, idx=None: orc.fill_u16(9, f, m, idx),
        lambda f, m, idx=None: orc.fill_bool(9, f, m, idx),
        lambda f, m, idx=None: orc.fill_f16_bits(9, f, m, idx),
        lambda f, m, idx=None: orc.fill_randn_paired(9, f, m, idx),
        lambda f, m, idx=None: orc.fill_exponential_f32(9, f, m, idx),
        lambda f, m, idx=None: orc.fill_exponential_f32_own(9, f, m, idx),
        lambda f, m, idx=None: orc.fill_randn_precise(9, f, m, idx),
        lambda f, m, idx=None: orc.fill_exponential_f64(9, f, m, idx),
        lambda f, m, idx=None: orc.fill_u32(9, f, m, idx),
        lambda f, m, idx=None: orc.fill_u64(9, f, m, idx),
        lambda f, m, idx=None: orc.fill_f32(9, f, m, idx),
        lambda f, m, idx=None: orc.fill_f64(9, f, m, idx),
        lambda f, m, idx=None: orc.fill_u32_below(9, f, (1 << 31) + 1, m, idx),
        lambda f, m, idx=None: orc.fill_u64_below(9, f, (1 << 63) + 1, m, idx),
        lambda f, m, idx=None: orc.fill_i32_range(9, f, -500, 1000, m, idx),
        lambda f, m, idx=None: orc.fill_i64_range32(9, f, -500, 1000, m, idx),
        lambda f, m, idx=None: orc.fill_i64_range(9, f, -500, 1000, m, idx),
        lambda f, m, idx=None: orc.fill_randn(9, f, m, idx),
        lambda f, m, idx=None: orc.fill_normal_f64(9, f, m, idx),
    ]
    for first in (0, 1, 3, U32 - 5):
        for fill in fills:
            whole = fill(first, n)
            for _ in range(3):
                a, b = sorted(rng.integers(0, n, 2))
                part = fill((first + int(a)) % U32, int(b - a))
                assert np.array_equal(part.view(np.uint8), whole[a:b].view(np.uint8))
            sel = rng.integers(0, n, 257)
            assert np.array_equal(fill(first, None, sel).view(np.uint8), whole[sel].view(np.uint8))


ALL_PINS = [
    pin_tile_mean, pin_uniform_grid, pin_hash_bijective, pin_draw64_words, pin_narrow_fills,
    pin_lemire_exhaustive_8bit, pin_lemire_exhaustive_16bit, pin_lemire_wide_words,
    pin_below_distributions, pin_ranges_wrap, pin_randn_special_angles, pin_box_muller_closed_forms,
    pin_randn_tail_end, pin_randn_distribution, pin_randn_paired, pin_exponentials,
    pin_neglog_f32_exhaustive, pin_neglog_f32_maps_back, pin_neglog_f32_table, pin_exponential_f32_fill,
    pin_cos2pi_exhaustive, pin_cos2pi_coefficients, pin_randn_precise,
    pin_neglog64_accuracy, pin_neglog64_powers_of_two, pin_neglog64_table, pin_exponential_f64_fill,
    pin_dropout, pin_zexp_zlog,
    pin_zig_table_published, pin_zig_table_invariants, pin_zig_candidate_rounding, pin_zig_miss_rate,
    pin_normal_f64_distribution, pin_zig_wedge_acceptance,
    pin_substream_purposes, pin_substream_is_the_generator, pin_retries_take_substream_words_in_order,
    pin_slice_invariant,
]
