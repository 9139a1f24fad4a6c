"""CPU oracle for the lowbias32 counter-based random fills.

TEST INFRASTRUCTURE ONLY.  The tests, the package's ``smoke()`` check and the
benchmark's CPU-baseline leg are the only users; the product path never
imports this package.  ``oracle.c`` holds the arithmetic (plain C, one element
at a time); this module only compiles it with gcc and marshals numpy arrays
through ctypes.
"""
from __future__ import annotations

import ctypes as C
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (if stale) and return its path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    cmd = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off",
           "-fexcess-precision=standard", "-fno-fast-math", "-fPIC", "-shared",
           _SRC, "-o", _LIB + ".tmp", "-lm"]
    if platform.machine() in ("x86_64", "AMD64"):
        cmd.append("-lquadmath")
    subprocess.run(cmd, check=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


_u32, _u64, _i32, _i64 = C.c_uint32, C.c_uint64, C.c_int32, C.c_int64
_sz, _f32, _f64, _p = C.c_size_t, C.c_float, C.c_double, C.c_void_p

_SIGS = {
    "orc_hash32": (_u32, [_u32]),
    "orc_draw32": (_u32, [_u32, _u32]),
    "orc_draw64": (_u64, [_u32, _u32]),
    "orc_uniform_f32": (_f32, [_u32, _u32]),
    "orc_uniform_f64": (_f64, [_u32, _u32]),
    "orc_lemire_step": (C.c_int, [_u64, _u64, C.c_uint, C.POINTER(_u64)]),
    "orc_below32": (_u32, [_u32, _u32, _u32]),
    "orc_below64": (_u64, [_u32, _u32, _u64]),
    "orc_randn": (_f64, [_u32, _u32]),
    "orc_box_muller": (_f64, [_u32, _u32]),
    "orc_box_muller_sin": (_f64, [_u32, _u32]),
    "orc_box_muller_fill": (None, [_p, _p, _sz, _p, _p]),
    "orc_dropout": (_f32, [_f32, _f32, _u32, _u32]),
    "orc_zexp": (_f64, [_f64]),
    "orc_zlog": (_f64, [_f64]),
    "orc_zig_table": (C.c_int, [C.c_uint, _p, _p, C.POINTER(_f64), C.POINTER(_f64)]),
    "orc_zig1024": (None, [_p, _p]),
    "orc_zig_first_draw_fast": (C.c_int, [_u32, _u32]),
    "orc_substream_keys": (None, [_u32, C.c_int, _p, _sz, _p]),
    "orc_substream_words32": (None, [_u32, _u32, _sz, _p]),
    "orc_substream_words64": (None, [_u32, _u32, _sz, _p]),
    "orc_zig_candidates": (None, [_p, _sz, _p]),
    "orc_normal_f64": (_f64, [_u32, _u32]),
    "orc_fill_u32": (None, [_u32, _u32, _sz, _p, _p]),
    "orc_fill_u64": (None, [_u32, _u32, _sz, _p, _p]),
    "orc_fill_f32": (None, [_u32, _u32, _sz, _p, _p]),
    "orc_fill_f64": (None, [_u32, _u32, _sz, _p, _p]),
    "orc_fill_u8": (None, [_u32, _u32, _sz, _p, _p]),
    "orc_fill_u16": (None, [_u32, _u32, _sz, _p, _p]),
    "orc_fill_bool": (None, [_u32, _u32, _sz, _p, _p]),
    "orc_fill_f16_bits": (None, [_u32, _u32, _sz, _p, _p]),
    "orc_fill_u32_below": (None, [_u32, _u32, _sz, _p, _u32, _p]),
    "orc_fill_u64_below": (None, [_u32, _u32, _sz, _p, _u64, _p]),
    "orc_fill_i32_range": (None, [_u32, _u32, _sz, _p, _i32, _u32, _p]),
    "orc_fill_i64_range32": (None, [_u32, _u32, _sz, _p, _i64, _u32, _p]),
    "orc_fill_i64_range": (None, [_u32, _u32, _sz, _p, _i64, _u64, _p]),
    "orc_fill_randn": (None, [_u32, _u32, _sz, _p, _p]),
    "orc_fill_randn_paired": (None, [_u32, _u32, _sz, _p, _p]),
    "orc_fill_exponential_f32": (None, [_u32, _u32, _sz, _p, _p]),
    "orc_fill_exponential_f64": (None, [_u32, _u32, _sz, _p, _p]),
    "orc_fill_exponential_f32_own": (None, [_u32, _u32, _sz, _p, _p]),
    "orc_neglog_fill": (None, [_p, _sz, _p]),
    "orc_fill_randn_precise": (None, [_u32, _u32, _sz, _p, _p]),
    "orc_cos2pi_fill": (None, [_p, _sz, _p]),
    "orc_cos2pi_coefficients": (None, [_p]),
    "orc_neglog64_fill": (None, [_p, _sz, _p]),
    "orc_neglog64_table": (None, [_p, _p, _p, _p, _p]),
    "orc_neglog_table": (None, [_p, _p, _p, _p]),
    "orc_randn_paired": (_f64, [_u32, _u32]),
    "orc_fill_normal_f64": (None, [_u32, _u32, _sz, _p, _p]),
    "orc_dropout_fill": (None, [_p, _f32, _u32, _u32, _sz, _p, _p]),
    "orc_fill_zig_fast": (None, [_u32, _u32, _sz, _p, _p]),
    "orc_zexp_fill": (None, [_p, _sz, _p]),
    "orc_zlog_fill": (None, [_p, _sz, _p]),
}


def _bind(handle: C.CDLL) -> C.CDLL:
    for name, (res, args) in _SIGS.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    return handle


def compile_variant(source_text: str, out_dir: str) -> str:
    """Compile a modified copy of oracle.c (used by the tests that plant a
    mistake in the oracle and check that a pin catches it)."""
    src = os.path.join(out_dir, "oracle_variant.c")
    so = os.path.join(out_dir, "liboracle_variant.so")
    with open(src, "w") as fh:
        fh.write(source_text)
    cmd = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off",
           "-fexcess-precision=standard", "-fno-fast-math", "-fPIC", "-shared",
           src, "-o", so, "-lm"]
    if platform.machine() in ("x86_64", "AMD64"):
        cmd.append("-lquadmath")
    subprocess.run(cmd, check=True)
    return so


def source() -> str:
    with open(_SRC) as fh:
        return fh.read()


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def _idx(n: int | None, idx) -> tuple[int, np.ndarray | None]:
    if idx is None:
        return int(n), None
    idx = np.ascontiguousarray(idx, dtype=np.uint64)
    return idx.size, idx


class Oracle:
    """numpy front end over one loaded copy of the oracle library."""

    def __init__(self, path: str):
        self.path = os.path.abspath(path)  # identifies the compiled library (each variant has its own file)
        self.lib = _bind(C.CDLL(path))

    # Scalar definitions ------------------------------------------------------
    def hash32(self, x: int) -> int:
        return self.lib.orc_hash32(x & 0xFFFFFFFF)

    def draw32(self, seed: int, c: int) -> int:
        return self.lib.orc_draw32(seed & 0xFFFFFFFF, c & 0xFFFFFFFF)

    def draw64(self, seed: int, c: int) -> int:
        return self.lib.orc_draw64(seed & 0xFFFFFFFF, c & 0xFFFFFFFF)

    def lemire_step(self, x: int, b: int, w: int) -> tuple[bool, int]:
        v = C.c_uint64()
        ok = self.lib.orc_lemire_step(x, b, w, C.byref(v))
        return bool(ok), v.value

    def below32(self, seed: int, c: int, b: int) -> int:
        return self.lib.orc_below32(seed & 0xFFFFFFFF, c & 0xFFFFFFFF, b)

    def below64(self, seed: int, c: int, b: int) -> int:
        return self.lib.orc_below64(seed & 0xFFFFFFFF, c & 0xFFFFFFFF, b)

    # Substreams (bounded retries and ziggurat misses) -------------------------
    PURPOSES = ("B32", "B64", "N64")

    def substream_keys(self, seed: int, purpose: str, counters) -> np.ndarray:
        """The element keys of `counters` for one purpose ("B32", "B64", "N64")."""
        g = np.ascontiguousarray(counters, dtype=np.uint32)
        out = np.empty(g.size, np.uint32)
        self.lib.orc_substream_keys(seed & 0xFFFFFFFF, self.PURPOSES.index(purpose), _ptr(g), g.size, _ptr(out))
        return out

    def substream_words32(self, key: int, n: int, k0: int = 0) -> np.ndarray:
        out = np.empty(n, np.uint32)
        self.lib.orc_substream_words32(key & 0xFFFFFFFF, k0 & 0xFFFFFFFF, n, _ptr(out))
        return out

    def substream_words64(self, key: int, n: int, k0: int = 0) -> np.ndarray:
        out = np.empty(n, np.uint64)
        self.lib.orc_substream_words64(key & 0xFFFFFFFF, k0 & 0xFFFFFFFF, n, _ptr(out))
        return out

    def randn(self, seed: int, c: int) -> float:
        return self.lib.orc_randn(seed & 0xFFFFFFFF, c & 0xFFFFFFFF)

    def normal_f64(self, seed: int, c: int) -> float:
        return self.lib.orc_normal_f64(seed & 0xFFFFFFFF, c & 0xFFFFFFFF)

    def zexp(self, t: float) -> float:
        return self.lib.orc_zexp(t)

    def zlog(self, x: float) -> float:
        return self.lib.orc_zlog(x)

    def zig_table(self, N: int):
        """(X, F, r, v) for an N-layer ziggurat; X and F have N+1 entries."""
        X = np.empty(N + 1, np.float64)
        F = np.empty(N + 1, np.float64)
        r, v = C.c_double(), C.c_double()
        if self.lib.orc_zig_table(N, _ptr(X), _ptr(F), C.byref(r), C.byref(v)) != 0:
            raise ValueError("N must be at least 2")
        return X, F, r.value, v.value

    def zig_candidates(self, w):
        """The ziggurat fast path's magnitude RNE((w >> 11) 2^-53 X[w & 1023])
        of each 64-bit draw w, fast or not."""
        w = np.ascontiguousarray(w, dtype=np.uint64)
        x = np.empty(w.size, dtype=np.float64)
        self.lib.orc_zig_candidates(_ptr(w), w.size, _ptr(x))
        return x

    def zig1024(self):
        X = np.empty(1025, np.float64)
        F = np.empty(1025, np.float64)
        self.lib.orc_zig1024(_ptr(X), _ptr(F))
        return X, F

    # Fills (element i at counter first + i, or first + idx[i]) ---------------
    def _fill(self, fn, dtype, seed, first, n, idx, *extra):
        n, idx = _idx(n, idx)
        out = np.empty(n, dtype)
        getattr(self.lib, fn)(seed & 0xFFFFFFFF, first & 0xFFFFFFFF, n, _ptr(idx),
                              *extra, _ptr(out))
        return out

    def fill_u32(self, seed, first, n=None, idx=None):
        return self._fill("orc_fill_u32", np.uint32, seed, first, n, idx)

    def fill_u64(self, seed, first, n=None, idx=None):
        return self._fill("orc_fill_u64", np.uint64, seed, first, n, idx)

    def fill_f32(self, seed, first, n=None, idx=None):
        return self._fill("orc_fill_f32", np.float32, seed, first, n, idx)

    def fill_f64(self, seed, first, n=None, idx=None):
        return self._fill("orc_fill_f64", np.float64, seed, first, n, idx)

    def fill_u8(self, seed, first, n=None, idx=None):
        return self._fill("orc_fill_u8", np.uint8, seed, first, n, idx)

    def fill_u16(self, seed, first, n=None, idx=None):
        return self._fill("orc_fill_u16", np.uint16, seed, first, n, idx)

    def fill_bool(self, seed, first, n=None, idx=None):
        return self._fill("orc_fill_bool", np.uint8, seed, first, n, idx)

    def fill_f16_bits(self, seed, first, n=None, idx=None):
        return self._fill("orc_fill_f16_bits", np.uint16, seed, first, n, idx)

    def fill_u32_below(self, seed, first, bound, n=None, idx=None):
        return self._fill("orc_fill_u32_below", np.uint32, seed, first, n, idx, bound)

    def fill_u64_below(self, seed, first, bound, n=None, idx=None):
        return self._fill("orc_fill_u64_below", np.uint64, seed, first, n, idx, bound)

    def fill_i32_range(self, seed, first, low, bound, n=None, idx=None):
        return self._fill("orc_fill_i32_range", np.int32, seed, first, n, idx, low, bound)

    def fill_i64_range32(self, seed, first, low, bound, n=None, idx=None):
        return self._fill("orc_fill_i64_range32", np.int64, seed, first, n, idx, low, bound)

    def fill_i64_range(self, seed, first, low, bound, n=None, idx=None):
        return self._fill("orc_fill_i64_range", np.int64, seed, first, n, idx, low, bound)

    def fill_randn(self, seed, first, n=None, idx=None):
        """binary64 values of the randn definition (not rounded to f32)."""
        return self._fill("orc_fill_randn", np.float64, seed, first, n, idx)

    def box_muller_array(self, d0, d1, sine=False):
        """binary64 Box-Muller values of the draw pairs (d0[i], d1[i]): the
        cosine branch, or (cosine, sine) with sine=True."""
        d0 = np.ascontiguousarray(d0, dtype=np.uint32)
        d1 = np.ascontiguousarray(d1, dtype=np.uint32)
        assert d0.shape == d1.shape
        out = np.empty(d0.size, dtype=np.float64)
        out_sin = np.empty(d0.size, dtype=np.float64) if sine else None
        self.lib.orc_box_muller_fill(_ptr(d0), _ptr(d1), d0.size, _ptr(out), _ptr(out_sin))
        return (out, out_sin) if sine else out

    def fill_randn_paired(self, seed, first, n=None, idx=None):
        """binary64 values of the paired Box-Muller definition."""
        return self._fill("orc_fill_randn_paired", np.float64, seed, first, n, idx)

    def fill_exponential_f32(self, seed, first, n=None, idx=None):
        """binary64 values of -ln(1 - u) on the f32 uniform (not rounded to f32)."""
        return self._fill("orc_fill_exponential_f32", np.float64, seed, first, n, idx)

    def fill_randn_precise(self, seed, first, n=None, idx=None):
        """binary32 values of the precise f32 normal fill (randn's definition to a few ulp)."""
        return self._fill("orc_fill_randn_precise", np.float32, seed, first, n, idx)

    def fill_exponential_f32_own(self, seed, first, n=None, idx=None):
        """binary32 values of the f32 exponential fill (the own table-driven log)."""
        return self._fill("orc_fill_exponential_f32_own", np.float32, seed, first, n, idx)

    def fill_exponential_f64(self, seed, first, n=None, idx=None):
        return self._fill("orc_fill_exponential_f64", np.float64, seed, first, n, idx)

    def fill_normal_f64(self, seed, first, n=None, idx=None):
        return self._fill("orc_fill_normal_f64", np.float64, seed, first, n, idx)

    def fill_zig_fast(self, seed, first, n=None, idx=None):
        """1 where the element's first draw takes the ziggurat's fast path."""
        return self._fill("orc_fill_zig_fast", np.uint8, seed, first, n, idx)

    def dropout(self, x, p, seed, first, idx=None):
        """dropout of f32 x, x[i] at counter first + i (or first + idx[i])."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        n, idx = _idx(x.size, idx)
        if n != x.size:
            raise ValueError("x and idx differ in length")
        out = np.empty(n, np.float32)
        self.lib.orc_dropout_fill(_ptr(x), float(np.float32(p)), seed & 0xFFFFFFFF,
                                  first & 0xFFFFFFFF, n, _ptr(idx), _ptr(out))
        return out

    def zexp_array(self, t):
        t = np.ascontiguousarray(t, dtype=np.float64)
        out = np.empty_like(t)
        self.lib.orc_zexp_fill(_ptr(t), t.size, _ptr(out))
        return out

    def neglog_array(self, m):
        """-ln(1 - m 2^-23) in binary32 by the own log, for 23-bit integers m."""
        m = np.ascontiguousarray(m, dtype=np.uint32)
        if m.size and int(m.max()) >= 1 << 23:
            raise ValueError("m must be below 2^23")
        out = np.empty(m.size, np.float32)
        self.lib.orc_neglog_fill(_ptr(m), m.size, _ptr(out))
        return out

    def cos2pi_array(self, m):
        """cos(2 pi m 2^-23) in binary32 by the own routine, for 23-bit integers m."""
        m = np.ascontiguousarray(m, dtype=np.uint32)
        if m.size and int(m.max()) >= 1 << 23:
            raise ValueError("m must be below 2^23")
        out = np.empty(m.size, np.float32)
        self.lib.orc_cos2pi_fill(_ptr(m), m.size, _ptr(out))
        return out

    def cos2pi_coefficients(self):
        """s1_hi s1_lo s3 s5 s7 s9 c2_hi c2_lo c4 c6 c8 c10 (binary32)."""
        out = np.empty(12, np.float32)
        self.lib.orc_cos2pi_coefficients(_ptr(out))
        return out

    def neglog64_array(self, m):
        """-ln(1 - m 2^-53) in binary64 by the own fixed-point log, for 53-bit integers m."""
        m = np.ascontiguousarray(m, dtype=np.uint64)
        if m.size and int(m.max()) >= 1 << 53:
            raise ValueError("m must be below 2^53")
        out = np.empty(m.size, np.float64)
        self.lib.orc_neglog64_fill(_ptr(m), m.size, _ptr(out))
        return out

    def neglog64_table(self):
        """I_j (2048), ln inv_j at 2^96 as Python ints (2048), ln 2 at 2^96, and the
        Horner constants 1/k (index k = 1 .. 6): 1 at 2^63, 1/2 and 1/3 at 2^64,
        1/4 .. 1/6 at 2^33."""
        inv = np.empty(2048, np.int32)
        hi, lo = np.empty(2048, np.int64), np.empty(2048, np.uint64)
        ln2, coef = np.empty(2, np.int64), np.empty(7, np.uint64)
        self.lib.orc_neglog64_table(_ptr(inv), _ptr(hi), _ptr(lo), _ptr(ln2), _ptr(coef))
        lninv = [(int(h) << 64) + int(l) for h, l in zip(hi, lo)]
        return ([int(x) for x in inv], lninv, (int(ln2[0]) << 64) + (int(ln2[1]) & ((1 << 64) - 1)),
                [int(c) for c in coef])

    def neglog_table(self):
        """The own log's table: inv, hi, lo (257 binary32 each) and (ln2_hi, ln2_lo)."""
        inv, hi, lo = (np.empty(257, np.float32) for _ in range(3))
        ln2 = np.empty(2, np.float32)
        self.lib.orc_neglog_table(_ptr(inv), _ptr(hi), _ptr(lo), _ptr(ln2))
        return inv, hi, lo, ln2

    def zlog_array(self, x):
        x = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty_like(x)
        self.lib.orc_zlog_fill(_ptr(x), x.size, _ptr(out))
        return out


_default: Oracle | None = None


def default() -> Oracle:
    """The oracle built from oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def variant(source_text: str, out_dir: str) -> Oracle:
    return Oracle(compile_variant(source_text, out_dir))


def __getattr__(name):
    # oracle.fill_u32(...) etc. forward to the default instance.
    if not name.startswith("_") and hasattr(Oracle, name):
        return getattr(default(), name)
    raise AttributeError(name)
