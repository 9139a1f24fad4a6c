"""Stateless counter-based random fills (lowbias32 hash32) for GB300.

A thin ctypes binding of the C ABI in include/rng.h: every function here
carries the C entry point's name, marshals a CUDA tensor's pointer, length
and the current stream, and raises on a non-OK status.  All work runs in the
library's sm_103a kernels; there is no fallback: if the library has not been
built, importing this package fails.

    import torch, dropout_lowbias32_hash32_gb300 as rng
    out = torch.empty(1 << 28, dtype=torch.float32, device="cuda")
    rng.rng_fill_f32(seed=1, first_counter=0, out=out)
"""
from __future__ import annotations

import ctypes as C
import os

from . import sharding  # noqa: F401  (counter ranges for multi-process fills)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIBRARY_PATH = os.path.join(_PKG, "_lib", "librng_lowbias32.so")

if not os.path.exists(LIBRARY_PATH):
    raise ImportError(
        f"{LIBRARY_PATH} is missing: build the CUDA library first "
        "(python dropout_lowbias32_hash32_gb300/build.py, or __graft_entry__.build())")

_lib = C.CDLL(LIBRARY_PATH)

_u32, _u64, _i32, _i64, _sz = C.c_uint32, C.c_uint64, C.c_int32, C.c_int64, C.c_size_t
_p, _f32, _int = C.c_void_p, C.c_float, C.c_int

# name -> argument types (every entry point returns rng_status = int)
_FILL_SIGS = {
    "rng_fill_u32": [_u32, _u32, _sz, _p, _p],
    "rng_fill_u64": [_u32, _u32, _sz, _p, _p],
    "rng_fill_f32": [_u32, _u32, _sz, _p, _p],
    "rng_fill_f64": [_u32, _u32, _sz, _p, _p],
    "rng_fill_u8": [_u32, _u32, _sz, _p, _p],
    "rng_fill_u16": [_u32, _u32, _sz, _p, _p],
    "rng_fill_f16": [_u32, _u32, _sz, _p, _p],
    "rng_fill_bool": [_u32, _u32, _sz, _p, _p],
    "rng_fill_u32_below": [_u32, _u32, _sz, _u32, _p, _p],
    "rng_fill_u64_below": [_u32, _u32, _sz, _u64, _p, _p],
    "rng_fill_i32_range": [_u32, _u32, _sz, _i32, _u32, _p, _p],
    "rng_fill_i64_range32": [_u32, _u32, _sz, _i64, _u32, _p, _p],
    "rng_fill_i64_range": [_u32, _u32, _sz, _i64, _u64, _p, _p],
    "rng_fill_normal_f32": [_u32, _u32, _sz, _p, _p],
    "rng_fill_normal_f32_pairs": [_u32, _u32, _sz, _p, _p],
    "rng_fill_normal_f32_precise": [_u32, _u32, _sz, _p, _p],
    "rng_fill_exponential_f32": [_u32, _u32, _sz, _p, _p],
    "rng_fill_exponential_f64": [_u32, _u32, _sz, _p, _p],
    "rng_fill_normal_f64": [_u32, _u32, _sz, _p, _p],
    "rng_fill_normal_f64_noalloc": [_u32, _u32, _sz, _p, _p],
    "rng_dropout_fwd": [_p, _p, _f32, _u32, _u32, _sz, _p],
    "rng_dropout_bwd": [_p, _p, _f32, _u32, _u32, _sz, _p],
    "rng_debug_set_miss_capacity": [_sz],
    "rng_debug_last_miss_count": [C.POINTER(_u64)],
    "rng_debug_eval_f64": [_int, _p, _p, _sz, _p],
    "rng_debug_write_ceiling": [_int, _p, _sz, _p],
}
for _name, _args in _FILL_SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _int
_lib.rng_status_string.argtypes = [_int]
_lib.rng_status_string.restype = C.c_char_p
_lib.rng_last_error.argtypes = []
_lib.rng_last_error.restype = C.c_char_p
_lib.rng_debug_launch_count.argtypes = []
_lib.rng_debug_launch_count.restype = _u64

RNG_OK, RNG_EINVAL, RNG_ECUDA, RNG_ENOMEM = 0, 1, 2, 3


class RngError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.rng_status_string(status).decode()
        detail = _lib.rng_last_error().decode()
        super().__init__(f"{where}: {msg}" + (f" ({detail})" if detail else ""))


def _check(status: int, where: str) -> None:
    if status != RNG_OK:
        raise RngError(status, where)


def raw(name: str):
    """The ctypes function of a C entry point (plain pointers and sizes)."""
    return getattr(_lib, name)


# ---- tensor marshalling -------------------------------------------------------
_ALLOWED = {
    "u32": ("uint32", "int32"), "u64": ("uint64", "int64"), "i32": ("int32",), "i64": ("int64",),
    "f32": ("float32",), "f64": ("float64",), "u8": ("uint8", "int8", "bool"), "u16": ("uint16", "int16"),
    "f16": ("float16", "uint16", "int16"),
}


def _ptr(t, kind: str, name: str = "out") -> tuple[int, int]:
    if not getattr(t, "is_cuda", False):
        raise TypeError(f"{name} must be a CUDA tensor")
    if str(t.dtype).replace("torch.", "") not in _ALLOWED[kind]:
        raise TypeError(f"{name} must have dtype {' or '.join(_ALLOWED[kind])}, not {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr(), t.numel()


def _stream(stream, t) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream(t.device).cuda_stream or None
    return int(getattr(stream, "cuda_stream", stream)) or None


def _on_device(t):
    """The library launches on the CUDA runtime's current device: make it the
    tensor's for the duration of a call."""
    import torch
    return torch.cuda.device(t.device)


def _fill(name, kind, seed, first_counter, out, stream, *extra):
    p, n = _ptr(out, kind)
    with _on_device(out):
        _check(getattr(_lib, name)(seed & 0xFFFFFFFF, first_counter & 0xFFFFFFFF, n, *extra, p,
                                   _stream(stream, out)), name)
    return out


def rng_fill_u32(seed, first_counter, out, stream=None):
    return _fill("rng_fill_u32", "u32", seed, first_counter, out, stream)


def rng_fill_u64(seed, first_counter, out, stream=None):
    return _fill("rng_fill_u64", "u64", seed, first_counter, out, stream)


def rng_fill_f32(seed, first_counter, out, stream=None):
    return _fill("rng_fill_f32", "f32", seed, first_counter, out, stream)


def rng_fill_f64(seed, first_counter, out, stream=None):
    return _fill("rng_fill_f64", "f64", seed, first_counter, out, stream)


def rng_fill_u8(seed, first_counter, out, stream=None):
    return _fill("rng_fill_u8", "u8", seed, first_counter, out, stream)


def rng_fill_u16(seed, first_counter, out, stream=None):
    return _fill("rng_fill_u16", "u16", seed, first_counter, out, stream)


def rng_fill_f16(seed, first_counter, out, stream=None):
    return _fill("rng_fill_f16", "f16", seed, first_counter, out, stream)


def rng_fill_bool(seed, first_counter, out, stream=None):
    return _fill("rng_fill_bool", "u8", seed, first_counter, out, stream)


def rng_fill_u32_below(seed, first_counter, bound, out, stream=None):
    return _fill("rng_fill_u32_below", "u32", seed, first_counter, out, stream, bound)


def rng_fill_u64_below(seed, first_counter, bound, out, stream=None):
    return _fill("rng_fill_u64_below", "u64", seed, first_counter, out, stream, bound)


def rng_fill_i32_range(seed, first_counter, low, bound, out, stream=None):
    return _fill("rng_fill_i32_range", "i32", seed, first_counter, out, stream, low, bound)


def rng_fill_i64_range32(seed, first_counter, low, bound, out, stream=None):
    return _fill("rng_fill_i64_range32", "i64", seed, first_counter, out, stream, low, bound)


def rng_fill_i64_range(seed, first_counter, low, bound, out, stream=None):
    return _fill("rng_fill_i64_range", "i64", seed, first_counter, out, stream, low, bound)


def rng_fill_normal_f32(seed, first_counter, out, stream=None):
    return _fill("rng_fill_normal_f32", "f32", seed, first_counter, out, stream)


def rng_fill_normal_f32_pairs(seed, first_counter, out, stream=None):
    return _fill("rng_fill_normal_f32_pairs", "f32", seed, first_counter, out, stream)


def rng_fill_normal_f32_precise(seed, first_counter, out, stream=None):
    return _fill("rng_fill_normal_f32_precise", "f32", seed, first_counter, out, stream)


def rng_fill_exponential_f32(seed, first_counter, out, stream=None):
    return _fill("rng_fill_exponential_f32", "f32", seed, first_counter, out, stream)


def rng_fill_exponential_f64(seed, first_counter, out, stream=None):
    return _fill("rng_fill_exponential_f64", "f64", seed, first_counter, out, stream)


def rng_fill_normal_f64(seed, first_counter, out, stream=None):
    return _fill("rng_fill_normal_f64", "f64", seed, first_counter, out, stream)


def rng_fill_normal_f64_noalloc(seed, first_counter, out, stream=None):
    """rng_fill_normal_f64 without any device allocation (n <= 2^28); see rng.h."""
    return _fill("rng_fill_normal_f64_noalloc", "f64", seed, first_counter, out, stream)


def _dropout(name, x, y, p, seed, first_counter, stream):
    px, n = _ptr(x, "f32", "x")
    py, ny = _ptr(y, "f32", "y")
    if n != ny:
        raise ValueError(f"{name}: x has {n} elements, y has {ny}")
    if x.device != y.device:
        raise ValueError(f"{name}: x is on {x.device}, y on {y.device}")
    with _on_device(y):
        _check(getattr(_lib, name)(px, py, float(p), seed & 0xFFFFFFFF, first_counter & 0xFFFFFFFF, n,
                                   _stream(stream, y)), name)
    return y


def rng_dropout_fwd(x, y, p, seed, first_counter, stream=None):
    return _dropout("rng_dropout_fwd", x, y, p, seed, first_counter, stream)


def rng_dropout_bwd(dy, dx, p, seed, first_counter, stream=None):
    return _dropout("rng_dropout_bwd", dy, dx, p, seed, first_counter, stream)


def rng_status_string(status: int) -> str:
    return _lib.rng_status_string(status).decode()


def rng_last_error() -> str:
    return _lib.rng_last_error().decode()


def rng_debug_set_miss_capacity(capacity: int | None) -> None:
    _check(_lib.rng_debug_set_miss_capacity((1 << 64) - 1 if capacity is None else capacity),
           "rng_debug_set_miss_capacity")


def rng_debug_last_miss_count() -> int:
    c = _u64()
    _check(_lib.rng_debug_last_miss_count(C.byref(c)), "rng_debug_last_miss_count")
    return c.value


def rng_debug_launch_count() -> int:
    return _lib.rng_debug_launch_count()


def rng_debug_write_ceiling(which: int, buf, stream=None):
    """which = 0: cudaMemsetAsync over buf; 1: the plain 16-byte store kernel."""
    if not buf.is_contiguous():
        raise ValueError("rng_debug_write_ceiling: buf must be contiguous")
    nbytes = buf.numel() * buf.element_size()
    with _on_device(buf):
        _check(_lib.rng_debug_write_ceiling(which, buf.data_ptr(), nbytes, _stream(stream, buf)),
               "rng_debug_write_ceiling")
    return buf


def rng_debug_eval_f64(which: int, inp, out, stream=None):
    pi, n = _ptr(inp, "f64", "in")
    po, no = _ptr(out, "f64", "out")
    if n != no:
        raise ValueError("in and out differ in length")
    if inp.device != out.device:
        raise ValueError(f"rng_debug_eval_f64: in is on {inp.device}, out on {out.device}")
    with _on_device(out):
        _check(_lib.rng_debug_eval_f64(which, pi, po, n, _stream(stream, out)), "rng_debug_eval_f64")
    return out
