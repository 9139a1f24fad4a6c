"""The C-ABI library loads and exports every entry point include/rng.h
declares, and rejects bad arguments before touching the GPU (no GPU needed:
every call here returns before any CUDA call)."""
import ctypes as C
import math
import os
import re

import pytest

from helpers import ROOT

HEADER = os.path.join(ROOT, "include", "rng.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rng_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def rng():
    import dropout_lowbias32_hash32_gb300 as rng
    return rng


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("rng_fill_u32", "rng_fill_u64", "rng_fill_f32", "rng_fill_f64",
                     "rng_fill_u32_below", "rng_fill_u64_below", "rng_fill_i32_range",
                     "rng_fill_i64_range32", "rng_fill_i64_range", "rng_fill_normal_f32",
                     "rng_fill_normal_f64", "rng_dropout_fwd", "rng_dropout_bwd",
                     "rng_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(rng):
    lib = C.CDLL(rng.LIBRARY_PATH)
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing


def test_status_strings(rng):
    assert rng.rng_status_string(0) == "RNG_OK"
    for st in (1, 2, 3):
        assert rng.rng_status_string(st).startswith("RNG_E")
    assert "unknown" in rng.rng_status_string(99)


def test_null_output_rejected(rng):
    for name in ("rng_fill_u32", "rng_fill_u64", "rng_fill_f32", "rng_fill_f64",
                 "rng_fill_normal_f32", "rng_fill_normal_f64"):
        assert rng.raw(name)(1, 0, 7, None, None) == rng.RNG_EINVAL
        assert "NULL" in rng.rng_last_error()
    assert rng.raw("rng_fill_u32_below")(1, 0, 7, 10, None, None) == rng.RNG_EINVAL


def test_zero_length_is_a_noop(rng):
    assert rng.raw("rng_fill_u32")(1, 0, 0, None, None) == rng.RNG_OK
    assert rng.raw("rng_fill_normal_f64")(1, 0, 0, None, None) == rng.RNG_OK
    assert rng.raw("rng_dropout_fwd")(None, None, 0.5, 1, 0, 0, None) == rng.RNG_OK


def test_misaligned_output_rejected(rng):
    # a pointer that is not a multiple of the element size (never dereferenced)
    assert rng.raw("rng_fill_u64")(1, 0, 4, 0x1004, None) == rng.RNG_EINVAL
    assert rng.raw("rng_fill_f32")(1, 0, 4, 0x1002, None) == rng.RNG_EINVAL
    assert "aligned" in rng.rng_last_error()


def test_length_past_the_address_space_rejected(rng):
    # pointers never dereferenced: the range check runs before anything is enqueued
    assert rng.raw("rng_fill_u32")(1, 0, 1 << 62, 0x1000, None) == rng.RNG_EINVAL
    assert "address space" in rng.rng_last_error()
    assert rng.raw("rng_fill_u64")(1, 0, 1 << 61, 0x1000, None) == rng.RNG_EINVAL
    assert rng.raw("rng_fill_u8")(1, 0, (1 << 64) - 0x1000, 0x1000, None) == rng.RNG_EINVAL
    assert rng.raw("rng_fill_normal_f64")(1, 0, 1 << 61, 0x1000, None) == rng.RNG_EINVAL
    assert rng.raw("rng_dropout_fwd")(0x1000, 0x2000, 0.5, 1, 0, 1 << 62, None) == rng.RNG_EINVAL
    assert rng.raw("rng_debug_write_ceiling")(1, 0x1000, (1 << 64) - 16, None) == rng.RNG_EINVAL
    assert "address space" in rng.rng_last_error()


def test_zero_bound_rejected(rng):
    assert rng.raw("rng_fill_u32_below")(1, 0, 4, 0, 0x1000, None) == rng.RNG_EINVAL
    assert rng.raw("rng_fill_u64_below")(1, 0, 4, 0, 0x1000, None) == rng.RNG_EINVAL
    assert rng.raw("rng_fill_i32_range")(1, 0, 4, -5, 0, 0x1000, None) == rng.RNG_EINVAL
    assert rng.raw("rng_fill_i64_range32")(1, 0, 4, -5, 0, 0x1000, None) == rng.RNG_EINVAL
    assert rng.raw("rng_fill_i64_range")(1, 0, 4, -5, 0, 0x1000, None) == rng.RNG_EINVAL


@pytest.mark.parametrize("p", [-0.1, 1.0, 1.5, math.nan, math.inf])
def test_dropout_probability_rejected(rng, p):
    assert rng.raw("rng_dropout_fwd")(0x1000, 0x2000, p, 1, 0, 4, None) == rng.RNG_EINVAL
    assert rng.raw("rng_dropout_bwd")(0x1000, 0x2000, p, 1, 0, 4, None) == rng.RNG_EINVAL


def test_dropout_partial_overlap_rejected(rng):
    # y starts 4 elements into x's 16: overlapping but not the same array
    assert rng.raw("rng_dropout_fwd")(0x1000, 0x1010, 0.5, 1, 0, 16, None) == rng.RNG_EINVAL
    assert "overlap" in rng.rng_last_error()
    assert rng.raw("rng_dropout_fwd")(None, 0x1000, 0.5, 1, 0, 16, None) == rng.RNG_EINVAL


def test_debug_hooks_without_gpu(rng):
    assert rng.raw("rng_debug_eval_f64")(5, None, None, 0, None) == rng.RNG_EINVAL
    assert rng.raw("rng_debug_eval_f64")(-1, None, None, 0, None) == rng.RNG_EINVAL
    assert rng.raw("rng_debug_last_miss_count")(None) == rng.RNG_EINVAL
    assert rng.rng_debug_launch_count() >= 0
    rng.rng_debug_set_miss_capacity(None)
    ceiling = rng.raw("rng_debug_write_ceiling")
    assert ceiling(2, 0x1000, 16, None) == rng.RNG_EINVAL
    assert ceiling(0, None, 16, None) == rng.RNG_EINVAL
    assert ceiling(1, 0x1008, 16, None) == rng.RNG_EINVAL  # misaligned for the store kernel
    assert ceiling(1, 0x1000, 24, None) == rng.RNG_EINVAL  # not whole 16-byte vectors
    assert ceiling(1, 0x1000, 0, None) == rng.RNG_OK


def test_python_names_match_c_names(rng):
    for name in declared_symbols():
        assert hasattr(rng, name), name


def test_package_fails_loudly_without_its_library(tmp_path):
    """There is no CPU fallback: a copy of the package without the built
    library refuses to import, naming the missing file."""
    import shutil
    import subprocess
    import sys
    src = os.path.join(ROOT, "dropout_lowbias32_hash32_gb300")
    dst = tmp_path / "dropout_lowbias32_hash32_gb300"
    shutil.copytree(src, dst, ignore=shutil.ignore_patterns("_lib", "_build", "__pycache__"))
    res = subprocess.run([sys.executable, "-c", "import dropout_lowbias32_hash32_gb300"], cwd=tmp_path,
                         capture_output=True, text=True, env={**os.environ, "PYTHONPATH": str(tmp_path)})
    assert res.returncode != 0
    assert "ImportError" in res.stderr and "librng_lowbias32.so" in res.stderr
