"""The public device header (include/rng_device.cuh) used the way a fused
user kernel would use it: kernels compiled against the header alone must
draw what the oracle defines and what the library's fills write, and the
Phobos page's dropout_rows tile kernel must equal rng_dropout_fwd."""
import ctypes as C
import os
import shutil
import subprocess

import numpy as np
import pytest

from helpers import ROOT

SRC = os.path.join(ROOT, "tests", "device_api", "device_api_kernels.cu")
BUILD = os.path.join(ROOT, "tests", "device_api", "_build")
U32 = 1 << 32


def _nvcc():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


@pytest.fixture(scope="module")
def devlib():
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not available")
    os.makedirs(BUILD, exist_ok=True)
    so = os.path.join(BUILD, "libdevice_api_kernels.so")
    deps = [SRC] + [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))]
    if not os.path.exists(so) or os.path.getmtime(so) < max(os.path.getmtime(d) for d in deps):
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                        "-I" + os.path.join(ROOT, "include"), "-Xcompiler", "-fPIC", "-shared", SRC,
                        "-o", so + ".tmp"], check=True)
        os.replace(so + ".tmp", so)
    lib = C.CDLL(so)
    lib.device_api_draws.argtypes = [C.c_uint32, C.c_uint32, C.c_uint32] + [C.c_void_p] * 6
    lib.device_api_neglog.argtypes = [C.c_void_p, C.c_void_p, C.c_uint32, C.c_int]
    lib.device_api_cos2pi.argtypes = [C.c_void_p, C.c_void_p, C.c_uint32, C.c_int]
    lib.device_api_box_muller.argtypes = [C.c_void_p] * 5 + [C.c_uint32]
    lib.device_api_dropout_rows.argtypes = [C.c_void_p, C.c_void_p, C.c_uint32, C.c_uint32, C.c_float, C.c_uint32,
                                            C.c_int, C.POINTER(C.c_int), C.POINTER(C.c_float)]
    lib.device_api_host_hash32.argtypes = [C.c_uint32]
    lib.device_api_host_hash32.restype = C.c_uint32
    return lib


def test_header_neglog_table_matches_the_oracle(orc):
    """The header's generated table (gen_neglog_table.py: exact rationals and
    mpmath) equals the oracle's own (binary64 and binary128 in C), entry by
    entry: two derivations from the same definition."""
    import re
    txt = open(os.path.join(ROOT, "include", "lowbias32_neglog_table.inc")).read()

    def val(t):
        t = t.strip()
        assert t.endswith("f"), t
        return float.fromhex(t[:-1]) if "x" in t else float(t[:-1])

    rows = re.findall(r"^    \{([^}]*)\},", txt, re.M)
    table = np.array([[val(x) for x in r.split(",")] for r in rows])
    inv, hi, lo, ln2 = orc.neglog_table()
    assert table.shape == (257, 4)
    assert np.array_equal(table[:, 0], inv) and np.array_equal(table[:, 1], hi) and np.array_equal(table[:, 2], lo)
    consts = dict(re.findall(r"kNegLogLn2(Hi|Lo) = ([^;]+);", txt))
    assert val(consts["Hi"]) == ln2[0] and val(consts["Lo"]) == ln2[1]


@pytest.mark.gpu
def test_header_neglog_on_every_input(devlib, orc):
    """neg_log_grid on all 2^23 inputs equals the oracle's own f32 log, bit for
    bit, alone and in the paired f32x2 form the fills use (each input paired
    with its neighbour and, reversed, with another)."""
    import torch
    m = np.arange(1 << 23, dtype=np.uint32)
    want = orc.neglog_array(m).view(np.uint32)
    out = torch.empty(m.size, dtype=torch.float32, device="cuda")
    for order, paired in ((m, 0), (m, 1), (m[::-1].copy(), 1)):
        mg = torch.from_numpy(order.view(np.int32)).cuda()
        assert devlib.device_api_neglog(mg.data_ptr(), out.data_ptr(), m.size, paired) == 0
        got = out.cpu().numpy().view(np.uint32)
        bad = np.nonzero(got != want[order])[0]
        assert bad.size == 0, (paired, bad.size, [(int(i), int(order[i]), hex(int(got[i])), hex(int(want[order][i])))
                                                  for i in bad[:8]])


def test_header_cos2pi_coefficients_match_the_oracle(orc):
    """The header's generated coefficients (gen_cos2pi_coefficients.py, mpmath)
    equal the oracle's own (binary128 in C), in the oracle's order."""
    import re
    txt = open(os.path.join(ROOT, "include", "lowbias32_cos2pi.inc")).read()
    vals = dict(re.findall(r"constexpr float (kCos2Pi\w+) = ([^;]+);", txt))
    names = ["S1Hi", "S1Lo", "S3", "S5", "S7", "S9", "C2Hi", "C2Lo", "C4", "C6", "C8", "C10"]
    got = np.array([float.fromhex(vals["kCos2Pi" + k][:-1]) for k in names])
    assert np.array_equal(got, orc.cos2pi_coefficients().astype(np.float64))


@pytest.mark.gpu
def test_header_cos2pi_on_every_input(devlib, orc):
    """cos2pi_grid on all 2^23 inputs equals the oracle's own cosine, bit for
    bit, alone and in the paired f32x2 form the precise fill uses."""
    import torch
    m = np.arange(1 << 23, dtype=np.uint32)
    want = orc.cos2pi_array(m).view(np.uint32)
    out = torch.empty(m.size, dtype=torch.float32, device="cuda")
    for order, paired in ((m, 0), (m, 1), (m[::-1].copy(), 1)):
        mg = torch.from_numpy(order.view(np.int32)).cuda()
        assert devlib.device_api_cos2pi(mg.data_ptr(), out.data_ptr(), m.size, paired) == 0
        got = out.cpu().numpy().view(np.uint32)
        bad = np.nonzero(got != want[order])[0]
        assert bad.size == 0, (paired, bad.size, [(int(i), int(order[i]), hex(int(got[i])), hex(int(want[order][i])))
                                                  for i in bad[:8]])


@pytest.mark.gpu
def test_header_randn_on_every_u0(devlib, orc):
    """randn_of_draws and randn_pair_of_draws for all 2^23 grid values of u0,
    within 4e-6 (1 + |z|) of the oracle's binary64 Box-Muller branches: with
    u1 = 0 (cos = 1, so z is the radius: the series below u0 = 2^-7 and the
    hardware log2 above it, unmasked), with every u1 against one large radius,
    and with seeded random angles and random bits above the 23-bit grid.  The
    pair's cosine branch is randn_of_draws' value bit for bit."""
    import torch
    m = np.arange(1 << 23, dtype=np.uint32)
    gen = np.random.default_rng(20261202)
    high = gen.integers(0, 1 << 9, m.size, dtype=np.uint32) << np.uint32(23)
    cases = {"u1 = 0": (m, np.zeros_like(m)),
             "u0 = 1 - 2^-23, every u1": (np.full_like(m, 0x7FFFFF), m),
             "random u1": (m | high, gen.integers(0, 1 << 32, m.size, dtype=np.uint64).astype(np.uint32))}
    out, px, py = (torch.empty(m.size, dtype=torch.float32, device="cuda") for _ in range(3))
    for name, (d0, d1) in cases.items():
        g0 = torch.from_numpy(d0.view(np.int32)).cuda()
        g1 = torch.from_numpy(d1.view(np.int32)).cuda()
        assert devlib.device_api_box_muller(g0.data_ptr(), g1.data_ptr(), out.data_ptr(), px.data_ptr(),
                                            py.data_ptr(), m.size) == 0
        assert torch.equal(out.view(torch.int32), px.view(torch.int32)), name
        ref_x, ref_y = orc.box_muller_array(d0, d1, sine=True)
        for got, ref, branch in ((out, ref_x, "cos"), (py, ref_y, "sin")):
            err = np.abs(got.cpu().numpy().astype(np.float64) - ref) / (1 + np.abs(ref))
            print(f"randn of draws, {name}, {branch}: worst |err| / (1 + |z|) = {err.max():.3e}")
            assert err.max() <= 4e-6, (name, branch, int(np.argmax(err)), float(err.max()))


def test_header_hash_on_the_host_matches_the_oracle(devlib, orc):
    for x in (0, 1, 2, 0x9E3779B9, U32 - 1, 123456789):
        assert devlib.device_api_host_hash32(x) == orc.hash32(x)


@pytest.mark.gpu
@pytest.mark.parametrize("first", [0, 3, U32 - 5])
def test_header_draws_match_the_oracle_and_the_fills(devlib, orc, first):
    import torch

    import dropout_lowbias32_hash32_gb300 as rng
    n, seed = 100003, 0x9E3779B9
    d32 = torch.empty(n, dtype=torch.int32, device="cuda")
    d64 = torch.empty(n, dtype=torch.int64, device="cuda")
    u = torch.empty(n, dtype=torch.float32, device="cuda")
    z = torch.empty(n, dtype=torch.float32, device="cuda")
    ex = torch.empty(n, dtype=torch.float32, device="cuda")
    zp = torch.empty(n, dtype=torch.float32, device="cuda")
    assert devlib.device_api_draws(seed, first, n, d32.data_ptr(), d64.data_ptr(), u.data_ptr(), z.data_ptr(),
                                   ex.data_ptr(), zp.data_ptr()) == 0
    assert np.array_equal(d32.cpu().numpy().view(np.uint32), orc.fill_u32(seed, first, n))
    assert np.array_equal(d64.cpu().numpy().view(np.uint64), orc.fill_u64(seed, first, n))
    assert np.array_equal(u.cpu().numpy().view(np.uint32), orc.fill_f32(seed, first, n).view(np.uint32))
    ref = orc.fill_randn(seed, first, n)
    zz = z.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(zz - ref) / (1 + np.abs(ref))) <= 4e-6
    # the fused draw is the library fill's element, bit for bit
    lib_z = rng.rng_fill_normal_f32(seed, first, torch.empty(n, dtype=torch.float32, device="cuda"))
    assert torch.equal(lib_z.view(torch.int32), z.view(torch.int32))
    assert np.array_equal(ex.cpu().numpy().view(np.uint32),
                          orc.fill_exponential_f32_own(seed, first, n).view(np.uint32))
    lib_ex = rng.rng_fill_exponential_f32(seed, first, torch.empty(n, dtype=torch.float32, device="cuda"))
    assert torch.equal(lib_ex.view(torch.int32), ex.view(torch.int32))
    assert np.array_equal(zp.cpu().numpy().view(np.uint32), orc.fill_randn_precise(seed, first, n).view(np.uint32))
    lib_zp = rng.rng_fill_normal_f32_precise(seed, first, torch.empty(n, dtype=torch.float32, device="cuda"))
    assert torch.equal(lib_zp.view(torch.int32), zp.view(torch.int32))


CANDIDATES = (1, 2, 4, 8, 16, 32)


@pytest.mark.gpu
@pytest.mark.parametrize("p", [0.1, 0.5])
@pytest.mark.parametrize("R", CANDIDATES)
def test_dropout_rows_tile_kernel_equals_the_fused_fill(devlib, orc, p, R):
    import torch

    import dropout_lowbias32_hash32_gb300 as rng
    from dropout_lowbias32_hash32_gb300 import workloads
    rows = 1003  # a ragged last tile for every R > 1
    x = workloads.dropout_x(rows * 256)
    xg = torch.from_numpy(x).cuda()
    y = torch.empty_like(xg)
    chosen = C.c_int(-1)
    assert devlib.device_api_dropout_rows(xg.data_ptr(), y.data_ptr(), rows, 42, p, 0, R, C.byref(chosen), None) == 0
    assert chosen.value == R
    assert np.array_equal(y.cpu().numpy().view(np.uint32), orc.dropout(x, p, 42, 0).view(np.uint32))
    y_lib = rng.rng_dropout_fwd(xg, torch.empty_like(xg), p, 42, 0)
    assert torch.equal(y.view(torch.int32), y_lib.view(torch.int32))


@pytest.mark.gpu
def test_dropout_rows_autotune_picks_a_candidate_and_keeps_the_values(devlib, orc):
    """The listing's @autotune over R: every candidate is timed on the caller's
    buffers, the fastest is returned, and the output is the same whatever R
    (a first counter near the 2^32 wrap)."""
    import torch

    from dropout_lowbias32_hash32_gb300 import workloads
    rows, first = 1 << 16, U32 - 1000  # 64 MiB; counters wrap
    x = workloads.dropout_x(rows * 256)
    xg = torch.from_numpy(x).cuda()
    y = torch.empty_like(xg)
    chosen = C.c_int(-1)
    ms = (C.c_float * len(CANDIDATES))()
    assert devlib.device_api_dropout_rows(xg.data_ptr(), y.data_ptr(), rows, 7, 0.25, first, 0,
                                          C.byref(chosen), ms) == 0
    assert chosen.value in CANDIDATES
    assert all(t > 0 for t in ms) and ms[CANDIDATES.index(chosen.value)] == min(ms)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), orc.dropout(x, 0.25, 7, first).view(np.uint32))


@pytest.mark.gpu
def test_dropout_rows_in_place(devlib, orc):
    import torch

    from dropout_lowbias32_hash32_gb300 import workloads
    rows = 517
    x = workloads.dropout_x(rows * 256)
    yg = torch.from_numpy(x).cuda()
    assert devlib.device_api_dropout_rows(yg.data_ptr(), yg.data_ptr(), rows, 3, 0.5, 11, 16, None, None) == 0
    assert np.array_equal(yg.cpu().numpy().view(np.uint32), orc.dropout(x, 0.5, 3, 11).view(np.uint32))
