"""rng_fill_normal_f64_noalloc: the f64 normal fill for callers that cannot
call cudaMalloc -- code whose device memory belongs to another allocator (a
caching allocator that reserved the pool up front) or that cannot take
cudaMalloc's implicit device synchronisation.  It keeps its miss list in the
library's static device array instead of allocating one.

Called through the C ABI with plain pointers and checked bit for bit (the
f64 normal's parity bar) against the CPU oracle and against
rng_fill_normal_f64, on two calls in a row; this file runs last so that a
failure here leaves every other test run.
"""
import ctypes as C

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

U32 = 1 << 32
MAX_N = 1 << 28


@pytest.fixture(scope="module")
def torch():
    import torch
    assert torch.cuda.is_available(), "these tests need the GB300"
    return torch


@pytest.fixture(scope="module")
def rng(torch):
    import dropout_lowbias32_hash32_gb300 as rng
    return rng


def _noalloc(rng, torch, seed, first, out):
    fn = rng.raw("rng_fill_normal_f64_noalloc")
    stream = torch.cuda.current_stream().cuda_stream
    return fn(seed, first, out.numel(), out.data_ptr(), C.c_void_p(stream or None))


def _reference(rng, torch, seed, first, n, offset=0):
    ref = torch.empty(n + offset, dtype=torch.float64, device="cuda")[offset:]
    return rng.rng_fill_normal_f64(seed, first, ref)


def _bits(a):
    return np.ascontiguousarray(a).view(np.int64)


def test_two_calls_in_a_row_match_the_oracle_and_the_allocating_fill(rng, torch, orc):
    cases = [(7, 3, (1 << 20) + 3, 1), (11, U32 - 5, (1 << 22) + 1, 0)]
    outs = []
    for seed, first, n, offset in cases:
        out = torch.empty(n + offset, dtype=torch.float64, device="cuda")[offset:]
        assert _noalloc(rng, torch, seed, first, out) == rng.RNG_OK, rng.rng_last_error()
        outs.append(out)
    torch.cuda.synchronize()
    for (seed, first, n, offset), out in zip(cases, outs):
        got = out.cpu().numpy()
        want = orc.fill_normal_f64(seed, first, n)
        bad = np.nonzero(_bits(got) != _bits(want))[0]
        assert bad.size == 0, (seed, first, n, bad[:5])
        ref = _reference(rng, torch, seed, first, n, offset)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int64), ref.view(torch.int64)), (seed, first, n)


def _oracle_at_every_miss_and_a_sample(torch, orc, out, seed, first, n):
    """The oracle's values at every element whose first draw misses the fast
    path and at 2^18 random positions plus both ends."""
    fast = np.empty(n, np.uint8)
    step = 1 << 24
    for a in range(0, n, step):
        fast[a:a + step] = orc.fill_zig_fast(seed, first + a, min(step, n - a))
    g = np.random.default_rng(5)
    idx = np.unique(np.concatenate([np.nonzero(fast == 0)[0], g.integers(0, n, 1 << 18),
                                    np.arange(4096), np.arange(n - 4096, n)]).astype(np.int64))
    got = out[torch.from_numpy(idx).cuda()].cpu().numpy()
    want = orc.fill_normal_f64(seed, first, idx=idx)
    bad = np.nonzero(_bits(got) != _bits(want))[0]
    assert bad.size == 0, (idx[bad[:5]], bad.size)


def test_maximum_size_twice_and_no_device_allocation(rng, torch, orc):
    out = torch.empty(MAX_N, dtype=torch.float64, device="cuda")
    ref = _reference(rng, torch, 7, 0, MAX_N)
    assert _noalloc(rng, torch, 7, 0, out) == rng.RNG_OK  # set-up on this device happens by now
    torch.cuda.synchronize()
    _oracle_at_every_miss_and_a_sample(torch, orc, out, 7, 0, MAX_N)
    assert torch.equal(out.view(torch.int64), ref.view(torch.int64))
    free_before, _ = torch.cuda.mem_get_info()
    out.fill_(0)
    assert _noalloc(rng, torch, 7, 0, out) == rng.RNG_OK
    assert _noalloc(rng, torch, 7, 0, out) == rng.RNG_OK
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    assert torch.equal(out.view(torch.int64), ref.view(torch.int64))
    del out, ref
    torch.cuda.empty_cache()


def test_sizes_beyond_the_maximum_are_rejected(rng, torch):
    fn = rng.raw("rng_fill_normal_f64_noalloc")
    assert fn(7, 0, MAX_N + 1, 0x1000, None) == rng.RNG_EINVAL
    assert "2^28" in rng.rng_last_error()
    assert fn(7, 0, 0, None, None) == rng.RNG_OK
