"""Out-of-bounds guard: every fill writes exactly its n elements.

The output slice sits inside a larger buffer pre-filled with a canary byte
pattern; after the fill, every byte before and after the slice must still
hold the canary (a stand-in for a bounds-checking sanitizer, which is not
available here).  Sizes bracket the vector width and one block's run of each
generator (up to 32768 elements); offsets cover every start within a 16-byte
vector (within 32 bytes for dropout)."""
import numpy as np
import pytest

from test_gpu_parity import fills

pytestmark = pytest.mark.gpu
U32 = 1 << 32
CANARY = 0xA5
GUARD = 4096  # bytes on each side
SIZES = (0, 1, 3, 17, 2047, 2049, 4095, 4097, 8191, 8193, 16383, 16385, 32767, 32769, 3 * 152 * 8 * 256 * 4 + 13)
NAMES = ["u32", "u64", "f32", "f64", "u32_below_1000", "u64_below_1000", "i32_range", "i64_range32", "i64_range",
         "normal_f64", "u8", "u16", "f16", "bool", "exponential_f32", "exponential_f64", "normal_f32_precise",
         "normal_f32", "normal_f32_pairs"]


def _gpu_fill(rng, torch, orc, name):
    """The fill's call and output dtype (the f32 Box-Muller fills are held to a
    tolerance, so the bit-exact parity table does not list them)."""
    if name == "normal_f32":
        return (lambda out, first: rng.rng_fill_normal_f32(7, first, out)), torch.float32
    if name == "normal_f32_pairs":
        return (lambda out, first: rng.rng_fill_normal_f32_pairs(7, first, out)), torch.float32
    gpu, dtype, _ = fills(rng, torch, orc)[name]
    return gpu, dtype


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


@pytest.fixture(scope="module")
def rng(torch):
    import dropout_lowbias32_hash32_gb300 as r
    return r


@pytest.mark.parametrize("name", NAMES)
def test_fill_writes_only_its_elements(rng, torch, orc, name):
    gpu, dtype = _gpu_fill(rng, torch, orc, name)
    size = torch.empty(0, dtype=dtype).element_size()
    for n in SIZES:
        for offset in range(16 // size):
            total = GUARD + (offset + n) * size + GUARD
            buf = torch.full((total,), CANARY, dtype=torch.uint8, device="cuda")
            start = GUARD + offset * size
            out = buf[start:start + n * size].view(dtype)
            for first in (0, U32 - 5):
                gpu(out, first)
            host = buf.cpu().numpy()
            assert np.all(host[:start] == CANARY), (name, n, offset, "before")
            assert np.all(host[start + n * size:] == CANARY), (name, n, offset, "after")
            if n >= 16:
                assert not np.all(host[start:start + n * size] == CANARY), (name, n, offset, "not written")


def test_dropout_writes_only_its_elements(rng, torch):
    """y at every offset within 32 bytes, x aligned (the 32-byte kernel at
    offset 0, the 16-byte one at offset 4, the scalar one otherwise) and x at
    y's offset (the 32-byte kernel with a head of 0..7 elements)."""
    from dropout_lowbias32_hash32_gb300 import workloads
    for n in SIZES:
        xh = torch.from_numpy(workloads.dropout_x(max(n, 1) + 8)).cuda()
        for offset in range(8):
            for x in (xh[:n], xh[offset:offset + n]):
                buf = torch.full((GUARD + (offset + n) * 4 + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
                start = GUARD + offset * 4
                y = buf[start:start + n * 4].view(torch.float32)
                rng.rng_dropout_fwd(x, y, 0.3, 42, 0)
                host = buf.cpu().numpy()
                assert np.all(host[:start] == CANARY) and np.all(host[start + n * 4:] == CANARY), (n, offset)
                if n >= 16:
                    assert not np.all(host[start:start + n * 4] == CANARY), (n, offset, "not written")
