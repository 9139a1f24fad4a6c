"""The library's generated tables against the oracle's own derivations.

Each table used by a kernel is computed twice from its definition, by a
generator script of the CUDA side (mpmath, exact rationals) and by the oracle
in C (binary128 arithmetic); neither uses the other.  They must agree entry by
entry, which is what makes the kernels' bit-exact parity possible."""
import os
import re

import numpy as np

from helpers import ROOT

CSRC = os.path.join(ROOT, "dropout_lowbias32_hash32_gb300", "csrc")


def _hex_floats(block: str) -> np.ndarray:
    return np.array([float.fromhex(t) for t in re.findall(r"-?0x[0-9a-f.]+p[+-]\d+", block)])


def _macro(text: str, name: str) -> str:
    start = text.index(f"#define {name} \\")
    end = text.index("\n#define", start + 1)
    return text[start:end]


def test_ziggurat_table_equals_the_oracle(orc):
    """X[0..1024] and F[0..1024] of the 1024-layer Marsaglia-Tsang table:
    gen_zig_tables.py (mpmath, Anderson root finder) and the oracle (binary128
    bisection on the closure residual), all 2050 entries bit for bit; the
    fast-path and wedge pairs are built from them."""
    text = open(os.path.join(CSRC, "zig_tables.inc")).read()
    X = _hex_floats(_macro(text, "ZIG_X_VALUES"))
    F = _hex_floats(_macro(text, "ZIG_F_VALUES"))
    ox, of = orc.zig1024()
    assert X.size == 1025 and F.size == 1025
    assert np.array_equal(X.view(np.uint64), ox.view(np.uint64))
    assert np.array_equal(F.view(np.uint64), of.view(np.uint64))
    pairs = _hex_floats(_macro(text, "ZIG_HALFX_XNEXT_VALUES")).reshape(-1, 2)
    assert np.array_equal(pairs[:, 0], X[:1024] / 2) and np.array_equal(pairs[:, 1], X[1:])


def test_f64_log_table_equals_the_oracle(orc):
    """The f64 exponential's fixed-point log: I_j, ln(inv_j) 2^96, ln 2 2^96 and
    the Horner constants 1/k, gen_neglog64_table.py (mpmath, exact rationals)
    against the oracle (binary128), entry by entry."""
    text = open(os.path.join(CSRC, "neglog64_table.inc")).read()
    rows = re.findall(r"\{0x([0-9a-f]+)ull, 0x([0-9a-f]+)ull\}", text)
    inv, lninv, ln2, coef = orc.neglog64_table()
    assert len(rows) == 2048
    for j, (lo, packed) in enumerate(rows):
        lo, packed = int(lo, 16), int(packed, 16)
        hi = packed & ((1 << 48) - 1)
        hi -= (hi >> 47) << 48  # the signed 48-bit field
        assert packed >> 48 == inv[j], j
        assert (hi << 64) + lo == lninv[j], j
    lo = int(re.search(r"kNegLog64Ln2Lo = 0x([0-9a-f]+)ull", text).group(1), 16)
    hi = int(re.search(r"kNegLog64Ln2Hi = (-?\d+)ll", text).group(1))
    assert (hi << 64) + lo == ln2
    for k in range(1, 7):
        assert int(re.search(rf"kNegLog64D{k} = (\d+)u", text).group(1)) == coef[k], k
