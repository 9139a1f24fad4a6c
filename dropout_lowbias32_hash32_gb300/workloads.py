"""Synthetic workloads: the configurations the fills are measured and
checked on, and seeded generators for the inputs dropout reads.

The generators draw from numpy's PCG64 and hold none of the lowbias32
arithmetic, so the same inputs serve the CUDA path and the CPU oracle.

Configurations (sizes, seeds, counters) follow the measured workloads:
  uniform fills   2^28 elements of u32, u64, f32, f64; seed 0x9E3779B9;
                  first counter in {0, 1, 3, 2^32 - 5} (unaligned starts and
                  the counter wrap);
  bounded         2^28 elements; u32_below(1000), u32_below(2^32 - 2),
                  u64_below(1000), u64_below(2^64 - 2), low + u32_below(1000)
                  into int32 and int64 (low = -500), low + u64_below(1000)
                  into int64; seeds 1..4;
  normals         2^24 and 2^28 elements, f32 Box-Muller and the f64
                  ziggurat, seed 7, first counter in {0, 1, 3};
  dropout         X of shape [2^20, 256] f32 ~ U(-1, 1), p in {0.1, 0.5},
                  seed 42, counter = flat index; dY ~ N(0, 1) f32.
"""
from __future__ import annotations

import numpy as np

N_FULL = 1 << 28
UNIFORM_SEED = 0x9E3779B9
FIRST_COUNTERS = (0, 1, 3, (1 << 32) - 5)
BOUNDED_SEEDS = (1, 2, 3, 4)
LOW = -500
NORMAL_SEED = 7
NORMAL_SIZES = (1 << 24, 1 << 28)
DROPOUT_SHAPE = (1 << 20, 256)
DROPOUT_P = (0.1, 0.5)
DROPOUT_SEED = 42
X_SEED = 11
DY_SEED = 12


def dropout_x(n: int, seed: int = X_SEED) -> np.ndarray:
    """X ~ U(-1, 1) as f32."""
    return np.random.default_rng(seed).uniform(-1.0, 1.0, n).astype(np.float32)


def dropout_dy(n: int, seed: int = DY_SEED) -> np.ndarray:
    """dY ~ N(0, 1) as f32."""
    return np.random.default_rng(seed).standard_normal(n, dtype=np.float32)


def special_floats() -> np.ndarray:
    """Signed zeros, subnormals, extremes, infinities and NaN (f32)."""
    f = np.finfo(np.float32)
    vals = [0.0, -0.0, f.tiny, -f.tiny, f.smallest_subnormal, -f.smallest_subnormal,
            f.smallest_subnormal * 3, f.max, -f.max, f.eps, 1.0, -1.0, np.inf, -np.inf, np.nan]
    return np.array(vals, dtype=np.float32)
