"""Seeded synthetic inputs for the scan, compaction and split workloads.

This module only draws inputs: it holds none of the scan's arithmetic and is
the one piece of Python shared by the tests, the benchmark and the oracle
checks.  All draws use NumPy's ``default_rng(seed)`` (PCG64) on the host.

Workloads (sizes and distributions as the pages' applications use them;
the pages fix no generator, so the seeds are this library's convention):

* ``small_digits``  -- int32 uniform in [0, 9], N = 65,536, seed 0;
* ``unit_floats``   -- fp32 uniform in [0, 1), N = 2^24, seed 1;
* ``compaction``    -- int32 uniform over the whole int32 range, N = 2^26,
  seed 2, with the predicate x > t at selectivities 1 %, 50 %, 99 %;
* ``brackets``      -- int32 +1/-1 with p = 0.5 each, N = 2^28, seed 3
  (the bracket sequence of geek-doc.cn section 一);
* ``radix_keys``    -- uint32 uniform over [0, 2^32), N = 2^26, seed 4;
* ``max_values``    -- int32 uniform over the whole range, N = 2^28, seed 5;
* ``xor_values``    -- uint32 uniform over [0, 2^32), N = 2^28, seed 6;
* ``segmented``     -- int32 uniform in [0, 9] with segment heads drawn
  independently with p = 1/1024 (mean segment length 1,024; element 0 a
  head), N = 2^28, seed 7 (the pages give no segmented workload: the size
  follows the operator sweep, the values the 65,536-element case).
"""
from __future__ import annotations

import numpy as np

N_SMALL = 65_536
N_F32 = 1 << 24
N_COMPACT = 1 << 26
N_SWEEP = 1 << 28
N_SORT = 1 << 26

SELECTIVITIES = (0.01, 0.50, 0.99)


def small_digits(n: int = N_SMALL, seed: int = 0) -> np.ndarray:
    return np.random.default_rng(seed).integers(0, 10, n, dtype=np.int32)


def unit_floats(n: int = N_F32, seed: int = 1) -> np.ndarray:
    return np.random.default_rng(seed).random(n, dtype=np.float32)


def full_range_i32(n: int, seed: int) -> np.ndarray:
    return np.random.default_rng(seed).integers(-2**31, 2**31, n, dtype=np.int32)


def full_range_u32(n: int, seed: int) -> np.ndarray:
    return np.random.default_rng(seed).integers(0, 2**32, n, dtype=np.uint32)


def compaction_values(n: int = N_COMPACT, seed: int = 2) -> np.ndarray:
    return full_range_i32(n, seed)


def threshold_for(selectivity: float) -> int:
    """t such that P(x > t) is closest to ``selectivity`` for x uniform over
    all 2^32 int32 values, where P(x > t) = (2^31 - 1 - t) / 2^32."""
    t = round((2**31 - 1) - selectivity * 2**32)
    return int(max(-2**31, min(2**31 - 1, t)))


def predicate_flags(values: np.ndarray, t: int) -> np.ndarray:
    """uint8 flags, 1 where values > t (signed compare), else 0."""
    return (values > np.int32(t)).astype(np.uint8)


def brackets(n: int = N_SWEEP, seed: int = 3) -> np.ndarray:
    bits = np.random.default_rng(seed).integers(0, 2, n, dtype=np.int32)
    return (2 * bits - 1).astype(np.int32)


def radix_keys(n: int = N_SORT, seed: int = 4) -> np.ndarray:
    return full_range_u32(n, seed)


def max_values(n: int = N_SWEEP, seed: int = 5) -> np.ndarray:
    return full_range_i32(n, seed)


def xor_values(n: int = N_SWEEP, seed: int = 6) -> np.ndarray:
    return full_range_u32(n, seed)


def segmented(n: int = N_SWEEP, seed: int = 7, mean_len: int = 1024) -> tuple[np.ndarray, np.ndarray]:
    """(values, heads): int32 digits and uint8 segment heads."""
    rng = np.random.default_rng(seed)
    values = rng.integers(0, 10, n, dtype=np.int32)
    heads = (rng.random(n, dtype=np.float32) < np.float32(1.0 / mean_len)).astype(np.uint8)
    if n:
        heads[0] = 1
    return values, heads


def random_input(dtype, n: int, seed: int, op: str = "add") -> np.ndarray:
    """A test input of any size: small non-negative digits for add (so
    int32 prefix sums stay readable), full-range values for max and xor,
    [0, 1) for fp32."""
    dtype = np.dtype(dtype)
    rng = np.random.default_rng(seed)
    if dtype == np.float32:
        if op == "max":
            return (rng.standard_normal(n, dtype=np.float32) * 1000).astype(np.float32)
        return rng.random(n, dtype=np.float32)
    if op == "add":
        return rng.integers(0, 10, n, dtype=dtype)
    if dtype == np.int32:
        return rng.integers(-2**31, 2**31, n, dtype=np.int32)
    return rng.integers(0, 2**32, n, dtype=np.uint32)
