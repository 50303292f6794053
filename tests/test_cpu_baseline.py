"""The multithreaded CPU baseline (oracle/mt_baseline.c: the blocked
three-phase scan of geek-doc.cn "并行前缀和 scan ..." section 四 on host
threads, chunks of at least 16 KB per lpnh.cn "并行扫描" section 5.1)
against the serial oracle, bit for bit.  It is a timed baseline only; parity
of the CUDA path is always judged against the serial oracle."""
import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("threads", [1, 2, 3, 8, 64])
def test_mt_baseline_matches_oracle(threads):
    rng = np.random.default_rng(threads)
    for n in (0, 1, 7, 4095, 4096, 4097, 8193, 100_003, (1 << 20) + 5):
        x = rng.integers(-2**31, 2**31, n, dtype=np.int32)   # full range: the sums wrap
        y, used = oracle.mt_scan_exclusive_add(x, threads)
        assert 1 <= used <= threads
        assert used <= max(1, n // 4096)                    # at least 16 KB per thread
        assert np.array_equal(y, oracle.scan(x, "add", False)), (n, threads)


def test_mt_baseline_uses_every_core_on_large_inputs():
    import os
    x = np.ones(1 << 22, dtype=np.int32)
    y, used = oracle.mt_scan_exclusive_add(x)
    assert used == min(os.cpu_count() or 1, 256)
    assert y[-1] == (1 << 22) - 1
