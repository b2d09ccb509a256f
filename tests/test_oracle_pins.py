"""The CPU oracle against its pins (no GPU)."""
import pytest

import oracle
import pins

ORACLE = oracle.Oracle()


@pytest.mark.parametrize("check", pins.CONVERSION_CHECKS, ids=lambda f: f.__name__)
def test_conversion_pins(check):
    check(ORACLE)


@pytest.mark.parametrize("check", pins.GEMM_CHECKS, ids=lambda f: f.__name__)
def test_gemm_pins(check):
    check(ORACLE)


def test_threaded_split_matches_single_thread():
    import numpy as np
    rng = np.random.default_rng(3)
    M, N, K = 300, 70, 256
    A = pins.half_bits(rng.uniform(-1, 1, (M, K)))
    B = pins.half_bits(rng.uniform(-1, 1, (N, K)))
    d1 = ORACLE.gemm_tn(A, B, None, M, N, K, 1.0, 0.0, threads=1)
    d8 = ORACLE.gemm_tn(A, B, None, M, N, K, 1.0, 0.0, threads=8)
    assert np.array_equal(d1, d8)
