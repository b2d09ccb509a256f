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


@pytest.mark.parametrize("check", pins.SOFTMAX_CHECKS, ids=lambda f: f.__name__)
def test_softmax_pins(check):
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


def test_softmax_threaded_split_matches_single_thread():
    import numpy as np
    rng = np.random.default_rng(4)
    M, N, d = 500, 300, 64
    Q = pins.half_bits(rng.standard_normal((M, d)))
    K = pins.half_bits(rng.standard_normal((N, d)))
    m1, l1 = ORACLE.score_softmax_stats(Q, K, M, N, d, 0.125, threads=1)
    m8, l8 = ORACLE.score_softmax_stats(Q, K, M, N, d, 0.125, threads=8)
    assert np.array_equal(m1, m8) and np.array_equal(l1, l8)
