"""Shapes at the edges of the tile scheduler, against the oracle: a very long K (2048
k-blocks per tile; small-integer inputs keep every fp32 sum exact, so the result must
match bit for bit) on the automatic K-slice plan, stream-K and fixed slices, swapped
small-M problems with long K, many batch entries of tiny matrices, tall matrices with a
handful of columns, and K shorter than one k-block on many tiles."""
import numpy as np
import pytest

import oracle
from dense_fp16_gemm_tn_gb300 import inputs
from gpu_util import assert_close, assert_device_ok, options, run_problem, to_dev, to_host, torch

import dense_fp16_gemm_tn_gb300 as G

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("opts", [{}, {"stream_k": 1}, {"force_splits": 8, "force_pair": 1}],
                         ids=["auto", "stream_k", "split8"])
def test_long_k_small_integers_bit_exact_on_samples(opts):
    t = torch()
    M, N, K = 256, 384, 131072
    A = inputs.small_int_half(3, M, K)
    B = inputs.small_int_half(4, N, K)
    D = t.empty(M * N, dtype=t.float16, device="cuda")
    with options(**opts):
        G.gemm_tn_f16(to_dev(A), K, to_dev(B), K, None, N, D, N, M, N, K, 1.0, 0.0)
        t.cuda.synchronize()
    assert_device_ok()
    got = to_host(D).reshape(M, N)
    rng = np.random.default_rng(5)
    m = np.concatenate([rng.integers(0, M, 1500), [0, 0, M - 1, M - 1]])
    n = np.concatenate([rng.integers(0, N, 1500), [0, N - 1, 0, N - 1]])
    ref = oracle.gemm_tn_entries(A, B, None, K, 1.0, 0.0, np.zeros_like(m), m, n, lda=K, ldb=K)
    assert np.array_equal(got[m, n], ref), "long-K sums are exact: results must match bit for bit"


def test_many_batch_entries_of_tiny_matrices():
    run_problem(64, 72, 64, batch=1024, alpha=0.5, beta=1.0, seed=21)


def test_tall_matrix_with_few_columns():
    run_problem(8192, 16, 1024, alpha=1.0, beta=-0.5, seed=22)
    run_problem(4000, 40, 300, seed=23)


def test_k_shorter_than_one_block_on_many_tiles():
    run_problem(1500, 1800, 8, alpha=2.0, beta=0.5, seed=24)
    run_problem(1024, 1032, 24, seed=25, dist="int", compare="exact")


def test_swapped_long_k_slices():
    """Small M with long K: swapped operands, K slices (the plan's automatic choice)."""
    t = torch()
    M, N, K = 48, 1024, 32768
    plan = G.gemm_tn_f16_plan(M, N, K, 1, K, K, N, N, 0, 0, 0, 0, 0.0, 15, 152)
    assert plan["swap_ab"] == 1 and plan["splits"] > 1
    A = inputs.small_int_half(6, M, K)
    B = inputs.small_int_half(7, N, K)
    D = t.empty(M * N, dtype=t.float16, device="cuda")
    G.gemm_tn_f16(to_dev(A), K, to_dev(B), K, None, N, D, N, M, N, K, 1.0, 0.0)
    t.cuda.synchronize()
    assert_device_ok()
    got = to_host(D).reshape(M, N)
    rng = np.random.default_rng(8)
    m = rng.integers(0, M, 2000)
    n = rng.integers(0, N, 2000)
    ref = oracle.gemm_tn_entries(A, B, None, K, 1.0, 0.0, np.zeros_like(m), m, n, lda=K, ldb=K)
    assert np.array_equal(got[m, n], ref)
    run_problem(24, 1500, 16384, alpha=0.5, beta=1.5, seed=26)


@pytest.mark.parametrize("M,N,K,beta", [(640, 1024, 8192, 0.75), (128, 8192, 8192, -1.25)])
def test_automatic_two_or_three_k_slices_unswapped(M, N, K, beta):
    """Tiles that fill at most half the SMs with 128-255 k-blocks take a few K slices on
    the automatic plan (no forced option); the slices and their sum kernel, with C read
    by the sum, must agree with the oracle element by element."""
    plan = G.gemm_tn_f16_plan(M, N, K, 1, K, K, N, N, 0, 0, 0, 0, beta, 15, 152)
    assert plan["swap_ab"] == 0 and plan["splits"] > 1 and plan["stream_k"] == 0
    run_problem(M, N, K, alpha=0.5, beta=beta, seed=27)
