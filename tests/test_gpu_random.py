"""Seeded random problems across the planner's decisions (tile shapes, CTA pairs,
operand swap, stream-K, repacked operands, C / D of any alignment, batches,
broadcast operands, operand majors), each against the oracle element by element."""
import numpy as np
import pytest

import dense_fp16_gemm_tn_gb300 as G
import oracle
from dense_fp16_gemm_tn_gb300 import inputs
from gpu_util import SENTINEL, assert_close, assert_device_ok, run_problem, to_dev, to_host, torch

pytestmark = pytest.mark.gpu


def _draw(rng):
    M = int(rng.choice([1, 7, 16, 48, 100, 255, 256, 300, 640, 1024, 1100, 1500]))
    N = int(rng.choice([8, 16, 33, 128, 257, 512, 777, 1000, 1030, 1500]))
    K = int(rng.choice([1, 15, 64, 100, 256, 513, 1024, 2047]))
    batch = int(rng.choice([1, 1, 1, 2, 3]))
    pad = lambda: int(rng.choice([0, 0, 1, 3, 8]))
    return dict(M=M, N=N, K=K, batch=batch, lda=K + pad(), ldb=K + pad(), ldc=N + pad(), ldd=N + pad(),
                alpha=float(rng.choice([1.0, 0.5, -1.25])), beta=float(rng.choice([0.0, 0.0, 1.0, -0.5])))


CASES = [_draw(np.random.default_rng(1000 + i)) for i in range(24)]


@pytest.mark.parametrize("case", CASES, ids=[f"r{i}" for i in range(len(CASES))])
def test_random_problem(case):
    work = case["M"] * case["N"] * case["K"] * case["batch"]
    if work > 1.5e9:  # keep the oracle's share of the suite short
        case = dict(case, K=min(case["K"], 256))
    bc = np.random.default_rng(case["M"] * 7 + case["N"]).integers(0, 3) if case["batch"] > 1 else 0
    run_problem(case["M"], case["N"], case["K"], batch=case["batch"], lda=case["lda"], ldb=case["ldb"],
                ldc=case["ldc"], ldd=case["ldd"], alpha=case["alpha"], beta=case["beta"], seed=case["M"] + case["K"],
                bcast_a=bool(bc == 1), bcast_b=bool(bc == 2), d_pad_rows=2)


MAJOR_CASES = [(int(a), int(b), m, n, k) for a, b, m, n, k in
               [(1, 0, 300, 520, 200), (0, 1, 1100, 640, 384), (1, 1, 257, 1030, 129), (1, 1, 1024, 1024, 1024)]]


@pytest.mark.parametrize("a_mn,b_mn,M,N,K", MAJOR_CASES, ids=[f"m{i}" for i in range(len(MAJOR_CASES))])
def test_random_majors_with_misaligned_d(a_mn, b_mn, M, N, K):
    """MN-major operands with an odd leading dimension for D."""
    t = torch()
    lda = (M if a_mn else K) + 8
    ldb = (N if b_mn else K) + 8
    ldd = N + 3
    a_rows, a_len = (K, M) if a_mn else (M, K)
    b_rows, b_len = (K, N) if b_mn else (N, K)
    A = inputs.with_ld(inputs.uniform_half(M + 1, a_rows, a_len), lda)
    B = inputs.with_ld(inputs.uniform_half(N + 2, b_rows, b_len), ldb)
    dD = t.full((M * ldd + 2 * ldd,), 0, dtype=t.int16, device="cuda")
    dD.fill_(np.int16(np.uint16(SENTINEL).view(np.int16)))
    dD = dD.view(t.float16)
    G.gemm_f16(a_mn, b_mn, to_dev(A), lda, 0, to_dev(B), ldb, 0, None, N, 0, dD, ldd, 0, M, N, K, 1, 0.5, 0.0)
    t.cuda.synchronize()
    assert_device_ok()
    got = to_host(dD)
    a_st = (1, lda) if a_mn else (lda, 1)
    b_st = (1, ldb) if b_mn else (ldb, 1)
    ref = oracle.gemm_strided(A, a_st, B, b_st, None, M, N, K, 0.5, 0.0, ldd=ldd).reshape(M, ldd)
    body = got[: M * ldd].reshape(M, ldd)
    assert (body[:, N:] == SENTINEL).all() and (got[M * ldd:] == SENTINEL).all()
    assert_close(body[:, :N], ref[:, :N], K, what=f"majors {a_mn}{b_mn}")
