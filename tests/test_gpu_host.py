"""gemm_tn_f16_host: the GEMM on host buffers (staged and pipelined by the library)
against the oracle, with page-locked and pageable host memory."""
import numpy as np
import pytest

import dense_fp16_gemm_tn_gb300 as G
import oracle
from dense_fp16_gemm_tn_gb300 import inputs
from gpu_util import SENTINEL, assert_close, assert_device_ok, torch

pytestmark = pytest.mark.gpu


def host_case(M, N, K, *, lda=None, ldb=None, ldc=None, ldd=None, alpha=1.0, beta=0.0, pinned=True, seed=0):
    t = torch()
    lda, ldb, ldc, ldd = lda or K, ldb or K, ldc or N, ldd or N
    A = inputs.with_ld(inputs.uniform_half(seed, M, K), lda) if K else np.zeros((M, lda), np.uint16)
    B = inputs.with_ld(inputs.uniform_half(seed + 1, N, K), ldb) if K else np.zeros((N, ldb), np.uint16)
    C = inputs.with_ld(inputs.uniform_half(seed + 2, M, N), ldc) if beta != 0 else None
    D = np.full((M + 2) * ldd, SENTINEL, dtype=np.uint16)  # two guard rows after the matrix

    def host(x):
        if x is None:
            return None
        if not pinned:
            return np.ascontiguousarray(x)
        h = t.empty(x.size, dtype=t.int16).pin_memory()
        h.numpy()[:] = np.ascontiguousarray(x).reshape(-1).view(np.int16)
        return h

    hA, hB, hC = host(A), host(B), host(C)
    hD = host(D)
    G.gemm_tn_f16_host(hA, lda, hB, ldb, hC, ldc, hD, ldd, M, N, K, alpha, beta)
    t.cuda.synchronize()
    assert_device_ok()
    got = (hD.numpy().view(np.uint16) if pinned else hD).reshape(M + 2, ldd)
    ref = oracle.gemm_tn(A, B, C, M, N, K, alpha, beta, lda=lda, ldb=ldb, ldc=ldc, ldd=ldd).reshape(M, ldd)
    assert (got[:M, N:] == SENTINEL).all(), "host D padding written"
    assert (got[M:] == SENTINEL).all(), "host D written past its last row"
    assert_close(got[:M, :N], ref[:, :N], K, what=f"host M={M} N={N} K={K}")


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_gemm_one_block(pinned):
    host_case(300, 264, 130, pinned=pinned)


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_gemm_one_block_with_beta_and_padding(pinned):
    # one row block: copies and GEMM in order on the caller's stream
    host_case(200, 136, 72, lda=80, ldb=75, ldc=140, ldd=139, alpha=-0.5, beta=1.5, pinned=pinned, seed=11)


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_gemm_several_row_blocks_with_beta_and_padding(pinned):
    # 2100 rows -> row blocks of 768: three blocks, the last one ragged
    host_case(2100, 777, 513, lda=520, ldb=515, ldc=780, ldd=790, alpha=0.5, beta=1.5, pinned=pinned, seed=7)


def test_host_gemm_k_zero_and_empty():
    host_case(130, 70, 0, beta=2.0, seed=3)
    t = torch()
    D = np.full(16, SENTINEL, dtype=np.uint16)
    assert G.gemm_tn_f16_host(None, 8, None, 8, None, 8, D, 8, 0, 8, 8, 1.0, 0.0) == G.GEMM_OK
    t.cuda.synchronize()
    assert (D == SENTINEL).all()


def test_host_gemm_matches_device_call_bitwise():
    """The staged call runs the same kernels on the same data: bit-identical to gemm_tn_f16."""
    t = torch()
    M, N, K = 1500, 640, 384
    A = t.randn((M, K)).half()
    B = t.randn((N, K)).half()
    hD = t.empty((M, N), dtype=t.float16).pin_memory()
    G.gemm_tn_f16_host(A.pin_memory(), K, B.pin_memory(), K, None, N, hD, N, M, N, K, 1.0, 0.0)
    dD = t.empty((M, N), dtype=t.float16, device="cuda")
    G.gemm_tn_f16(A.cuda(), K, B.cuda(), K, None, N, dD, N, M, N, K, 1.0, 0.0)
    t.cuda.synchronize()
    assert t.equal(hD, dD.cpu())
