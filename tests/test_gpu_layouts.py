"""gemm_f16 with MN-major operands (A stored K x M and/or B stored K x N) against the
stride-generic oracle, element by element, through the C ABI."""
import zlib

import numpy as np
import pytest

import dense_fp16_gemm_tn_gb300 as G
import oracle
from dense_fp16_gemm_tn_gb300 import inputs
from gpu_util import SENTINEL, assert_close, assert_device_ok, options, to_dev, to_host, torch

pytestmark = pytest.mark.gpu

LAYOUTS = [(1, 0), (0, 1), (1, 1)]


def run_layout(M, N, K, a_mn, b_mn, *, batch=1, alpha=1.0, beta=0.0, lda=None, ldb=None, ldc=None, ldd=None,
               dist="uniform", seed=0, opts=None, compare="tol"):
    t = torch()
    gen = {"uniform": inputs.uniform_half, "int": inputs.small_int_half}[dist]
    lda = lda or (M if a_mn else K)
    ldb = ldb or (N if b_mn else K)
    ldc = ldc or N
    ldd = ldd or N
    a_rows, a_len = (K, M) if a_mn else (M, K)
    b_rows, b_len = (K, N) if b_mn else (N, K)
    A = np.stack([inputs.with_ld(x, lda) for x in inputs.batched(gen, seed, batch, a_rows, a_len)])
    B = np.stack([inputs.with_ld(x, ldb) for x in inputs.batched(gen, seed + 1, batch, b_rows, b_len)])
    C = None
    if beta != 0:
        C = np.stack([inputs.with_ld(x, ldc) for x in inputs.batched(gen, seed + 2, batch, M, N)])
    sA, sB, sC, sD = a_rows * lda, b_rows * ldb, M * ldc, M * ldd
    dA, dB = to_dev(A), to_dev(B)
    dC = to_dev(C) if C is not None else None
    dD = t.full((batch * sD + 2 * ldd,), 0, dtype=t.int16, device="cuda")
    dD.fill_(np.int16(np.uint16(SENTINEL).view(np.int16)))
    dD = dD.view(t.float16)
    with options(**(opts or {})):
        G.gemm_f16(a_mn, b_mn, dA, lda, sA, dB, ldb, sB, dC, ldc, sC, dD, ldd, sD, M, N, K, batch, alpha, beta)
        t.cuda.synchronize()
        assert_device_ok()
    got = to_host(dD)
    a_st = (1, lda) if a_mn else (lda, 1)
    b_st = (1, ldb) if b_mn else (ldb, 1)
    ref = oracle.gemm_strided(A, a_st, B, b_st, C, M, N, K, alpha, beta, ldc=ldc, ldd=ldd, batch=batch,
                              strideA=sA, strideB=sB, strideC=sC, strideD=sD)
    body = got[: batch * sD].reshape(batch, M, ldd)
    refb = ref[: batch * sD].reshape(batch, M, ldd)
    assert (body[:, :, N:] == SENTINEL).all(), "store into D's padding columns"
    assert (got[batch * sD:] == SENTINEL).all(), "store past the end of D"
    if compare == "exact":
        assert np.array_equal(body[:, :, :N], refb[:, :, :N]), "not bit-exact"
    else:
        assert_close(body[:, :, :N], refb[:, :, :N], K, what=f"a_mn={a_mn} b_mn={b_mn} M={M} N={N} K={K}")


CASES = [
    ("pair256", dict(M=600, N=776, K=520, opts=dict(force_pair=2, force_bn=256))),
    ("pair128", dict(M=600, N=776, K=520, opts=dict(force_pair=2, force_bn=128))),
    ("single256", dict(M=300, N=520, K=200, opts=dict(force_pair=1, force_bn=256))),
    ("single128", dict(M=300, N=264, K=130, opts=dict(force_pair=1, force_bn=128))),
    ("tma_c_beta", dict(M=300, N=520, K=200, alpha=0.5, beta=1.5)),
    ("generic_packed", dict(M=257, N=263, K=129, alpha=0.5, beta=1.5)),
    ("padded_ld", dict(M=200, N=136, K=100, lda=None, ldb=None, ldc=140, ldd=144, beta=-1.0)),
    ("streamk", dict(M=1280, N=1280, K=1024, opts=dict(stream_k=1))),
    ("batched", dict(M=200, N=136, K=72, batch=3, alpha=0.125, beta=1.0)),
    ("k65", dict(M=130, N=136, K=65)),
    ("k7", dict(M=130, N=136, K=7)),
    ("small_m", dict(M=16, N=1000, K=300)),
]


@pytest.mark.parametrize("a_mn,b_mn", LAYOUTS, ids=["MN_K", "K_MN", "MN_MN"])
@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_layout_parity(name, kw, a_mn, b_mn):
    run_layout(a_mn=a_mn, b_mn=b_mn, seed=zlib.crc32(name.encode()) % 1000, **kw)


@pytest.mark.parametrize("a_mn,b_mn", LAYOUTS, ids=["MN_K", "K_MN", "MN_MN"])
def test_layout_small_integers_bit_exact(a_mn, b_mn):
    run_layout(512, 384, 256, a_mn, b_mn, dist="int", compare="exact", opts=dict(force_pair=2, force_bn=256))
    run_layout(200, 136, 200, a_mn, b_mn, beta=1.0, dist="int", compare="exact")


def test_k_major_through_gemm_f16_matches_gemm_tn_f16():
    t = torch()
    M, N, K = 300, 264, 130
    A = t.randn((M, K), device="cuda").half()
    B = t.randn((N, K), device="cuda").half()
    D1 = t.empty((M, N), dtype=t.float16, device="cuda")
    D2 = t.empty((M, N), dtype=t.float16, device="cuda")
    G.gemm_tn_f16(A, K, B, K, None, N, D1, N, M, N, K, 1.0, 0.0)
    G.gemm_f16(G.GEMM_K_MAJOR, G.GEMM_K_MAJOR, A, K, 0, B, K, 0, None, N, 0, D2, N, 0, M, N, K, 1, 1.0, 0.0)
    t.cuda.synchronize()
    assert t.equal(D1, D2)
    assert G.gemm_f16(2, 0, A, K, 0, B, K, 0, None, N, 0, D2, N, 0, M, N, K, 1, 1.0, 0.0, check=False) == \
        G.GEMM_ERR_INVALID_VALUE
