"""gemm_f16_acc16 (fp16 accumulation on the tensor core, the smem_gemm page's
F16F16F16F16 atom) against the oracle.

Small integers keep every partial sum an integer below 2048, exactly representable
in fp16, so the result must match bit for bit.  For uniform inputs the bound comes
from the arithmetic: each 16-wide K step may round the running sum once to fp16,
an error of at most one fp16 ulp of the largest partial sum, itself at most
S_abs = sum_k |A_mk B_nk|; so |D - D_ref| <= 2 ulp(D_ref) + |alpha| ceil(K/16) ulp(S_abs)."""
import math

import numpy as np
import pytest

import dense_fp16_gemm_tn_gb300 as G
import oracle
from dense_fp16_gemm_tn_gb300 import inputs
from gpu_util import assert_device_ok, bits_to_f64, options, to_dev, to_host, torch, ulp16

pytestmark = pytest.mark.gpu


def run_acc16(M, N, K, *, alpha=1.0, beta=0.0, dist="uniform", seed=0, opts=None, a_mn=0, b_mn=0):
    t = torch()
    gen = inputs.small_int_half if dist == "int" else inputs.uniform_half
    A = gen(seed, K, M) if a_mn else gen(seed, M, K)
    B = gen(seed + 1, K, N) if b_mn else gen(seed + 1, N, K)
    C = gen(seed + 2, M, N) if beta != 0 else None
    lda, ldb = (M if a_mn else K), (N if b_mn else K)
    D = t.full((M, N), float("nan"), dtype=t.float16, device="cuda")
    with options(**(opts or {})):
        G.gemm_f16_acc16(a_mn, b_mn, to_dev(A), lda, 0, to_dev(B), ldb, 0, to_dev(C) if C is not None else None, N, 0,
                         D, N, 0, M, N, K, 1, alpha, beta)
        t.cuda.synchronize()
        assert_device_ok()
    got = to_host(D).reshape(M, N)
    a_st, b_st = ((1, M) if a_mn else (K, 1)), ((1, N) if b_mn else (K, 1))
    ref = oracle.gemm_strided(A, a_st, B, b_st, C, M, N, K, alpha, beta).reshape(M, N)
    s_abs = oracle.gemm_strided(A & np.uint16(0x7FFF), a_st, B & np.uint16(0x7FFF), b_st, None, M, N, K, 1.0,
                                0.0).reshape(M, N)
    return got, ref, s_abs


CASES = [
    ("tma_single", dict(M=300, N=520, K=256, opts=dict(force_pair=1, force_bn=256))),
    ("tma_pair", dict(M=600, N=776, K=256, opts=dict(force_pair=2, force_bn=256))),
    ("tma_bn128", dict(M=300, N=264, K=192, opts=dict(force_pair=1, force_bn=128))),
    ("generic_beta", dict(M=257, N=263, K=256, alpha=0.5, beta=1.5)),
    ("mn_major", dict(M=300, N=520, K=256, a_mn=1, b_mn=1)),
]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_acc16_small_integers_bit_exact(name, kw):
    got, ref, _ = run_acc16(dist="int", seed=3, **kw)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_acc16_uniform_within_fp16_accumulation_bound(name, kw):
    got, ref, s_abs = run_acc16(dist="uniform", seed=5, **kw)
    g, r, sa = bits_to_f64(got), bits_to_f64(ref), bits_to_f64(s_abs)
    alpha = abs(kw.get("alpha", 1.0))
    K = kw["K"]
    tol = 2 * ulp16(r) + alpha * math.ceil(K / 16) * ulp16(sa * 1.01)
    err = np.abs(g - r)
    assert (err <= tol).all(), f"worst excess {float((err - tol).max())}"
    # and it is a genuinely lower-precision result than the fp32-accumulating path
    assert float(err.max()) > 0.0
