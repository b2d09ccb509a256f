"""Run only under the checked build (GEMM_TN_F16_CHECKED=1, from test_gpu_checked.py):
a range for D trimmed by GEMM_TN_OPT_CHECK_TRIM_D makes the kernels' own stores past
it fail their bounds check.  Each path that writes D itself -- the row-word epilogue,
the predicated epilogue, the swapped epilogue, the split-K sum, the K == 0 scale, the
small-problem kernel's 16-byte and element stores --
must report GEMM_ERR_BOUNDS, leave the bytes past the trimmed range unwritten, and
still write every other element correctly.  Nothing here touches memory outside the
real buffers: the trimmed range is smaller than the allocation."""
import numpy as np
import pytest

import dense_fp16_gemm_tn_gb300 as G
import oracle
from dense_fp16_gemm_tn_gb300 import inputs
from gpu_util import SENTINEL, assert_close, options, to_dev, to_host, torch

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not G.checked_requested(), reason="needs the checked build (GEMM_TN_F16_CHECKED=1)")]

CASES = [
    # name, M, N, K, ldd, opts
    ("row_word_epilogue", 300, 520, 200, 523, {}),
    ("predicated_epilogue", 300, 520, 200, 520, {"force_generic": 1}),
    ("swapped_epilogue", 16, 1000, 300, 1000, {}),
    ("split_k_sum", 200, 136, 1000, 136, {"force_splits": 3, "force_pair": 1}),
    ("k_zero_scale", 130, 136, 0, 139, {}),
    ("small_kernel_vector_stores", 300, 264, 128, 264, {"small": 128}),
    ("small_kernel_element_stores", 300, 263, 128, 265, {"small": 64}),
]


def test_the_checked_build_is_loaded():
    assert G.gemm_tn_f16_is_checked() == 1


@pytest.mark.parametrize("name,M,N,K,ldd,opts", CASES, ids=[c[0] for c in CASES])
def test_trimmed_d_range_is_reported_and_skipped(name, M, N, K, ldd, opts):
    t = torch()
    trim = 6  # bytes: the last three elements of D fall outside the declared range
    A = inputs.uniform_half(81, M, max(K, 1))[:, :K].copy() if K else np.zeros((M, 1), np.uint16)
    B = inputs.uniform_half(82, N, max(K, 1))[:, :K].copy() if K else np.zeros((N, 1), np.uint16)
    beta = 0.5 if K == 0 else 0.0
    C = inputs.uniform_half(83, M, N) if beta else None
    dA, dB = to_dev(np.ascontiguousarray(A)), to_dev(np.ascontiguousarray(B))
    dC = to_dev(C) if C is not None else None
    D = t.full((M * ldd,), 0, dtype=t.int16, device="cuda")
    D.fill_(np.int16(np.uint16(SENTINEL).view(np.int16)))
    D = D.view(t.float16)
    with options(**opts):
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_CHECK_TRIM_D, trim)
        try:
            G.gemm_tn_f16(dA, max(K, 1), dB, max(K, 1), dC, N, D, ldd, M, N, K, 1.0, beta)
            t.cuda.synchronize()
            st = G.gemm_tn_f16_last_device_error()
        finally:
            G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_CHECK_TRIM_D, 0)
    assert st == G.GEMM_ERR_BOUNDS, G.gemm_status_string(st)
    got = to_host(D).reshape(M, ldd)
    # the last row's final three elements were outside the range: not written
    assert (got[M - 1, N - 3:N] == SENTINEL).all()
    ref = oracle.gemm_tn(A, B, C, M, N, K, 1.0, beta, lda=max(K, 1), ldb=max(K, 1), ldd=ldd).reshape(M, ldd)
    # a row-word store is checked (and skipped) as a whole 64-element row segment; element
    # stores one by one: in the last row's last 64 columns an element is either correct
    # or untouched, everywhere else it is correct
    body = got[:, :N].copy()
    tail = body[M - 1, max(0, N - 64):]
    untouched = tail == SENTINEL
    tail[untouched] = ref[M - 1, max(0, N - 64):N][untouched]
    assert_close(body, ref[:, :N], K, what=name)
    # the library keeps working afterwards
    G.gemm_tn_f16(dA, max(K, 1), dB, max(K, 1), dC, N, D, ldd, M, N, K, 1.0, beta)
    t.cuda.synchronize()
    assert G.gemm_tn_f16_last_device_error() == G.GEMM_OK
    assert_close(to_host(D).reshape(M, ldd)[:, :N], ref[:, :N], K, what=name + " after")
