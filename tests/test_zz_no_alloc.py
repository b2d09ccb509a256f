"""gemm_tn_f16_splitk_static: the split-K GEMM whose scratch is a fixed device
array inside the library, for callers that must not allocate device memory at
call time (an allocator calling from its own internals, or a service whose
memory budget is fixed at start-up).  Its results must agree with the regular
entry point's, within the parity tolerance, on two calls in a row that share
the array.  This file is collected last on purpose."""
import numpy as np
import pytest

import dense_fp16_gemm_tn_gb300 as G
from dense_fp16_gemm_tn_gb300 import inputs
from gpu_util import assert_close, assert_device_ok, to_dev, to_host, torch

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed, with_c):
    A = to_dev(inputs.uniform_half(seed, M, K))
    B = to_dev(inputs.uniform_half(seed + 1, N, K))
    C = to_dev(inputs.uniform_half(seed + 2, M, N)) if with_c else None
    return A, B, C


def test_static_scratch_matches_regular_entry_two_calls_in_a_row():
    t = torch()
    cases = [  # (M, N, K, alpha, beta, splits): swapped split-K, then plain split-K with beta
        (16, 2048, 4096, 1.0, 0.0, 0),
        (200, 136, 1000, 0.5, 1.5, 3),
    ]
    outs = []
    for i, (M, N, K, alpha, beta, splits) in enumerate(cases):
        A, B, C = _operands(M, N, K, 500 + 10 * i, beta != 0)
        D_static = t.full((M, N), float("nan"), dtype=t.float16, device="cuda")
        G.gemm_tn_f16_splitk_static(A, K, B, K, C, N, D_static, N, M, N, K, alpha, beta, splits)
        outs.append((A, B, C, D_static, M, N, K, alpha, beta))
    t.cuda.synchronize()
    assert_device_ok()
    for A, B, C, D_static, M, N, K, alpha, beta in outs:
        D_reg = t.empty((M, N), dtype=t.float16, device="cuda")
        G.gemm_tn_f16(A, K, B, K, C, N, D_reg, N, M, N, K, alpha, beta)
        t.cuda.synchronize()
        assert_device_ok()
        assert_close(to_host(D_static), to_host(D_reg), K, what=f"static split-K M={M} N={N} K={K}")


def test_static_scratch_rejects_oversize_and_unaligned_without_launching():
    t = torch()
    M, N, K = 1024, 1024, 4096
    A, B, _ = _operands(M, N, K, 900, False)
    D = t.zeros((M, N), dtype=t.float16, device="cuda")
    # 8 slices x 1024 x 1024 x 4 bytes = 32 MiB > the 16 MiB array
    assert 8 * M * N * 4 > G.GEMM_TN_STATIC_SCRATCH_BYTES
    st = G.gemm_tn_f16_splitk_static(A, K, B, K, None, N, D, N, M, N, K, 1.0, 0.0, 8, check=False)
    assert st == G.GEMM_ERR_WORKSPACE
    # an operand whose rows are not 16-byte aligned would need a repacked copy: rejected
    A_odd = t.zeros((64 * 1001,), dtype=t.float16, device="cuda")
    st = G.gemm_tn_f16_splitk_static(A_odd, 1001, B, K, None, N, D, N, 64, N, 1000, 1.0, 0.0, 0, check=False)
    assert st == G.GEMM_ERR_MISALIGNED
    t.cuda.synchronize()
    assert bool((D == 0).all())
