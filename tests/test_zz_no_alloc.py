"""gemm_tn_f16_splitk_static: the split-K GEMM whose scratch is a fixed device
array inside the library, for callers that must not allocate device memory at
call time (an allocator calling from its own internals, or a service whose
memory budget is fixed at start-up).  Its results must agree with the oracle
element by element, and with the regular entry point's, within the parity
tolerance, on two calls in a row that share the array; a second round of the
same calls must leave the device's free memory unchanged.  This file is
collected last on purpose."""
import numpy as np
import pytest

import dense_fp16_gemm_tn_gb300 as G
import oracle
from dense_fp16_gemm_tn_gb300 import inputs
from gpu_util import assert_close, assert_device_ok, to_dev, to_host, torch

pytestmark = pytest.mark.gpu

# (M, N, K, alpha, beta, splits): swapped split-K on the automatic slice count; plain
# split-K with beta and three slices; seven slices whose fp32 partials fill 98 % of the
# array (7 x 512 x 1152 x 4 bytes of 16 MiB).
CASES = [
    (16, 2048, 4096, 1.0, 0.0, 0),
    (200, 136, 1000, 0.5, 1.5, 3),
    (512, 1152, 4096, 1.0, -0.75, 7),
]


def _host_operands(M, N, K, seed, with_c):
    A = inputs.uniform_half(seed, M, K)
    B = inputs.uniform_half(seed + 1, N, K)
    C = inputs.uniform_half(seed + 2, M, N) if with_c else None
    return A, B, C


def _outputs():
    t = torch()
    return [t.full((M, N), float("nan"), dtype=t.float16, device="cuda") for M, N, *_ in CASES]


def _run_static(cases_dev, outs):
    t = torch()
    for (A, B, C), D, (M, N, K, alpha, beta, splits) in zip(cases_dev, outs, CASES):
        G.gemm_tn_f16_splitk_static(A, K, B, K, C, N, D, N, M, N, K, alpha, beta, splits)
    t.cuda.synchronize()
    assert_device_ok()
    return outs


def test_static_scratch_matches_oracle_and_regular_entry_two_calls_in_a_row():
    t = torch()
    assert 7 * 512 * 1152 * 4 <= G.GEMM_TN_STATIC_SCRATCH_BYTES
    host = [_host_operands(M, N, K, 500 + 10 * i, beta != 0) for i, (M, N, K, _, beta, _) in enumerate(CASES)]
    dev = [(to_dev(A), to_dev(B), to_dev(C) if C is not None else None) for A, B, C in host]
    # the calls follow each other on one stream and share the array
    outs = _run_static(dev, _outputs())
    for (A, B, C), (dA, dB, dC), D_static, (M, N, K, alpha, beta, _) in zip(host, dev, outs, CASES):
        got = to_host(D_static)
        ref = oracle.gemm_tn(A, B, C, M, N, K, alpha, beta)
        assert_close(got, ref, K, what=f"static split-K vs oracle M={M} N={N} K={K}")
        D_reg = t.empty((M, N), dtype=t.float16, device="cuda")
        G.gemm_tn_f16(dA, K, dB, K, dC, N, D_reg, N, M, N, K, alpha, beta)
        t.cuda.synchronize()
        assert_device_ok()
        assert_close(got, to_host(D_reg), K, what=f"static split-K vs gemm_tn_f16 M={M} N={N} K={K}")
    # A second round: same results, and no device memory taken (kernels are loaded by now).
    again_bufs = _outputs()
    t.cuda.synchronize()
    free0, _ = t.cuda.mem_get_info()
    again = _run_static(dev, again_bufs)
    free1, _ = t.cuda.mem_get_info()
    assert free1 == free0, f"device free memory moved by {free0 - free1} bytes across allocation-free calls"
    for a, b in zip(outs, again):
        assert np.array_equal(to_host(a), to_host(b)), "the same call must give the same bits"


def test_static_scratch_rejects_oversize_and_unaligned_without_launching():
    t = torch()
    M, N, K = 1024, 1024, 4096
    A = to_dev(inputs.uniform_half(900, M, K))
    B = to_dev(inputs.uniform_half(901, N, K))
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
