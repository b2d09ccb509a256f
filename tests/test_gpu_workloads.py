"""The six measured workloads at full size, in the launch configuration the
bench times (the library's automatic plan): every output element against the
oracle.  A sample of outputs (computed one by one) plus the edge rows and
columns is checked first, as a quick pre-check, together with a property that
holds at any size (every output finite); then the whole result is compared with
the full oracle evaluation, a few batch entries at a time."""
import numpy as np
import pytest

import oracle
from dense_fp16_gemm_tn_gb300 import inputs
import dense_fp16_gemm_tn_gb300 as G
from gpu_util import assert_close, assert_close_full, assert_device_ok, to_dev, to_host, torch

pytestmark = pytest.mark.gpu


def _sample_positions(w, rng, n=3000):
    b = rng.integers(0, w.batch, n)
    m = rng.integers(0, w.M, n)
    nn = rng.integers(0, w.N, n)
    # corners and the ragged last row / column of the first and last batch entry
    edge_b, edge_m, edge_n = [], [], []
    for bb in {0, w.batch - 1}:
        for mm in (0, w.M - 1):
            cols = np.unique(np.concatenate([np.arange(min(w.N, 64)), np.arange(max(0, w.N - 64), w.N)]))
            edge_b += [bb] * len(cols); edge_m += [mm] * len(cols); edge_n += list(cols)
        for nn_ in (0, w.N - 1):
            rows = np.unique(np.concatenate([np.arange(min(w.M, 64)), np.arange(max(0, w.M - 64), w.M)]))
            edge_b += [bb] * len(rows); edge_m += list(rows); edge_n += [nn_] * len(rows)
    return (np.concatenate([b, edge_b]).astype(np.int64), np.concatenate([m, edge_m]).astype(np.int64),
            np.concatenate([nn, edge_n]).astype(np.int64))


@pytest.mark.parametrize("key", list(inputs.WORKLOADS))
def test_workload_full_parity(key):
    t = torch()
    w = inputs.WORKLOADS[key]
    A, B, C = w.make()
    sA, sB, sC, sD = w.M * w.lda_, w.N * w.ldb_, w.M * w.ldc_, w.M * w.ldd_
    dA, dB = to_dev(A), to_dev(B)
    dC = to_dev(C) if C is not None else None
    dD = t.empty((w.batch * sD,), dtype=t.float16, device="cuda")
    if w.batch == 1:
        G.gemm_tn_f16(dA, w.lda_, dB, w.ldb_, dC, w.ldc_, dD, w.ldd_, w.M, w.N, w.K, w.alpha, w.beta)
    else:
        G.gemm_tn_f16_batched(dA, w.lda_, sA, dB, w.ldb_, sB, dC, w.ldc_, sC, dD, w.ldd_, sD,
                              w.M, w.N, w.K, w.batch, w.alpha, w.beta)
    t.cuda.synchronize()
    assert_device_ok()
    # property at full size: all outputs finite (inputs are bounded, no overflow possible)
    view = dD.view(w.batch, w.M, w.ldd_)[:, :, : w.N]
    assert bool(t.isfinite(view).all())
    rng = np.random.default_rng(123)
    b, m, n = _sample_positions(w, rng)
    idx = t.from_numpy(b * sD + m * w.ldd_ + n).cuda()
    got = to_host(dD[idx])
    ref = oracle.gemm_tn_entries(A, B, C, w.K, w.alpha, w.beta, b, m, n, lda=w.lda_, ldb=w.ldb_, ldc=w.ldc_,
                                 strideA=sA, strideB=sB, strideC=sC)
    assert_close(got, ref, w.K, what=key)

    # every element: the oracle over a few batch entries at a time (bounded host memory)
    plan = G.gemm_tn_f16_plan(w.M, w.N, w.K, w.batch, w.lda_, w.ldb_, w.ldc_, w.ldd_, sA, sB, sC, sD, w.beta, 15,
                              t.cuda.get_device_properties(0).multi_processor_count)
    per = max(1, (1 << 26) // (w.M * w.ldd_))
    for b0 in range(0, w.batch, per):
        nb = min(per, w.batch - b0)
        got_b = to_host(dD[b0 * sD:(b0 + nb) * sD]).reshape(nb, w.M, w.ldd_)[:, :, : w.N]
        ref_b = oracle.gemm_tn(A[b0:b0 + nb], B[b0:b0 + nb], None if C is None else C[b0:b0 + nb],
                               w.M, w.N, w.K, w.alpha, w.beta, lda=w.lda_, ldb=w.ldb_, ldc=w.ldc_, ldd=w.ldd_,
                               batch=nb, strideA=sA, strideB=sB, strideC=sC, strideD=sD)
        ref_b = ref_b[: nb * sD].reshape(nb, w.M, w.ldd_)[:, :, : w.N]
        assert_close_full(got_b, ref_b, w.K, what=f"{key} batch entries {b0}..{b0 + nb - 1} (plan {plan})")
