"""Operands whose rows TMA cannot address, rewritten by kernels earlier on the stream:
either repacked, with the GEMM launched as a programmatic dependent of the repack (its
set-up overlaps the repack, and its loads must still see the repacked copies), or read
row by row by the GEMM's own loader warps, which must see the fresh rows.
Several rounds of (overwrite A and B on the device, GEMM) are queued without any
synchronisation in between; every round's D must match the oracle on that round's
operands."""
import numpy as np
import pytest

import dense_fp16_gemm_tn_gb300 as G
import oracle
from dense_fp16_gemm_tn_gb300 import inputs
from gpu_util import assert_close, assert_device_ok, options, to_dev, to_host, torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("opts,row_load", [({}, False), ({"force_pack": 1}, False), ({"force_bn": 512, "force_pair": 2}, False),
                                           ({"stream_k": 1, "force_pack": 1}, False),
                                           ({"force_bn": 128, "force_pair": 1, "row_loader": 1}, True),
                                           ({"force_bn": 256, "force_pair": 2, "row_loader": 1}, True)],
                         ids=["auto", "repack", "wide_repack", "stream_k_repack", "row_loader", "row_loader_pair"])
def test_rounds_of_fresh_operands_through_the_repack(opts, row_load):
    t = torch()
    M, N, K, lda, ldb = 700, 1032, 520, 523, 521  # odd leading dimensions: A and B are repacked
    rounds = 4
    hostA = [inputs.with_ld(inputs.uniform_half(100 + r, M, K), lda) for r in range(rounds)]
    hostB = [inputs.with_ld(inputs.uniform_half(200 + r, N, K), ldb) for r in range(rounds)]
    srcA = [to_dev(a).reshape(-1) for a in hostA]
    srcB = [to_dev(b).reshape(-1) for b in hostB]
    dA = t.empty(M * lda, dtype=t.float16, device="cuda")
    dB = t.empty(N * ldb, dtype=t.float16, device="cuda")
    outs = [t.empty(M * N, dtype=t.float16, device="cuda") for _ in range(rounds)]
    with options(**opts):
        plan = G.gemm_tn_f16_plan(M, N, K, 1, lda, ldb, N, N, 0, 0, 0, 0, 0.0, 15, 152)
        if not row_load:  # repacked copies, the GEMM a programmatic dependent of the repack
            assert plan["pack_a"] == 1 and plan["pack_b"] == 1 and plan["row_load"] == 0
        else:  # the GEMM's loader warps read the freshly written rows themselves
            assert plan["pack_a"] == 0 and plan["pack_b"] == 0 and plan["row_load"] == 3
        t.cuda.synchronize()
        for r in range(rounds):
            dA.copy_(srcA[r])  # a kernel on the stream writes the operands ...
            dB.copy_(srcB[r])
            G.gemm_tn_f16(dA, lda, dB, ldb, None, N, outs[r], N, M, N, K, 1.0, 0.0)  # ... the GEMM reads them
        t.cuda.synchronize()
    assert_device_ok()
    for r in range(rounds):
        ref = oracle.gemm_tn(hostA[r].reshape(-1), hostB[r].reshape(-1), None, M, N, K, 1.0, 0.0, lda=lda, ldb=ldb)
        assert_close(to_host(outs[r]).reshape(M, N), ref.reshape(M, N), K, what=f"round {r}")


def test_wide_tile_with_repacked_operands_and_beta():
    from gpu_util import run_problem
    run_problem(600, 1096, 520, lda=523, ldb=521, alpha=0.5, beta=1.5, seed=31,
                opts=dict(force_bn=512, force_pair=2))
