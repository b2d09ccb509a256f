"""Problems whose C or D rows TMA cannot address, at sizes past 2^20 outputs and with
misaligned C beside an aligned D.  C is read where it is by the epilogue's own aligned
loads, shifted into place per row (TMA epilogue, plan epi_tma 1, when D is aligned); a
misaligned D is written in place by the row-word epilogue (epi_tma 0); nothing is staged
(stage_cd 0).  Against the oracle element by element, with guard bands around D, and
against the predicated epilogue bit for bit."""
import numpy as np
import pytest

import dense_fp16_gemm_tn_gb300 as G
import oracle
from dense_fp16_gemm_tn_gb300 import inputs
from gpu_util import SENTINEL, assert_close, assert_device_ok, options, run_problem, to_dev, to_host, torch

pytestmark = pytest.mark.gpu

CASES = [
    # name, M, N, K, batch, ldc, ldd, beta
    ("d_odd_ld_beta0", 1100, 1000, 320, 1, 1000, 1003, 0.0),
    ("cd_odd_ld_beta", 1100, 1000, 320, 1, 1001, 1003, 1.5),
    ("c_odd_ld_only", 1030, 1040, 200, 1, 1043, 1040, -0.5),
    ("d_odd_ld_only_beta", 1030, 1040, 200, 1, 1040, 1047, 2.0),
    ("batched_odd_ld", 600, 900, 256, 3, 905, 907, 0.75),
    ("packed_everything", 1500, 1003, 777, 1, 1003, 1003, 1.5),
]


@pytest.mark.parametrize("name,M,N,K,batch,ldc,ldd,beta", CASES, ids=[c[0] for c in CASES])
def test_large_misaligned_c_d(name, M, N, K, batch, ldc, ldd, beta):
    run_problem(M, N, K, batch=batch, ldc=ldc, ldd=ldd, alpha=0.5, beta=beta, seed=len(name), d_pad_rows=2)


def test_large_misaligned_plan():
    p = G.gemm_tn_f16_plan(1100, 1000, 320, 1, 320, 320, 1001, 1003, 0, 0, 0, 0, 1.5, 15, 152)
    assert p["stage_cd"] == 0 and p["epi_tma"] == 0 and p["workspace_bytes"] == 0


C_CASES = [
    # name, M, N, K, batch, ldc, beta, stream-K expected
    ("small_odd_ldc", 256, 256, 192, 1, 257, 1.0, None),
    ("ragged_n_odd_ldc", 300, 1000, 256, 1, 1001, -0.5, None),
    ("single_stream_k", 1280, 1280, 1024, 1, 1283, 0.75, 1),
    ("pair_stream_k", 2560, 2560, 1024, 1, 2563, -1.5, 1),
    ("batched_odd_stride", 200, 392, 128, 3, 395, 1.25, None),
    ("narrow_n", 520, 72, 96, 1, 75, 2.0, None),
]


@pytest.mark.parametrize("name,M,N,K,batch,ldc,beta,sk", C_CASES, ids=[c[0] for c in C_CASES])
def test_c_read_in_place(name, M, N, K, batch, ldc, beta, sk):
    """Misaligned C with an aligned D: the TMA epilogue reads C itself, nothing is staged
    (the stream-K cases force the split, so that the fix-up path reads C too)."""
    opts = dict(stream_k=1) if sk else {}
    with options(**opts):
        p = G.gemm_tn_f16_plan(M, N, K, batch, K, K, ldc, N, M * K, N * K, M * ldc, M * N, beta, 15, 152)
    assert p["epi_tma"] == 1 and p["stage_cd"] == 0
    if sk is not None:
        assert p["stream_k"] == sk
    run_problem(M, N, K, batch=batch, ldc=ldc, ldd=N, alpha=0.5, beta=beta, seed=len(name) + 40, d_pad_rows=2,
                opts=opts)


def test_c_read_in_place_misaligned_base_every_row_shift():
    """C starts 2 bytes past a 16-byte boundary and its leading dimension is odd, so the
    eight possible shifts occur row after row; the last row ends at the end of C's buffer."""
    t = torch()
    M, N, K, ldc = 1031, 520, 200, 523
    A = inputs.uniform_half(21, M, K)
    B = inputs.uniform_half(22, N, K)
    C = inputs.with_ld(inputs.uniform_half(23, M, N), ldc).reshape(-1)[: (M - 1) * ldc + N]
    ref = oracle.gemm_tn(A, B, C, M, N, K, -0.75, 1.5, ldc=ldc, ldd=N)
    cbuf = t.zeros((C.size + 1,), dtype=t.int16, device="cuda")
    cbuf[1:] = t.from_numpy(C.view(np.int16)).cuda()
    dC = cbuf.view(t.float16)[1:]
    dD = t.full((M * N + 2 * N,), 0, dtype=t.int16, device="cuda")
    dD.fill_(np.int16(np.uint16(SENTINEL).view(np.int16)))
    dD = dD.view(t.float16)
    G.gemm_tn_f16(to_dev(A), K, to_dev(B), K, dC, ldc, dD, N, M, N, K, -0.75, 1.5)
    t.cuda.synchronize()
    assert_device_ok()
    got = to_host(dD)
    assert (got[M * N:] == SENTINEL).all(), "store past the end of D"
    assert_close(got[: M * N], ref, K, what="misaligned C base")


def test_c_read_in_place_small_integers_bit_exact():
    run_problem(1100, 1000, 256, ldc=1001, ldd=1000, beta=-1.0, dist="int", compare="exact", seed=6, d_pad_rows=2)
    run_problem(600, 640, 512, ldc=645, ldd=640, beta=1.0, dist="int", compare="exact", seed=7, d_pad_rows=2,
                opts=dict(stream_k=1))


def test_large_misaligned_small_integers_bit_exact():
    run_problem(1100, 1000, 256, ldc=1001, ldd=1003, beta=1.0, dist="int", compare="exact", seed=5, d_pad_rows=2)


def test_large_misaligned_matches_predicated_epilogue_bitwise():
    """Both epilogues compute alpha*acc + beta*c in fp32 and round once: same bits."""
    t = torch()
    M, N, K, ldc, ldd = 1100, 1000, 384, 1001, 1003
    A = t.randn((M, K), device="cuda").half()
    B = t.randn((N, K), device="cuda").half()
    C = t.randn((M * ldc,), device="cuda").half()
    D1 = t.zeros((M * ldd,), device="cuda", dtype=t.float16)
    D2 = t.zeros((M * ldd,), device="cuda", dtype=t.float16)
    G.gemm_tn_f16(A, K, B, K, C, ldc, D1, ldd, M, N, K, 0.5, 1.5)
    with options(force_generic=1):
        G.gemm_tn_f16(A, K, B, K, C, ldc, D2, ldd, M, N, K, 0.5, 1.5)
    t.cuda.synchronize()
    assert_device_ok()
    assert t.equal(D1, D2)


def test_large_misaligned_in_place_and_misaligned_base():
    """D == C (same odd leading dimension), and a D whose base is 2 bytes off 16."""
    t = torch()
    M, N, K, ld = 1024, 1027, 256, 1027
    A = inputs.uniform_half(11, M, K)
    B = inputs.uniform_half(12, N, K)
    C = inputs.with_ld(inputs.uniform_half(13, M, N), ld)
    ref = oracle.gemm_tn(A, B, C, M, N, K, 0.5, 1.0, ldc=ld, ldd=ld).reshape(M, ld)
    dCD = to_dev(C.reshape(-1))
    G.gemm_tn_f16(to_dev(A), K, to_dev(B), K, dCD, ld, dCD, ld, M, N, K, 0.5, 1.0)
    t.cuda.synchronize()
    assert_device_ok()
    got = to_host(dCD).reshape(M, ld)
    assert_close(got[:, :N], ref[:, :N], K, what="in place")
    # misaligned base: D starts one half into a buffer of sentinels
    M2, N2, ld2 = 1100, 1000, 1000
    buf = t.full((M2 * ld2 + 16,), 0, dtype=t.int16, device="cuda")
    buf.fill_(np.int16(np.uint16(SENTINEL).view(np.int16)))
    bufh = buf.view(t.float16)
    A2 = inputs.uniform_half(14, M2, K)
    B2 = inputs.uniform_half(15, N2, K)
    plan = G.gemm_tn_f16_plan(M2, N2, K, 1, K, K, N2, ld2, 0, 0, 0, 0, 0.0, 0b0111, 152)
    assert plan["stage_cd"] == 0 and plan["epi_tma"] == 0
    G.gemm_tn_f16(to_dev(A2), K, to_dev(B2), K, None, N2, bufh[1:], ld2, M2, N2, K, 1.0, 0.0)
    t.cuda.synchronize()
    assert_device_ok()
    got = to_host(bufh)
    assert got[0] == SENTINEL and (got[1 + M2 * ld2:] == SENTINEL).all()
    ref2 = oracle.gemm_tn(A2, B2, None, M2, N2, K, 1.0, 0.0, ldd=ld2)
    assert_close(got[1:1 + M2 * ld2], ref2, K, what="misaligned base")
