"""The row-word epilogue (plan: epi_tma 0, stage_cd 0 for problems whose D rows TMA cannot
address, at any size): each thread writes its row of D, and reads its row of C, through
the 16-byte-aligned words that cover the row segment, with element stores at the two edges.
Against the oracle element by element with sentinels in D's padding columns and after its
last row, and against the predicated epilogue bit for bit."""
import numpy as np
import pytest

import dense_fp16_gemm_tn_gb300 as G
import oracle
from dense_fp16_gemm_tn_gb300 import inputs
from gpu_util import SENTINEL, assert_close, assert_device_ok, options, run_problem, to_dev, to_host, torch

pytestmark = pytest.mark.gpu

CASES = [
    # name, M, N, K, batch, ldc, ldd, beta, opts
    ("odd_ldd_beta0", 300, 520, 256, 1, 520, 523, 0.0, {}),
    ("odd_ldc_ldd", 257, 391, 200, 1, 393, 397, 1.5, {}),
    ("even_misaligned_ldd", 512, 512, 512, 1, 514, 516, -1.0, {}),
    ("ragged_n", 200, 1000, 96, 1, 1001, 1003, 0.5, {}),
    ("narrow_n", 640, 40, 64, 1, 41, 45, 2.0, {}),
    ("batched", 130, 300, 128, 3, 303, 305, 0.75, {}),
    ("batched_stride8", 128, 600, 136, 3, 601, 605, -0.5, {}),
    ("many_tiles_odd_ld", 1100, 1800, 320, 1, 1801, 1803, 1.5, {}),
    ("stream_k", 700, 700, 1024, 1, 701, 703, 1.0, {"stream_k": 1}),
    ("pair", 768, 768, 1024, 1, 769, 771, -0.5, {"force_pair": 2, "force_bn": 256}),
    ("pair_stream_k", 520, 776, 2048, 1, 777, 779, 1.25, {"force_pair": 2, "force_bn": 256, "stream_k": 1}),
    ("bn128", 300, 264, 130, 1, 265, 267, 1.0, {"force_bn": 128}),
    ("bn256_single", 300, 520, 200, 1, 521, 523, 1.0, {"force_bn": 256, "force_pair": 1}),
]


@pytest.mark.parametrize("name,M,N,K,batch,ldc,ldd,beta,opts", CASES, ids=[c[0] for c in CASES])
def test_row_word_epilogue(name, M, N, K, batch, ldc, ldd, beta, opts):
    with options(**opts):
        p = G.gemm_tn_f16_plan(M, N, K, batch, K, K, ldc, ldd, M * K, N * K, M * ldc, M * ldd, beta, 15, 152)
    assert p["epi_tma"] == 0 and p["stage_cd"] == 0 and p["swap_ab"] == 0
    run_problem(M, N, K, batch=batch, ldc=ldc, ldd=ldd, alpha=0.5, beta=beta, seed=len(name) + 70, opts=opts,
                d_pad_rows=2)


def test_row_word_small_integers_bit_exact():
    run_problem(300, 520, 256, ldc=521, ldd=523, beta=1.0, dist="int", compare="exact", seed=9, d_pad_rows=2)
    run_problem(700, 700, 1024, ldc=701, ldd=703, beta=-1.0, dist="int", compare="exact", seed=10, d_pad_rows=2,
                opts=dict(stream_k=1))


def test_row_word_matches_predicated_epilogue_bitwise():
    t = torch()
    M, N, K, ldc, ldd = 600, 500, 384, 503, 505
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


def test_row_word_in_place_and_misaligned_base():
    """D == C with an odd leading dimension; then a D whose base is 2 bytes past a 16-byte
    boundary, inside a buffer of sentinels."""
    t = torch()
    M, N, K, ld = 500, 517, 256, 517
    A = inputs.uniform_half(31, M, K)
    B = inputs.uniform_half(32, N, K)
    C = inputs.with_ld(inputs.uniform_half(33, M, N), ld)
    ref = oracle.gemm_tn(A, B, C, M, N, K, 0.5, 1.0, ldc=ld, ldd=ld).reshape(M, ld)
    dCD = to_dev(C.reshape(-1))
    G.gemm_tn_f16(to_dev(A), K, to_dev(B), K, dCD, ld, dCD, ld, M, N, K, 0.5, 1.0)
    t.cuda.synchronize()
    assert_device_ok()
    got = to_host(dCD).reshape(M, ld)
    assert_close(got[:, :N], ref[:, :N], K, what="in place")
    M2, N2, ld2 = 600, 640, 640
    buf = t.full((M2 * ld2 + 16,), 0, dtype=t.int16, device="cuda")
    buf.fill_(np.int16(np.uint16(SENTINEL).view(np.int16)))
    bufh = buf.view(t.float16)
    A2 = inputs.uniform_half(34, M2, K)
    B2 = inputs.uniform_half(35, N2, K)
    plan = G.gemm_tn_f16_plan(M2, N2, K, 1, K, K, N2, ld2, 0, 0, 0, 0, 0.0, 0b0111, 152)
    assert plan["epi_tma"] == 0 and plan["stage_cd"] == 0
    G.gemm_tn_f16(to_dev(A2), K, to_dev(B2), K, None, N2, bufh[1:], ld2, M2, N2, K, 1.0, 0.0)
    t.cuda.synchronize()
    assert_device_ok()
    got = to_host(bufh)
    assert got[0] == SENTINEL and (got[1 + M2 * ld2:] == SENTINEL).all()
    ref2 = oracle.gemm_tn(A2, B2, None, M2, N2, K, 1.0, 0.0, ldd=ld2)
    assert_close(got[1:1 + M2 * ld2], ref2, K, what="misaligned base")


OFFSETS = [0, 1, 3, 7]


@pytest.mark.parametrize("oc", OFFSETS)
@pytest.mark.parametrize("od", OFFSETS)
def test_row_word_base_offsets(oc, od):
    """C and D starting 0, 2, 6 or 14 bytes past a 16-byte boundary, with odd leading
    dimensions, one problem with a stream-K split and one without; sentinels before D,
    in its padding columns and after it."""
    t = torch()
    for M, N, K, ldc, ldd, sk in ((200, 330, 96, 333, 335, 0), (300, 520, 1024, 521, 527, 1)):
        A = inputs.uniform_half(40 + oc, M, K)
        B = inputs.uniform_half(50 + od, N, K)
        C = inputs.with_ld(inputs.uniform_half(60 + oc + od, M, N), ldc).reshape(-1)
        ref = oracle.gemm_tn(A, B, C, M, N, K, 0.75, -1.25, ldc=ldc, ldd=ldd).reshape(M, ldd)
        cbuf = t.zeros((C.size + 8,), dtype=t.int16, device="cuda")
        cbuf[oc:oc + C.size] = t.from_numpy(C.view(np.int16)).cuda()
        dbuf = t.full((M * ldd + 16,), 0, dtype=t.int16, device="cuda")
        dbuf.fill_(np.int16(np.uint16(SENTINEL).view(np.int16)))
        dC = cbuf.view(t.float16)[oc:]
        dD = dbuf.view(t.float16)[od:]
        with options(stream_k=1 if sk else -1):
            p = G.gemm_tn_f16_plan(M, N, K, 1, K, K, ldc, ldd, 0, 0, 0, 0, -1.25, 0b0011, 152)
            G.gemm_tn_f16(to_dev(A), K, to_dev(B), K, dC, ldc, dD, ldd, M, N, K, 0.75, -1.25)
            t.cuda.synchronize()
        assert_device_ok()
        assert p["epi_tma"] == 0 and p["stream_k"] == sk
        got = to_host(dbuf.view(t.float16))
        assert (got[:od] == SENTINEL).all() and (got[od + M * ldd:] == SENTINEL).all(), "store outside D"
        body = got[od:od + M * ldd].reshape(M, ldd)
        assert (body[:, N:] == SENTINEL).all(), "store into D's padding columns"
        assert_close(body[:, :N], ref[:, :N], K, what=f"C offset {oc}, D offset {od}, stream-K {sk}")
