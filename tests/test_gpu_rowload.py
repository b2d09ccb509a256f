"""Operands whose rows TMA cannot address (a leading dimension, batch stride or base
that is not a multiple of 16 bytes), read by the GEMM's own loader warps (the
GEMM_TN_OPT_ROW_LOADER option; by default such operands are repacked): each loader
thread fetches the aligned 16-byte words covering its row's 64 halves of a k-block,
shifts them into place, zeroes the halves past K and writes the 128-byte-swizzled
shared-memory image the tensor core reads.  Nothing is repacked and no scratch is taken.
Against the oracle element by element (guard bands around D), on CTA pairs and single
CTAs, with every whole-tile epilogue, K tails, batches, broadcast operands, one operand
misaligned and the other fetched by TMA, serpentine K order, and base pointers at every
2-byte offset in a 16-byte word; small-integer inputs bit for bit, also against the
repacking path."""
import numpy as np
import pytest

import dense_fp16_gemm_tn_gb300 as G
import oracle
from dense_fp16_gemm_tn_gb300 import inputs
from gpu_util import SENTINEL, assert_close, assert_device_ok, options, run_problem, to_dev, to_host, torch

pytestmark = pytest.mark.gpu

CASES = [
    # name, kw for run_problem, expected row_load bits
    ("pair_vec_beta", dict(M=600, N=776, K=520, lda=523, ldb=521, ldc=781, ldd=779, alpha=0.5, beta=1.5,
                           opts=dict(row_loader=1, force_pair=2, force_bn=256)), 3),
    ("pair_tma", dict(M=600, N=776, K=520, lda=523, ldb=521, opts=dict(row_loader=1, force_pair=2, force_bn=256)), 3),
    ("pair_tma_c", dict(M=600, N=776, K=520, lda=523, ldb=521, alpha=-1.0, beta=0.25,
                        opts=dict(row_loader=1, force_pair=2, force_bn=256)), 3),
    ("pair_tma_cg", dict(M=600, N=776, K=520, lda=523, ldb=521, ldc=777, alpha=0.5, beta=1.5,
                         opts=dict(row_loader=1, force_pair=2, force_bn=256)), 3),
    ("single_vec_beta", dict(M=300, N=520, K=200, lda=201, ldb=203, ldc=523, ldd=521, alpha=0.5, beta=1.5,
                             opts=dict(row_loader=1, force_pair=1, force_bn=128)), 3),
    ("single_tma", dict(M=300, N=520, K=200, lda=201, ldb=203, opts=dict(row_loader=1, force_pair=1, force_bn=128)), 3),
    ("single_tma_c", dict(M=300, N=520, K=200, lda=201, ldb=203, beta=-2.0, opts=dict(row_loader=1, force_pair=1, force_bn=128)), 3),
    ("only_a_misaligned", dict(M=600, N=776, K=520, lda=523, opts=dict(row_loader=1, force_pair=2, force_bn=256)), 1),
    ("only_b_misaligned", dict(M=300, N=520, K=200, ldb=203, beta=0.5, opts=dict(row_loader=1, force_pair=1, force_bn=128)), 2),
    ("k1", dict(M=130, N=136, K=1, lda=3, ldb=5, opts=dict(row_loader=1, force_pair=1, force_bn=128)), 3),
    ("k7", dict(M=260, N=264, K=7, lda=9, ldb=7, opts=dict(row_loader=1, force_pair=2, force_bn=256)), 3),
    ("k63", dict(M=130, N=136, K=63, lda=63, ldb=65, opts=dict(row_loader=1, force_pair=1, force_bn=128)), 3),
    ("k65_beta", dict(M=257, N=263, K=65, lda=65, ldb=67, ldc=263, ldd=263, alpha=2.0, beta=0.25,
                      opts=dict(row_loader=1)), 3),
    ("k129_ragged", dict(M=257, N=263, K=129, lda=129, ldb=131, ldc=263, ldd=263, alpha=0.5, beta=1.5,
                         opts=dict(row_loader=1)), 3),
    ("batched", dict(M=200, N=136, K=100, batch=3, lda=103, ldb=101, ldc=140, ldd=139, beta=-1.0,
                     opts=dict(row_loader=1, force_pair=1, force_bn=128)), 3),
    ("batched_pair", dict(M=520, N=520, K=600, batch=2, lda=601, ldb=603, opts=dict(row_loader=1, force_pair=2, force_bn=256)), 3),
    ("broadcast_b", dict(M=130, N=136, K=66, batch=4, lda=67, ldb=69, bcast_b=True,
                         opts=dict(row_loader=1, force_pair=1, force_bn=128)), 3),
    ("many_waves_serpentine", dict(M=3000, N=2900, K=700, lda=701, ldb=703, alpha=0.5, beta=1.5, ldc=2901,
                                   ldd=2903, opts=dict(row_loader=1, serpentine=1, force_pair=2, force_bn=256)), 3),
    ("many_waves_single", dict(M=2600, N=2000, K=330, lda=331, ldb=333, opts=dict(row_loader=1, force_pair=1, force_bn=128)), 3),
]


def _plan(kw):
    M, N, K = kw["M"], kw["N"], kw["K"]
    batch = kw.get("batch", 1)
    lda, ldb = kw.get("lda") or K, kw.get("ldb") or K
    ldc, ldd = kw.get("ldc") or N, kw.get("ldd") or N
    sB = 0 if kw.get("bcast_b") else N * ldb
    with options(**kw.get("opts", {})):
        return G.gemm_tn_f16_plan(M, N, K, batch, lda, ldb, ldc, ldd, M * lda, sB, M * ldc, M * ldd,
                                  kw.get("beta", 0.0), 15, 152)


@pytest.mark.parametrize("name,kw,rl", CASES, ids=[c[0] for c in CASES])
def test_row_loader_parity(name, kw, rl):
    p = _plan(kw)
    assert p["row_load"] == rl and p["pack_a"] == 0 and p["pack_b"] == 0, p
    run_problem(seed=len(name) * 7 + 3, **kw)


@pytest.mark.parametrize("pair", [1, 2])
def test_row_loader_small_integers_bit_exact_and_equal_to_repack(pair):
    kw = dict(M=700, N=1032, K=520, lda=523, ldb=521, dist="int", compare="exact", seed=41)
    bn = 256 if pair == 2 else 128
    got = run_problem(opts=dict(row_loader=1, force_pair=pair, force_bn=bn), **kw)
    packed = run_problem(opts=dict(force_pair=pair, force_bn=bn), **kw)
    assert np.array_equal(got, packed)


@pytest.mark.parametrize("off_a,off_b", [(1, 0), (0, 3), (5, 7), (2, 6), (7, 1)])
def test_row_loader_base_pointer_offsets(off_a, off_b):
    """A and B whose base pointers sit 2*off bytes past a 16-byte boundary (aligned leading
    dimensions): every row is misaligned the same way."""
    t = torch()
    M, N, K = 520, 600, 328
    A = inputs.uniform_half(61 + off_a, M, K)
    B = inputs.uniform_half(71 + off_b, N, K)
    bufA = t.full((M * K + 16,), float("nan"), dtype=t.float16, device="cuda")
    bufB = t.full((N * K + 16,), float("nan"), dtype=t.float16, device="cuda")
    bufA[off_a:off_a + M * K] = to_dev(A).reshape(-1)
    bufB[off_b:off_b + N * K] = to_dev(B).reshape(-1)
    dA, dB = bufA[off_a:], bufB[off_b:]
    D = t.full((M * N + 64,), 0, dtype=t.int16, device="cuda")
    D.fill_(np.int16(np.uint16(SENTINEL).view(np.int16)))
    D = D.view(t.float16)
    align = (1 if off_a == 0 else 0) | (2 if off_b == 0 else 0) | 4 | 8
    with options(row_loader=1):
        p = G.gemm_tn_f16_plan(M, N, K, 1, K, K, N, N, 0, 0, 0, 0, 0.0, align, 152)
        assert p["row_load"] == ((1 if off_a else 0) | (2 if off_b else 0)) and p["pack_a"] == 0 and p["pack_b"] == 0
        G.gemm_tn_f16(dA, K, dB, K, None, N, D, N, M, N, K, 1.0, 0.0)
        t.cuda.synchronize()
    assert_device_ok()
    got = to_host(D)
    assert (got[M * N:] == SENTINEL).all(), "store past the end of D"
    ref = oracle.gemm_tn(A, B, None, M, N, K, 1.0, 0.0)
    assert_close(got[:M * N], ref, K, what=f"offsets {off_a}/{off_b}")
