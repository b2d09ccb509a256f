"""score_softmax_stats_f16 (fused score GEMM + scale + online softmax statistics)
against the oracle, row by row, through the C ABI.

Tolerance, derived from the arithmetic of the kernel (fp32 tensor-core
accumulation of the score, base-2 exponent with ex2.approx, fp32 running sums):
  - score: |acc - exact dot| <= E = (d + 1) 2^-23 max_j sum_k |q_ik k_jk|
    (d roundings, truncation allowed), so
    |row_max - m| <= |alpha| E + 2^-22 |m|;
  - each exp term's argument x = t_j - t_max is off by at most
    dx = 2 |sc| E + 5 * 2^-24 T  (sc = alpha log2 e, T = |sc| max_j |acc_ij|),
    its value by ln2 dx + 2^-21 (ex2.approx) relative;
  - the running sum: one rescale per 32-column chunk at most (each 2^-21 +
    2^-23 + ln2 2^-23 T relative) and (chunks + 12) fp32 additions of positive
    terms (2^-24 each), plus the merge of the two partial states (2 * 2^-21).
Rows whose statistics are fixed by structure (equal keys, dominant keys, small
integers) are checked much more tightly."""
import math

import numpy as np
import pytest

import dense_fp16_gemm_tn_gb300 as G
import oracle
from dense_fp16_gemm_tn_gb300 import inputs
from gpu_util import assert_device_ok, bits_to_f64, to_dev, torch

pytestmark = pytest.mark.gpu

LOG2E = 1.4426950408889634
SENT = np.float32(-12345.0)


def _bounds(Qf, Kf, alpha, m_ref):
    """Per-row (tol_m, rel_l) from the derivation in the module docstring."""
    M, d = Qf.shape
    N = Kf.shape[0]
    A = (np.abs(Qf) @ np.abs(Kf).T).max(axis=1)
    E = (d + 1) * 2.0 ** -23 * A
    sc = abs(alpha) * LOG2E
    T = sc * A
    tol_m = abs(alpha) * E + 2.0 ** -22 * np.abs(m_ref) + 1e-30
    dx = 2 * sc * E + 5 * 2.0 ** -24 * T
    chunks = math.ceil(N / 32)
    rel_l = (math.log(2) * dx + 2.0 ** -21 + chunks * (2.0 ** -21 + 2.0 ** -23 + math.log(2) * 2.0 ** -23 * T)
             + (chunks + 12) * 2.0 ** -24 + 2 * 2.0 ** -21)
    return tol_m, rel_l


def _operands(M, N, d, batch, ldq, ldk, seed, dist):
    gen = {"normal": inputs.normal_half, "uniform": inputs.uniform_half, "int": inputs.small_int_half}[dist]
    Q = np.stack([inputs.with_ld(x, ldq) for x in inputs.batched(gen, seed, batch, M, d)])
    K = np.stack([inputs.with_ld(x, ldk) for x in inputs.batched(gen, seed + 1, batch, N, d)])
    return Q, K


def run_softmax(Q, K, M, N, d, batch, alpha, ldq, ldk, strideQ, strideK, rows_pad=64):
    """GPU statistics (float32 arrays of batch*M) with sentinel guard entries after them."""
    t = torch()
    dQ, dK = to_dev(Q), to_dev(K)
    n = batch * M
    dm = t.full((n + rows_pad,), float(SENT), dtype=t.float32, device="cuda")
    dl = t.full((n + rows_pad,), float(SENT), dtype=t.float32, device="cuda")
    G.score_softmax_stats_f16(dQ, ldq, strideQ, dK, ldk, strideK, dm, dl, M, N, d, batch, alpha)
    t.cuda.synchronize()
    assert_device_ok()
    m, l = dm.cpu().numpy(), dl.cpu().numpy()
    assert (m[n:] == SENT).all() and (l[n:] == SENT).all(), "store past the last row"
    return m[:n], l[:n]


def check_rows(Q, K, m_gpu, l_gpu, M, N, d, batch, alpha, ldq, ldk, strideQ, strideK, rows=None, what=""):
    """Compare GPU rows (all, or the flattened indices `rows`) with the oracle under the derived bounds."""
    if rows is None:
        m_ref, l_ref = oracle.score_softmax_stats(Q, K, M, N, d, alpha, ldq=ldq, ldk=ldk, batch=batch,
                                                  strideQ=strideQ, strideK=strideK)
        rows = np.arange(batch * M)
    else:
        m_ref = np.empty(len(rows))
        l_ref = np.empty(len(rows))
        for i, r in enumerate(rows):
            mm, ll = oracle.score_softmax_stats(Q, K, M, N, d, alpha, ldq=ldq, ldk=ldk, batch=batch,
                                                strideQ=strideQ, strideK=strideK, rows=(int(r), int(r) + 1))
            m_ref[i], l_ref[i] = mm[r], ll[r]
        m_gpu, l_gpu = m_gpu[rows], l_gpu[rows]
    Qflat = bits_to_f64(Q.ravel())
    Kflat = bits_to_f64(K.ravel())
    tol_m = np.empty(len(rows))
    rel_l = np.empty(len(rows))
    for b in np.unique(rows // M):
        sel = rows // M == b
        i = rows[sel] % M
        qb = Qflat[b * strideQ: b * strideQ + M * ldq].reshape(M, ldq)[i, :d]
        kb = Kflat[b * strideK: b * strideK + N * ldk].reshape(N, ldk)[:, :d]
        tol_m[sel], rel_l[sel] = _bounds(qb, kb, alpha, m_ref[sel])
    em = np.abs(m_gpu.astype(np.float64) - m_ref)
    el = np.abs(l_gpu.astype(np.float64) - l_ref) / l_ref
    assert np.isfinite(m_gpu).all() and np.isfinite(l_gpu).all(), f"{what}: non-finite output"
    bad = em > tol_m
    assert not bad.any(), f"{what}: row_max off in {bad.sum()} rows, worst {em.max():.3g} (tol {tol_m[np.argmax(em)]:.3g})"
    bad = el > rel_l
    assert not bad.any(), f"{what}: row_sum off in {bad.sum()} rows, worst rel {el.max():.3g}"
    return em, el


CASES = [
    # name, M, N, d, batch, alpha, ldq, ldk, dist, broadcast_k
    ("d64_ragged", 300, 700, 64, 3, 0.125, 64, 64, "normal", False),
    ("d32", 130, 300, 32, 2, 0.3, 32, 40, "normal", False),
    ("d128", 200, 513, 128, 2, 0.088, 128, 128, "normal", False),
    ("d200_padded", 129, 257, 200, 2, 0.07, 208, 216, "normal", False),
    ("d256", 256, 1024, 256, 1, 1.0 / 16, 256, 256, "normal", False),
    ("keys_fewer_than_half_tile", 64, 100, 64, 2, 0.125, 64, 64, "normal", False),
    ("one_key", 5, 1, 64, 1, 0.125, 64, 64, "normal", False),
    ("negative_alpha", 200, 600, 64, 2, -0.2, 64, 64, "normal", False),
    ("alpha_zero", 100, 333, 64, 1, 0.0, 64, 64, "normal", False),
    ("rows_not_16B_aligned", 100, 300, 60, 2, 0.125, 62, 61, "uniform", False),
    ("broadcast_keys", 150, 400, 64, 3, 0.125, 64, 64, "normal", True),
    ("persistent_units", 4096, 512, 64, 8, 0.125, 64, 64, "normal", False),
]


@pytest.mark.parametrize("name,M,N,d,batch,alpha,ldq,ldk,dist,bk", CASES, ids=[c[0] for c in CASES])
def test_softmax_parity(name, M, N, d, batch, alpha, ldq, ldk, dist, bk):
    Q, K = _operands(M, N, d, batch, ldq, ldk, seed=len(name) * 7 + M, dist=dist)
    strideQ, strideK = M * ldq, (0 if bk else N * ldk)
    if bk:
        K = K[:1]
    m, l = run_softmax(Q, K, M, N, d, batch, alpha, ldq, ldk, strideQ, strideK)
    em, el = check_rows(Q, K, m, l, M, N, d, batch, alpha, ldq, ldk, strideQ, strideK, what=name)
    # tripwire well inside the worst-case bound: a correct kernel's typical row_sum error is ~1e-6
    assert np.median(el) < 2e-5, f"{name}: median row_sum error {np.median(el):.3g}"


@pytest.mark.parametrize("order", ["increasing", "decreasing"])
def test_softmax_monotone_scores(order):
    """Scores that grow (or shrink) steadily along the keys by about 16 base-2 units
    per 256-key tile: growing ones move the row maximum on every tile, so every
    reference move and rescale is taken; shrinking ones never move it after the
    first tile."""
    from pins import half_bits
    M, N, d = 200, 4096, 64
    rng = np.random.default_rng(9)
    Q = half_bits(0.5 + 0.01 * rng.standard_normal((M, d)))
    ramp = 8.0 * np.arange(N) / N
    if order == "decreasing":
        ramp = ramp[::-1]
    K = half_bits(ramp[:, None] * np.ones((N, d)))
    m, l = run_softmax(Q, K, M, N, d, 1, 1.0, d, d, M * d, N * d)
    check_rows(Q, K, m, l, M, N, d, 1, 1.0, d, d, M * d, N * d, what=order)


def test_softmax_equal_keys_sum_is_the_key_count():
    """All keys equal: every score of a row is the same, so row_sum = N up to the rounding
    of one exp argument per term (no dropped or doubled key passes)."""
    M, N, d, alpha = 200, 700, 64, 0.125
    Q = inputs.normal_half(31, M, d)
    v = inputs.normal_half(32, 1, d)
    K = np.repeat(v, N, axis=0)
    m, l = run_softmax(Q, K, M, N, d, 1, alpha, d, d, M * d, N * d)
    m_ref, _ = oracle.score_softmax_stats(Q, K, M, N, d, alpha)
    assert np.allclose(m, m_ref, rtol=1e-5, atol=1e-5)
    assert np.abs(l / N - 1).max() < 1e-5, np.abs(l / N - 1).max()


def test_softmax_dominant_keys_are_counted():
    """Keys +v or -v with q.v = 1024: the -v terms underflow to 0, so row_sum counts the
    +v keys, including ones in the ragged last tile and in both column halves."""
    M, N, d = 130, 600, 16
    Q = np.full((M, d), 8.0)
    hot = np.zeros(N, bool)
    hot[[0, 31, 32, 127, 128, 255, 256, 300, 511, 512, 599]] = True
    K = np.where(hot[:, None], 8.0, -8.0) * np.ones((N, d))
    from pins import half_bits
    Qb, Kb = half_bits(Q), half_bits(K)
    m, l = run_softmax(Qb, Kb, M, N, d, 1, 1.0, d, d, M * d, N * d)
    assert (m == 1024.0).all()
    assert np.abs(l - hot.sum()).max() < 1e-4, l[:4]


def test_softmax_small_integers_row_max_exact():
    """Small integers with alpha a power of two: every score is exact in fp32, so row_max
    equals the oracle's bit for bit."""
    M, N, d, batch = 200, 520, 64, 2
    Q, K = _operands(M, N, d, batch, d, d, seed=40, dist="int")
    for alpha in (0.25, -0.5):
        m, l = run_softmax(Q, K, M, N, d, batch, alpha, d, d, M * d, N * d)
        m_ref, l_ref = oracle.score_softmax_stats(Q, K, M, N, d, alpha, batch=batch)
        assert np.array_equal(m.astype(np.float64), m_ref)
        assert (np.abs(l / l_ref - 1) < 1e-5).all()


def test_softmax_degenerate_sizes():
    t = torch()
    Q = to_dev(inputs.normal_half(1, 8, 64))
    K = to_dev(inputs.normal_half(2, 8, 64))
    m = t.full((16,), 7.0, dtype=t.float32, device="cuda")
    l = t.full((16,), 7.0, dtype=t.float32, device="cuda")
    G.score_softmax_stats_f16(Q, 64, 0, K, 64, 0, m, l, 8, 0, 64, 1, 0.125)   # no keys
    t.cuda.synchronize()
    assert (m[:8] == -math.inf).all() and (l[:8] == 0).all() and (m[8:] == 7).all()
    G.score_softmax_stats_f16(Q, 64, 0, K, 64, 0, m, l, 8, 5, 0, 2, 0.125)    # d == 0
    t.cuda.synchronize()
    assert (m == 0).all() and (l == 5).all()
    m.fill_(7.0)
    G.score_softmax_stats_f16(Q, 64, 0, K, 64, 0, m, l, 0, 5, 64, 2, 0.125)   # no rows
    t.cuda.synchronize()
    assert (m == 7).all()
    assert_device_ok()


def test_softmax_score_workload_every_row():
    """The batched score workload (8 x 16 heads, Q, K 4096 x 64, N(0,1), alpha 1/8) in one
    call: 384 sampled rows against the oracle first (first and last rows of the first and
    last heads included), then every one of the 524288 rows."""
    w = inputs.WORKLOADS["score_qk"]
    batch, M, N, d = w.batch, w.M, w.N, w.K
    Q, K, _ = w.make()
    m, l = run_softmax(Q, K, M, N, d, batch, w.alpha, d, d, M * d, N * d)
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([rng.integers(0, batch * M, 376),
                                     [0, M - 1, M, (batch - 1) * M, batch * M - 128, batch * M - 1]]))
    check_rows(Q, K, m, l, M, N, d, batch, w.alpha, d, d, M * d, N * d, rows=rows, what="score workload (sample)")
    check_rows(Q, K, m, l, M, N, d, batch, w.alpha, d, d, M * d, N * d, what="score workload (every row)")
