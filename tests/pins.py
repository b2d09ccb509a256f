"""Checks that pin the CPU oracle to facts outside itself.

Each ``check_*`` function takes an oracle instance (``oracle.Oracle``) and
raises AssertionError when the oracle disagrees with what IEEE 754 binary16
and the mathematics of the TN GEMM fix:

- binary16 decode/encode against numpy's IEEE conversions (a library routine),
  exhaustively, including every rounding tie;
- exact rational brute force on tiny shapes (Python integers, then the
  nearest binary16 found by searching every finite value, ties to even);
- identity and permutation matrices, the all-ones closed form, the transpose
  invariant D(A,B)^T = D(B,A), small-integer exactness against numpy's
  integer matmul, beta == 0 not reading C, leading-dimension padding never
  being read, batched == per-batch;
- softmax row statistics: exact scores from integer matmul with math.fsum of
  math.exp, scipy's logsumexp, equal keys (l = N), the shift invariance of
  softmax, dominant keys whose rivals underflow (l counts them), degenerate
  sizes.

The same checks run against deliberately broken copies of the oracle
(tests/test_oracle_mutants.py) to show that each plausible slip fails at
least one of them.
"""
from __future__ import annotations

from bisect import bisect_left
from fractions import Fraction

import numpy as np

# ---------------------------------------------------------------- helpers

_POS_VALUES = None


def _pos_values():
    """All non-negative finite binary16 values as exact Fractions, indexed by bit pattern."""
    global _POS_VALUES
    if _POS_VALUES is None:
        f = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
        _POS_VALUES = [Fraction(float(v)) for v in f]
    return _POS_VALUES


def exact_rne_half(x: Fraction) -> int:
    """Nearest binary16 to the exact rational x (ties to even), found by search."""
    vals = _pos_values()
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    if a >= Fraction(65520):  # max finite 65504 plus half an ulp (16)
        return sign | 0x7C00
    i = bisect_left(vals, a)
    best = None
    for j in (i - 1, i):
        if 0 <= j < len(vals):
            key = (abs(vals[j] - a), j & 1)
            if best is None or key < best[0]:
                best = (key, j)
    return sign | best[1]


def half_bits(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def bits_to_f64(b) -> np.ndarray:
    return np.asarray(b, dtype=np.uint16).view(np.float16).astype(np.float64)


def same_bits(a, b) -> bool:
    """Bitwise equality, except that +0 and -0 compare equal and NaNs match NaNs."""
    a = np.asarray(a, dtype=np.uint16).ravel()
    b = np.asarray(b, dtype=np.uint16).ravel()
    if a.shape != b.shape:
        return False
    za, zb = (a & 0x7FFF) == 0, (b & 0x7FFF) == 0
    na = ((a & 0x7C00) == 0x7C00) & ((a & 0x3FF) != 0)
    nb = ((b & 0x7C00) == 0x7C00) & ((b & 0x3FF) != 0)
    ok = (a == b) | (za & zb) | (na & nb)
    return bool(ok.all())


def narrow_halves(rng, shape, emin=-8, emax=-1, zero_frac=0.05):
    """Random binary16 values +-(1 + f/1024) * 2^e with e in [emin, emax] (and a few zeros).
    Their products are multiples of 2^(2*emin - 20), so fp64 sums of a few
    dozen of them are exact."""
    n = int(np.prod(shape))
    e = rng.integers(emin, emax + 1, size=n)
    f = rng.integers(0, 1024, size=n)
    s = rng.integers(0, 2, size=n)
    bits = (s << 15) | ((e + 15) << 10) | f
    bits = np.where(rng.random(n) < zero_frac, 0, bits)
    return bits.astype(np.uint16).reshape(shape)


# ---------------------------------------------------------------- binary16 conversions

def check_decode_exhaustive(o):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = h.view(np.float16).astype(np.float64)
    got = np.array([o.half_to_double(int(x)) for x in h])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def check_encode_roundtrip(o):
    for h in range(65536):
        if (h & 0x7C00) == 0x7C00 and (h & 0x3FF):
            continue  # NaN payloads are not preserved (one quiet NaN)
        x = float(np.uint16(h).view(np.float16))
        assert o.double_to_half(x) == h, hex(h)


def check_encode_ties_and_neighbours(o):
    """Every midpoint between adjacent positive finite halves rounds to the even
    one; one fp64 ulp either side rounds to the nearer one."""
    lo = np.arange(0, 0x7BFF, dtype=np.uint16)
    a = lo.view(np.float16).astype(np.float64)
    b = (lo + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    mid = (a + b) / 2  # exact: both have at most 11 significant bits
    for i in range(len(lo)):
        even = int(lo[i]) if (int(lo[i]) & 1) == 0 else int(lo[i]) + 1
        for sgn in (1.0, -1.0):
            sbit = 0 if sgn > 0 else 0x8000
            assert o.double_to_half(sgn * mid[i]) == sbit | even, (hex(int(lo[i])), sgn)
            assert o.double_to_half(sgn * np.nextafter(mid[i], np.inf)) == sbit | (int(lo[i]) + 1)
            assert o.double_to_half(sgn * np.nextafter(mid[i], 0.0)) == sbit | int(lo[i])
    # Against numpy's correctly rounded float64 -> float16 on the same points.
    got = np.array([o.double_to_half(float(x)) for x in mid], dtype=np.uint16)
    assert np.array_equal(got, mid.astype(np.float16).view(np.uint16))


def check_encode_specials(o):
    assert o.double_to_half(65504.0) == 0x7BFF
    assert o.double_to_half(65519.999) == 0x7BFF
    assert o.double_to_half(65520.0) == 0x7C00          # tie at the top goes to "even" = infinity
    assert o.double_to_half(-65520.0) == 0xFC00
    assert o.double_to_half(1e300) == 0x7C00
    assert o.double_to_half(float("inf")) == 0x7C00
    assert o.double_to_half(float("-inf")) == 0xFC00
    n = o.double_to_half(float("nan"))
    assert (n & 0x7C00) == 0x7C00 and (n & 0x3FF)
    assert o.double_to_half(2.0 ** -24) == 0x0001       # smallest subnormal
    assert o.double_to_half(2.0 ** -25) == 0x0000       # tie to even -> zero
    assert o.double_to_half(np.nextafter(2.0 ** -25, 1)) == 0x0001
    assert o.double_to_half(-(2.0 ** -26)) == 0x8000    # negative underflow keeps the sign
    assert o.double_to_half(2.0 ** -14) == 0x0400       # smallest normal
    assert o.double_to_half(2.0 ** -14 - 2.0 ** -25) == 0x0400  # tie 0x3FF/0x400 -> even 0x400
    assert o.double_to_half(1.0 + 2.0 ** -11) == 0x3C00  # tie -> even
    assert o.double_to_half(1.0 + 3 * 2.0 ** -11) == 0x3C02
    assert o.double_to_half(0.0) == 0 and o.double_to_half(-0.0) == 0x8000


def check_encode_random_vs_numpy(o, seed=11, n=60000):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(n) * np.exp2(rng.uniform(-30, 18, n))
    got = np.array([o.double_to_half(float(v)) for v in x], dtype=np.uint16)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


# ---------------------------------------------------------------- GEMM definition

def check_bruteforce_exact(o, seed=5, cases=40):
    """Tiny shapes: the oracle equals RNE(exact rational value) bit for bit."""
    rng = np.random.default_rng(seed)
    alphas = [1.0, 0.5, -2.0, 0.25]
    betas = [0.0, 1.5, -0.75, 3.0]
    for t in range(cases):
        M, N = int(rng.integers(1, 8)), int(rng.integers(1, 8))
        K = int(rng.integers(1, 65))
        alpha, beta = alphas[t % 4], betas[(t // 4) % 4]
        A = narrow_halves(rng, (M, K))
        B = narrow_halves(rng, (N, K))
        C = narrow_halves(rng, (M, N))
        D = o.gemm_tn(A, B, C, M, N, K, alpha, beta).reshape(M, N)
        Af = [[Fraction(float(v)) for v in row] for row in bits_to_f64(A)]
        Bf = [[Fraction(float(v)) for v in row] for row in bits_to_f64(B)]
        Cf = [[Fraction(float(v)) for v in row] for row in bits_to_f64(C)]
        for m in range(M):
            for n in range(N):
                s = sum(Af[m][k] * Bf[n][k] for k in range(K))
                x = Fraction(alpha) * s + (Fraction(beta) * Cf[m][n] if beta != 0 else 0)
                want = exact_rne_half(x)
                assert same_bits(D[m, n], want), (t, m, n, hex(int(D[m, n])), hex(want))


def check_identity(o, seed=6):
    rng = np.random.default_rng(seed)
    M = K = 37
    N = 23
    A = half_bits(np.eye(M))
    B = half_bits(rng.uniform(-1, 1, (N, K)))
    for alpha in (1.0, 2.0, -0.5):
        D = o.gemm_tn(A, B, None, M, N, K, alpha, 0.0).reshape(M, N)
        want = half_bits(alpha * bits_to_f64(B).T)  # scaling by a power of two is exact
        assert np.array_equal(D, want)


def check_permutation(o, seed=7):
    rng = np.random.default_rng(seed)
    M = K = 29
    N = 41
    p = rng.permutation(M)
    P = np.zeros((M, K))
    P[np.arange(M), p] = 1.0
    A = half_bits(P)
    B = half_bits(rng.uniform(-1, 1, (N, K)))
    D = o.gemm_tn(A, B, None, M, N, K, 1.0, 0.0).reshape(M, N)
    assert np.array_equal(D, np.ascontiguousarray(B.T[p, :]))


def check_all_ones(o):
    """A = B = C = 1: every entry is RNE(alpha*K + beta)."""
    for (M, N, K, alpha, beta) in [(5, 7, 2047, 0.5, 1.5), (3, 4, 4096, 1.0, 0.0),
                                   (2, 3, 2049, 1.0, 0.0), (4, 4, 3, -1.0, 0.25),
                                   (3, 2, 0, 1.0, 2.0), (2, 2, 70000, 1.0, 0.0)]:
        one = 0x3C00
        A = np.full((M, max(K, 1)), one, dtype=np.uint16)
        B = np.full((N, max(K, 1)), one, dtype=np.uint16)
        C = np.full((M, N), one, dtype=np.uint16)
        D = o.gemm_tn(A, B, C, M, N, K, alpha, beta, lda=max(K, 1), ldb=max(K, 1)).reshape(M, N)
        want = exact_rne_half(Fraction(alpha) * K + Fraction(beta))
        assert (D == want).all(), (M, N, K, alpha, beta, hex(int(D[0, 0])), hex(want))
    # the ragged workload's value: 0.5*2047 + 1.5 = 1025 exactly; 2049 ties to 2048
    assert exact_rne_half(Fraction(1025)) == half_bits(1025.0)
    assert exact_rne_half(Fraction(2049)) == half_bits(2048.0)


def check_transpose_invariant(o, seed=8):
    rng = np.random.default_rng(seed)
    M, N, K = 19, 33, 77
    A = half_bits(rng.uniform(-1, 1, (M, K)))
    B = half_bits(rng.uniform(-1, 1, (N, K)))
    D1 = o.gemm_tn(A, B, None, M, N, K, 0.75, 0.0).reshape(M, N)
    D2 = o.gemm_tn(B, A, None, N, M, K, 0.75, 0.0).reshape(N, M)
    assert np.array_equal(D1.T, D2)


def check_small_integers(o, seed=9):
    """Entries in {-2..2}, K <= 256: every partial sum is an integer below 2^11,
    so the result is exact; numpy's integer matmul gives it."""
    rng = np.random.default_rng(seed)
    M, N, K = 45, 38, 256
    Ai = rng.integers(-2, 3, (M, K))
    Bi = rng.integers(-2, 3, (N, K))
    Ci = rng.integers(-8, 9, (M, N))
    ref = Ai @ Bi.T
    D = o.gemm_tn(half_bits(Ai), half_bits(Bi), None, M, N, K, 1.0, 0.0).reshape(M, N)
    assert np.array_equal(bits_to_f64(D), ref.astype(np.float64))
    D = o.gemm_tn(half_bits(Ai), half_bits(Bi), half_bits(Ci), M, N, K, 1.0, 1.0).reshape(M, N)
    assert np.array_equal(bits_to_f64(D), (ref + Ci).astype(np.float64))
    D = o.gemm_tn(half_bits(Ai), half_bits(Bi), half_bits(Ci), M, N, K, 2.0, -1.0).reshape(M, N)
    assert np.array_equal(bits_to_f64(D), (2 * ref - Ci).astype(np.float64))


def check_beta_zero_does_not_read_c(o):
    M, N, K = 6, 5, 9
    A = np.full((M, K), 0x3C00, dtype=np.uint16)
    B = np.full((N, K), 0x3C00, dtype=np.uint16)
    C = np.full((M, N), 0x7E00, dtype=np.uint16)  # NaN
    D = o.gemm_tn(A, B, C, M, N, K, 1.0, 0.0).reshape(M, N)
    assert (D == half_bits(9.0)).all()
    D = o.gemm_tn(A, B, C, M, N, K, 1.0, 1.0).reshape(M, N)
    assert ((D & 0x7C00) == 0x7C00).all() and ((D & 0x3FF) != 0).all()  # NaN propagates


def check_leading_dims(o, seed=10):
    """Padding columns (NaN) beyond K / N are never read nor written."""
    rng = np.random.default_rng(seed)
    M, N, K = 13, 11, 21
    lda, ldb, ldc, ldd = 24, 29, 17, 15
    Ai = rng.integers(-2, 3, (M, K))
    Bi = rng.integers(-2, 3, (N, K))
    Ci = rng.integers(-2, 3, (M, N))
    A = np.full((M, lda), 0x7E00, dtype=np.uint16); A[:, :K] = half_bits(Ai)
    B = np.full((N, ldb), 0x7E00, dtype=np.uint16); B[:, :K] = half_bits(Bi)
    C = np.full((M, ldc), 0x7E00, dtype=np.uint16); C[:, :N] = half_bits(Ci)
    D = np.full(M * ldd, 0x1234, dtype=np.uint16)
    o.gemm_tn(A, B, C, M, N, K, 1.0, 1.0, lda=lda, ldb=ldb, ldc=ldc, ldd=ldd, D=D)
    D = D.reshape(M, ldd)
    assert np.array_equal(bits_to_f64(D[:, :N]), (Ai @ Bi.T + Ci).astype(np.float64))
    assert (D[:, N:] == 0x1234).all()


def check_batched(o, seed=12):
    rng = np.random.default_rng(seed)
    batch, M, N, K = 3, 7, 10, 33
    Ai = rng.integers(-2, 3, (batch, M, K))
    Bi = rng.integers(-2, 3, (batch, N, K))
    Ci = rng.integers(-2, 3, (batch, M, N))
    D = o.gemm_tn(half_bits(Ai), half_bits(Bi), half_bits(Ci), M, N, K, 1.0, -1.0, batch=batch)
    want = np.einsum("bmk,bnk->bmn", Ai, Bi) - Ci
    assert np.array_equal(bits_to_f64(D).reshape(batch, M, N), want.astype(np.float64))


def check_entries_match_full(o, seed=13):
    rng = np.random.default_rng(seed)
    batch, M, N, K = 2, 17, 12, 40
    A = half_bits(rng.uniform(-1, 1, (batch, M, K)))
    B = half_bits(rng.uniform(-1, 1, (batch, N, K)))
    C = half_bits(rng.uniform(-1, 1, (batch, M, N)))
    D = o.gemm_tn(A, B, C, M, N, K, 0.5, 1.5, batch=batch).reshape(batch, M, N)
    b = rng.integers(0, batch, 50); m = rng.integers(0, M, 50); n = rng.integers(0, N, 50)
    e = o.gemm_tn_entries(A, B, C, K, 0.5, 1.5, b, m, n, lda=K, ldb=K, ldc=N,
                          strideA=M * K, strideB=N * K, strideC=M * N)
    assert np.array_equal(e, D[b, m, n])


def check_degenerate(o):
    D = np.full(12, 0x1234, dtype=np.uint16)
    A = np.zeros(12, dtype=np.uint16)
    o.gemm_tn(A, A, None, 0, 4, 3, 1.0, 0.0, D=D)
    o.gemm_tn(A, A, None, 4, 0, 3, 1.0, 0.0, D=D, ldd=3)
    assert (D == 0x1234).all()
    C = half_bits(np.arange(6, dtype=np.float64).reshape(2, 3))
    D = o.gemm_tn(np.zeros(1, np.uint16), np.zeros(1, np.uint16), C, 2, 3, 0, 1.0, 0.5, lda=1, ldb=1)
    assert np.array_equal(bits_to_f64(D).reshape(2, 3), 0.5 * np.arange(6).reshape(2, 3))


def check_strided_layouts(o, seed=14):
    """Generic strides: with TN strides it is the TN oracle bit for bit; with A or B
    stored transposed it equals the TN oracle on explicitly transposed copies; small
    integers give numpy's exact integer matmul for every layout."""
    rng = np.random.default_rng(seed)
    M, N, K = 23, 17, 45
    A = half_bits(rng.uniform(-1, 1, (M, K)))
    B = half_bits(rng.uniform(-1, 1, (N, K)))
    C = half_bits(rng.uniform(-1, 1, (M, N)))
    ref = o.gemm_tn(A, B, C, M, N, K, 0.5, 1.5).reshape(M, N)
    got = o.gemm_strided(A, (K, 1), B, (K, 1), C, M, N, K, 0.5, 1.5).reshape(M, N)
    assert np.array_equal(got, ref)
    At = np.ascontiguousarray(A.T)  # stored K x M (M contiguous)
    Bt = np.ascontiguousarray(B.T)  # stored K x N
    for a_store, a_st, b_store, b_st in ((At, (1, M), B, (K, 1)), (A, (K, 1), Bt, (1, N)), (At, (1, M), Bt, (1, N))):
        got = o.gemm_strided(a_store, a_st, b_store, b_st, C, M, N, K, 0.5, 1.5).reshape(M, N)
        assert np.array_equal(got, ref)
    Ai = rng.integers(-2, 3, (M, K)); Bi = rng.integers(-2, 3, (N, K))
    want = (Ai @ Bi.T).astype(np.float64)
    for a_store, a_st in ((half_bits(Ai), (K, 1)), (half_bits(np.ascontiguousarray(Ai.T)), (1, M))):
        for b_store, b_st in ((half_bits(Bi), (K, 1)), (half_bits(np.ascontiguousarray(Bi.T)), (1, N))):
            got = o.gemm_strided(a_store, a_st, b_store, b_st, None, M, N, K, 1.0, 0.0).reshape(M, N)
            assert np.array_equal(bits_to_f64(got), want)


def check_transpose(o, seed=15):
    """y = x^T: equals numpy's transpose element for element, twice is the identity,
    and padding beyond ld is neither read into nor written."""
    rng = np.random.default_rng(seed)
    for dt in (np.uint32, np.uint16):
        rows, cols = 37, 53
        x = rng.integers(0, np.iinfo(dt).max, (rows, cols), dtype=dt)
        y = o.transpose(x, rows, cols).reshape(cols, rows)
        assert np.array_equal(y, x.T)
        assert np.array_equal(o.transpose(y, cols, rows).reshape(rows, cols), x)
        xp = np.full((rows, cols + 5), 7, dtype=dt); xp[:, :cols] = x
        yp = np.full(cols * (rows + 3), 9, dtype=dt)
        o.transpose(xp, rows, cols, ldx=cols + 5, ldy=rows + 3, Y=yp)
        yp = yp.reshape(cols, rows + 3)
        assert np.array_equal(yp[:, :rows], x.T) and (yp[:, rows:] == 9).all()


# ------------------------------------------------- softmax row statistics

def _small_ints(rng, shape, lo=-2, hi=2):
    return rng.integers(lo, hi + 1, shape).astype(np.int64)


def _padded_bits(x_int, ld):
    """Rows of small integers as binary16 bits with NaN (0x7E00) padding up to ld."""
    rows, cols = x_int.shape
    out = np.full((rows, ld), 0x7E00, dtype=np.uint16)
    out[:, :cols] = half_bits(x_int.astype(np.float64))
    return out


def check_softmax_exact_small_int(o, seed=21):
    """Small integers, power-of-two alpha: every score is exact, so m must equal
    alpha * max of numpy's integer matmul exactly, and l the correctly rounded sum
    of exp over those exact scores (math.fsum of math.exp) to fp64 summation error.
    Batched, with NaN-padded leading dimensions that must never be read."""
    import math
    rng = np.random.default_rng(seed)
    batch, M, N, d = 2, 7, 29, 23
    ldq, ldk = d + 3, d + 5
    for alpha in (0.25, -0.5, 2.0):
        Qi = _small_ints(rng, (batch, M, d))
        Ki = _small_ints(rng, (batch, N, d))
        Q = np.concatenate([_padded_bits(Qi[b], ldq).ravel() for b in range(batch)])
        K = np.concatenate([_padded_bits(Ki[b], ldk).ravel() for b in range(batch)])
        m, l = o.score_softmax_stats(Q, K, M, N, d, alpha, ldq=ldq, ldk=ldk, batch=batch)
        for b in range(batch):
            S = Qi[b] @ Ki[b].T  # exact integers
            for i in range(M):
                row = [alpha * float(v) for v in S[i]]
                mref = max(row)
                assert m[b * M + i] == mref, (b, i, m[b * M + i], mref)
                lref = math.fsum(math.exp(v - mref) for v in row)
                assert abs(l[b * M + i] - lref) <= 1e-13 * lref, (b, i, l[b * M + i], lref)


def check_softmax_logsumexp(o, seed=22):
    """N(0,1) fp16 inputs at the head width of the retile_D page (64): m against the
    row maximum of numpy's fp64 matmul and m + log(l) against scipy's logsumexp."""
    from scipy.special import logsumexp
    rng = np.random.default_rng(seed)
    M, N, d, alpha = 6, 333, 64, 0.125
    Q = half_bits(rng.standard_normal((M, d)))
    K = half_bits(rng.standard_normal((N, d)))
    S = alpha * (bits_to_f64(Q).reshape(M, d) @ bits_to_f64(K).reshape(N, d).T)
    m, l = o.score_softmax_stats(Q, K, M, N, d, alpha)
    assert np.allclose(m, S.max(axis=1), rtol=1e-13, atol=1e-13)
    assert np.allclose(m + np.log(l), logsumexp(S, axis=1), rtol=1e-13, atol=1e-13)
    # every term is at most 1 and the largest is 1
    assert (l >= 1.0).all() and (l <= N).all()


def check_softmax_equal_keys(o, seed=23):
    """All keys equal: every score of a row is the same, so l = N exactly and m is
    that score (rows of both signs, so an m started at 0 instead of -inf shows)."""
    rng = np.random.default_rng(seed)
    M, N, d, alpha = 9, 41, 16, 0.5
    Qi = _small_ints(rng, (M, d))
    v = _small_ints(rng, (d,))
    Ki = np.tile(v, (N, 1))
    m, l = o.score_softmax_stats(half_bits(Qi.astype(float)), half_bits(Ki.astype(float)), M, N, d, alpha)
    s = alpha * (Qi @ v).astype(np.float64)
    assert (s < 0).any() and (s > 0).any()
    assert np.array_equal(m, s)
    assert np.array_equal(l, np.full(M, float(N)))


def check_softmax_shift_invariance(o, seed=24):
    """Adding one vector c to every key shifts each row's scores by alpha*q.c:
    m moves by exactly that and l does not change (all exact with small integers)."""
    rng = np.random.default_rng(seed)
    M, N, d, alpha = 8, 37, 19, 0.25
    Qi = _small_ints(rng, (M, d))
    Ki = _small_ints(rng, (N, d))
    c = _small_ints(rng, (d,))
    m0, l0 = o.score_softmax_stats(half_bits(Qi.astype(float)), half_bits(Ki.astype(float)), M, N, d, alpha)
    m1, l1 = o.score_softmax_stats(half_bits(Qi.astype(float)), half_bits((Ki + c).astype(float)), M, N, d, alpha)
    assert np.array_equal(m1, m0 + alpha * (Qi @ c).astype(np.float64))
    assert np.array_equal(l1, l0)


def check_softmax_dominant_keys(o):
    """Keys are +v or -v with q.v = 1024: the -v terms underflow to exactly 0 in
    exp, so l counts the +v keys, wherever they sit (first and last included)."""
    M, N, d = 3, 50, 16
    Q = np.full((M, d), 8.0)
    hot = np.zeros(N, bool)
    hot[[0, 7, 8, 23, N - 1]] = True
    K = np.where(hot[:, None], 8.0, -8.0) * np.ones((N, d))
    m, l = o.score_softmax_stats(half_bits(Q), half_bits(K), M, N, d, 1.0)
    assert np.array_equal(m, np.full(M, 1024.0))
    assert np.array_equal(l, np.full(M, float(hot.sum())))


def check_softmax_degenerate(o):
    """N = 1: l = 1, m = the score.  N = 0: m = -inf, l = 0.  d = 0: all scores 0."""
    Q = half_bits(np.array([[1.0, 2.0, -3.0]]))
    K = half_bits(np.array([[0.5, 0.25, 1.0]]))
    m, l = o.score_softmax_stats(Q, K, 1, 1, 3, 2.0)
    assert m[0] == 2.0 * (0.5 + 0.5 - 3.0) and l[0] == 1.0
    m, l = o.score_softmax_stats(Q, K, 1, 0, 3, 2.0)
    assert m[0] == -np.inf and l[0] == 0.0
    m, l = o.score_softmax_stats(Q, np.zeros(4, np.uint16), 1, 4, 0, 2.0, ldq=3, ldk=1)
    assert m[0] == 0.0 and l[0] == 4.0
    m, l = o.score_softmax_stats(Q, K, 0, 1, 3, 2.0)
    assert m.size == 0 and l.size == 0


SOFTMAX_CHECKS = [check_softmax_exact_small_int, check_softmax_logsumexp, check_softmax_equal_keys,
                  check_softmax_shift_invariance, check_softmax_dominant_keys, check_softmax_degenerate]

GEMM_CHECKS = [check_bruteforce_exact, check_strided_layouts, check_identity, check_permutation, check_all_ones,
               check_transpose_invariant, check_small_integers, check_beta_zero_does_not_read_c,
               check_leading_dims, check_batched, check_entries_match_full, check_degenerate, check_transpose]
CONVERSION_CHECKS = [check_decode_exhaustive, check_encode_specials, check_encode_random_vs_numpy,
                     check_encode_ties_and_neighbours, check_encode_roundtrip]
