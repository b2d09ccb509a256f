"""Helpers for the GPU parity tests: move binary16 bit arrays to and from the
device, run the library through its C ABI, and compare with the oracle under
the stated tolerance |D_gpu - D_ref| <= 2 ulp_fp16(D_ref) + 1e-3 * sqrt(K)."""
from __future__ import annotations

import contextlib
import math

import numpy as np

import dense_fp16_gemm_tn_gb300 as G
import oracle
from dense_fp16_gemm_tn_gb300 import inputs

SENTINEL = 0x5A5A  # value planted around D to catch out-of-bounds stores


def torch():
    import torch as _t
    return _t


def to_dev(bits: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(t.float16).cuda()


def to_host(x) -> np.ndarray:
    t = torch()
    return x.detach().cpu().view(t.int16).numpy().view(np.uint16)


def bits_to_f64(b) -> np.ndarray:
    return np.asarray(b, dtype=np.uint16).view(np.float16).astype(np.float64)


def ulp16(x: np.ndarray) -> np.ndarray:
    """Spacing of binary16 numbers at |x|: 2^(e-10) for |x| in [2^e, 2^(e+1)), e >= -14; else 2^-24."""
    a = np.abs(x)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.clip(e, -14, 15)
    u = np.exp2(e - 10)
    return np.where(a < 2.0 ** -14, 2.0 ** -24, u)


def tolerance(ref_f64: np.ndarray, K: int) -> np.ndarray:
    return 2.0 * ulp16(ref_f64) + 1e-3 * math.sqrt(max(K, 0))


def assert_close(got_bits, ref_bits, K, what=""):
    g = bits_to_f64(got_bits).ravel()
    r = bits_to_f64(ref_bits).ravel()
    nan_r = np.isnan(r)
    assert np.array_equal(np.isnan(g), nan_r), f"{what}: NaN mismatch ({int(np.isnan(g).sum())} vs {int(nan_r.sum())})"
    inf_r = np.isinf(r)
    assert np.array_equal(g[inf_r], r[inf_r]), f"{what}: infinity mismatch"
    fin = ~nan_r & ~inf_r
    err = np.abs(g[fin] - r[fin])
    tol = tolerance(r[fin], K)
    bad = err > tol
    if bad.any():
        i = int(np.argmax(err - tol))
        raise AssertionError(f"{what}: {int(bad.sum())} of {fin.sum()} entries outside tolerance; worst "
                             f"got {g[fin][i]!r} want {r[fin][i]!r} tol {tol[i]:.3g}")


def assert_close_full(got_bits, ref_bits, K, what=""):
    """assert_close for large arrays: entries whose bits already agree pass at once, the
    tolerance is evaluated on the others only."""
    g = np.ascontiguousarray(got_bits).ravel()
    r = np.ascontiguousarray(ref_bits).ravel()
    assert g.shape == r.shape, f"{what}: shape mismatch"
    diff = np.flatnonzero(g != r)
    if diff.size:
        assert_close(g[diff], r[diff], K, what=f"{what} ({diff.size} of {g.size} entries not bit-identical)")


def assert_device_ok():
    st = G.gemm_tn_f16_last_device_error()
    assert st == G.GEMM_OK, G.gemm_status_string(st)


@contextlib.contextmanager
def options(**kw):
    names = {"force_bn": G.GEMM_TN_OPT_FORCE_BN, "force_pair": G.GEMM_TN_OPT_FORCE_PAIR,
             "force_splits": G.GEMM_TN_OPT_FORCE_SPLITS, "force_swap": G.GEMM_TN_OPT_FORCE_SWAP,
             "force_generic": G.GEMM_TN_OPT_FORCE_GENERIC_EPI, "force_pack": G.GEMM_TN_OPT_FORCE_PACK,
             "skip_first_load": G.GEMM_TN_OPT_SKIP_FIRST_LOAD, "timeout_ns": G.GEMM_TN_OPT_WAIT_TIMEOUT_NS,
             "stream_k": G.GEMM_TN_OPT_STREAM_K, "group_m": G.GEMM_TN_OPT_GROUP_M,
             "serpentine": G.GEMM_TN_OPT_SERPENTINE,
             "row_loader": G.GEMM_TN_OPT_ROW_LOADER,
             "k_cluster": G.GEMM_TN_OPT_K_CLUSTER,
             "small": G.GEMM_TN_OPT_SMALL}
    old = {k: G.gemm_tn_f16_get_option(names[k]) for k in kw}
    try:
        for k, v in kw.items():
            G.gemm_tn_f16_set_option(names[k], v)
        yield
    finally:
        for k, v in old.items():
            G.gemm_tn_f16_set_option(names[k], v)


def make_operands(M, N, K, batch, lda, ldb, ldc, beta, seed, dist="uniform", bcast_a=False, bcast_b=False):
    gen = {"uniform": inputs.uniform_half, "normal": inputs.normal_half, "int": inputs.small_int_half}[dist]
    na = 1 if bcast_a else batch
    nb = 1 if bcast_b else batch
    A = np.stack([inputs.with_ld(a, lda) for a in inputs.batched(gen, seed, na, M, max(K, 1))[:, :, :K]]) \
        if K > 0 else np.zeros((na, M, lda), np.uint16)
    B = np.stack([inputs.with_ld(b, ldb) for b in inputs.batched(gen, seed + 1, nb, N, max(K, 1))[:, :, :K]]) \
        if K > 0 else np.zeros((nb, N, ldb), np.uint16)
    C = None
    if beta != 0:
        C = np.stack([inputs.with_ld(c, ldc) for c in inputs.batched(gen, seed + 2, batch, M, N)])
    return A, B, C


def run_problem(M, N, K, *, batch=1, alpha=1.0, beta=0.0, lda=None, ldb=None, ldc=None, ldd=None,
                dist="uniform", seed=0, bcast_a=False, bcast_b=False, opts=None, compare="tol",
                d_pad_rows=3):
    """Run one problem on the GPU and on the oracle and compare; returns the plan used."""
    t = torch()
    lda = lda or max(K, 1)
    ldb = ldb or max(K, 1)
    ldc = ldc or N
    ldd = ldd or N
    A, B, C = make_operands(M, N, K, batch, lda, ldb, ldc, beta, seed, dist, bcast_a, bcast_b)
    sA = 0 if bcast_a else M * lda
    sB = 0 if bcast_b else N * ldb
    sC = M * ldc
    sD = M * ldd
    dA, dB = to_dev(A), to_dev(B)
    dC = to_dev(C) if C is not None else None
    # D with a guard band of sentinel rows after the last entry and sentinel padding columns.
    d_elems = batch * sD + d_pad_rows * ldd
    dD = t.full((d_elems,), 0, dtype=t.int16, device="cuda")
    dD.fill_(np.int16(np.uint16(SENTINEL).view(np.int16)))
    dD = dD.view(t.float16)
    with options(**(opts or {})):
        if batch == 1 and not (bcast_a or bcast_b):
            G.gemm_tn_f16(dA, lda, dB, ldb, dC, ldc, dD, ldd, M, N, K, alpha, beta)
        else:
            G.gemm_tn_f16_batched(dA, lda, sA, dB, ldb, sB, dC, ldc, sC, dD, ldd, sD, M, N, K, batch, alpha, beta)
        t.cuda.synchronize()
        assert_device_ok()
    got = to_host(dD)
    ref = oracle.gemm_tn(A, B, C, M, N, K, alpha, beta, lda=lda, ldb=ldb, ldc=ldc, ldd=ldd, batch=batch,
                         strideA=sA, strideB=sB, strideC=sC, strideD=sD)
    body = got[: batch * sD].reshape(batch, M, ldd)
    refb = ref[: batch * sD].reshape(batch, M, ldd)
    # padding columns and rows after D must still hold the sentinel
    assert (body[:, :, N:] == SENTINEL).all(), "store into D's padding columns"
    assert (got[batch * sD:] == SENTINEL).all(), "store past the end of D"
    if compare == "exact":
        assert np.array_equal(body[:, :, :N], refb[:, :, :N]), "not bit-exact"
    else:
        assert_close(body[:, :, :N], refb[:, :, :N], K, what=f"M={M} N={N} K={K} batch={batch}")
    return got
