"""CPU oracle for the half-precision TN GEMM — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs
(``cpu_baseline`` and ``--impl reference``) may import this package.  The
product (``dense_fp16_gemm_tn_gb300``) never imports it, and the two share no
code: this package compiles and loads its own plain C file
(``gemm_tn_oracle.c``) and nothing else.

What it computes::

    D[b,m,n] = RNE_fp16(alpha * sum_k A[b,m,k] * B[b,n,k] + beta * C[b,m,n])

and, for the fused score + softmax step, the softmax row statistics of
S = alpha * Q K^T: m[b,i] = max_j S[b,i,j], l[b,i] = sum_j exp(S[b,i,j] - m[b,i]);

in fp64 with one final rounding (see ``gemm_tn_oracle.h`` for the passages of
the pages it follows: the TN inner product and ``axpby`` epilogue of the
``gemm_device`` walk-through, section 3, and the (M,K)/(N,K) stride-(K,1)
operand views of "cute(8) smem_gemm", section "代码实现").

Arrays cross this interface as numpy ``uint16`` arrays holding binary16 bit
patterns, so nothing here depends on a library's half-precision arithmetic.
Large problems are split by output rows over a thread pool; ctypes releases
the GIL for the duration of each C call, so the threads run in parallel.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_tn_oracle.c")
_LIB = os.path.join(_HERE, "libgemm_tn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc.  -ffp-contract=off keeps a*b+c unfused, so
    x86 and Arm hosts give bit-identical results."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "gemm_tn_oracle.h"))
    ):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _bind(path):
    lib = ctypes.CDLL(path)
    i64, u16p, i64p = ctypes.c_int64, ctypes.POINTER(ctypes.c_uint16), ctypes.POINTER(ctypes.c_int64)
    lib.gto_half_to_double.argtypes = [ctypes.c_uint16]
    lib.gto_half_to_double.restype = ctypes.c_double
    lib.gto_double_to_half.argtypes = [ctypes.c_double]
    lib.gto_double_to_half.restype = ctypes.c_uint16
    lib.gto_gemm_tn_f16.argtypes = [u16p, i64, i64, u16p, i64, i64, u16p, i64, i64,
                                    u16p, i64, i64, i64, i64, i64,
                                    ctypes.c_float, ctypes.c_float, i64, i64]
    lib.gto_gemm_tn_f16.restype = None
    lib.gto_gemm_tn_f16_entries.argtypes = [u16p, i64, i64, u16p, i64, i64, u16p, i64, i64,
                                            i64, ctypes.c_float, ctypes.c_float,
                                            i64p, i64p, i64p, i64, u16p]
    lib.gto_gemm_tn_f16_entries.restype = None
    lib.gto_gemm_f16_strided.argtypes = [u16p, i64, i64, i64, u16p, i64, i64, i64, u16p, i64, i64,
                                         u16p, i64, i64, i64, i64, i64,
                                         ctypes.c_float, ctypes.c_float, i64, i64]
    lib.gto_gemm_f16_strided.restype = None
    u32p = ctypes.POINTER(ctypes.c_uint32)
    lib.gto_transpose_u32.argtypes = [u32p, i64, u32p, i64, i64, i64]
    lib.gto_transpose_u32.restype = None
    lib.gto_transpose_u16.argtypes = [u16p, i64, u16p, i64, i64, i64]
    lib.gto_transpose_u16.restype = None
    f64p = ctypes.POINTER(ctypes.c_double)
    lib.gto_score_softmax_stats.argtypes = [u16p, i64, i64, u16p, i64, i64, i64, i64, i64, ctypes.c_float,
                                            f64p, f64p, i64, i64]
    lib.gto_score_softmax_stats.restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(_LIB)
    return _lib


def compile_source(src_path: str, out_path: str) -> str:
    """Compile an oracle source file (same flags as build()) to out_path.
    Used by the pin tests to check that deliberately broken copies of the
    oracle fail the pins."""
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-I", _HERE, "-o", out_path, src_path, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    return out_path


class Oracle:
    """The oracle API bound to one compiled copy of the oracle (the default
    build, or a test's deliberately broken variant)."""

    def __init__(self, lib=None):
        self._lib = lib

    @classmethod
    def from_path(cls, path):
        return cls(_bind(path))

    @property
    def lib(self):
        return self._lib if self._lib is not None else _load()

    def half_to_double(self, h: int) -> float:
        return self.lib.gto_half_to_double(int(h))

    def double_to_half(self, x: float) -> int:
        return int(self.lib.gto_double_to_half(float(x)))

    def gemm_tn(self, *args, **kw):
        return _gemm_tn(self.lib, *args, **kw)

    def gemm_tn_entries(self, *args, **kw):
        return _gemm_tn_entries(self.lib, *args, **kw)

    def gemm_strided(self, *args, **kw):
        return _gemm_strided(self.lib, *args, **kw)

    def transpose(self, *args, **kw):
        return _transpose(self.lib, *args, **kw)

    def score_softmax_stats(self, *args, **kw):
        return _score_softmax_stats(self.lib, *args, **kw)


def _u16ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_uint16)()
    assert a.dtype == np.uint16 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def half_to_double(h: int) -> float:
    return _load().gto_half_to_double(int(h))


def double_to_half(x: float) -> int:
    return int(_load().gto_double_to_half(float(x)))


def gemm_tn(*args, **kw):
    return _gemm_tn(_load(), *args, **kw)


def gemm_tn_entries(*args, **kw):
    return _gemm_tn_entries(_load(), *args, **kw)


def gemm_strided(*args, **kw):
    return _gemm_strided(_load(), *args, **kw)


def transpose(*args, **kw):
    return _transpose(_load(), *args, **kw)


def score_softmax_stats(*args, **kw):
    return _score_softmax_stats(_load(), *args, **kw)


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _gemm_tn(lib, A, B, C, M, N, K, alpha, beta, *, lda=None, ldb=None, ldc=None, ldd=None,
            batch=1, strideA=None, strideB=None, strideC=None, strideD=None,
            D=None, threads=None):
    """Full oracle GEMM.  A, B, C are flat (or any-shape, C-contiguous) uint16
    arrays of binary16 bits laid out with the given leading dimensions and batch
    strides (elements).  Returns D (uint16, flat ``batch*strideD`` elements
    unless ``D`` is supplied)."""
    lda = K if lda is None else lda
    ldb = K if ldb is None else ldb
    ldc = N if ldc is None else ldc
    ldd = N if ldd is None else ldd
    strideA = M * lda if strideA is None else strideA
    strideB = N * ldb if strideB is None else strideB
    strideC = M * ldc if strideC is None else strideC
    strideD = M * ldd if strideD is None else strideD
    if D is None:
        D = np.zeros(max(batch * strideD, 1), dtype=np.uint16)
    rows = batch * M
    if rows == 0 or N == 0:
        return D
    Cp = _u16ptr(C) if beta != 0 else _u16ptr(None)
    args_pre = (_u16ptr(A), lda, strideA, _u16ptr(B), ldb, strideB, Cp, ldc, strideC,
                _u16ptr(D), ldd, strideD, M, N, K, float(alpha), float(beta))
    nthr = default_threads() if threads is None else threads
    work = rows * N * max(K, 1)
    if nthr <= 1 or work < (1 << 22):
        lib.gto_gemm_tn_f16(*args_pre, 0, rows)
        return D
    chunk = max(1, (rows + 4 * nthr - 1) // (4 * nthr))
    spans = [(r, min(rows, r + chunk)) for r in range(0, rows, chunk)]
    with ThreadPoolExecutor(max_workers=nthr) as ex:
        list(ex.map(lambda s: lib.gto_gemm_tn_f16(*args_pre, s[0], s[1]), spans))
    return D


def _gemm_tn_entries(lib, A, B, C, K, alpha, beta, b_idx, m_idx, n_idx, *, lda, ldb, ldc=0,
                    strideA=0, strideB=0, strideC=0, threads=None):
    """Oracle values at chosen output positions (arrays of equal length)."""
    b_idx = np.ascontiguousarray(b_idx, dtype=np.int64)
    m_idx = np.ascontiguousarray(m_idx, dtype=np.int64)
    n_idx = np.ascontiguousarray(n_idx, dtype=np.int64)
    count = len(m_idx)
    out = np.zeros(max(count, 1), dtype=np.uint16)
    i64p = ctypes.POINTER(ctypes.c_int64)
    Cp = _u16ptr(C) if beta != 0 else _u16ptr(None)
    nthr = default_threads() if threads is None else threads

    def run(lo, hi):
        lib.gto_gemm_tn_f16_entries(
            _u16ptr(A), lda, strideA, _u16ptr(B), ldb, strideB, Cp, ldc, strideC,
            K, float(alpha), float(beta),
            b_idx[lo:].ctypes.data_as(i64p), m_idx[lo:].ctypes.data_as(i64p),
            n_idx[lo:].ctypes.data_as(i64p), hi - lo,
            out[lo:].ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)))

    if nthr <= 1 or count * max(K, 1) < (1 << 20):
        run(0, count)
    else:
        chunk = (count + nthr - 1) // nthr
        with ThreadPoolExecutor(max_workers=nthr) as ex:
            list(ex.map(lambda lo: run(lo, min(count, lo + chunk)), range(0, count, chunk)))
    return out[:count]


def _gemm_strided(lib, A, a_strides, B, b_strides, C, M, N, K, alpha, beta, *, ldc=None, ldd=None,
                  batch=1, strideA=0, strideB=0, strideC=None, strideD=None, D=None, threads=None):
    """Oracle GEMM with generic element strides: A(m,k) = A[b*strideA + m*a_strides[0] +
    k*a_strides[1]], B(n,k) likewise; C and D row-major with ldc / ldd."""
    ldc = N if ldc is None else ldc
    ldd = N if ldd is None else ldd
    strideC = M * ldc if strideC is None else strideC
    strideD = M * ldd if strideD is None else strideD
    if D is None:
        D = np.zeros(max(batch * strideD, 1), dtype=np.uint16)
    rows = batch * M
    if rows == 0 or N == 0:
        return D
    Cp = _u16ptr(C) if beta != 0 else _u16ptr(None)
    args_pre = (_u16ptr(A), a_strides[0], a_strides[1], strideA, _u16ptr(B), b_strides[0], b_strides[1], strideB,
                Cp, ldc, strideC, _u16ptr(D), ldd, strideD, M, N, K, float(alpha), float(beta))
    nthr = default_threads() if threads is None else threads
    if nthr <= 1 or rows * N * max(K, 1) < (1 << 22):
        lib.gto_gemm_f16_strided(*args_pre, 0, rows)
        return D
    chunk = max(1, (rows + 4 * nthr - 1) // (4 * nthr))
    spans = [(r, min(rows, r + chunk)) for r in range(0, rows, chunk)]
    with ThreadPoolExecutor(max_workers=nthr) as ex:
        list(ex.map(lambda s: lib.gto_gemm_f16_strided(*args_pre, s[0], s[1]), spans))
    return D


def _transpose(lib, X, rows, cols, *, ldx=None, ldy=None, Y=None):
    """y = x^T for a rows x cols row-major x of uint32 (fp32 bits) or uint16 (fp16 bits).
    Returns Y, a flat array of cols * ldy elements unless Y is supplied."""
    ldx = cols if ldx is None else ldx
    ldy = rows if ldy is None else ldy
    X = np.ascontiguousarray(X)
    if Y is None:
        Y = np.zeros(max(cols * ldy, 1), dtype=X.dtype)
    if X.dtype == np.uint32:
        p = ctypes.POINTER(ctypes.c_uint32)
        lib.gto_transpose_u32(X.ctypes.data_as(p), ldx, Y.ctypes.data_as(p), ldy, rows, cols)
    elif X.dtype == np.uint16:
        lib.gto_transpose_u16(_u16ptr(X), ldx, _u16ptr(Y), ldy, rows, cols)
    else:
        raise TypeError("uint32 or uint16 bit patterns expected")
    return Y


def _score_softmax_stats(lib, Q, Kmat, M, N, d, alpha, *, ldq=None, ldk=None, batch=1, strideQ=None,
                         strideK=None, rows=None, threads=None):
    """Softmax row statistics of S = alpha * Q K^T per batch entry: returns (m, l), two
    float64 arrays indexed r = b*M + i, with m = max_j S[i, j] and l = sum_j exp(S[i, j] - m).
    Q, K are uint16 arrays of binary16 bits (M x d and N x d per batch entry, leading
    dimensions ldq / ldk, batch strides strideQ / strideK).  ``rows`` = (r_begin, r_end)
    restricts the work to those flattened rows (the others stay NaN)."""
    ldq = d if ldq is None else ldq
    ldk = d if ldk is None else ldk
    strideQ = M * ldq if strideQ is None else strideQ
    strideK = N * ldk if strideK is None else strideK
    total = batch * M
    m = np.full(max(total, 1), np.nan)
    l = np.full(max(total, 1), np.nan)
    r0, r1 = (0, total) if rows is None else rows
    if r1 <= r0:
        return m[:total], l[:total]
    f64p = ctypes.POINTER(ctypes.c_double)
    args_pre = (_u16ptr(Q), ldq, strideQ, _u16ptr(Kmat), ldk, strideK, M, N, d, float(alpha),
                m.ctypes.data_as(f64p), l.ctypes.data_as(f64p))
    nthr = default_threads() if threads is None else threads
    if nthr <= 1 or (r1 - r0) * max(N, 1) * max(d, 1) < (1 << 21):
        lib.gto_score_softmax_stats(*args_pre, r0, r1)
        return m[:total], l[:total]
    chunk = max(1, (r1 - r0 + 4 * nthr - 1) // (4 * nthr))
    spans = [(r, min(r1, r + chunk)) for r in range(r0, r1, chunk)]
    with ThreadPoolExecutor(max_workers=nthr) as ex:
        list(ex.map(lambda sp: lib.gto_score_softmax_stats(*args_pre, sp[0], sp[1]), spans))
    return m[:total], l[:total]
