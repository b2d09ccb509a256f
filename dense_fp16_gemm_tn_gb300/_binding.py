"""ctypes binding to ``libgemm_tn_f16.so`` — argument marshalling only.

Each function has the name and argument order of the C function it calls
(see ``include/gemm_tn_f16.h``).  Pointer arguments accept an integer
address, ``None`` (NULL) or any object with ``data_ptr()`` (a torch tensor);
``stream`` accepts an integer handle, ``None`` (the legacy default stream) or
an object with a ``cuda_stream`` attribute (a torch stream).  All arithmetic
happens in the library's CUDA kernels; there is no fallback: if the library
is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

GEMM_OK = 0
GEMM_ERR_INVALID_VALUE = 1
GEMM_ERR_MISALIGNED = 2
GEMM_ERR_UNSUPPORTED = 3
GEMM_ERR_CUDA = 4
GEMM_ERR_TIMEOUT = 5
GEMM_ERR_WORKSPACE = 6
GEMM_ERR_BOUNDS = 7

GEMM_TN_OPT_WAIT_TIMEOUT_NS = 1
GEMM_TN_OPT_SKIP_FIRST_LOAD = 2
GEMM_TN_OPT_FORCE_BN = 3
GEMM_TN_OPT_FORCE_PAIR = 4
GEMM_TN_OPT_FORCE_SPLITS = 5
GEMM_TN_OPT_FORCE_SWAP = 6
GEMM_TN_OPT_FORCE_GENERIC_EPI = 7
GEMM_TN_OPT_FORCE_PACK = 8
GEMM_TN_OPT_STREAM_K = 9
GEMM_TN_OPT_GROUP_M = 10
GEMM_TN_OPT_SERPENTINE = 11
GEMM_TN_OPT_ROW_LOADER = 12
GEMM_TN_OPT_CHECK_TRIM_D = 13
GEMM_TN_OPT_K_CLUSTER = 14
GEMM_TN_OPT_SMALL = 15

EXPORTED = ["gemm_tn_f16", "gemm_tn_f16_batched", "gemm_status_string", "gemm_tn_f16_last_device_error",
            "gemm_tn_f16_last_cuda_error", "gemm_tn_f16_shutdown", "gemm_tn_f16_version", "gemm_tn_f16_plan",
            "gemm_tn_f16_set_option", "gemm_tn_f16_get_option", "gemm_tn_f16_splitk_static", "gemm_f16", "transpose_f32", "transpose_f16", "gemm_f16_acc16",
            "score_softmax_stats_f16", "gemm_tn_f16_host", "gemm_tn_f16_is_checked"]

GEMM_K_MAJOR = 0
GEMM_MN_MAJOR = 1

GEMM_TN_STATIC_SCRATCH_BYTES = 16 * 1024 * 1024


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {gemm_status_string(status)} (status {status})"
        if status == GEMM_ERR_CUDA:
            msg += f", cudaError_t {gemm_tn_f16_last_cuda_error()}"
        super().__init__(msg)


class gemm_tn_plan_t(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32),
                ("cta_pair", ctypes.c_int32), ("swap_ab", ctypes.c_int32), ("splits", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("epi_tma", ctypes.c_int32), ("pack_a", ctypes.c_int32),
                ("pack_b", ctypes.c_int32), ("units", ctypes.c_int64), ("grid", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_int64), ("stream_k", ctypes.c_int32), ("sk_maxc", ctypes.c_int32),
                ("dp_tiles", ctypes.c_int64), ("sk_tiles", ctypes.c_int64), ("stage_cd", ctypes.c_int32),
                ("row_load", ctypes.c_int32), ("k_cluster", ctypes.c_int32), ("reserved", ctypes.c_int32)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


_lock = threading.Lock()
_lib = None


def checked_requested() -> bool:
    """True when GEMM_TN_F16_CHECKED=1: this process loads the checked build (device-side
    bounds checks on the kernels' own loads and stores) instead of the regular library."""
    return os.environ.get("GEMM_TN_F16_CHECKED", "") == "1"


def library_path() -> str:
    return _build.LIB_PATH_CHECKED if checked_requested() else _build.LIB_PATH


def load_library(build_if_missing: bool = True):
    """Load (building first if needed) the shared library.  Raises if it cannot."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        checked = checked_requested()
        path = library_path()
        if not os.path.exists(path) or not _build.up_to_date(checked=checked):
            if not build_if_missing:
                raise RuntimeError(f"{path} is missing; run dense_fp16_gemm_tn_gb300.build.build()")
            _build.build(checked=checked)
        lib = ctypes.CDLL(path)
        vp, i64, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float
        lib.gemm_tn_f16.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, i64, i64, i64, f32, f32, vp]
        lib.gemm_tn_f16.restype = ctypes.c_int
        lib.gemm_tn_f16_batched.argtypes = [vp, i64, i64, vp, i64, i64, vp, i64, i64, vp, i64, i64,
                                            i64, i64, i64, i64, f32, f32, vp]
        lib.gemm_tn_f16_batched.restype = ctypes.c_int
        lib.gemm_status_string.argtypes = [ctypes.c_int]
        lib.gemm_status_string.restype = ctypes.c_char_p
        lib.gemm_tn_f16_last_device_error.argtypes = []
        lib.gemm_tn_f16_last_device_error.restype = ctypes.c_int
        lib.gemm_tn_f16_last_cuda_error.argtypes = []
        lib.gemm_tn_f16_last_cuda_error.restype = ctypes.c_int
        lib.gemm_tn_f16_shutdown.argtypes = []
        lib.gemm_tn_f16_shutdown.restype = None
        lib.gemm_tn_f16_version.argtypes = []
        lib.gemm_tn_f16_version.restype = ctypes.c_int
        lib.gemm_tn_f16_is_checked.argtypes = []
        lib.gemm_tn_f16_is_checked.restype = ctypes.c_int
        lib.gemm_tn_f16_plan.argtypes = [i64] * 12 + [f32, ctypes.c_uint32, ctypes.c_int32,
                                                       ctypes.POINTER(gemm_tn_plan_t)]
        lib.gemm_tn_f16_plan.restype = ctypes.c_int
        lib.gemm_tn_f16_set_option.argtypes = [ctypes.c_int32, i64]
        lib.gemm_tn_f16_set_option.restype = ctypes.c_int
        lib.gemm_tn_f16_get_option.argtypes = [ctypes.c_int32]
        lib.gemm_tn_f16_get_option.restype = ctypes.c_int64
        lib.gemm_tn_f16_splitk_static.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, i64, i64, i64, f32, f32,
                                                  ctypes.c_int32, vp]
        lib.gemm_tn_f16_splitk_static.restype = ctypes.c_int
        lib.gemm_f16.argtypes = [ctypes.c_int32, ctypes.c_int32, vp, i64, i64, vp, i64, i64, vp, i64, i64,
                                 vp, i64, i64, i64, i64, i64, i64, f32, f32, vp]
        lib.gemm_f16.restype = ctypes.c_int
        lib.gemm_f16_acc16.argtypes = lib.gemm_f16.argtypes
        lib.gemm_f16_acc16.restype = ctypes.c_int
        lib.score_softmax_stats_f16.argtypes = [vp, i64, i64, vp, i64, i64, vp, vp, i64, i64, i64, i64, f32, vp]
        lib.score_softmax_stats_f16.restype = ctypes.c_int
        lib.gemm_tn_f16_host.argtypes = lib.gemm_tn_f16.argtypes
        lib.gemm_tn_f16_host.restype = ctypes.c_int
        for name in ("transpose_f32", "transpose_f16"):
            getattr(lib, name).argtypes = [vp, i64, vp, i64, i64, i64, vp]
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(x):
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):  # numpy array (host memory)
        return x.ctypes.data
    return int(x)


def _stream(s):
    if s is None:
        return None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    return int(s)


def _check(status, where, check):
    if check and status != GEMM_OK:
        raise GemmError(status, where)
    return status


def gemm_tn_f16(A, lda, B, ldb, C, ldc, D, ldd, M, N, K, alpha, beta, stream=None, *, check=True):
    st = load_library().gemm_tn_f16(_ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, _ptr(D), ldd, M, N, K,
                                    float(alpha), float(beta), _stream(stream))
    return _check(st, "gemm_tn_f16", check)


def gemm_tn_f16_batched(A, lda, strideA, B, ldb, strideB, C, ldc, strideC, D, ldd, strideD,
                        M, N, K, batch, alpha, beta, stream=None, *, check=True):
    st = load_library().gemm_tn_f16_batched(_ptr(A), lda, strideA, _ptr(B), ldb, strideB, _ptr(C), ldc, strideC,
                                            _ptr(D), ldd, strideD, M, N, K, batch, float(alpha), float(beta),
                                            _stream(stream))
    return _check(st, "gemm_tn_f16_batched", check)


def gemm_f16(a_major, b_major, A, lda, strideA, B, ldb, strideB, C, ldc, strideC, D, ldd, strideD,
             M, N, K, batch, alpha, beta, stream=None, *, check=True):
    st = load_library().gemm_f16(int(a_major), int(b_major), _ptr(A), lda, strideA, _ptr(B), ldb, strideB,
                                 _ptr(C), ldc, strideC, _ptr(D), ldd, strideD, M, N, K, batch,
                                 float(alpha), float(beta), _stream(stream))
    return _check(st, "gemm_f16", check)


def gemm_f16_acc16(a_major, b_major, A, lda, strideA, B, ldb, strideB, C, ldc, strideC, D, ldd, strideD,
                   M, N, K, batch, alpha, beta, stream=None, *, check=True):
    st = load_library().gemm_f16_acc16(int(a_major), int(b_major), _ptr(A), lda, strideA, _ptr(B), ldb, strideB,
                                       _ptr(C), ldc, strideC, _ptr(D), ldd, strideD, M, N, K, batch,
                                       float(alpha), float(beta), _stream(stream))
    return _check(st, "gemm_f16_acc16", check)


def gemm_tn_f16_host(A, lda, B, ldb, C, ldc, D, ldd, M, N, K, alpha, beta, stream=None, *, check=True):
    """gemm_tn_f16 on host buffers (numpy arrays or CPU tensors; page-locked memory overlaps
    the copies).  Asynchronous on `stream`: synchronize before reading D."""
    st = load_library().gemm_tn_f16_host(_ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, _ptr(D), ldd, M, N, K,
                                         float(alpha), float(beta), _stream(stream))
    return _check(st, "gemm_tn_f16_host", check)


def score_softmax_stats_f16(Q, ldq, strideQ, K, ldk, strideK, row_max, row_sum, M, N, d, batch, alpha,
                            stream=None, *, check=True):
    """Softmax row statistics of S = alpha * Q K^T (fp32 row_max, row_sum); S is never stored."""
    st = load_library().score_softmax_stats_f16(_ptr(Q), ldq, strideQ, _ptr(K), ldk, strideK, _ptr(row_max),
                                                _ptr(row_sum), M, N, d, batch, float(alpha), _stream(stream))
    return _check(st, "score_softmax_stats_f16", check)


def transpose_f32(X, ldx, Y, ldy, rows, cols, stream=None, *, check=True):
    st = load_library().transpose_f32(_ptr(X), ldx, _ptr(Y), ldy, rows, cols, _stream(stream))
    return _check(st, "transpose_f32", check)


def transpose_f16(X, ldx, Y, ldy, rows, cols, stream=None, *, check=True):
    st = load_library().transpose_f16(_ptr(X), ldx, _ptr(Y), ldy, rows, cols, _stream(stream))
    return _check(st, "transpose_f16", check)


def gemm_tn_f16_splitk_static(A, lda, B, ldb, C, ldc, D, ldd, M, N, K, alpha, beta, splits=0, stream=None, *,
                              check=True):
    """Split-K GEMM whose scratch is a fixed array inside the library: allocates nothing."""
    st = load_library().gemm_tn_f16_splitk_static(_ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, _ptr(D), ldd, M, N, K,
                                                  float(alpha), float(beta), int(splits), _stream(stream))
    return _check(st, "gemm_tn_f16_splitk_static", check)


def gemm_status_string(status: int) -> str:
    return load_library().gemm_status_string(int(status)).decode()


def gemm_tn_f16_last_device_error() -> int:
    return load_library().gemm_tn_f16_last_device_error()


def gemm_tn_f16_last_cuda_error() -> int:
    return load_library().gemm_tn_f16_last_cuda_error()


def gemm_tn_f16_shutdown() -> None:
    load_library().gemm_tn_f16_shutdown()


def gemm_tn_f16_version() -> int:
    return load_library().gemm_tn_f16_version()


def gemm_tn_f16_is_checked() -> int:
    return load_library().gemm_tn_f16_is_checked()


def gemm_tn_f16_plan(M, N, K, batch, lda, ldb, ldc, ldd, strideA, strideB, strideC, strideD,
                     beta, align_flags, num_sms):
    plan = gemm_tn_plan_t()
    st = load_library().gemm_tn_f16_plan(M, N, K, batch, lda, ldb, ldc, ldd, strideA, strideB, strideC, strideD,
                                         float(beta), align_flags, num_sms, ctypes.byref(plan))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_tn_f16_plan")
    return plan.as_dict()


def gemm_tn_f16_set_option(option: int, value: int) -> None:
    _check(load_library().gemm_tn_f16_set_option(int(option), int(value)), "gemm_tn_f16_set_option", True)


def gemm_tn_f16_get_option(option: int) -> int:
    return load_library().gemm_tn_f16_get_option(int(option))
