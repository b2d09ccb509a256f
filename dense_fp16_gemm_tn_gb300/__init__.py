"""GB300-native half-precision TN GEMM: D = alpha * A . B^T + beta * C.

The compute path is the C-ABI library ``libgemm_tn_f16.so`` (hand-written
sm_103a kernels: TMA, mbarrier rings, tcgen05 tensor cores with tensor-memory
accumulators).  This package holds its sources (``csrc/``), its build step
(``build``), a ctypes binding with the C function names (``_binding``) and the
seeded input generators (``inputs``).  There is no CPU or library fallback.
"""
from ._binding import (  # noqa: F401
    EXPORTED,
    GEMM_ERR_CUDA,
    GEMM_ERR_INVALID_VALUE,
    GEMM_ERR_MISALIGNED,
    GEMM_ERR_TIMEOUT,
    GEMM_ERR_UNSUPPORTED,
    GEMM_ERR_WORKSPACE,
    GEMM_K_MAJOR,
    GEMM_MN_MAJOR,
    GEMM_OK,
    GEMM_TN_OPT_FORCE_BN,
    GEMM_TN_OPT_FORCE_GENERIC_EPI,
    GEMM_TN_OPT_FORCE_PACK,
    GEMM_TN_OPT_FORCE_PAIR,
    GEMM_TN_OPT_FORCE_SPLITS,
    GEMM_TN_OPT_FORCE_SWAP,
    GEMM_TN_OPT_GROUP_M,
    GEMM_TN_OPT_ROW_LOADER,
    GEMM_TN_OPT_SERPENTINE,
    GEMM_TN_OPT_SKIP_FIRST_LOAD,
    GEMM_TN_OPT_STREAM_K,
    GEMM_TN_OPT_WAIT_TIMEOUT_NS,
    GEMM_TN_STATIC_SCRATCH_BYTES,
    GemmError,
    gemm_f16,
    gemm_f16_acc16,
    gemm_status_string,
    gemm_tn_f16,
    gemm_tn_f16_batched,
    gemm_tn_f16_get_option,
    gemm_tn_f16_host,
    gemm_tn_f16_last_cuda_error,
    gemm_tn_f16_last_device_error,
    gemm_tn_f16_plan,
    gemm_tn_f16_set_option,
    score_softmax_stats_f16,
    gemm_tn_f16_shutdown,
    gemm_tn_f16_splitk_static,
    gemm_tn_f16_version,
    library_path,
    load_library,
    transpose_f16,
    transpose_f32,
)
