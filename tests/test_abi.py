"""The C-ABI library without a GPU: it loads, exports every function the
header declares, and its host-only logic (argument checks, planning, options)
behaves as documented.  No compute call is made here."""
import ctypes
import os
import re
import subprocess

import pytest

import dense_fp16_gemm_tn_gb300 as G
from dense_fp16_gemm_tn_gb300 import build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "gemm_tn_f16.h")


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"GEMM_TN_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)))


def test_library_builds_and_loads():
    G.load_library()
    assert os.path.exists(G.library_path())


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 10
    lib = ctypes.CDLL(G.library_path())
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(G.EXPORTED)
    out = subprocess.run(["nm", "-D", "--defined-only", G.library_path()], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == set(names), exported ^ set(names)


def test_checked_build_exports_the_same_symbols():
    """The checked build (device-side bounds checks) is the same library: same exports,
    and it says it is the checked one; the regular build says it is not."""
    path = B.build(checked=True)
    assert path == B.LIB_PATH_CHECKED and path != B.LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == set(declared_functions())
    lib = ctypes.CDLL(path)
    lib.gemm_tn_f16_is_checked.restype = ctypes.c_int
    assert lib.gemm_tn_f16_is_checked() == 1
    assert G.gemm_tn_f16_is_checked() == (1 if G.checked_requested() else 0)
    assert G.gemm_status_string(G.GEMM_ERR_BOUNDS).startswith("device-side bounds check")


def test_built_for_sm103a_only():
    assert B.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings_and_version():
    for s in range(8):
        assert G.gemm_status_string(s)
    assert "unknown" in G.gemm_status_string(99)
    assert G.gemm_tn_f16_version() >= 10000


@pytest.mark.parametrize("args", [
    dict(M=-1, N=8, K=8, lda=8, ldb=8, ldd=8),
    dict(M=8, N=8, K=8, lda=7, ldb=8, ldd=8),     # lda < K
    dict(M=8, N=8, K=8, lda=8, ldb=7, ldd=8),     # ldb < K
    dict(M=8, N=8, K=8, lda=8, ldb=8, ldd=7),     # ldd < N
])
def test_invalid_sizes_rejected_before_any_cuda_call(args):
    a = dict(A=0x1000, B=0x2000, C=None, ldc=8, D=0x3000, alpha=1.0, beta=0.0)
    a.update(args)
    st = G.gemm_tn_f16(a["A"], a["lda"], a["B"], a["ldb"], a["C"], a["ldc"], a["D"], a["ldd"],
                       a["M"], a["N"], a["K"], a["alpha"], a["beta"], check=False)
    assert st == G.GEMM_ERR_INVALID_VALUE


def test_null_and_misaligned_pointers_rejected():
    assert G.gemm_tn_f16(None, 8, 0x2000, 8, None, 8, 0x3000, 8, 8, 8, 8, 1.0, 0.0, check=False) == \
        G.GEMM_ERR_INVALID_VALUE
    assert G.gemm_tn_f16(0x1000, 8, 0x2000, 8, None, 8, 0x3000, 8, 8, 8, 8, 1.0, 1.0, check=False) == \
        G.GEMM_ERR_INVALID_VALUE  # beta != 0 needs C
    assert G.gemm_tn_f16(0x1001, 8, 0x2000, 8, None, 8, 0x3000, 8, 8, 8, 8, 1.0, 0.0, check=False) == \
        G.GEMM_ERR_MISALIGNED
    # D overlapping A, and C overlapping D without being identical
    assert G.gemm_tn_f16(0x1000, 8, 0x2000, 8, None, 8, 0x1010, 8, 8, 8, 8, 1.0, 0.0, check=False) == \
        G.GEMM_ERR_INVALID_VALUE
    assert G.gemm_tn_f16(0x1000, 8, 0x2000, 8, 0x3010, 8, 0x3000, 8, 8, 8, 8, 1.0, 1.0, check=False) == \
        G.GEMM_ERR_INVALID_VALUE
    assert G.gemm_tn_f16(0x1000, 8, 0x2000, 8, 0x3000, 16, 0x3000, 8, 8, 8, 8, 1.0, 1.0, check=False) == \
        G.GEMM_ERR_INVALID_VALUE  # C == D but different leading dimensions


def test_batched_output_entries_must_be_disjoint():
    st = G.gemm_tn_f16_batched(0x100000, 8, 64, 0x200000, 8, 64, None, 8, 0, 0x300000, 8, 32,
                               8, 8, 8, 2, 1.0, 0.0, check=False)
    assert st == G.GEMM_ERR_INVALID_VALUE
    st = G.gemm_tn_f16_batched(0x100000, 8, -64, 0x200000, 8, 64, None, 8, 0, 0x300000, 8, 64,
                               8, 8, 8, 2, 1.0, 0.0, check=False)
    assert st == G.GEMM_ERR_INVALID_VALUE


def test_empty_problems_are_no_ops_without_touching_cuda():
    assert G.gemm_tn_f16(None, 1, None, 1, None, 1, None, 1, 0, 5, 5, 1.0, 0.0, check=False) == G.GEMM_OK
    assert G.gemm_tn_f16_batched(None, 1, 0, None, 1, 0, None, 1, 0, None, 1, 0, 4, 4, 4, 0, 1.0, 0.0,
                                 check=False) == G.GEMM_OK


def test_sizes_beyond_int32_unsupported():
    st = G.gemm_tn_f16(0x1000, 1 << 31, 0x2000, 1 << 31, None, 8, 0x3000, 8, 8, 8, 1 << 31, 1.0, 0.0, check=False)
    assert st == G.GEMM_ERR_UNSUPPORTED


def plan(M, N, K, batch=1, lda=None, ldb=None, ldc=None, ldd=None, sA=0, sB=0, sC=0, sD=0, beta=0.0,
         align=15, sms=148):
    return G.gemm_tn_f16_plan(M, N, K, batch, lda or K, ldb or K, ldc or N, ldd or N, sA, sB, sC, sD,
                              beta, align, sms)


def test_plan_large_square_uses_cta_pairs_and_tma_store():
    p = plan(5120, 5120, 4096, sms=152)
    assert p["kernel"] == 2 and p["cta_pair"] == 2 and p["tile_m"] == 256 and p["tile_n"] == 256
    assert p["epi_tma"] == 1 and p["splits"] == 1 and p["pack_a"] == 0 and p["pack_b"] == 0
    G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_FORCE_BN, 256)
    try:
        p = plan(8192, 8192, 8192, sms=152)
    finally:
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_FORCE_BN, 0)
    # 1024 tiles over 76 pairs = 13.5 waves; the half-empty last wave (68 k-blocks of 128 per
    # group) is shared out by k-block
    assert p["tile_n"] == 256 and p["stream_k"] == 1 and p["dp_tiles"] == 13 * 76 and p["grid"] == 152


def test_plan_wide_pair_tiles_only_for_many_full_waves_of_long_tiles():
    # 8192^3: 512 tiles of 256 x 512 over 76 pairs, 6.7 waves, data-parallel (8 waves of
    # 432-column tiles would save less than 5 % of the MMA work on the critical path)
    p = plan(8192, 8192, 8192, sms=152)
    assert p["cta_pair"] == 2 and p["tile_m"] == 256 and p["tile_n"] == 512 and p["epi_tma"] == 1
    assert p["stream_k"] == 0 and p["units"] == 512 and p["grid"] == 152 and p["stages"] == 4
    assert plan(16384, 16384, 8192, sms=152)["tile_n"] == 512
    # 6144 x 8192 x 8192, D = alpha A B^T: 5.05 waves of 512-column tiles, exactly 6 of
    # 256 x 432 tiles (24 x 19 = 456 = 6 x 76)
    p = plan(6144, 8192, 8192, sms=152)
    assert p["cta_pair"] == 2 and p["tile_n"] == 432 and p["units"] == 6 * 76 and p["stream_k"] == 0
    assert plan(6144, 8192, 8192, sms=152, beta=1.0)["tile_n"] == 256
    # too few waves, short K, a mostly empty last wave, or an epilogue without TMA stores
    for M, N, K, kw in ((4096, 4096, 4096, {}), (4096, 4096, 8192, {}), (8192, 8192, 4096, {}),
                        (8192, 6144, 8192, {}), (8192, 8192, 8192, dict(ldd=8193)),
                        (8192, 8192, 8192, dict(align=0b0111))):
        assert plan(M, N, K, sms=152, **kw)["tile_n"] == 256, (M, N, K, kw)
    # forced: 512 columns with CTA pairs and a TMA epilogue, else 256
    G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_FORCE_BN, 512)
    try:
        assert plan(4096, 4096, 4096, sms=152)["tile_n"] == 512
        assert plan(4096, 4096, 4096, sms=152, beta=1.0, ldc=4097)["tile_n"] == 512
        assert plan(4096, 4096, 4096, sms=152, ldd=4097)["tile_n"] == 256
    finally:
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_FORCE_BN, 0)
    # forced 432: D = alpha A B^T by TMA stores only, else 512, else 256
    G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_FORCE_BN, 432)
    try:
        assert plan(4096, 4096, 4096, sms=152)["tile_n"] == 432
        assert plan(4096, 4096, 4096, sms=152, beta=1.0)["tile_n"] == 512
        assert plan(4096, 4096, 4096, sms=152, ldd=4097)["tile_n"] == 256
        assert plan(16, 4096, 4096, sms=152)["tile_n"] == 16  # skinny problems stay swapped
    finally:
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_FORCE_BN, 0)


def test_plan_single_k_block_tiles_take_the_deep_store_queue_variant():
    # the attention score (K = 64, one k-block per tile, store-bound): 128 x 256 tiles with a
    # three-stage ring and four staging buffers per epilogue warp
    p = plan(4096, 4096, 64, batch=128, sA=4096 * 64, sB=4096 * 64, sD=4096 * 4096, sms=152)
    assert p["tile_m"] == 128 and p["tile_n"] == 256 and p["cta_pair"] == 1 and p["stages"] == 3
    assert p["epi_tma"] == 1
    # two k-blocks: the four-stage ring
    assert plan(4096, 4096, 128, batch=128, sA=4096 * 128, sB=4096 * 128, sD=4096 * 4096, sms=152)["stages"] == 4
    # beta != 0 (C by TMA): no such variant
    assert plan(4096, 4096, 64, batch=8, sA=4096 * 64, sB=4096 * 64, sC=4096 * 4096, sD=4096 * 4096, beta=1.0,
                sms=152)["stages"] == 4


def test_plan_forced_stream_k_splits_the_partial_wave():
    G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_STREAM_K, 1)
    G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_FORCE_BN, 256)
    try:
        p = plan(8192, 8192, 8192, sms=152)
        q = plan(8192, 8192, 8192, sms=128)  # 16 whole waves over 64 pairs: nothing to split
    finally:
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_STREAM_K, 0)
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_FORCE_BN, 0)
    # 13 whole waves run data-parallel, the remaining tiles are shared by k-block
    assert p["stream_k"] == 1 and p["dp_tiles"] == 13 * 76 and p["sk_tiles"] == 1024 - 13 * 76
    assert p["grid"] == 152 and p["units"] == 13 * 76
    assert q["stream_k"] == 0 and q["units"] == 1024
    G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_STREAM_K, -1)
    try:
        assert plan(16, 8192, 8192)["stream_k"] == 0
    finally:
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_STREAM_K, 0)


def test_plan_skinny_m_swaps_and_splits_k():
    # 64 swapped tiles of 128 rows: the two K halves of each tile on the two CTAs of a
    # cluster (one launch, no scratch) ...
    p = plan(16, 8192, 8192)
    assert p["kernel"] == 2 and p["swap_ab"] == 1 and p["tile_n"] == 16 and p["splits"] == 1
    assert p["k_cluster"] == 1 and p["grid"] == 128 and p["units"] == 64 and p["workspace_bytes"] == 0
    # ... or, without the cluster split, two K slices and the sum kernel
    G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_K_CLUSTER, -1)
    try:
        p = plan(16, 8192, 8192)
    finally:
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_K_CLUSTER, 0)
    assert p["kernel"] == 3 and p["swap_ab"] == 1 and p["tile_n"] == 16 and p["splits"] == 2
    assert p["k_cluster"] == 0 and p["workspace_bytes"] >= 2 * 16 * 8192 * 4
    # stream-K when no whole slices fit (128 tiles), and when asked for
    q = plan(16, 16384, 8192, sms=152)
    assert q["kernel"] == 2 and q["swap_ab"] == 1 and q["splits"] == 1 and q["stream_k"] == 1
    G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_STREAM_K, 1)
    try:
        r = plan(16, 8192, 8192)
    finally:
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_STREAM_K, 0)
    assert r["kernel"] == 2 and r["splits"] == 1 and r["stream_k"] == 1 and r["dp_tiles"] == 0
    assert r["sk_tiles"] == 64 and r["grid"] == 148 and 2 <= r["sk_maxc"] <= 4
    assert r["workspace_bytes"] >= 64 * r["sk_maxc"] * 128 * 16 * 4


def test_plan_stream_k_needs_one_iteration_per_group():
    G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_STREAM_K, 1)
    try:
        p = plan(128, 128, 512)  # one tile, 8 k-blocks: only 8 groups take part
        q = plan(128, 128, 448)  # 7 k-blocks: too few to share out
    finally:
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_STREAM_K, 0)
    assert p["stream_k"] == 1 and p["grid"] == 8 and p["sk_maxc"] == 8
    assert q["stream_k"] == 0 and q["grid"] == 1


def test_plan_automatic_stream_k_only_where_it_was_measured_to_pay():
    # long K or narrow swapped tiles: split the partial wave
    for M, N, K in ((4096, 4096, 4096), (4096, 4096, 8192), (2560, 2560, 8192), (256, 8192, 8192), (16, 16384, 8192),
                    (5120, 5120, 4096)):
        assert plan(M, N, K, sms=152)["stream_k"] == 1, (M, N, K)
    # 256 x 512 tiles: their 256 KB-per-CTA partials did not pay back (8192^3 603-612 against
    # 586-588 us data-parallel)
    assert plan(8192, 8192, 8192, sms=152)["stream_k"] == 0
    # short K, too few whole waves, or many contributors per split tile: data-parallel
    for M, N, K in ((1024, 1024, 1024), (2048, 2048, 1024), (4096, 4096, 2048), (1280, 4096, 4096),
                    (384, 4096, 4096), (2560, 2560, 1024), (4096, 8192, 4096)):
        assert plan(M, N, K, sms=152)["stream_k"] == 0, (M, N, K)


def test_plan_long_k_on_few_tiles_splits_k_to_fill_the_gpu():
    # K slices so that tiles x slices ~ the SM count (2..32, >= 8 k-blocks each), reduced
    # by the separate kernel
    for M, N, K, splits in ((256, 384, 131072, 25), (128, 128, 262144, 32), (512, 512, 65536, 9),
                            (256, 256, 8192, 16), (256, 256, 4096, 8), (512, 512, 2048, 4), (768, 768, 4096, 4),
                            # up to half the SMs busy, 128-255 k-blocks
                            (1024, 1024, 8192, 2), (128, 8192, 8192, 2), (640, 1024, 8192, 3)):
        p = plan(M, N, K, sms=152)
        assert p["kernel"] == 3 and p["splits"] == splits and p["tile_n"] == 128 and p["cta_pair"] == 1, (M, N, K)
        assert p["workspace_bytes"] >= splits * M * N * 4
    # swapped small-M problems with room for 3+ slices per tile: slices too
    for M, N, K, splits in ((48, 1024, 32768, 19), (64, 512, 131072, 32), (16, 1024, 65536, 19)):
        p = plan(M, N, K, sms=152)
        assert p["kernel"] == 3 and p["swap_ab"] == 1 and p["splits"] == splits, (M, N, K)
    # not for short K, many tiles, swapped skinny problems, or a forced stream-K choice
    for M, N, K in ((256, 256, 1024), (1024, 1024, 4096), (1024, 1024, 32768), (896, 1024, 16384), (16, 16384, 8192),
                    (4096, 4096, 4096)):
        assert plan(M, N, K, sms=152)["splits"] == 1, (M, N, K)
    G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_STREAM_K, 1)
    try:
        p = plan(256, 384, 131072, sms=152)
    finally:
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_STREAM_K, 0)
    assert p["splits"] == 1 and p["stream_k"] == 1


def test_plan_forced_splits_use_the_reduction_kernel():
    G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_FORCE_SPLITS, 4)
    try:
        p = plan(16, 8192, 8192)
    finally:
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_FORCE_SPLITS, 0)
    assert p["kernel"] == 3 and p["splits"] == 4 and p["stream_k"] == 0
    assert p["workspace_bytes"] >= 4 * 16 * 8192 * 4


def test_plan_ragged_packed_ld_repacks_operands_only():
    # A, B repacked; C read and D written where they are by the epilogue
    p = plan(4095, 3073, 2047, lda=2047, ldb=2047, ldc=3073, ldd=3073, beta=1.5)
    assert p["pack_a"] == 1 and p["pack_b"] == 1 and p["row_load"] == 0
    assert p["epi_tma"] == 0 and p["stage_cd"] == 0
    assert p["workspace_bytes"] >= 2 * (4095 + 3073) * 2048
    G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_FORCE_GENERIC_EPI, 1)
    try:
        p = plan(4095, 3073, 2047, lda=2047, ldb=2047, ldc=3073, ldd=3073, beta=1.5)
    finally:
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_FORCE_GENERIC_EPI, 0)
    assert p["epi_tma"] == 0 and p["stage_cd"] == 0


def test_plan_row_loader_option_reads_operand_rows_in_kernel():
    G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_ROW_LOADER, 1)
    try:
        # A, B read row by row by the loader warps (nothing repacked, no scratch)
        p = plan(4095, 3073, 2047, lda=2047, ldb=2047, ldc=3073, ldd=3073, beta=1.5)
        assert p["row_load"] == 3 and p["pack_a"] == 0 and p["pack_b"] == 0
        assert p["epi_tma"] == 0 and p["stage_cd"] == 0 and p["workspace_bytes"] == 0
        # only B misaligned: A still comes by TMA
        p = plan(4096, 3072, 2047, lda=2048, ldb=2047, ldc=3072, ldd=3072, beta=1.5)
        assert p["row_load"] == 2 and p["pack_a"] == 0 and p["pack_b"] == 0 and p["epi_tma"] == 1
        # forced repack, or an epilogue with no row-loader variant: repacked to scratch
        for opt in (G.GEMM_TN_OPT_FORCE_PACK, G.GEMM_TN_OPT_FORCE_GENERIC_EPI):
            G.gemm_tn_f16_set_option(opt, 1)
            try:
                p = plan(4095, 3073, 2047, lda=2047, ldb=2047, ldc=3073, ldd=3073, beta=1.5)
            finally:
                G.gemm_tn_f16_set_option(opt, 0)
            assert p["pack_a"] == 1 and p["pack_b"] == 1 and p["row_load"] == 0
        # swapped small-M problems have no row-loader variant either
        p = plan(16, 3073, 2047, lda=2047, ldb=2047, ldc=3073, ldd=3073)
        assert p["swap_ab"] == 1 and p["pack_a"] == 1 and p["pack_b"] == 1 and p["row_load"] == 0
    finally:
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_ROW_LOADER, 0)


def test_plan_score_batched_short_k():
    p = plan(4096, 4096, 64, batch=128, sA=4096 * 64, sB=4096 * 64, sD=4096 * 4096)
    assert p["kernel"] == 2 and p["cta_pair"] == 1 and p["tile_n"] == 256 and p["epi_tma"] == 1
    assert p["units"] == 32 * 16 * 128


def test_plan_misaligned_pointer_forces_pack_only():
    # A, B repacked; C and D accessed in place by the epilogue's row words
    p = plan(1024, 1024, 1024, align=0)
    assert p["pack_a"] == 1 and p["pack_b"] == 1 and p["row_load"] == 0
    assert p["epi_tma"] == 0 and p["stage_cd"] == 0
    p = plan(1024, 1024, 1024, align=0, beta=1.0)
    assert p["epi_tma"] == 0 and p["stage_cd"] == 0
    # aligned D, misaligned C: the TMA epilogue at any size, nothing staged
    p = plan(256, 256, 1024, ldc=257, beta=1.0)
    assert p["epi_tma"] == 1 and p["stage_cd"] == 0
    # small: the predicated epilogue reads C and writes D where they are
    p = plan(256, 256, 1024, align=0, beta=1.0)
    assert p["epi_tma"] == 0 and p["stage_cd"] == 0


def test_plan_k_zero_and_empty():
    assert plan(8, 8, 0)["kernel"] == 1
    assert plan(0, 8, 8)["kernel"] == 0


def test_plan_stream_k_grid_never_exceeds_iterations():
    for M, N, K in ((16, 1024, 512), (16, 1024, 1000), (300, 300, 4096), (1000, 1000, 65536)):
        p = plan(M, N, K)
        if p["stream_k"]:
            tiles = p["dp_tiles"] + p["sk_tiles"]
            assert p["grid"] // p["cta_pair"] <= tiles * ((K + 63) // 64)


def test_options_roundtrip_and_validation():
    G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_FORCE_BN, 128)
    assert G.gemm_tn_f16_get_option(G.GEMM_TN_OPT_FORCE_BN) == 128
    p = plan(8192, 8192, 8192)
    assert p["tile_n"] == 128
    G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_FORCE_BN, 0)
    assert plan(5120, 5120, 4096)["tile_n"] == 256
    G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_FORCE_BN, 512)
    assert G.gemm_tn_f16_get_option(G.GEMM_TN_OPT_FORCE_BN) == 512
    G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_FORCE_BN, 0)
    with pytest.raises(G.GemmError):
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_FORCE_BN, 100)
    with pytest.raises(G.GemmError):
        G.gemm_tn_f16_set_option(12345, 1)
    with pytest.raises(G.GemmError):
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_WAIT_TIMEOUT_NS, 10)


def test_gemm_f16_rejects_bad_majors_and_leading_dims():
    # unknown major
    assert G.gemm_f16(3, 0, 0x1000, 8, 0, 0x2000, 8, 0, None, 8, 0, 0x3000, 8, 0, 8, 8, 8, 1, 1.0, 0.0,
                      check=False) == G.GEMM_ERR_INVALID_VALUE
    # MN-major A needs lda >= M (A stored K x lda): M = 16 > lda = 8
    assert G.gemm_f16(G.GEMM_MN_MAJOR, 0, 0x1000, 8, 0, 0x2000, 8, 0, None, 8, 0, 0x3000, 8, 0, 16, 8, 8, 1,
                      1.0, 0.0, check=False) == G.GEMM_ERR_INVALID_VALUE
    # MN-major B needs ldb >= N
    assert G.gemm_f16(0, G.GEMM_MN_MAJOR, 0x1000, 8, 0, 0x2000, 8, 0, None, 16, 0, 0x3000, 16, 0, 8, 16, 8, 1,
                      1.0, 0.0, check=False) == G.GEMM_ERR_INVALID_VALUE


def test_transpose_host_checks_without_a_gpu():
    assert G.transpose_f32(None, 8, None, 8, 0, 8, check=False) == G.GEMM_OK
    assert G.transpose_f32(0x1000, 4, 0x9000, 8, 8, 8, check=False) == G.GEMM_ERR_INVALID_VALUE
    assert G.transpose_f16(0x1001, 8, 0x9000, 8, 8, 8, check=False) == G.GEMM_ERR_MISALIGNED
    assert G.transpose_f32(0x1000, 8, 0x1010, 8, 8, 8, check=False) == G.GEMM_ERR_INVALID_VALUE


def test_score_softmax_host_checks_without_a_gpu():
    f = G.score_softmax_stats_f16
    Q, K, m, l = 0x100000, 0x200000, 0x300000, 0x400000
    # empty problems: nothing to do, no CUDA call
    assert f(None, 64, 0, None, 64, 0, None, None, 0, 16, 64, 1, 0.125, check=False) == G.GEMM_OK
    assert f(None, 64, 0, None, 64, 0, None, None, 16, 16, 64, 0, 0.125, check=False) == G.GEMM_OK
    # negative sizes, missing outputs, short leading dimensions
    assert f(Q, 64, 0, K, 64, 0, m, l, -1, 16, 64, 1, 0.125, check=False) == G.GEMM_ERR_INVALID_VALUE
    assert f(Q, 64, 0, K, 64, 0, None, l, 16, 16, 64, 1, 0.125, check=False) == G.GEMM_ERR_INVALID_VALUE
    assert f(Q, 32, 0, K, 64, 0, m, l, 16, 16, 64, 1, 0.125, check=False) == G.GEMM_ERR_INVALID_VALUE
    assert f(Q, 64, 0, K, 32, 0, m, l, 16, 16, 64, 1, 0.125, check=False) == G.GEMM_ERR_INVALID_VALUE
    assert f(None, 64, 0, K, 64, 0, m, l, 16, 16, 64, 1, 0.125, check=False) == G.GEMM_ERR_INVALID_VALUE
    # head dimension limit and output alignment
    assert f(Q, 512, 0, K, 512, 0, m, l, 16, 16, 257, 1, 0.125, check=False) == G.GEMM_ERR_UNSUPPORTED
    assert f(Q, 64, 0, K, 64, 0, m + 2, l, 16, 16, 64, 1, 0.125, check=False) == G.GEMM_ERR_MISALIGNED
    assert f(Q + 1, 64, 0, K, 64, 0, m, l, 16, 16, 64, 1, 0.125, check=False) == G.GEMM_ERR_MISALIGNED
    # outputs overlapping each other or an input
    assert f(Q, 64, 0, K, 64, 0, m, m + 32, 16, 16, 64, 1, 0.125, check=False) == G.GEMM_ERR_INVALID_VALUE
    assert f(Q, 64, 0, K, 64, 0, Q + 64, l, 16, 16, 64, 1, 0.125, check=False) == G.GEMM_ERR_INVALID_VALUE
    assert f(Q, 64, 0, K, 64, 0, m, K + 128, 16, 16, 64, 1, 0.125, check=False) == G.GEMM_ERR_INVALID_VALUE


def test_host_gemm_checks_without_a_gpu():
    f = G.gemm_tn_f16_host
    assert f(None, 8, None, 8, None, 8, None, 8, 0, 8, 8, 1.0, 0.0, check=False) == G.GEMM_OK
    assert f(0x1000, 8, 0x2000, 8, None, 8, 0x3000, 8, -1, 8, 8, 1.0, 0.0, check=False) == G.GEMM_ERR_INVALID_VALUE
    assert f(0x1000, 4, 0x2000, 8, None, 8, 0x3000, 8, 8, 8, 8, 1.0, 0.0, check=False) == G.GEMM_ERR_INVALID_VALUE
    assert f(0x1000, 8, 0x2000, 8, None, 8, None, 8, 8, 8, 8, 1.0, 0.0, check=False) == G.GEMM_ERR_INVALID_VALUE
    assert f(0x1001, 8, 0x2000, 8, None, 8, 0x3000, 8, 8, 8, 8, 1.0, 0.0, check=False) == G.GEMM_ERR_MISALIGNED


def test_host_gemm_rejects_overlapping_buffers_without_a_gpu():
    f = G.gemm_tn_f16_host
    # D overlapping A, and C overlapping D without being D
    assert f(0x1000, 8, 0x8000, 8, None, 8, 0x1010, 8, 8, 8, 8, 1.0, 0.0, check=False) == G.GEMM_ERR_INVALID_VALUE
    assert f(0x1000, 8, 0x8000, 8, 0x20010, 8, 0x20000, 8, 8, 8, 8, 1.0, 1.0, check=False) == G.GEMM_ERR_INVALID_VALUE


def test_plan_small_problem_kernel_when_forced():
    # every k-block at once (K <= 512 / 384 for widths 64 / 128); tile width 64 while a wave of 128-wide tiles
    # would fill at most half the SMs, else 128; forced widths honoured
    G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_SMALL, 1)
    try:
        p = plan(128, 128, 128, sms=152)
        q = plan(1000, 2000, 256, sms=152)  # 8 x 16 tiles of 128 x 128: more than half the SMs
        r = plan(128, 128, 513, sms=152)  # nine k-blocks: the persistent kernel
        s = plan(128, 128, 128, lda=129, sms=152)  # rows tensor copies cannot address
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_FORCE_BN, 256)
        t = plan(128, 128, 128, sms=152)  # an option of the persistent kernel wins
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_FORCE_BN, 0)
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_SMALL, 128)
        u = plan(200, 136, 72, batch=3, sA=200 * 72, sB=136 * 72, sD=200 * 136, sms=152)
    finally:
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_FORCE_BN, 0)
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_SMALL, 0)
    assert p["kernel"] == 4 and p["tile_m"] == 128 and p["tile_n"] == 64 and p["stages"] == 2
    assert p["units"] == 2 and p["grid"] == 2 and p["workspace_bytes"] == 0
    assert q["kernel"] == 4 and q["tile_n"] == 128 and q["units"] == 8 * 16 and q["stages"] == 4
    assert r["kernel"] == 2 and s["kernel"] == 2 and t["kernel"] == 2
    assert u["kernel"] == 4 and u["tile_n"] == 128 and u["units"] == 2 * 2 * 3
    with pytest.raises(G.GemmError):
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_SMALL, 32)


def test_plan_small_problem_kernel_automatic_rule():
    # 64-wide tiles while they fit one wave; larger problems stay on the persistent kernel
    p = plan(1000, 1000, 96, sms=152)  # 8 x 16 = 128 tiles of 128 x 64
    q = plan(1536, 1536, 128, sms=152)  # 12 x 24 = 288: more than a wave
    r = plan(128, 128, 576, sms=152)  # nine k-blocks
    s = plan(1024, 1024, 512, sms=152)  # eight k-blocks, 128 tiles of 128 x 64
    assert p["kernel"] == 4 and p["tile_n"] == 64 and p["units"] == 128
    assert q["kernel"] == 2 and r["kernel"] == 2
    assert s["kernel"] == 4 and s["tile_n"] == 64 and s["stages"] == 8
