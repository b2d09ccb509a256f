"""GPU vs oracle, element by element, through the C ABI.

Sizes span several tiles with ragged tails; forced options reach every compiled
kernel variant (single CTA / CTA pair, 128 / 256 columns, TMA or predicated
epilogue, swapped operands, split-K, repacked operands).  Tolerance:
|D_gpu - D_ref| <= 2 ulp_fp16(D_ref) + 1e-3 sqrt(K); small-integer inputs must
match bit for bit (the fp32 accumulation is then exact).
"""
import zlib

import numpy as np
import pytest

import dense_fp16_gemm_tn_gb300 as G
from gpu_util import assert_device_ok, options, run_problem, to_dev, to_host, torch

pytestmark = pytest.mark.gpu

CASES = [
    ("single_tile_128", dict(M=128, N=128, K=128)),
    ("tma_bn256_ragged", dict(M=300, N=520, K=200, opts=dict(force_bn=256, force_pair=1))),
    ("tma_bn128_ragged", dict(M=300, N=520, K=200, opts=dict(force_bn=128, force_pair=1))),
    ("tma_pair256", dict(M=600, N=776, K=520, opts=dict(force_bn=256, force_pair=2))),
    ("tma_pair128", dict(M=600, N=776, K=520, opts=dict(force_bn=128, force_pair=2))),
    ("tma_many_units", dict(M=1100, N=1032, K=1000)),
    ("generic_beta_bn256", dict(M=300, N=520, K=200, alpha=0.5, beta=1.5, opts=dict(force_bn=256, force_pair=1))),
    ("generic_beta_bn128", dict(M=300, N=520, K=200, alpha=0.5, beta=1.5, opts=dict(force_bn=128, force_pair=1))),
    ("generic_beta_pair", dict(M=600, N=776, K=520, alpha=0.5, beta=1.5, opts=dict(force_bn=256, force_pair=2))),
    ("generic_forced_beta0", dict(M=260, N=390, K=70, opts=dict(force_generic=1))),
    # TMA-store epilogue with beta != 0: C tiles fetched by TMA (aligned C)
    ("tma_beta_single", dict(M=300, N=520, K=200, alpha=0.5, beta=1.5, opts=dict(force_bn=256, force_pair=1))),
    ("tma_beta_bn128", dict(M=300, N=264, K=130, alpha=-1.0, beta=0.25, opts=dict(force_bn=128, force_pair=1))),
    ("tma_beta_pair", dict(M=600, N=776, K=520, alpha=0.5, beta=1.5, opts=dict(force_bn=256, force_pair=2))),
    ("tma_beta_ldc_padded", dict(M=257, N=264, K=96, alpha=0.5, beta=1.5, ldc=272, ldd=280)),
    ("tma_beta_streamk", dict(M=1280, N=1280, K=1024, alpha=0.5, beta=1.5, opts=dict(stream_k=1))),
    ("tma_beta_batched", dict(M=200, N=136, K=72, batch=3, alpha=0.125, beta=1.0)),
    ("tma_beta_batched_bcast_c_free", dict(M=256, N=256, K=128, batch=2, beta=-0.5)),
    ("packed_ragged", dict(M=257, N=263, K=129, alpha=0.5, beta=1.5)),
    ("packed_padded_ld", dict(M=200, N=136, K=100, lda=103, ldb=101, ldc=140, ldd=139, beta=-1.0)),
    ("packed_forced", dict(M=256, N=256, K=256, opts=dict(force_pack=1))),
    ("packed_pair", dict(M=513, N=515, K=517, alpha=0.5, beta=1.5, opts=dict(force_pair=2, force_bn=256))),
    ("swap_m16", dict(M=16, N=1000, K=300)),
    ("swap_m1", dict(M=1, N=777, K=64)),
    ("swap_m40_beta", dict(M=40, N=1024, K=256, alpha=0.5, beta=1.5)),
    ("swap_m64", dict(M=64, N=600, K=64)),
    ("swap_m33_packed", dict(M=33, N=400, K=77)),
    ("splitk_swap_auto", dict(M=16, N=512, K=2048)),
    ("splitk_swap_beta", dict(M=24, N=700, K=1500, alpha=0.5, beta=1.5, opts=dict(force_splits=5))),
    ("splitk_normal", dict(M=256, N=256, K=4096, opts=dict(force_splits=4, force_pair=1))),
    ("splitk_normal_beta", dict(M=200, N=136, K=1000, alpha=0.5, beta=1.5, opts=dict(force_splits=3, force_pair=1))),
    # tiles of one k-block with D = alpha A B^T by TMA stores: the four-staging-buffer variant
    # (three-stage ring), ragged edges, a K tail inside the k-block, batches
    ("store_queue_k40_batched", dict(M=1000, N=2104, K=40, batch=2, alpha=0.125)),
    ("store_queue_k64_single_row_block", dict(M=100, N=1104, K=64)),
    ("k1", dict(M=130, N=136, K=1)),
    ("k7", dict(M=130, N=136, K=7)),
    ("k63", dict(M=130, N=136, K=63)),
    ("k65", dict(M=130, N=136, K=65)),
    ("k130_beta", dict(M=130, N=136, K=130, alpha=2.0, beta=0.25)),
    ("batched", dict(M=200, N=136, K=72, batch=3)),
    ("batched_beta", dict(M=200, N=136, K=72, batch=3, alpha=0.125, beta=1.0)),
    ("batched_bcast_b", dict(M=130, N=136, K=64, batch=4, bcast_b=True)),
    ("batched_bcast_a_packed", dict(M=130, N=130, K=66, batch=3, bcast_a=True)),
    ("batched_pair", dict(M=520, N=520, K=600, batch=2, opts=dict(force_pair=2, force_bn=256))),
    ("batched_swap", dict(M=16, N=300, K=128, batch=3)),
    ("batched_short_k_normal", dict(M=512, N=512, K=64, batch=4, alpha=0.125, dist="normal")),
    # stream-K: the k-blocks of the tiles that do not fill a whole wave are spread over all CTA groups
    ("streamk_pair_no_dp_wave", dict(M=1280, N=1280, K=1024, opts=dict(stream_k=1))),
    ("streamk_pair_dp_plus_sk", dict(M=2560, N=2560, K=512, opts=dict(stream_k=1))),
    ("streamk_pair_generic_forced", dict(M=2000, N=1800, K=900, alpha=0.5, beta=1.5,
                                         opts=dict(stream_k=1, force_pair=2, force_bn=256))),
    ("streamk_single_tma_forced", dict(M=1100, N=1032, K=1000, opts=dict(stream_k=1, force_pair=1))),
    ("streamk_pair_generic_beta", dict(M=1290, N=1288, K=1000, alpha=0.5, beta=1.5, opts=dict(stream_k=1))),
    ("streamk_single_packed_beta", dict(M=1500, N=1100, K=700, alpha=0.5, beta=1.5, opts=dict(stream_k=1))),
    ("streamk_swap_skinny", dict(M=16, N=1024, K=4096)),
    ("streamk_swap_beta", dict(M=40, N=2000, K=1000, alpha=0.5, beta=1.5, opts=dict(stream_k=1))),
    ("streamk_batched", dict(M=600, N=600, K=640, batch=3, opts=dict(stream_k=1))),
    # K halves on the two CTAs of a cluster, the partial added through distributed shared memory
    ("kcluster_m16", dict(M=16, N=1000, K=3000, opts=dict(k_cluster=1))),
    ("kcluster_m40_beta", dict(M=40, N=2000, K=1000, alpha=0.5, beta=1.5, opts=dict(k_cluster=1))),
    ("kcluster_m24_three_kblocks", dict(M=24, N=777, K=130, opts=dict(k_cluster=1))),
    ("kcluster_many_tiles_per_cluster", dict(M=16, N=40000, K=512, beta=-0.75, opts=dict(k_cluster=1))),
    ("kcluster_batched", dict(M=16, N=600, K=256, batch=3, alpha=0.25, beta=1.0, opts=dict(k_cluster=1))),
    ("kcluster_packed", dict(M=33, N=400, K=777, lda=779, ldb=781, opts=dict(k_cluster=1))),
    ("kcluster_auto_skinny", dict(M=16, N=8192, K=4096)),
    # serpentine K order: odd waves of whole tiles walk K backwards
    ("serpentine_pair_waves", dict(M=3000, N=2900, K=700, alpha=0.5, beta=1.5,
                                   opts=dict(serpentine=1, stream_k=-1, force_pair=2, force_bn=256))),
    ("serpentine_single_waves", dict(M=2600, N=2000, K=330, opts=dict(serpentine=1, stream_k=-1, force_pair=1))),
    ("serpentine_wide_streamk", dict(M=4608, N=4608, K=640, opts=dict(serpentine=1, stream_k=1, force_bn=512))),
    ("serpentine_splitk", dict(M=300, N=1300, K=3000, opts=dict(serpentine=1, force_splits=3, force_pair=1))),
]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_parity(name, kw):
    run_problem(seed=zlib.crc32(name.encode()) % 1000, **kw)


@pytest.mark.parametrize("bn_m", [16, 32, 64])
def test_k_cluster_small_integers_bit_exact(bn_m):
    """K halves summed through distributed shared memory: exact sums must match bit for bit."""
    run_problem(bn_m, 3000, 2048, dist="int", compare="exact", seed=33, opts=dict(k_cluster=1))


@pytest.mark.parametrize("serp", [1, -1])
def test_serpentine_small_integers_bit_exact(serp):
    """Reversed K order must not change an exact sum: several waves of pair tiles with
    small-integer operands, bit for bit against the oracle."""
    run_problem(2600, 2400, 512, dist="int", compare="exact", seed=31,
                opts=dict(serpentine=serp, stream_k=-1, force_pair=2, force_bn=256))


EXACT = [
    ("exact_tma", dict(M=256, N=384, K=256)),
    ("exact_pair", dict(M=512, N=512, K=256, opts=dict(force_pair=2, force_bn=256))),
    ("exact_generic_beta", dict(M=200, N=136, K=200, beta=1.0)),
    ("exact_swap", dict(M=16, N=600, K=256)),
    ("exact_splitk", dict(M=16, N=256, K=256, opts=dict(force_splits=4))),
    ("exact_packed", dict(M=129, N=131, K=255)),
    ("exact_streamk_pair", dict(M=2560, N=2304, K=512, opts=dict(stream_k=1))),
    ("exact_streamk_swap", dict(M=16, N=1024, K=2048)),
    ("exact_store_queue", dict(M=700, N=1304, K=64, batch=2)),
]


@pytest.mark.parametrize("name,kw", EXACT, ids=[c[0] for c in EXACT])
def test_small_integers_bit_exact(name, kw):
    run_problem(seed=7, dist="int", compare="exact", **kw)


def test_k_zero_scales_c():
    run_problem(M=70, N=90, K=0, alpha=1.0, beta=0.5)
    run_problem(M=70, N=90, K=0, alpha=1.0, beta=0.0)


def test_empty_problem_touches_nothing():
    t = torch()
    D = t.full((64,), 3.0, dtype=t.float16, device="cuda")
    A = t.zeros(64, dtype=t.float16, device="cuda")
    G.gemm_tn_f16(A, 8, A, 8, None, 8, D, 8, 0, 8, 8, 1.0, 0.0)
    G.gemm_tn_f16(A, 8, A, 8, None, 8, D, 8, 8, 0, 8, 1.0, 0.0)
    G.gemm_tn_f16_batched(A, 8, 64, A, 8, 64, None, 8, 64, D, 8, 64, 8, 8, 8, 0, 1.0, 0.0)
    t.cuda.synchronize()
    assert (D == 3.0).all()


def test_beta_zero_ignores_nan_c():
    t = torch()
    M, N, K = 130, 136, 64
    A = t.ones((M, K), dtype=t.float16, device="cuda")
    B = t.ones((N, K), dtype=t.float16, device="cuda")
    C = t.full((M, N), float("nan"), dtype=t.float16, device="cuda")
    for opts in ({}, {"force_generic": 1}):
        D = t.empty((M, N), dtype=t.float16, device="cuda")
        with options(**opts):
            G.gemm_tn_f16(A, K, B, K, C, N, D, N, M, N, K, 1.0, 0.0)
        t.cuda.synchronize()
        assert (D == 64.0).all()


def test_c_aliases_d():
    t = torch()
    M, N, K = 257, 264, 96
    rng = np.random.default_rng(0)
    A = t.from_numpy(rng.integers(-2, 3, (M, K)).astype(np.float16)).cuda()
    B = t.from_numpy(rng.integers(-2, 3, (N, K)).astype(np.float16)).cuda()
    C = t.from_numpy(rng.integers(-4, 5, (M, N)).astype(np.float16)).cuda()
    want = (A.float() @ B.float().T) * 2.0 - C.float()
    for opts in ({}, {"force_generic": 1}):  # TMA-loaded C, then predicated loads
        D = C.clone()
        with options(**opts):
            G.gemm_tn_f16(A, K, B, K, D, N, D, N, M, N, K, 2.0, -1.0)
        t.cuda.synchronize()
        assert t.equal(D.float(), want)


def test_all_ones_closed_form_ragged_workload_shape():
    """A = B = C = 1 at the ragged workload's shape: every entry is 0.5*2047 + 1.5 = 1025."""
    t = torch()
    M, N, K = 4095, 3073, 2047
    A = t.ones((M, K), dtype=t.float16, device="cuda")
    B = t.ones((N, K), dtype=t.float16, device="cuda")
    C = t.ones((M, N), dtype=t.float16, device="cuda")
    D = t.empty((M, N), dtype=t.float16, device="cuda")
    G.gemm_tn_f16(A, K, B, K, C, N, D, N, M, N, K, 0.5, 1.5)
    t.cuda.synchronize()
    assert_device_ok()
    assert (D == 1025.0).all()


def test_timeout_is_reported_and_context_survives():
    """A CTA that never issues its first load makes its MMA wait run out: the
    kernel reports GEMM_ERR_TIMEOUT and exits, and the next call works."""
    t = torch()
    M, N, K = 256, 256, 256
    A = t.ones((M, K), dtype=t.float16, device="cuda")
    B = t.ones((N, K), dtype=t.float16, device="cuda")
    D = t.zeros((M, N), dtype=t.float16, device="cuda")
    assert G.gemm_tn_f16_last_device_error() == G.GEMM_OK
    with options(skip_first_load=1, timeout_ns=50_000_000, force_pair=1, force_bn=128):
        G.gemm_tn_f16(A, K, B, K, None, N, D, N, M, N, K, 1.0, 0.0)
        t.cuda.synchronize()
    assert G.gemm_tn_f16_last_device_error() == G.GEMM_ERR_TIMEOUT
    assert G.gemm_tn_f16_last_device_error() == G.GEMM_OK  # reading clears the word
    G.gemm_tn_f16(A, K, B, K, None, N, D, N, M, N, K, 1.0, 0.0)
    t.cuda.synchronize()
    assert_device_ok()
    assert (D == 256.0).all()


def test_stream_argument_is_honoured():
    t = torch()
    M, N, K = 300, 264, 128
    A = t.randn((M, K), device="cuda").half()
    B = t.randn((N, K), device="cuda").half()
    D1 = t.empty((M, N), dtype=t.float16, device="cuda")
    D2 = t.empty((M, N), dtype=t.float16, device="cuda")
    G.gemm_tn_f16(A, K, B, K, None, N, D1, N, M, N, K, 1.0, 0.0)
    s = t.cuda.Stream()
    s.wait_stream(t.cuda.current_stream())
    with t.cuda.stream(s):
        G.gemm_tn_f16(A, K, B, K, None, N, D2, N, M, N, K, 1.0, 0.0, stream=s)
    s.synchronize()
    t.cuda.synchronize()
    assert t.equal(D1, D2)


def test_invalid_arguments_rejected_on_device_path():
    t = torch()
    A = t.ones((16, 16), dtype=t.float16, device="cuda")
    st = G.gemm_tn_f16(A, 8, A, 16, None, 16, A, 16, 16, 16, 16, 1.0, 0.0, check=False)
    assert st == G.GEMM_ERR_INVALID_VALUE  # lda < K
    st = G.gemm_tn_f16(A.data_ptr() + 1, 16, A, 16, None, 16, t.empty_like(A), 16, 16, 16, 16, 1.0, 0.0,
                       check=False)
    assert st == G.GEMM_ERR_MISALIGNED
    st = G.gemm_tn_f16(A, 16, A, 16, None, 16, A, 16, 16, 16, 16, 1.0, 0.0, check=False)
    assert st == G.GEMM_ERR_INVALID_VALUE  # D overlaps A
