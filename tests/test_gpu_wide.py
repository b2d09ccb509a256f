"""256 x 512 CTA-pair tiles (two N=256 MMAs per K step into one 512-column accumulator,
whose first half is handed back to the MMA before the second is read) against the oracle,
element by element: ragged tails in every dimension, each TMA epilogue (beta == 0, C by
TMA, C at any alignment), stream-K with and without data-parallel waves, batches, and
MN-major operands."""
import zlib

import pytest

import dense_fp16_gemm_tn_gb300 as G
from gpu_util import options, run_problem
from test_gpu_layouts import LAYOUTS, run_layout

pytestmark = pytest.mark.gpu

WIDE = dict(force_bn=512, force_pair=2)


def plan_for(M, N, K, batch=1, ldc=None, beta=0.0, opts=None, **_):
    ldc = ldc or N
    with options(**opts):
        return G.gemm_tn_f16_plan(M, N, K, batch, K, K, ldc, N, M * K, N * K, M * ldc, M * N, beta, 15, 152)


CASES = [
    ("one_tile", dict(M=256, N=512, K=128)),
    ("ragged_all", dict(M=600, N=1096, K=520)),
    ("k_tail", dict(M=300, N=712, K=65)),
    ("beta_tma_c", dict(M=600, N=1096, K=520, alpha=0.5, beta=1.5)),
    ("beta_c_misaligned", dict(M=600, N=1096, K=520, ldc=1097, alpha=-0.75, beta=1.25)),
    ("batched", dict(M=520, N=1040, K=600, batch=2, alpha=0.125, beta=1.0)),
    ("many_tiles", dict(M=2100, N=2600, K=384)),
    ("streamk_no_dp_wave", dict(M=1280, N=1536, K=1024, opts=dict(stream_k=1))),
    ("streamk_dp_plus_sk", dict(M=3072, N=3584, K=1024, opts=dict(stream_k=1))),
    ("streamk_beta", dict(M=1290, N=1544, K=1000, alpha=0.5, beta=1.5, opts=dict(stream_k=1))),
    ("streamk_beta_c_misaligned", dict(M=1290, N=1544, K=1000, ldc=1545, alpha=0.5, beta=1.5,
                                       opts=dict(stream_k=1))),
]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_wide_tile_parity(name, kw):
    kw = dict(kw)
    opts = dict(WIDE, **kw.pop("opts", {}))
    plan = plan_for(opts=opts, **kw)
    assert plan["tile_n"] == 512 and plan["cta_pair"] == 2 and plan["epi_tma"] == 1
    run_problem(seed=zlib.crc32(name.encode()) % 1000, opts=opts, **kw)


EXACT = [
    ("exact", dict(M=512, N=1024, K=256)),
    ("exact_beta", dict(M=600, N=1096, K=200, beta=1.0)),
    ("exact_streamk", dict(M=3072, N=3584, K=1024, opts=dict(stream_k=1))),
]


@pytest.mark.parametrize("name,kw", EXACT, ids=[c[0] for c in EXACT])
def test_wide_tile_small_integers_bit_exact(name, kw):
    kw = dict(kw)
    opts = dict(WIDE, **kw.pop("opts", {}))
    assert plan_for(opts=opts, **kw)["tile_n"] == 512
    run_problem(seed=11, dist="int", compare="exact", opts=opts, **kw)


@pytest.mark.parametrize("a_mn,b_mn", LAYOUTS, ids=["MN_K", "K_MN", "MN_MN"])
def test_wide_tile_mn_major(a_mn, b_mn):
    run_layout(600, 1096, 520, a_mn, b_mn, alpha=0.5, beta=1.5, seed=5 + 2 * a_mn + b_mn, opts=WIDE)
    run_layout(1280, 1536, 1024, a_mn, b_mn, seed=9 + 2 * a_mn + b_mn, opts=dict(WIDE, stream_k=1))


# 256 x 432 pair tiles: MMAs of N = 256 and 176 into one accumulator (the first part handed
# back after its four 64-column chunks), six TMA-stored chunks and a 48-column tail written
# from registers.  The last tile column ends inside the first MMA's part, inside the
# second's, inside the tail chunk, and exactly on the tile.  (D rows 16-byte aligned: N and
# ldd multiples of 8, which the 432-column variant needs.)
W432 = dict(force_bn=432, force_pair=2)
CASES_432 = [
    ("one_tile", dict(M=256, N=432, K=128)),
    ("end_in_first_part", dict(M=600, N=536, K=520)),
    ("end_in_second_part", dict(M=300, N=1168, K=200)),
    ("end_in_tail_chunk", dict(M=520, N=832, K=136)),
    ("k_tail", dict(M=300, N=712, K=65)),
    ("k1", dict(M=260, N=440, K=1)),
    ("ldd_padded", dict(M=600, N=1000, K=264, ldd=1008, alpha=0.25)),
    ("batched", dict(M=520, N=904, K=200, batch=3, alpha=-0.5)),
    ("many_tiles_serpentine", dict(M=2100, N=2600, K=384, opts=dict(serpentine=1))),
]


@pytest.mark.parametrize("name,kw", CASES_432, ids=[c[0] for c in CASES_432])
def test_432_column_tile_parity(name, kw):
    kw = dict(kw)
    opts = dict(W432, **kw.pop("opts", {}))
    plan = plan_for(opts=opts, **kw)
    assert plan["tile_n"] == 432 and plan["cta_pair"] == 2 and plan["epi_tma"] == 1, plan
    run_problem(seed=zlib.crc32(name.encode()) % 1000, opts=opts, **kw)


@pytest.mark.parametrize("N", [864, 1168, 832])
def test_432_column_tile_small_integers_bit_exact(N):
    assert plan_for(M=512, N=N, K=256, opts=W432)["tile_n"] == 432
    run_problem(seed=13, M=512, N=N, K=256, dist="int", compare="exact", opts=W432)


def test_432_column_tile_falls_back_where_it_has_no_variant():
    # beta != 0 and MN-major operands take the 512-column tiles instead
    assert plan_for(M=600, N=1096, K=520, beta=1.5, opts=W432)["tile_n"] == 512
    run_problem(seed=17, M=600, N=1096, K=520, alpha=0.5, beta=1.5, opts=W432)
    run_layout(600, 1096, 520, 0, 1, seed=19, opts=W432)
