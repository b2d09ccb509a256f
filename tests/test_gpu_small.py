"""The small-problem kernel (K <= 512 / 384, one CTA per 128 x 64 or 128 x 128 tile, every
k-block loaded at once, D written from registers) against the oracle, element by
element: one tile and several, ragged M, N and K (tails inside a k-block, K = 1),
beta != 0 with C and D rows 16-byte aligned and not (the element path), batches
with a broadcast operand, and small-integer inputs bit for bit.  Each case runs with
the kernel forced at both tile widths; the plan must report it (kernel 4)."""
import numpy as np
import pytest

import dense_fp16_gemm_tn_gb300 as G
from gpu_util import options, run_problem

pytestmark = pytest.mark.gpu

CASES = [
    ("one_tile_128", dict(M=128, N=128, K=128)),
    ("ragged_tiny", dict(M=100, N=37, K=9, lda=16, ldb=24)),
    ("k1", dict(M=130, N=136, K=1, lda=8, ldb=8)),
    ("k65_beta", dict(M=200, N=136, K=65, alpha=0.5, beta=1.5, lda=72, ldb=80)),
    ("four_kblocks_beta", dict(M=300, N=264, K=256, alpha=-0.75, beta=0.25)),
    ("ragged_k_tail_in_last_block", dict(M=257, N=200, K=250, lda=256, ldb=256)),
    ("odd_ld_c_d_element_path", dict(M=129, N=131, K=64, beta=-1.0, ldc=133, ldd=135)),
    ("padded_ld_vector_path", dict(M=140, N=72, K=192, alpha=2.0, beta=0.5, lda=200, ldb=256, ldc=80, ldd=88)),
    ("batched_beta", dict(M=200, N=136, K=72, batch=3, alpha=0.125, beta=1.0)),
    ("batched_bcast_b", dict(M=130, N=136, K=64, batch=4, bcast_b=True)),
    ("many_tiles", dict(M=1000, N=1000, K=96, alpha=0.5)),
    ("six_kblocks_beta", dict(M=300, N=264, K=384, alpha=0.5, beta=-1.5)),
    ("k_tail_in_sixth_block", dict(M=129, N=200, K=330, lda=336, ldb=344)),
]


# eight k-blocks fit the 64-wide tiles only
CASES_64 = [
    ("eight_kblocks_beta", dict(M=260, N=136, K=512, alpha=0.25, beta=1.0)),
    ("k_tail_in_eighth_block", dict(M=200, N=77, K=500, lda=504, ldb=512)),
]


@pytest.mark.parametrize("name,case", CASES_64, ids=[c[0] for c in CASES_64])
def test_small_kernel_parity_long_k(name, case):
    case = dict(case)
    with options(small=64):
        p = _plan_kernel(case["M"], case["N"], case["K"], case.get("batch", 1), case.get("lda"), case.get("ldb"),
                         case.get("ldc"), case.get("ldd"), case.get("beta", 0.0))
    assert p["kernel"] == 4 and p["tile_n"] == 64 and p["stages"] == (case["K"] + 63) // 64, p
    run_problem(**case, opts=dict(small=64))


def _plan_kernel(M, N, K, batch=1, lda=None, ldb=None, ldc=None, ldd=None, beta=0.0):
    lda, ldb, ldc, ldd = lda or K, ldb or K, ldc or N, ldd or N
    return G.gemm_tn_f16_plan(M, N, K, batch, lda, ldb, ldc, ldd, M * lda, N * ldb, M * ldc, M * ldd, beta, 15,
                              152)


@pytest.mark.parametrize("width", [64, 128])
@pytest.mark.parametrize("name,case", CASES, ids=[c[0] for c in CASES])
def test_small_kernel_parity(name, case, width):
    case = dict(case)
    with options(small=width):
        p = _plan_kernel(case["M"], case["N"], case["K"], case.get("batch", 1), case.get("lda"), case.get("ldb"),
                         case.get("ldc"), case.get("ldd"), case.get("beta", 0.0))
    assert p["kernel"] == 4 and p["tile_n"] == width, p
    run_problem(**case, opts=dict(small=width))


@pytest.mark.parametrize("width", [64, 128])
def test_small_kernel_small_integers_bit_exact(width):
    for M, N, K, beta, ld in [(128, 128, 128, 0.0, 128), (300, 264, 256, 2.0, 256), (77, 45, 33, -1.0, 40)]:
        run_problem(M, N, K, beta=beta, lda=ld, ldb=ld, dist="int", compare="exact", opts=dict(small=width))


def test_small_kernel_off_reaches_the_persistent_kernel():
    with options(small=-1):
        p = _plan_kernel(128, 128, 128)
    assert p["kernel"] == 2
    run_problem(128, 128, 128, opts=dict(small=-1))


AUTO = [
    ("auto_single_tile", dict(M=128, N=128, K=128)),
    ("auto_small_m", dict(M=16, N=1024, K=128, alpha=0.5, beta=1.5)),
    ("auto_batched", dict(M=200, N=136, K=72, batch=3, alpha=0.125, beta=1.0)),
    ("auto_one_wave_of_64_wide_tiles", dict(M=1000, N=1000, K=200)),
    ("auto_eight_kblocks", dict(M=1024, N=1024, K=512, alpha=0.5)),
]


@pytest.mark.parametrize("name,case", AUTO, ids=[c[0] for c in AUTO])
def test_small_kernel_is_the_automatic_choice(name, case):
    case = dict(case)
    p = _plan_kernel(case["M"], case["N"], case["K"], case.get("batch", 1), beta=case.get("beta", 0.0))
    assert p["kernel"] == 4, p
    run_problem(**case)


def _draw(rng):
    """A seeded problem in the small kernel's reach at both widths: K <= 256, rows of A and B 16-byte
    aligned, C and D at any leading dimension, batches with broadcast operands."""
    K = int(rng.choice([1, 8, 40, 64, 100, 129, 192, 256]))
    ld = lambda k: 8 * ((k + 7) // 8) + 8 * int(rng.choice([0, 0, 1]))
    return dict(M=int(rng.choice([1, 5, 64, 127, 128, 200, 333, 520])), N=int(rng.choice([1, 9, 64, 65, 200, 511])),
                K=K, batch=int(rng.choice([1, 1, 2, 3])), lda=ld(K), ldb=ld(K),
                ldc_pad=int(rng.choice([0, 1, 7, 8])), ldd_pad=int(rng.choice([0, 1, 3, 8])),
                alpha=float(rng.choice([1.0, -0.5, 2.0])), beta=float(rng.choice([0.0, 1.0, -0.25])),
                bcast=int(rng.integers(0, 3)))


RANDOM = [_draw(np.random.default_rng(2000 + i)) for i in range(16)]


@pytest.mark.parametrize("case", RANDOM, ids=[f"r{i}" for i in range(len(RANDOM))])
def test_small_kernel_random_problems(case):
    c = dict(case)
    M, N, K, batch = c["M"], c["N"], c["K"], c["batch"]
    bc = c["bcast"] if batch > 1 else 0
    kw = dict(batch=batch, alpha=c["alpha"], beta=c["beta"], lda=c["lda"], ldb=c["ldb"],
              ldc=N + c["ldc_pad"], ldd=N + c["ldd_pad"], bcast_a=bc == 1, bcast_b=bc == 2, seed=M + N + K)
    with options(small=1):
        p = G.gemm_tn_f16_plan(M, N, K, batch, c["lda"], c["ldb"], kw["ldc"], kw["ldd"],
                               0 if bc == 1 else M * c["lda"], 0 if bc == 2 else N * c["ldb"], M * kw["ldc"],
                               M * kw["ldd"], c["beta"], 15, 152)
    assert p["kernel"] == 4, (case, p)
    run_problem(M, N, K, opts=dict(small=1), **kw)
