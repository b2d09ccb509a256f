"""The checked build on the GPU: the misaligned-operand, row-word, row-loader, repack,
split-K, swapped, wide-tile, small-problem and K == 0 paths run again in a child process that loads
libgemm_tn_f16_checked.so (GEMM_TN_F16_CHECKED=1), where every load and store the
kernels issue themselves is first tested against the byte range of its matrix.  Every
result must still match the oracle and no check may fire; and in that build a trimmed
range for D (GEMM_TN_OPT_CHECK_TRIM_D) must be reported as GEMM_ERR_BOUNDS with the
out-of-range stores skipped (test_gpu_checked_inner.py)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SELECTION = [
    "tests/test_gpu_checked_inner.py",
    "tests/test_gpu_misaligned_cd.py",
    "tests/test_gpu_rowword.py",
    "tests/test_gpu_rowload.py",
    "tests/test_gpu_dependent_launch.py",
    "tests/test_gpu_parity.py",
    "tests/test_gpu_wide.py",  # (the 432-column tile's tail chunk is stored from registers)
    "tests/test_gpu_small.py",  # (D stored from registers)
]


def test_paths_with_own_loads_and_stores_pass_under_device_bounds_checks():
    env = dict(os.environ, GEMM_TN_F16_CHECKED="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "gpu", *SELECTION,
           "-k", "not test_parity or packed or swap or generic or splitk or kcluster or k1 or k7 or k63 or k65 or batched"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    tail = (r.stdout + r.stderr)[-4000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and "skipped" not in r.stdout.splitlines()[-1], tail
