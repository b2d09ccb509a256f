import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


# Modules whose GPU tests take the library's automatic choice between the small-problem
# kernel and the persistent kernel; every other GPU module was written for the persistent
# kernel's paths (epilogues, swaps, K slices on small shapes too) and keeps them.
AUTOMATIC_SMALL_KERNEL_MODULES = {"test_gpu_small", "test_gpu_workloads", "test_gpu_random"}


@pytest.fixture(autouse=True)
def _persistent_kernel_on_small_shapes(request):
    if request.node.get_closest_marker("gpu") is None or \
            request.module.__name__.rsplit(".", 1)[-1] in AUTOMATIC_SMALL_KERNEL_MODULES:
        yield
        return
    import dense_fp16_gemm_tn_gb300 as G
    old = G.gemm_tn_f16_get_option(G.GEMM_TN_OPT_SMALL)
    G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_SMALL, -1)
    try:
        yield
    finally:
        G.gemm_tn_f16_set_option(G.GEMM_TN_OPT_SMALL, old)
