"""transpose_f32 / transpose_f16 through the C ABI against the oracle, bit for bit:
aligned (vectorised) and unaligned (scalar) paths, ragged edge tiles, padded ld."""
import numpy as np
import pytest

import dense_fp16_gemm_tn_gb300 as G
import oracle
from gpu_util import torch

pytestmark = pytest.mark.gpu


def dev_bits(x):
    t = torch()
    dt = {np.uint32: t.int32, np.uint16: t.int16}[x.dtype.type]
    signed = x.view(np.int32 if x.dtype == np.uint32 else np.int16)
    return t.from_numpy(np.ascontiguousarray(signed)).to("cuda").view(dt)


def host_bits(x, dtype):
    return x.cpu().numpy().view(dtype)


@pytest.mark.parametrize("dtype", [np.uint32, np.uint16], ids=["f32", "f16"])
@pytest.mark.parametrize("rows,cols,ldx_pad,ldy_pad,offset", [
    (1024, 1024, 0, 0, 0),     # the page's workload
    (1000, 777, 0, 0, 0),      # ragged edges, unaligned ld -> scalar path
    (640, 576, 8, 16, 0),      # padded, aligned leading dimensions
    (1, 1, 0, 0, 0),
    (3, 70, 0, 0, 0),
    (130, 66, 0, 0, 1),        # base pointers off 16-byte alignment -> scalar path
    (4096, 64, 0, 0, 0),
])
def test_transpose_matches_oracle(dtype, rows, cols, ldx_pad, ldy_pad, offset):
    t = torch()
    rng = np.random.default_rng(rows * 131 + cols)
    ldx, ldy = cols + ldx_pad, rows + ldy_pad
    x = rng.integers(0, np.iinfo(dtype).max, (rows, ldx), dtype=dtype)
    x_dev = dev_bits(np.concatenate([np.zeros(offset, dtype), x.ravel()]))
    y_dev = dev_bits(np.full(offset + cols * ldy + 64, 0x5A5A, dtype=dtype))
    fn = G.transpose_f32 if dtype == np.uint32 else G.transpose_f16
    esz = np.dtype(dtype).itemsize
    fn(x_dev.data_ptr() + offset * esz, ldx, y_dev.data_ptr() + offset * esz, ldy, rows, cols)
    t.cuda.synchronize()
    got = host_bits(y_dev, dtype)
    ref = np.full(cols * ldy, 0x5A5A, dtype=dtype)
    oracle.transpose(np.ascontiguousarray(x), rows, cols, ldx=ldx, ldy=ldy, Y=ref)
    assert np.array_equal(got[offset:offset + cols * ldy], ref)
    assert (got[:offset] == 0x5A5A).all() and (got[offset + cols * ldy:] == 0x5A5A).all()


def test_transpose_argument_checks():
    t = torch()
    x = t.zeros(64 * 64, dtype=t.float32, device="cuda")
    assert G.transpose_f32(x, 64, x, 64, 64, 64, check=False) == G.GEMM_ERR_INVALID_VALUE  # in place
    y = t.zeros(64 * 64, dtype=t.float32, device="cuda")
    assert G.transpose_f32(x, 32, y, 64, 64, 64, check=False) == G.GEMM_ERR_INVALID_VALUE  # ldx < cols
    assert G.transpose_f32(x.data_ptr() + 2, 64, y, 64, 8, 8, check=False) == G.GEMM_ERR_MISALIGNED
    assert G.transpose_f32(x, 64, y, 64, 0, 64, check=False) == G.GEMM_OK
