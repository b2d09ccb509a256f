"""Seeded synthetic inputs for the TN GEMM workloads.

This module is shared by the tests, the bench and the oracle's callers.  It
holds none of the GEMM's arithmetic: it only draws random numbers with numpy's
PCG64 generator, converts them to binary16 with numpy's own conversion, and
lays the bit patterns out with the requested leading dimensions.  Everything
it returns is a numpy ``uint16`` array of binary16 bit patterns.

Padding columns (``ld > cols``) are filled with a quiet NaN (0x7E00), so a
kernel that reads outside the logical matrix produces NaNs that the parity
checks catch.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

PAD_BITS = 0x7E00  # quiet NaN


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def uniform_half(seed: int, rows: int, cols: int, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    """rows x cols binary16 values, uniform in [lo, hi), as uint16 bits."""
    g = _rng(seed)
    x = g.random((rows, cols), dtype=np.float32)
    x = x * np.float32(hi - lo) + np.float32(lo)
    return x.astype(np.float16).view(np.uint16)


def normal_half(seed: int, rows: int, cols: int) -> np.ndarray:
    """rows x cols binary16 values drawn from N(0, 1), as uint16 bits."""
    g = _rng(seed)
    x = g.standard_normal((rows, cols), dtype=np.float32)
    return x.astype(np.float16).view(np.uint16)


def small_int_half(seed: int, rows: int, cols: int, lo: int = -2, hi: int = 2) -> np.ndarray:
    """Integers in [lo, hi] stored as binary16 bits (exact)."""
    g = _rng(seed)
    x = g.integers(lo, hi + 1, size=(rows, cols)).astype(np.float16)
    return x.view(np.uint16)


def with_ld(bits: np.ndarray, ld: int, pad_bits: int = PAD_BITS) -> np.ndarray:
    """Copy a (rows, cols) bit matrix into a (rows, ld) buffer, padding with NaN."""
    rows, cols = bits.shape
    assert ld >= cols
    out = np.full((rows, ld), pad_bits, dtype=np.uint16)
    out[:, :cols] = bits
    return out


def batched(gen, seed: int, batch: int, rows: int, cols: int) -> np.ndarray:
    """A (batch, rows, cols) stack; the whole stack comes from one stream."""
    flat = gen(seed, batch * rows, cols)
    return flat.reshape(batch, rows, cols)


@dataclass(frozen=True)
class Workload:
    """One GEMM problem: D = alpha * A . B^T + beta * C (per batch entry)."""
    name: str
    M: int
    N: int
    K: int
    batch: int = 1
    alpha: float = 1.0
    beta: float = 0.0
    lda: int | None = None
    ldb: int | None = None
    ldc: int | None = None
    ldd: int | None = None
    dist: str = "uniform"  # "uniform" in [-1,1] or "normal" N(0,1)
    seed: int = 0

    @property
    def lda_(self): return self.K if self.lda is None else self.lda
    @property
    def ldb_(self): return self.K if self.ldb is None else self.ldb
    @property
    def ldc_(self): return self.N if self.ldc is None else self.ldc
    @property
    def ldd_(self): return self.N if self.ldd is None else self.ldd

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K * self.batch

    @property
    def algorithmic_bytes(self) -> float:
        """Compulsory traffic: A and B read once, C read once if beta != 0, D written once."""
        mn = self.M * self.N * (2 if self.beta != 0 else 1)
        return 2.0 * (self.M * self.K + self.N * self.K + mn) * self.batch

    def make(self):
        """Return (A, B, C) as uint16 arrays shaped (batch, rows, ld); C is None if beta == 0."""
        gen = uniform_half if self.dist == "uniform" else normal_half
        A = batched(gen, self.seed * 3 + 0, self.batch, self.M, self.K)
        B = batched(gen, self.seed * 3 + 1, self.batch, self.N, self.K)
        A = np.stack([with_ld(a, self.lda_) for a in A]) if self.lda_ != self.K else A
        B = np.stack([with_ld(b, self.ldb_) for b in B]) if self.ldb_ != self.K else B
        C = None
        if self.beta != 0:
            C = batched(gen, self.seed * 3 + 2, self.batch, self.M, self.N)
            C = np.stack([with_ld(c, self.ldc_) for c in C]) if self.ldc_ != self.N else C
        return np.ascontiguousarray(A), np.ascontiguousarray(B), C if C is None else np.ascontiguousarray(C)


# The six measured problems.  Shapes, distributions, alpha and beta follow the
# workloads the method is studied on; seeds 1..6 are fixed per problem.
WORKLOADS = {
    "gemm_128": Workload("TN GEMM M=N=K=128, U[-1,1], alpha=1, beta=0", 128, 128, 128, seed=1),
    "gemm_4096": Workload("TN GEMM M=N=K=4096, U[-1,1], alpha=1, beta=0", 4096, 4096, 4096, seed=2),
    "gemm_ragged": Workload("TN GEMM M=4095 N=3073 K=2047 packed (lda=ldb=2047, ldc=ldd=3073), "
                            "U[-1,1], alpha=0.5, beta=1.5", 4095, 3073, 2047,
                            alpha=0.5, beta=1.5, seed=3),
    "score_qk": Workload("batched score S=Q.K^T, 8x16 heads, Q,K [4096,64] N(0,1), alpha=1/8, beta=0",
                         4096, 4096, 64, batch=128, alpha=0.125, beta=0.0, dist="normal", seed=4),
    "gemm_8192": Workload("TN GEMM M=N=K=8192, U[-1,1], alpha=1, beta=0", 8192, 8192, 8192, seed=5),
    "skinny_16": Workload("TN GEMM M=16 N=8192 K=8192 (split-K), U[-1,1], alpha=1, beta=0",
                          16, 8192, 8192, seed=6),
}
