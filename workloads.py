"""Seeded synthetic inputs for the SGEMM workloads.

This module only draws random numbers and names the problem shapes.  It holds
none of the GEMM arithmetic, so both the CUDA path and the CPU oracle can take
their inputs from it without sharing any computation.

Every array is row-major float32 (C order).  A leading dimension larger than the
logical width is realised as a wider backing array whose extra columns are
filled with a fixed pad value, so a kernel that reads or writes past the
logical width is caught by the tests.

Workloads (the shapes and value distributions of the method's benchmark
problems; see "Micro_gemm_4x4 - cuBLAS micro GEMM skeleton", section 2, for the
operand shapes (M,K), (K,N), (M,N)):

  square256      M=N=K=256, U[-1,1) seed 0, alpha=1, beta=0 (+ integer copy)
  square1024ab   M=N=K=1024, N(0,1) seed 1 for A, B and C0, alpha=1.5, beta=0.5
  ragged         M=1023, N=777, K=513, lda=513, ldb=ldc=777, U[-1,1) seed 2
  gpt2_qkv       X[1024,768] N(0,1), W[768,2304] N(0,0.02), seed 3
  gpt2_mlp_up    X[1024,768] N(0,1), W[768,3072] N(0,0.02), seed 3
  gpt2_mlp_down  H[1024,3072] N(0,1), W[3072,768] N(0,0.02), seed 3
  square2048/4096/8192, skinny_k64 (8192x8192x64), long_k (1024x1024x16384),
                 U[-1,1) seed 4, alpha=1, beta=0
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

PAD_VALUE = np.float32(-777.0)


@dataclass
class Problem:
    name: str
    M: int
    N: int
    K: int
    lda: int
    ldb: int
    ldc: int
    alpha: float
    beta: float
    A: np.ndarray            # (M, lda) backing array, float32
    B: np.ndarray            # (K, ldb) backing array, float32
    C0: np.ndarray           # (M, ldc) backing array, float32 (initial C)
    meta: dict = field(default_factory=dict)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


# name -> (M, N, K, dist, seed, alpha, beta, extra)
WORKLOADS = {
    "square256": (256, 256, 256, "uniform", 0, 1.0, 0.0, {}),
    "square256_int": (256, 256, 256, "int4", 0, 1.0, 0.0, {}),
    "square1024ab": (1024, 1024, 1024, "normal", 1, 1.5, 0.5, {}),
    "ragged": (1023, 777, 513, "uniform", 2, 1.0, 0.0, {}),
    "gpt2_qkv": (1024, 2304, 768, "gpt2", 3, 1.0, 0.0, {}),
    "gpt2_mlp_up": (1024, 3072, 768, "gpt2", 3, 1.0, 0.0, {}),
    "gpt2_mlp_down": (1024, 768, 3072, "gpt2", 3, 1.0, 0.0, {}),
    "square2048": (2048, 2048, 2048, "uniform", 4, 1.0, 0.0, {}),
    "square4096": (4096, 4096, 4096, "uniform", 4, 1.0, 0.0, {}),
    "square8192": (8192, 8192, 8192, "uniform", 4, 1.0, 0.0, {}),
    "skinny_k64": (8192, 8192, 64, "uniform", 4, 1.0, 0.0, {}),
    "long_k": (1024, 1024, 16384, "uniform", 4, 1.0, 0.0, {}),
}


def _padded(rng_fill, rows: int, cols: int, ld: int) -> np.ndarray:
    """A (rows, ld) float32 array: the first `cols` columns from `rng_fill`,
    the rest PAD_VALUE."""
    out = np.full((rows, max(ld, 1)), PAD_VALUE, dtype=np.float32)
    if rows and cols:
        out[:, :cols] = rng_fill((rows, cols))
    return out


def uniform_fill(rng: np.random.Generator, lo: float = -1.0, hi: float = 1.0):
    def fill(shape):
        return rng.uniform(lo, hi, size=shape).astype(np.float32)
    return fill


def normal_fill(rng: np.random.Generator, std: float = 1.0):
    def fill(shape):
        return (rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float32)
    return fill


def int_fill(rng: np.random.Generator, lo: int = -4, hi: int = 4):
    def fill(shape):
        return rng.integers(lo, hi + 1, size=shape).astype(np.float32)
    return fill


def make(M: int, N: int, K: int, *, dist: str = "uniform", seed: int = 0,
         alpha: float = 1.0, beta: float = 0.0, lda: int | None = None,
         ldb: int | None = None, ldc: int | None = None, name: str = "custom",
         c0_dist: str | None = None) -> Problem:
    """Draw one seeded problem.  `dist` picks the value distribution of A and B
    ("uniform" U[-1,1), "normal" N(0,1), "int4" integers in {-4..4},
    "gpt2" A ~ N(0,1) and B ~ N(0,0.02)).  C0 is drawn only when beta != 0
    (else it is filled with NaN, which a correct kernel never reads)."""
    lda = max(K, 1) if lda is None else lda
    ldb = max(N, 1) if ldb is None else ldb
    ldc = max(N, 1) if ldc is None else ldc
    rng = np.random.default_rng(seed)
    if dist == "uniform":
        fa = fb = fc = uniform_fill(rng)
    elif dist == "normal":
        fa = fb = fc = normal_fill(rng)
    elif dist == "int4":
        fa = fb = fc = int_fill(rng)
    elif dist == "gpt2":
        fa = fc = normal_fill(rng, 1.0)
        fb = normal_fill(rng, 0.02)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    if c0_dist is not None:
        fc = {"uniform": uniform_fill(rng), "normal": normal_fill(rng),
              "int4": int_fill(rng)}[c0_dist]
    A = _padded(fa, M, K, lda)
    B = _padded(fb, K, N, ldb)
    if beta != 0.0:
        C0 = _padded(fc, M, N, ldc)
    else:
        C0 = np.full((M, max(ldc, 1)), np.nan, dtype=np.float32)
        C0[:, N:] = PAD_VALUE
    return Problem(name, M, N, K, lda, ldb, ldc, float(alpha), float(beta), A, B, C0,
                   {"dist": dist, "seed": seed})


def operands(M: int, N: int, K: int, *, dist: str = "int4", seed: int = 0,
             lda: int | None = None, ldb: int | None = None):
    """A (M x lda) and B (K x ldb) only, drawn as make() draws them, for shapes
    whose C is too large to hold on the host (C0 is never read at beta = 0)."""
    lda = max(K, 1) if lda is None else lda
    ldb = max(N, 1) if ldb is None else ldb
    rng = np.random.default_rng(seed)
    fill = {"uniform": uniform_fill, "normal": normal_fill, "int4": int_fill}[dist](rng)
    return _padded(fill, M, K, lda), _padded(fill, K, N, ldb)


def workload(name: str, *, dist: str | None = None) -> Problem:
    """One of the named benchmark workloads (table in the module docstring)."""
    M, N, K, d, seed, alpha, beta, extra = WORKLOADS[name]
    return make(M, N, K, dist=dist or d, seed=seed, alpha=alpha, beta=beta,
                name=name, **extra)


def sample_indices(M: int, N: int, count: int, seed: int = 1234):
    """Seeded output coordinates for sampled checks at sizes the oracle cannot
    finish in full: the four corners, the last row and column, and `count`
    uniformly drawn (i, j) pairs."""
    rng = np.random.default_rng(seed)
    ii = [0, 0, M - 1, M - 1]
    jj = [0, N - 1, 0, N - 1]
    ii += list(rng.integers(0, M, size=count))
    jj += list(rng.integers(0, N, size=count))
    return np.asarray(ii, dtype=np.int64), np.asarray(jj, dtype=np.int64)
