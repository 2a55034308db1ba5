"""CPU oracle for the single-precision GEMM -- test infrastructure only.

Only the tests, the package's smoke check and the benchmark's CPU-baseline leg
may import this package.  The CUDA library never links, loads or calls it, and
the two share no code: the oracle is plain C (``oracle_sgemm.c``) compiled with
gcc, driven from here through ctypes.

Definition (see ``oracle_sgemm.c`` for the citations):

    C = fl32(alpha * (A @ B) + beta * C0), the sum over k in IEEE double,
    ascending k, one final rounding to float.

Parity is pinned, not assumed: ``tests/test_oracle_pins.py`` checks this
oracle against exact rational arithmetic, integer closed forms, identity and
permutation copies, rank-1 products and the inner-/outer-product
formulations, and shows that planted mistakes fail those pins.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_sgemm.c")
_LIB = os.path.join(_HERE, "liboracle_sgemm.so")
_lock = threading.Lock()
_lib = None

_f32p = ctypes.POINTER(ctypes.c_float)
_i64p = ctypes.POINTER(ctypes.c_int64)
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, IEEE double, no FMA contraction)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            common = [_i64, _i64, _i64, ctypes.c_float, _f32p, _i64, _f32p, _i64,
                      ctypes.c_float, _f32p, _i64]
            lib.oracle_sgemm.argtypes = common + [_f32p, _i64, ctypes.c_int]
            lib.oracle_sgemm.restype = ctypes.c_int
            lib.oracle_sgemm_rows.argtypes = common + [_i64p, _i64, _f32p, ctypes.c_int]
            lib.oracle_sgemm_rows.restype = ctypes.c_int
            lib.oracle_sgemm_entries.argtypes = common + [_i64p, _i64p, _i64, _f32p]
            lib.oracle_sgemm_entries.restype = ctypes.c_int
            lib.oracle_sgemm_ex.argtypes = [ctypes.c_int, ctypes.c_int, _i64, _i64, _i64,
                                            ctypes.c_float, _f32p, _i64, _i64, _f32p, _i64,
                                            _i64, ctypes.c_float, _f32p, _i64, _i64, _i64,
                                            _f32p, ctypes.c_int, _f32p, ctypes.c_int]
            lib.oracle_sgemm_ex.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _fp(a: np.ndarray):
    return a.ctypes.data_as(_f32p)


def _prep(M, N, K, A, lda, B, ldb, C0, ldc0, beta):
    A = np.ascontiguousarray(A, dtype=np.float32)
    B = np.ascontiguousarray(B, dtype=np.float32)
    if C0 is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C0")
        C0 = np.zeros((1,), dtype=np.float32)
    C0 = np.ascontiguousarray(C0, dtype=np.float32)
    lda = int(A.shape[1]) if lda is None and A.ndim == 2 else (lda or max(K, 1))
    ldb = int(B.shape[1]) if ldb is None and B.ndim == 2 else (ldb or max(N, 1))
    ldc0 = int(C0.shape[1]) if ldc0 is None and C0.ndim == 2 else (ldc0 or max(N, 1))
    return A, lda, B, ldb, C0, ldc0


def max_threads() -> int:
    """Threads one parallel oracle call uses on this host."""
    return int(_load().oracle_max_threads())


def sgemm(M: int, N: int, K: int, alpha: float, A: np.ndarray, B: np.ndarray,
          beta: float = 0.0, C0: np.ndarray | None = None, *, lda=None, ldb=None,
          ldc0=None, nthreads: int = 0) -> np.ndarray:
    """Full oracle product as a dense (M, N) float32 array."""
    lib = _load()
    A, lda, B, ldb, C0, ldc0 = _prep(M, N, K, A, lda, B, ldb, C0, ldc0, beta)
    out = np.empty((M, N), dtype=np.float32)
    if M and N:
        rc = lib.oracle_sgemm(M, N, K, float(alpha), _fp(A), lda, _fp(B), ldb,
                              float(beta), _fp(C0), ldc0, _fp(out), N, int(nthreads))
        if rc:
            raise RuntimeError("oracle_sgemm failed")
    return out


def sgemm_rows(M, N, K, alpha, A, B, beta, C0, rows, *, lda=None, ldb=None,
               ldc0=None, nthreads: int = 0) -> np.ndarray:
    """Oracle rows `rows` of C as a dense (len(rows), N) float32 array."""
    lib = _load()
    A, lda, B, ldb, C0, ldc0 = _prep(M, N, K, A, lda, B, ldb, C0, ldc0, beta)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((len(rows), N), dtype=np.float32)
    if len(rows) and N:
        rc = lib.oracle_sgemm_rows(M, N, K, float(alpha), _fp(A), lda, _fp(B), ldb,
                                   float(beta), _fp(C0), ldc0,
                                   rows.ctypes.data_as(_i64p), len(rows), _fp(out),
                                   int(nthreads))
        if rc:
            raise RuntimeError("oracle_sgemm_rows failed")
    return out


def sgemm_entries(M, N, K, alpha, A, B, beta, C0, ii, jj, *, lda=None, ldb=None,
                  ldc0=None) -> np.ndarray:
    """Oracle entries C[ii[t], jj[t]], each one inner product."""
    lib = _load()
    A, lda, B, ldb, C0, ldc0 = _prep(M, N, K, A, lda, B, ldb, C0, ldc0, beta)
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    out = np.empty(len(ii), dtype=np.float32)
    if len(ii):
        rc = lib.oracle_sgemm_entries(M, N, K, float(alpha), _fp(A), lda, _fp(B), ldb,
                                      float(beta), _fp(C0), ldc0,
                                      ii.ctypes.data_as(_i64p), jj.ctypes.data_as(_i64p),
                                      len(ii), _fp(out))
        if rc:
            raise RuntimeError("oracle_sgemm_entries failed")
    return out


def sgemm_ex(op_a: int, op_b: int, M: int, N: int, K: int, alpha: float, A: np.ndarray,
             lda: int, stride_a: int, B: np.ndarray, ldb: int, stride_b: int, beta: float,
             C0: np.ndarray | None, ldc0: int, stride_c0: int, batch: int,
             bias: np.ndarray | None = None, act: int = 0, *, nthreads: int = 0) -> np.ndarray:
    """The general form (see oracle_sgemm_ex in oracle_sgemm.c): batched,
    op(X) = X or X^T, + bias[j], act 0 (none) or 1 (tanh GELU).  A, B, C0 are
    the flat backing buffers the strides index.  Returns (batch, M, N)."""
    lib = _load()
    A = np.ascontiguousarray(A, dtype=np.float32).ravel()
    B = np.ascontiguousarray(B, dtype=np.float32).ravel()
    if C0 is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C0")
        C0 = np.zeros(1, np.float32)
    C0 = np.ascontiguousarray(C0, dtype=np.float32).ravel()
    bias_p = None
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float32).ravel()
        bias_p = _fp(bias)
    out = np.empty((batch, M, N), dtype=np.float32)
    if batch and M and N:
        rc = lib.oracle_sgemm_ex(int(op_a), int(op_b), M, N, K, float(alpha), _fp(A), lda,
                                 stride_a, _fp(B), ldb, stride_b, float(beta), _fp(C0), ldc0,
                                 stride_c0, batch, bias_p, int(act), _fp(out), int(nthreads))
        if rc:
            raise RuntimeError("oracle_sgemm_ex failed")
    return out


def problem(p, *, nthreads: int = 0) -> np.ndarray:
    """Oracle result for a `workloads.Problem`."""
    return sgemm(p.M, p.N, p.K, p.alpha, p.A, p.B, p.beta, p.C0, lda=p.lda,
                 ldb=p.ldb, ldc0=p.ldc, nthreads=nthreads)


def normalised_error(C: np.ndarray, C_ref: np.ndarray, K: int, A: np.ndarray,
                     B: np.ndarray, beta: float, C0: np.ndarray | None) -> float:
    """max|C - C_ref| / (K*max|A|*max|B| + |beta|*max|C0|): the error measure
    the parity tolerances are stated in (0 when the denominator is 0)."""
    den = float(K) * float(np.max(np.abs(A), initial=0.0)) * float(np.max(np.abs(B), initial=0.0))
    if beta != 0.0 and C0 is not None:
        den += abs(beta) * float(np.max(np.abs(C0), initial=0.0))
    num = float(np.max(np.abs(C.astype(np.float64) - C_ref.astype(np.float64)), initial=0.0))
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return num / den
