"""Pins for the oracle's general form (batched, transposed views, bias, GELU).

- With batch 1, op N/N, no bias and no activation it must equal the plain
  oracle (itself pinned in test_oracle_pins.py) bit for bit.
- A transposed view must equal the plain product on the explicitly
  transposed matrix; each batch slice must equal the plain product on that
  slice; stride 0 broadcasts one operand.
- Bias on integer inputs is exact (Python integers); tiny random cases are
  compared with exact rationals.
- The tanh GELU is checked against a library routine (torch's tanh-form GELU
  in float64) and the identity gelu(x) - gelu(-x) = x.
- Planted mistakes (ignored transpose, bias twice, erf-form GELU, ignored batch
  stride) fail at least one pin.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest

import oracle
from test_oracle_pins import f32_round


def ex(impl, op_a, op_b, M, N, K, alpha, A, lda, sa, B, ldb, sb, beta, C0, ldc0, sc, batch,
       bias=None, act=0):
    return impl(op_a, op_b, M, N, K, alpha, A, lda, sa, B, ldb, sb, beta, C0, ldc0, sc, batch,
                bias, act)


def real(*args):
    return oracle.sgemm_ex(*args)


def pin_plain_form(impl):
    rng = np.random.default_rng(61)
    M, N, K = 37, 29, 41
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    C0 = rng.uniform(-1, 1, (M, N)).astype(np.float32)
    got = ex(impl, 0, 0, M, N, K, 1.25, A, K, 0, B, N, 0, -0.5, C0, N, 0, 1)[0]
    assert np.array_equal(got, oracle.sgemm(M, N, K, 1.25, A, B, -0.5, C0))


def pin_transposed_views(impl):
    rng = np.random.default_rng(62)
    M, N, K = 23, 31, 17
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    plain = oracle.sgemm(M, N, K, 1.0, A, B)
    At = np.ascontiguousarray(A.T)     # stored K x M
    Bt = np.ascontiguousarray(B.T)     # stored N x K
    assert np.array_equal(ex(impl, 1, 0, M, N, K, 1.0, At, M, 0, B, N, 0, 0.0, None, N, 0, 1)[0], plain)
    assert np.array_equal(ex(impl, 0, 1, M, N, K, 1.0, A, K, 0, Bt, K, 0, 0.0, None, N, 0, 1)[0], plain)
    assert np.array_equal(ex(impl, 1, 1, M, N, K, 1.0, At, M, 0, Bt, K, 0, 0.0, None, N, 0, 1)[0], plain)


def pin_batches(impl):
    rng = np.random.default_rng(63)
    M, N, K, nb = 9, 11, 13, 4
    A = rng.uniform(-1, 1, (nb, M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (nb, K, N)).astype(np.float32)
    C0 = rng.uniform(-1, 1, (nb, M, N)).astype(np.float32)
    got = ex(impl, 0, 0, M, N, K, 0.5, A, K, M * K, B, N, K * N, 2.0, C0, N, M * N, nb)
    for b in range(nb):
        assert np.array_equal(got[b], oracle.sgemm(M, N, K, 0.5, A[b], B[b], 2.0, C0[b]))
    # stride 0: one B shared by every batch
    got = ex(impl, 0, 0, M, N, K, 1.0, A, K, M * K, B[0], N, 0, 0.0, None, N, M * N, nb)
    for b in range(nb):
        assert np.array_equal(got[b], oracle.sgemm(M, N, K, 1.0, A[b], B[0]))


def pin_integer_bias(impl):
    rng = np.random.default_rng(64)
    M, N, K = 7, 9, 5
    A = rng.integers(-4, 5, (M, K)).astype(np.float32)
    B = rng.integers(-4, 5, (K, N)).astype(np.float32)
    bias = rng.integers(-8, 9, N).astype(np.float32)
    got = ex(impl, 0, 0, M, N, K, 1.0, A, K, 0, B, N, 0, 0.0, None, N, 0, 1, bias)[0]
    want = [[sum(int(A[i, k]) * int(B[k, j]) for k in range(K)) + int(bias[j]) for j in range(N)]
            for i in range(M)]
    assert np.array_equal(got.astype(np.int64), np.array(want))


def pin_fraction_bruteforce(impl):
    rng = np.random.default_rng(65)
    for trial in range(12):
        M, N, K = (int(x) for x in rng.integers(1, 5, size=3))
        nb = int(rng.integers(1, 3))
        op_a, op_b = int(trial % 2), int((trial // 2) % 2)
        A = rng.uniform(-2, 2, (nb, K, M) if op_a else (nb, M, K)).astype(np.float32)
        B = rng.uniform(-2, 2, (nb, N, K) if op_b else (nb, K, N)).astype(np.float32)
        C0 = rng.uniform(-2, 2, (nb, M, N)).astype(np.float32)
        bias = rng.uniform(-2, 2, N).astype(np.float32)
        alpha, beta = float(np.float32(rng.uniform(-2, 2))), float(np.float32(rng.uniform(-2, 2)))
        got = ex(impl, op_a, op_b, M, N, K, alpha, A, M if op_a else K, A[0].size, B,
                 K if op_b else N, B[0].size, beta, C0, N, M * N, nb, bias)
        for b in range(nb):
            for i in range(M):
                for j in range(N):
                    s = Fraction(0)
                    for k in range(K):
                        a = A[b, k, i] if op_a else A[b, i, k]
                        bv = B[b, j, k] if op_b else B[b, k, j]
                        s += Fraction(float(a)) * Fraction(float(bv))
                    v = Fraction(alpha) * s + Fraction(beta) * Fraction(float(C0[b, i, j])) \
                        + Fraction(float(bias[j]))
                    assert got[b, i, j] == f32_round(v), (trial, b, i, j)


def pin_gelu(impl):
    torch = pytest.importorskip("torch")
    x = np.concatenate([np.linspace(-6, 6, 97), [0.0, 1.0, -1.0, 3.5e-3, 25.0, -25.0]])
    x = x.astype(np.float32)
    n = len(x)
    # C[i][0] = gelu(x_i * 1): K = 1, B = [[1]]
    got = ex(impl, 0, 0, n, 1, 1, 1.0, x.reshape(n, 1), 1, 0, np.ones((1, 1), np.float32), 1, 0,
             0.0, None, 1, 0, 1, None, 1)[0][:, 0]
    lib = torch.nn.functional.gelu(torch.from_numpy(x.astype(np.float64)), approximate="tanh")
    want = lib.numpy().astype(np.float32)
    assert np.all(np.abs(got.astype(np.float64) - want.astype(np.float64))
                  <= np.spacing(np.abs(want)).astype(np.float64) + 1e-30)
    # gelu(x) - gelu(-x) = x
    neg = ex(impl, 0, 0, n, 1, 1, 1.0, (-x).reshape(n, 1), 1, 0, np.ones((1, 1), np.float32), 1,
             0, 0.0, None, 1, 0, 1, None, 1)[0][:, 0]
    diff = got.astype(np.float64) - neg.astype(np.float64)
    assert np.all(np.abs(diff - x) <= 4 * np.spacing(np.abs(x)).astype(np.float64) + 1e-30)
    assert got[list(x).index(0.0)] == 0.0


PINS = [pin_plain_form, pin_transposed_views, pin_batches, pin_integer_bias,
        pin_fraction_bruteforce, pin_gelu]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_ex_pin(pin):
    pin(real)


def _mut_ignore_transpose(op_a, op_b, *rest):
    return real(0, 0, *rest)


def _mut_bias_twice(op_a, op_b, M, N, K, alpha, A, lda, sa, B, ldb, sb, beta, C0, ldc0, sc,
                    batch, bias=None, act=0):
    out = real(op_a, op_b, M, N, K, alpha, A, lda, sa, B, ldb, sb, beta, C0, ldc0, sc, batch,
               bias, act)
    if bias is not None and act == 0:
        out = (out + np.asarray(bias, np.float32)).astype(np.float32)
    return out


def _mut_erf_gelu(op_a, op_b, M, N, K, alpha, A, lda, sa, B, ldb, sb, beta, C0, ldc0, sc,
                  batch, bias=None, act=0):
    out = real(op_a, op_b, M, N, K, alpha, A, lda, sa, B, ldb, sb, beta, C0, ldc0, sc, batch,
               bias, 0)
    if act == 1:
        from math import erf, sqrt
        v = out.astype(np.float64)
        out = (0.5 * v * (1 + np.vectorize(erf)(v / sqrt(2)))).astype(np.float32)
    return out


def _mut_ignore_batch_stride(op_a, op_b, M, N, K, alpha, A, lda, sa, B, ldb, sb, beta, C0, ldc0,
                             sc, batch, bias=None, act=0):
    return real(op_a, op_b, M, N, K, alpha, A, lda, 0, B, ldb, sb, beta, C0, ldc0, sc, batch,
                bias, act)


MUTANTS = [_mut_ignore_transpose, _mut_bias_twice, _mut_erf_gelu, _mut_ignore_batch_stride]


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m.__name__ for m in MUTANTS])
def test_ex_pins_catch_planted_mistake(mutant):
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mutant)
        except (AssertionError, ValueError, IndexError, RuntimeError):
            failed.append(pin.__name__)
    assert failed, f"{mutant.__name__} passed every pin"
