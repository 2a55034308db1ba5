"""Pins for the CPU oracle: each check ties it to something other than itself.

- hand-worked fixtures under tests/golden/ (each with its citation);
- exact rational arithmetic (fractions.Fraction) on small inputs, correctly
  rounded to fp32 -- the plain definition, computed by a different route;
- integer inputs, where every summation order is exact, against Python ints
  in both formulations the pages derive (velog @levelstage "AutoMinepp4",
  section "행렬곱: by 벡터의 외적": inner products, and a sum of outer products);
- closed forms: identity and permutation copies, rank-1 products;
- the BLAS-style special cases (alpha == 0, beta == 0, K == 0, empty shapes).

The mutation tests at the end plant plausible mistakes in the oracle (on the
CPU) and check that at least one pin fails for each.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# helpers independent of the oracle
# --------------------------------------------------------------------------

def f32_round(q: Fraction) -> np.float32:
    """Correctly rounded (nearest, ties to even) fp32 value of a rational."""
    if q == 0:
        return np.float32(0.0)
    f = np.float32(float(q))
    best = None
    for cand in (np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))):
        d = abs(Fraction(float(cand)) - q)
        bits = int(np.array(cand, dtype=np.float32).view(np.uint32))
        key = (d, bits & 1)  # closer first; on a tie, even mantissa first
        if best is None or key < best[0]:
            best = (key, cand)
    return np.float32(best[1])


def exact_gemm(M, N, K, alpha, A, B, beta, C0):
    """alpha*A@B + beta*C0 in exact rationals, then one rounding to fp32."""
    out = np.empty((M, N), dtype=np.float32)
    al, be = Fraction(float(alpha)), Fraction(float(beta))
    for i in range(M):
        for j in range(N):
            s = Fraction(0)
            if alpha != 0:
                for k in range(K):
                    s += Fraction(float(A[i, k])) * Fraction(float(B[k, j]))
            v = al * s
            if beta != 0:
                v += be * Fraction(float(C0[i, j]))
            out[i, j] = f32_round(v)
    return out


def inner_product_form(A, B):
    """Each entry as a dot product of a row of A with a column of B (Python ints)."""
    M, K = A.shape
    N = B.shape[1]
    return [[sum(int(A[i, k]) * int(B[k, j]) for k in range(K)) for j in range(N)]
            for i in range(M)]


def outer_product_form(A, B):
    """Sum over k of outer(A[:, k], B[k, :]) (Python ints)."""
    M, K = A.shape
    N = B.shape[1]
    C = [[0] * N for _ in range(M)]
    for k in range(K):
        col = [int(A[i, k]) for i in range(M)]
        row = [int(B[k, j]) for j in range(N)]
        for i in range(M):
            for j in range(N):
                C[i][j] += col[i] * row[j]
    return C


def real_oracle(M, N, K, alpha, A, B, beta, C0, lda=None, ldb=None, ldc0=None):
    return oracle.sgemm(M, N, K, alpha, A, B, beta, C0, lda=lda, ldb=ldb, ldc0=ldc0)


# --------------------------------------------------------------------------
# the pins, written against an implementation `impl` so the mutation tests can
# run the same checks on a deliberately broken oracle
# --------------------------------------------------------------------------

def pin_golden(impl):
    for name in sorted(os.listdir(GOLDEN)):
        if not name.endswith(".json"):
            continue
        with open(os.path.join(GOLDEN, name)) as f:
            g = json.load(f)
        assert g.get("citation"), name

        def arr(x):
            def conv(v):
                if isinstance(v, str):
                    return float.fromhex(v) if v.startswith(("0x", "-0x")) else float(v)
                return float(v)
            return np.array([[conv(v) for v in row] for row in x], dtype=np.float32)

        A, B, C0, C = arr(g["A"]), arr(g["B"]), arr(g["C0"]), arr(g["C"])
        got = impl(g["M"], g["N"], g["K"], g["alpha"], A, B, g["beta"], C0)
        assert np.array_equal(got, C), (name, got, C)


def pin_fraction_bruteforce(impl):
    rng = np.random.default_rng(11)
    for trial in range(40):
        M, N, K = (int(x) for x in rng.integers(1, 7, size=3))
        A = rng.uniform(-2, 2, (M, K)).astype(np.float32)
        B = rng.uniform(-2, 2, (K, N)).astype(np.float32)
        C0 = rng.uniform(-2, 2, (M, N)).astype(np.float32)
        alpha = float(np.float32(rng.uniform(-2, 2)))
        beta = float(np.float32(rng.uniform(-2, 2))) if trial % 3 else 0.0
        got = impl(M, N, K, alpha, A, B, beta, C0)
        want = exact_gemm(M, N, K, alpha, A, B, beta, C0)
        assert np.array_equal(got, want), (trial, got, want)


def pin_integer_formulations(impl):
    rng = np.random.default_rng(12)
    for M, N, K in [(1, 1, 1), (5, 7, 3), (17, 9, 33), (64, 48, 80)]:
        A = rng.integers(-4, 5, (M, K)).astype(np.float32)
        B = rng.integers(-4, 5, (K, N)).astype(np.float32)
        got = impl(M, N, K, 1.0, A, B, 0.0, None)
        inner = np.array(inner_product_form(A, B), dtype=np.float64)
        outer = np.array(outer_product_form(A, B), dtype=np.float64)
        assert np.array_equal(inner, outer)
        assert np.array_equal(got.astype(np.float64), inner), (M, N, K)
        # alpha/beta on integers stays exact: multiples of 0.5 far below 2^23
        C0 = rng.integers(-4, 5, (M, N)).astype(np.float32)
        got = impl(M, N, K, 1.5, A, B, 0.5, C0)
        assert np.array_equal(got.astype(np.float64), 1.5 * inner + 0.5 * C0.astype(np.float64))


def pin_identity_permutation(impl):
    rng = np.random.default_rng(13)
    for M, N in [(1, 1), (7, 5), (33, 70)]:
        B = rng.uniform(-1, 1, (M, N)).astype(np.float32)
        eye = np.eye(M, dtype=np.float32)
        assert np.array_equal(impl(M, N, M, 1.0, eye, B, 0.0, None), B)
        A = rng.uniform(-1, 1, (N, M)).astype(np.float32)  # A (N x M) times I_M
        assert np.array_equal(impl(N, M, M, 1.0, A, eye, 0.0, None), A)
        perm = rng.permutation(M)
        P = np.zeros((M, M), dtype=np.float32)
        P[np.arange(M), perm] = 1.0
        assert np.array_equal(impl(M, N, M, 1.0, P, B, 0.0, None), B[perm])
        # P on the right permutes columns: (A @ P)[:, j] = A[:, q] where P[q, j] = 1
        assert np.array_equal(impl(N, M, M, 1.0, A, P, 0.0, None), A[:, np.argsort(perm)])


def pin_rank1(impl):
    rng = np.random.default_rng(14)
    for M, N in [(1, 9), (13, 1), (31, 47)]:
        u = rng.uniform(-1, 1, (M, 1)).astype(np.float32)
        v = rng.uniform(-1, 1, (1, N)).astype(np.float32)
        # K = 1: one correctly rounded fp32 product per entry
        assert np.array_equal(impl(M, N, 1, 1.0, u, v, 0.0, None), u * v)
        # alpha = 2 scales exactly
        assert np.array_equal(impl(M, N, 1, 2.0, u, v, 0.0, None), np.float32(2.0) * (u * v))
    # K > 1 with every column of A equal to u and every row of B equal to v:
    # C = K * u v^T, exact for integers
    for M, N, K in [(4, 6, 5), (9, 3, 64)]:
        u = rng.integers(-4, 5, (M, 1)).astype(np.float32)
        v = rng.integers(-4, 5, (1, N)).astype(np.float32)
        A = np.repeat(u, K, axis=1)
        B = np.repeat(v, K, axis=0)
        got = impl(M, N, K, 1.0, A, B, 0.0, None)
        assert np.array_equal(got.astype(np.float64), K * (u.astype(np.float64) @ v.astype(np.float64)))


def pin_special_cases(impl):
    rng = np.random.default_rng(15)
    M, N, K = 6, 5, 4
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    C0 = rng.uniform(-1, 1, (M, N)).astype(np.float32)
    # beta == 0: C0 is not read
    nanc = np.full((M, N), np.nan, dtype=np.float32)
    got = impl(M, N, K, 1.0, A, B, 0.0, nanc)
    assert np.all(np.isfinite(got))
    assert np.array_equal(got, exact_gemm(M, N, K, 1.0, A, B, 0.0, C0))
    # alpha == 0: A and B are not read; C = fl32(beta * C0)
    nanA = np.full_like(A, np.nan)
    nanB = np.full_like(B, np.nan)
    got = impl(M, N, K, 0.0, nanA, nanB, 0.75, C0)
    assert np.array_equal(got, (np.float64(0.75) * C0.astype(np.float64)).astype(np.float32))
    # K == 0: C = fl32(beta * C0); and 0 with beta == 0
    got = impl(M, N, 0, 1.0, np.zeros((M, 0), np.float32), np.zeros((0, N), np.float32), 0.5, C0)
    assert np.array_equal(got, (0.5 * C0.astype(np.float64)).astype(np.float32))
    got = impl(M, N, 0, 1.0, np.zeros((M, 0), np.float32), np.zeros((0, N), np.float32), 0.0, nanc)
    assert np.array_equal(got, np.zeros((M, N), np.float32))
    # empty outputs
    assert impl(0, N, K, 1.0, np.zeros((0, K), np.float32), B, 0.0, None).shape == (0, N)
    assert impl(M, 0, K, 1.0, A, np.zeros((K, 0), np.float32), 0.0, None).shape == (M, 0)


def pin_leading_dimensions(impl):
    p = workloads.make(37, 29, 23, seed=5, lda=40, ldb=31, ldc=33, beta=0.5)
    got = impl(p.M, p.N, p.K, p.alpha, p.A, p.B, p.beta, p.C0, p.lda, p.ldb, p.ldc)
    want = exact_gemm(p.M, p.N, p.K, p.alpha, p.A[:, :p.K], p.B[:, :p.N], p.beta, p.C0[:, :p.N])
    assert np.array_equal(got, want)


def pin_error_bound_long_k(impl):
    """At larger K, each entry is within the fp32 rounding of the exact value:
    |C - exact| <= ulp/2 + (K-1) * 2^-53 * sum|a_k b_k| (double summation)."""
    rng = np.random.default_rng(16)
    M, N, K = 3, 4, 2048
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    got = impl(M, N, K, 1.0, A, B, 0.0, None)
    for i in range(M):
        for j in range(N):
            terms = [Fraction(float(A[i, k])) * Fraction(float(B[k, j])) for k in range(K)]
            exact = sum(terms, Fraction(0))
            absum = float(sum(abs(t) for t in terms))
            r = f32_round(exact)
            ulp = float(np.spacing(np.float32(abs(r)))) if r != 0 else 2.0 ** -149
            bound = ulp / 2 + (K - 1) * 2.0 ** -53 * absum
            assert abs(Fraction(float(got[i, j])) - exact) <= Fraction(bound) * Fraction(1 + 2 ** -20)


PINS = [pin_golden, pin_fraction_bruteforce, pin_integer_formulations,
        pin_identity_permutation, pin_rank1, pin_special_cases,
        pin_leading_dimensions, pin_error_bound_long_k]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(real_oracle)


# --------------------------------------------------------------------------
# the oracle's other entry points agree with the full product
# --------------------------------------------------------------------------

def test_rows_and_entries_match_full():
    p = workloads.make(70, 45, 61, seed=6, lda=64, ldb=48, ldc=47, beta=-0.25)
    full = oracle.problem(p)
    rows = np.array([0, 5, 69, 33], dtype=np.int64)
    got_rows = oracle.sgemm_rows(p.M, p.N, p.K, p.alpha, p.A, p.B, p.beta, p.C0, rows,
                                 lda=p.lda, ldb=p.ldb, ldc0=p.ldc)
    assert np.array_equal(got_rows, full[rows])
    ii, jj = workloads.sample_indices(p.M, p.N, 50)
    got = oracle.sgemm_entries(p.M, p.N, p.K, p.alpha, p.A, p.B, p.beta, p.C0, ii, jj,
                               lda=p.lda, ldb=p.ldb, ldc0=p.ldc)
    assert np.array_equal(got, full[ii, jj])


def test_thread_count_does_not_change_result():
    p = workloads.make(64, 40, 300, seed=7)
    a = oracle.problem(p, nthreads=1)
    b = oracle.problem(p, nthreads=max(2, oracle.max_threads()))
    assert np.array_equal(a, b)


def test_normalised_error_measure():
    A = np.array([[1.0, -2.0]], np.float32)
    B = np.array([[0.5], [1.0]], np.float32)
    C = np.array([[3.0]], np.float32)
    ref = np.array([[2.0]], np.float32)
    # den = K*max|A|*max|B| = 2*2*1 = 4 ; num = 1
    assert oracle.normalised_error(C, ref, 2, A, B, 0.0, None) == 0.25
    C0 = np.array([[8.0]], np.float32)
    assert oracle.normalised_error(C, ref, 2, A, B, 0.5, C0) == 1.0 / 8.0


# --------------------------------------------------------------------------
# mutation tests: each planted mistake must fail at least one pin
# --------------------------------------------------------------------------

def _mutant_transposed_b(M, N, K, alpha, A, B, beta, C0, lda=None, ldb=None, ldc0=None):
    if B.ndim == 2 and B.shape[0] == B.shape[1]:
        B = np.ascontiguousarray(B.T)
    return real_oracle(M, N, K, alpha, A, B, beta, C0, lda, ldb, ldc0)


def _mutant_drop_last_k(M, N, K, alpha, A, B, beta, C0, lda=None, ldb=None, ldc0=None):
    lda = lda if lda is not None else (A.shape[1] if A.ndim == 2 else None)
    return real_oracle(M, N, max(K - 1, 0), alpha, A, B, beta, C0, lda, ldb, ldc0)


def _mutant_drop_beta(M, N, K, alpha, A, B, beta, C0, lda=None, ldb=None, ldc0=None):
    return real_oracle(M, N, K, alpha, A, B, 0.0, C0, lda, ldb, ldc0)


def _mutant_sign_beta(M, N, K, alpha, A, B, beta, C0, lda=None, ldb=None, ldc0=None):
    return real_oracle(M, N, K, alpha, A, B, -beta, C0, lda, ldb, ldc0)


def _mutant_fp32_accumulate(M, N, K, alpha, A, B, beta, C0, lda=None, ldb=None, ldc0=None):
    A2 = np.asarray(A, np.float32)[:, :K] if K else np.zeros((M, 0), np.float32)
    B2 = np.asarray(B, np.float32)[:K, :N]
    acc = np.zeros((M, N), np.float32)
    for k in range(K):
        acc = (acc + A2[:, k:k + 1] * B2[k:k + 1, :]).astype(np.float32)
    out = (np.float32(alpha) * acc).astype(np.float32)
    if beta != 0:
        out = (out + np.float32(beta) * np.asarray(C0, np.float32)[:, :N]).astype(np.float32)
    return out


def _mutant_alpha_twice(M, N, K, alpha, A, B, beta, C0, lda=None, ldb=None, ldc0=None):
    return real_oracle(M, N, K, alpha * alpha, A, B, beta, C0, lda, ldb, ldc0)


def _mutant_reads_c_when_beta_zero(M, N, K, alpha, A, B, beta, C0, lda=None, ldb=None, ldc0=None):
    out = real_oracle(M, N, K, alpha, A, B, beta, C0, lda, ldb, ldc0)
    if beta == 0 and C0 is not None and np.asarray(C0).size:
        out = out + 0.0 * np.asarray(C0, np.float32)[:M, :N]
    return out


def _mutant_ignores_lda(M, N, K, alpha, A, B, beta, C0, lda=None, ldb=None, ldc0=None):
    return real_oracle(M, N, K, alpha, A, B, beta, C0, K if K else None, ldb, ldc0)


MUTANTS = [_mutant_transposed_b, _mutant_drop_last_k, _mutant_drop_beta, _mutant_sign_beta,
           _mutant_fp32_accumulate, _mutant_alpha_twice, _mutant_reads_c_when_beta_zero,
           _mutant_ignores_lda]


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m.__name__ for m in MUTANTS])
def test_pins_catch_planted_mistake(mutant):
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mutant)
        except (AssertionError, ValueError, IndexError, RuntimeError):
            failed.append(pin.__name__)
    assert failed, f"{mutant.__name__} passed every pin"
