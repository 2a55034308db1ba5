"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Tolerances (the method's own statement of parity):
  * integer-valued inputs: bit-exact (every partial sum is an integer below
    2^24, so every summation order gives the same fp32 value);
  * otherwise: max|C - C_oracle| / (K*max|A|*max|B| + |beta|*max|C0|) <= 1e-6.
Every test also checks that C's padding and the memory around C are untouched.
"""
from __future__ import annotations

import dataclasses
import os

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

TOL_FFMA = 1e-6
SENTINEL = np.float32(-12345.5)


@pytest.fixture(scope="module")
def sg():
    import torch
    import dense_fp32_matrix_06_gb300 as pkg
    pkg.build()
    assert torch.cuda.is_available()
    pkg.load_library()
    return pkg


def _torch():
    import torch
    return torch


class DeviceProblem:
    """A workloads.Problem on the device, with C inside a guard band."""

    def __init__(self, p: workloads.Problem, a_offset: int = 0, b_offset: int = 0,
                 c_offset: int = 0):
        torch = _torch()
        self.p = p
        dev = torch.device("cuda")
        self.a_buf = torch.from_numpy(np.concatenate(
            [np.zeros(a_offset, np.float32), p.A.ravel()])).to(dev)
        self.b_buf = torch.from_numpy(np.concatenate(
            [np.zeros(b_offset, np.float32), p.B.ravel()])).to(dev)
        self.guard = 64 + c_offset
        c_host = np.full(self.guard + p.C0.size + 64, SENTINEL, np.float32)
        c_host[self.guard:self.guard + p.C0.size] = p.C0.ravel()
        # pad columns of C keep their own pad value (from workloads)
        self.c_host0 = c_host
        self.c_buf = torch.from_numpy(c_host.copy()).to(dev)
        self.a_ptr = self.a_buf.data_ptr() + 4 * a_offset
        self.b_ptr = self.b_buf.data_ptr() + 4 * b_offset
        self.c_ptr = self.c_buf.data_ptr() + 4 * self.guard

    def run(self, sg, alpha=None, beta=None):
        p = self.p
        sg.sgemm_ptr(p.M, p.N, p.K, p.alpha if alpha is None else alpha, self.a_ptr, p.lda,
                     self.b_ptr, p.ldb, p.beta if beta is None else beta, self.c_ptr, p.ldc,
                     _torch().cuda.current_stream().cuda_stream)

    def result(self):
        """(logical C, whole buffer) after a run."""
        _torch().cuda.synchronize()
        buf = self.c_buf.cpu().numpy()
        p = self.p
        C = buf[self.guard:self.guard + p.C0.size].reshape(p.C0.shape)[:, :p.N]
        return C.copy(), buf

    def check_untouched(self, buf):
        p = self.p
        want = self.c_host0.copy()
        region = want[self.guard:self.guard + p.C0.size].reshape(p.C0.shape)
        got_region = buf[self.guard:self.guard + p.C0.size].reshape(p.C0.shape)
        # everything outside the logical M x N block must be bit-identical
        mask = np.ones_like(region, dtype=bool)
        mask[:, :p.N] = False
        assert np.array_equal(got_region[mask].view(np.uint32), region[mask].view(np.uint32))
        assert np.array_equal(buf[:self.guard].view(np.uint32), want[:self.guard].view(np.uint32))
        tail = self.guard + p.C0.size
        assert np.array_equal(buf[tail:].view(np.uint32), want[tail:].view(np.uint32))


def logical(p):
    return p.A[:, :p.K], p.B[:, :p.N], (p.C0[:, :p.N] if p.beta != 0 else None)


def assert_parity(p, C, ref, exact: bool):
    if exact:
        assert np.array_equal(C, ref), f"{p.name}: not bit-exact on integer inputs"
    else:
        A, B, C0 = logical(p)
        err = oracle.normalised_error(C, ref, p.K, A, B, p.beta, C0)
        assert err <= TOL_FFMA, f"{p.name}: normalised error {err:.3e}"
        assert np.all(np.isfinite(C))


def run_and_check(sg, p, exact=False, **offsets):
    d = DeviceProblem(p, **offsets)
    d.run(sg)
    C, buf = d.result()
    d.check_untouched(buf)
    ref = oracle.problem(p)
    assert_parity(p, C, ref, exact)
    return C


SMALL = ["square256", "square256_int", "square1024ab", "ragged", "gpt2_qkv", "gpt2_mlp_up",
         "gpt2_mlp_down"]


@pytest.mark.parametrize("name", SMALL)
def test_workload_full_parity(sg, name):
    p = workloads.workload(name)
    run_and_check(sg, p, exact=(p.meta["dist"] == "int4"))


@pytest.mark.parametrize("name", SMALL)
def test_workload_integer_copy_bit_exact(sg, name):
    M, N, K, _, seed, alpha, beta, _ = workloads.WORKLOADS[name]
    p = workloads.make(M, N, K, dist="int4", seed=seed, alpha=alpha, beta=beta, name=name,
                       c0_dist="int4")
    run_and_check(sg, p, exact=True)


def test_ragged_leading_dimensions_and_alpha_beta(sg):
    p = workloads.make(1023, 777, 513, seed=2, lda=515, ldb=781, ldc=779, alpha=-0.75,
                       beta=1.25, c0_dist="uniform")
    run_and_check(sg, p)


@pytest.mark.parametrize("sched", [None, 0])   # as planned; the tiled kernels only
@pytest.mark.parametrize("seed", range(24))
def test_shape_fuzz(sg, tune, seed, sched):
    tune(schedule=sched)
    rng = np.random.default_rng(1000 + seed)
    M, N, K = (int(x) for x in rng.integers(1, 301, size=3))
    lda = K + int(rng.integers(0, 9))
    ldb = N + int(rng.integers(0, 9))
    ldc = N + int(rng.integers(0, 9))
    beta = 0.0 if seed % 2 == 0 else float(rng.uniform(-2, 2))
    alpha = float(rng.uniform(-2, 2))
    dist = "int4" if seed % 3 == 0 else "uniform"
    if dist == "int4":
        alpha, beta = 1.5, (0.5 if beta else 0.0)
    p = workloads.make(M, N, K, dist=dist, seed=seed, alpha=alpha, beta=beta, lda=lda,
                       ldb=ldb, ldc=ldc, c0_dist=dist if beta else None)
    offs = dict(a_offset=int(seed % 4 == 1), b_offset=int(seed % 5 == 2),
                c_offset=int(seed % 7 == 3))
    run_and_check(sg, p, exact=(dist == "int4"), **offs)


@pytest.mark.parametrize("sched", [None, 0])
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (1, 513, 17), (129, 1, 300), (128, 128, 16),
                                   (127, 129, 15), (256, 384, 1), (3, 5, 4096)])
def test_edge_shapes(sg, tune, M, N, K, sched):
    tune(schedule=sched)
    p = workloads.make(M, N, K, seed=M + N + K)
    run_and_check(sg, p)
    q = workloads.make(M, N, K, dist="int4", seed=M + N + K)
    run_and_check(sg, q, exact=True)


def test_beta_zero_never_reads_c(sg):
    p = workloads.make(200, 190, 70, seed=21)   # C0 is NaN where it is logical
    assert np.isnan(p.C0[:, :p.N]).all()
    C = run_and_check(sg, p)
    assert np.all(np.isfinite(C))


def test_alpha_zero_and_k_zero_scale_c(sg):
    p = workloads.make(130, 140, 50, seed=22, beta=0.75, c0_dist="uniform")
    p.A[:, :p.K] = np.nan
    p.B[:, :p.N] = np.nan
    p.alpha = 0.0
    d = DeviceProblem(p)
    d.run(sg)
    C, buf = d.result()
    d.check_untouched(buf)
    assert np.array_equal(C, oracle.problem(p))
    q = workloads.make(130, 140, 0, seed=23, beta=-0.5, c0_dist="uniform")
    d = DeviceProblem(q)
    d.run(sg)
    C, buf = d.result()
    d.check_untouched(buf)
    assert np.array_equal(C, oracle.problem(q))
    r = workloads.make(64, 64, 0, seed=24)   # K = 0, beta = 0: zeros, C not read
    d = DeviceProblem(r)
    d.run(sg)
    C, buf = d.result()
    assert np.array_equal(C, np.zeros((64, 64), np.float32))


def with_non_finite(p):
    """A copy of `p` with +inf, -inf and NaN planted in A and B (inside the
    logical block): row 5 meets +inf, row 9 -inf, row 40 NaN, row 70 both
    infinities (NaN in every column), column 7 a NaN of B."""
    A = p.A.copy()
    B = p.B.copy()
    A[5, 17] = np.inf
    A[9, 3] = -np.inf
    A[40, 60] = np.nan
    A[70, 10] = np.inf
    A[70, p.K - 1] = -np.inf
    B[10, :p.N] = np.abs(B[10, :p.N]) + 0.5       # so row 70's two infinite terms
    B[p.K - 1, :p.N] = np.abs(B[p.K - 1, :p.N]) + 0.5   # have opposite signs everywhere
    B[100, 7] = np.nan
    return dataclasses.replace(p, A=A, B=B, name=p.name + "+nonfinite")


def assert_same_specials(C, ref):
    """NaN, +inf and -inf exactly where the oracle has them."""
    assert np.array_equal(np.isnan(C), np.isnan(ref))
    assert np.array_equal(np.isposinf(C), np.isposinf(ref))
    assert np.array_equal(np.isneginf(C), np.isneginf(ref))


@pytest.mark.parametrize("knobs", [{}, {"tile": 64, "split_k": 3}, {"split_k": 4},
                                   {"transpose_a": 1, "tile": 128, "split_k": 1},
                                   {"transpose_a": 1, "tile": 128, "split_k": 3},
                                   {"schedule": 1}, {"schedule": 2}])
def test_non_finite_inputs_propagate_as_in_ieee_fp32(sg, tune, knobs):
    """IEEE semantics survive every path: a product with an infinity stays
    infinite with its sign, +inf and -inf in one sum give NaN, and a NaN
    spreads to its row or column -- the oracle (fp64 sums of the same
    products) fixes where.  The finite entries keep the usual tolerance."""
    tune(**knobs)
    M, N, K = (200, 256, 256) if knobs.get("schedule") == 2 else (300, 260, 1000)
    p = with_non_finite(workloads.make(M, N, K, seed=71, beta=0.5, c0_dist="uniform"))
    d = DeviceProblem(p)
    d.run(sg)
    C, buf = d.result()
    d.check_untouched(buf)
    ref = oracle.problem(p)
    assert_same_specials(C, ref)
    assert np.isposinf(ref[5]).any() and np.isneginf(ref[9]).any()
    assert np.isnan(ref[40]).all() and np.isnan(ref[70]).all() and np.isnan(ref[:, 7]).all()
    fin = np.isfinite(ref)
    A, B, C0 = logical(p)
    den = K * float(np.nanmax(np.abs(np.where(np.isfinite(A), A, 0)))) * \
        float(np.nanmax(np.abs(np.where(np.isfinite(B), B, 0)))) + 0.5 * float(np.abs(C0).max())
    assert float(np.abs(C[fin].astype(np.float64) - ref[fin]).max()) / den <= TOL_FFMA


@pytest.mark.parametrize("M,N,K,knobs", [
    (2048, 1024, 512, {}),                  # the A^T pass, then the grid
    (300, 260, 1000, {}),                   # 64-wide tiles, split K, reduction launch
    (256, 256, 256, {}),                    # the small-problem kernel
    (1024, 1024, 1024, {"transpose_a": 0, "tile": 128, "split_k": 4}),   # staged A, split
])
def test_subnormal_products_are_not_flushed(sg, tune, M, N, K, knobs):
    """Operands of magnitude up to 1e-19: every product is below the smallest
    normal float (1.18e-38), so a build that flushed subnormals to zero would
    turn each step's result into 0.  IEEE arithmetic keeps the usual
    tolerance against the oracle (its rounding of subnormal partial sums is
    absolute, 7e-46, far below K * max|A| * max|B|)."""
    tune(**knobs)
    p = workloads.make(M, N, K, seed=81)
    p = dataclasses.replace(p, A=(p.A * np.float32(1e-19)).astype(np.float32),
                            B=(p.B * np.float32(1e-19)).astype(np.float32))
    d = DeviceProblem(p)
    d.run(sg)
    C, buf = d.result()
    d.check_untouched(buf)
    ref = oracle.problem(p)
    A, B, _ = logical(p)
    den = K * float(np.abs(A).max()) * float(np.abs(B).max())
    assert np.abs(ref).max() > 1e-37                  # the results themselves are not tiny
    assert float(np.abs(C.astype(np.float64) - ref).max()) / den <= TOL_FFMA


def test_empty_shapes_are_no_ops(sg):
    torch = _torch()
    c = torch.full((4, 4), 3.0, device="cuda")
    sg.sgemm_ptr(0, 4, 4, 1.0, c.data_ptr(), 4, c.data_ptr(), 4, 0.0, c.data_ptr(), 4)
    sg.sgemm_ptr(4, 0, 4, 1.0, c.data_ptr(), 4, c.data_ptr(), 1, 0.0, c.data_ptr(), 1)
    torch.cuda.synchronize()
    assert bool((c == 3.0).all())


@pytest.mark.parametrize("kernel,tile", [("0", "128"), ("1", "128"), ("0", "64"), ("1", "64")])
@pytest.mark.parametrize("split", ["1", "2", "3", "7"])
def test_forced_kernel_and_split(sg, tune, kernel, tile, split):
    tune(kernel=kernel)
    tune(tile=tile)
    tune(split_k=split)
    p = workloads.make(300, 260, 1000, seed=31, beta=0.5, c0_dist="uniform")
    run_and_check(sg, p)
    q = workloads.make(256, 384, 1024, dist="int4", seed=32, alpha=1.5, beta=0.5,
                       c0_dist="int4")
    run_and_check(sg, q, exact=True)
    r = workloads.make(201, 77, 333, seed=33, lda=335, ldb=79, ldc=81)   # scalar path
    run_and_check(sg, r)


@pytest.mark.parametrize("M,N,K,dist,lds", [
    (2560, 2048, 1024, "int4", None),        # 320 tiles: the tail tiles split 4 ways
    (2560, 2048, 1040, "uniform", None),
    (2500, 2000, 777, "uniform", (781, 2003, 2001)),   # ragged tail tiles, scalar path
])
def test_tail_split_parity(sg, tune, M, N, K, dist, lds):
    lda, ldb, ldc = lds if lds else (None, None, None)
    p = workloads.make(M, N, K, dist=dist, seed=51, lda=lda, ldb=ldb, ldc=ldc,
                       alpha=1.5 if dist == "int4" else 0.75, beta=0.5,
                       c0_dist="int4" if dist == "int4" else "uniform")
    tune(tail_split="4")
    plan = sg.gemm_plan_for_sms(p.M, p.N, p.K, p.lda, p.ldb, p.ldc, sm_count=152)
    assert plan.tail_split > 1
    run_and_check(sg, p, exact=dist == "int4")
    tune(tail_split="0")
    run_and_check(sg, p, exact=dist == "int4")


@pytest.mark.parametrize("tile", ["64", "128"])
@pytest.mark.parametrize("name", ["square1024ab", "ragged", "gpt2_qkv", "square256_int"])
def test_forced_tile(sg, tune, tile, name):
    tune(tile=tile, schedule=0)
    p = workloads.workload(name)
    run_and_check(sg, p, exact=p.meta["dist"] == "int4")


@pytest.mark.parametrize("force", ["0", "1"])
@pytest.mark.parametrize("M,N,K,lds,dist", [
    (2048, 1024, 512, None, "uniform"),
    (2046, 1030, 515, (516, 1032, 1036), "uniform"),     # ragged: bounds-checked tiles
    (1024, 1536, 768, None, "int4"),
])
def test_transposed_a_path(sg, tune, force, M, N, K, lds, dist):
    tune(transpose_a=force)
    tune(split_k="1")
    tune(tile="128")
    lda, ldb, ldc = lds if lds else (None, None, None)
    p = workloads.make(M, N, K, dist=dist, seed=61, lda=lda, ldb=ldb, ldc=ldc,
                       alpha=1.5 if dist == "int4" else 0.75, beta=0.5,
                       c0_dist="int4" if dist == "int4" else "uniform")
    plan = sg.gemm_plan_for_sms(p.M, p.N, p.K, p.lda, p.ldb, p.ldc)
    assert plan.transpose_a == int(force)
    run_and_check(sg, p, exact=dist == "int4")


@pytest.mark.parametrize("split", ["2", "3"])
def test_transposed_a_with_split_k(sg, tune, split):
    tune(schedule=0, transpose_a="1")
    tune(split_k=split)
    tune(tile="128")
    p = workloads.make(512, 1024, 1000, seed=62, alpha=0.5, beta=-0.75, c0_dist="uniform")
    plan = sg.gemm_plan_for_sms(p.M, p.N, p.K, p.lda, p.ldb, p.ldc)
    assert plan.transpose_a == 1 and plan.split_k == int(split) and plan.bk == 32
    run_and_check(sg, p)
    q = workloads.make(384, 1152, 960, dist="int4", seed=63, alpha=1.5, beta=0.5, c0_dist="int4")
    run_and_check(sg, q, exact=True)


def test_transposed_a_with_caller_workspace(sg, tune):
    import torch
    p = workloads.workload("square4096")
    A = torch.from_numpy(p.A).cuda()
    B = torch.from_numpy(p.B).cuda()
    C = torch.empty((p.M, p.N), device="cuda")
    plan = sg.plan_for(A, B, C)
    assert plan.transpose_a == 1
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    sg.sgemm_with_plan(plan, A, B, C, 1.0, 0.0, ws)
    torch.cuda.synchronize()
    ii, jj = workloads.sample_indices(p.M, p.N, 2000, seed=5)
    ref = oracle.sgemm_entries(p.M, p.N, p.K, 1.0, p.A, p.B, 0.0, None, ii, jj)
    got = C.cpu().numpy()[ii, jj]
    den = p.K * float(np.abs(p.A).max()) * float(np.abs(p.B).max())
    assert float(np.abs(got.astype(np.float64) - ref).max()) / den <= TOL_FFMA
    with pytest.raises(sg.SgemmError) as e:
        sg.sgemm_with_plan(plan, A, B, C, 1.0, 0.0, ws[:1 << 20])
    assert e.value.status == 7


@pytest.mark.parametrize("tile", ["128", "64"])
def test_both_kernels_bit_identical(sg, tune, tile):
    tune(tile=tile)
    outs = []
    for kernel in ("0", "1"):
        tune(kernel=kernel)
        for name in ("square1024ab", "ragged", "long_k"):
            p = workloads.workload(name)
            d = DeviceProblem(p)
            d.run(sg)
            outs.append(d.result()[0])
    n = len(outs) // 2
    for a, b in zip(outs[:n], outs[n:]):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("M,N,K,lds,dist,knobs", [
    (2048, 1024, 512, None, "uniform", dict(transpose_a=1, schedule=0, split_k=1)),  # A^T grid
    (2046, 1030, 515, (516, 1032, 1036), "uniform", dict(transpose_a=1, schedule=0)),  # checked
    (1536, 1024, 1024, None, "int4", {}),                  # as planned: A^T + split-K
    (1024, 1024, 1024, None, "uniform", dict(transpose_a=1, schedule=1)),  # A^T + stream-K
    (1280, 2048, 2048, None, "int4", {}),                  # as planned: A^T + stream-K
])
def test_packed_issue_on_transposed_a_plans(sg, tune, M, N, K, lds, dist, knobs):
    """A^T plans issue their FMAs packed by default; scalar issue (tuning
    knob kernel = 0) gives the same C bit for bit, and both match the oracle."""
    tune(**knobs)
    lda, ldb, ldc = lds if lds else (None, None, None)
    p = workloads.make(M, N, K, dist=dist, seed=71, lda=lda, ldb=ldb, ldc=ldc,
                       alpha=1.5 if dist == "int4" else 0.75, beta=0.5,
                       c0_dist="int4" if dist == "int4" else "uniform")
    plan = sg.gemm_plan_for_sms(p.M, p.N, p.K, p.lda, p.ldb, p.ldc)
    assert plan.transpose_a == 1 and plan.kernel == 1
    outs = []
    for kernel in (None, 0):
        tune(kernel=kernel)
        outs.append(run_and_check(sg, p, exact=dist == "int4"))
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


@pytest.mark.parametrize("M,N,K,lda,a_offset,dist", [
    (2304, 1024, 515, 515, 0, "uniform"),     # odd lda: A's rows not 16-byte aligned
    (2304, 1024, 516, 516, 1, "int4"),        # A's pointer 4 bytes off
    (1280, 2048, 2047, 2047, 1, "uniform"),   # both, and A^T + stream-K
])
def test_transposed_a_path_with_unaligned_a(sg, M, N, K, lda, a_offset, dist):
    """Only B and C need 16-byte alignment for the A^T plans: A is copied into
    an aligned A^T first (the scalar transpose kernel reads it)."""
    p = workloads.make(M, N, K, dist=dist, seed=73, lda=lda, alpha=1.5 if dist == "int4" else 0.75,
                       beta=0.5, c0_dist="int4" if dist == "int4" else "uniform")
    plan = sg.gemm_plan_for_sms(p.M, p.N, p.K, p.lda, p.ldb, p.ldc, 4 * a_offset, 0, 0)
    assert plan.transpose_a == 1 and plan.vec == 1
    run_and_check(sg, p, exact=dist == "int4", a_offset=a_offset)


def test_deterministic_run_to_run(sg):
    for name in ("long_k", "ragged", "gpt2_mlp_down"):
        p = workloads.workload(name)
        d = DeviceProblem(p)
        first = None
        for _ in range(5):
            d.run(sg)
            C, _ = d.result()
            if first is None:
                first = C
            else:
                assert np.array_equal(C.view(np.uint32), first.view(np.uint32)), name


@pytest.mark.parametrize("name", ["long_k", "square1024ab"])
def test_sgemm_with_plan_caller_workspace(sg, name):
    """Caller-held workspace on a split plan: long_k (the A^T pass, then K
    ranges) and 1024^3 (64-wide tiles in eight K ranges, the balance rule)."""
    torch = _torch()
    p = workloads.workload(name)
    A = torch.from_numpy(p.A).cuda()
    B = torch.from_numpy(p.B).cuda()
    C = torch.empty((p.M, p.N), device="cuda")
    plan = sg.plan_for(A, B, C)
    # tiles share K ranges (split-K or stream-K), so the plan needs partials
    assert (plan.split_k > 1 or plan.sk_iters > 0) and plan.workspace_bytes > 0
    # the workspace needs no initialisation: start from garbage (NaN bytes)
    ws = torch.full((plan.workspace_bytes,), 0xFF, dtype=torch.uint8, device="cuda")
    if name == "square1024ab":
        assert (plan.bm, plan.split_k, plan.transpose_a) == (64, 8, 0)
    p0 = dataclasses.replace(p, alpha=1.0, beta=0.0)
    ref = oracle.problem(p0)
    for _ in range(3):   # and it can be reused as it is left
        C.fill_(float("nan"))
        sg.sgemm_with_plan(plan, A, B, C, 1.0, 0.0, ws)
        torch.cuda.synchronize()
        assert_parity(p0, C.cpu().numpy(), ref, exact=False)
    # the FFMA kernels leave the counter block (the 3xTF32 mode's) untouched
    assert bool((ws[:sg.WORKSPACE_COUNTER_BYTES] == 0xFF).all())
    with pytest.raises(sg.SgemmError) as e:
        sg.sgemm_with_plan(plan, A, B, C, 1.0, 0.0, ws[:16])
    assert e.value.status == 7


def test_torch_api_shapes_and_views(sg):
    torch = _torch()
    p = workloads.make(300, 200, 150, seed=41, lda=160, ldb=210)
    A = torch.from_numpy(p.A).cuda()[:, :p.K]     # row-strided views
    B = torch.from_numpy(p.B).cuda()[:, :p.N]
    C = sg.sgemm(A, B)
    torch.cuda.synchronize()
    assert_parity(p, C.cpu().numpy(), oracle.problem(p), exact=False)
    with pytest.raises(ValueError):
        sg.sgemm(A, B[:-1])
    with pytest.raises(ValueError):
        sg.sgemm(A[0], B)
    with pytest.raises(TypeError):
        sg.sgemm(A.double(), B)
    with pytest.raises(ValueError):   # column-strided operand
        sg.sgemm(A.t().contiguous().t(), B)


def test_status_errors_from_device_calls(sg):
    torch = _torch()
    x = torch.zeros(64, device="cuda")
    with pytest.raises(sg.SgemmError) as e:
        sg.sgemm_ptr(4, 4, 8, 1.0, x.data_ptr(), 7, x.data_ptr(), 4, 0.0, x.data_ptr(), 4)
    assert e.value.status == 1


# ---- full-size workloads: sampled entries against the oracle ----

LARGE = ["square2048", "square4096", "square8192", "skinny_k64", "long_k"]


@pytest.mark.parametrize("name", LARGE)
@pytest.mark.parametrize("dist", ["uniform", "int4"])
def test_large_workload_sampled(sg, name, dist):
    """The benchmark-size launches, checked where the oracle can afford it:
    3000 random entries, one random entry inside every output tile of the
    launch's plan, three single rows, and one whole block of tile rows."""
    p = workloads.workload(name, dist=None if dist == "uniform" else dist)
    d = DeviceProblem(p)
    plan = sg.gemm_plan(p.M, p.N, p.K, p.lda, p.ldb, p.ldc, d.a_ptr, d.b_ptr, d.c_ptr)
    d.run(sg)
    C, buf = d.result()
    d.check_untouched(buf)
    ii, jj = workloads.sample_indices(p.M, p.N, 3000, seed=7)
    # one entry per output tile (tile rows x tile columns of the plan)
    rng = np.random.default_rng(11)
    tm, tn = np.meshgrid(np.arange(plan.tiles_m), np.arange(plan.tiles_n), indexing="ij")
    ti = tm.ravel() * plan.bm + rng.integers(0, plan.bm, tm.size)
    tj = tn.ravel() * plan.bn + rng.integers(0, plan.bn, tn.size)
    keep = (ti < p.M) & (tj < p.N)
    assert keep.sum() >= plan.tiles_m * plan.tiles_n - plan.tiles_m - plan.tiles_n
    ii = np.concatenate([ii, ti[keep]])
    jj = np.concatenate([jj, tj[keep]])
    ref = oracle.sgemm_entries(p.M, p.N, p.K, p.alpha, p.A, p.B, p.beta, p.C0, ii, jj,
                               lda=p.lda, ldb=p.ldb, ldc0=p.ldc)
    got = C[ii, jj]
    # three rows, plus every row of one seeded tile row
    r0 = int(rng.integers(0, plan.tiles_m)) * plan.bm
    block = np.arange(r0, min(r0 + plan.bm, p.M), dtype=np.int64)
    rows = np.concatenate([np.array([0, p.M // 2 + 1, p.M - 1], np.int64), block])
    ref_rows = oracle.sgemm_rows(p.M, p.N, p.K, p.alpha, p.A, p.B, p.beta, p.C0, rows,
                                 lda=p.lda, ldb=p.ldb, ldc0=p.ldc)
    if dist == "int4":
        assert np.array_equal(got, ref)
        assert np.array_equal(C[rows], ref_rows)
    else:
        A, B, C0 = logical(p)
        den = p.K * float(np.abs(A).max()) * float(np.abs(B).max())
        assert float(np.abs(got.astype(np.float64) - ref).max()) / den <= TOL_FFMA
        assert float(np.abs(C[rows].astype(np.float64) - ref_rows).max()) / den <= TOL_FFMA
        assert np.all(np.isfinite(C))


@pytest.mark.parametrize("path", ["planned", "staged", "tf32x3"])
def test_output_beyond_two_to_the_31_elements(sg, tune, path):
    """A C of 131072 x 16400 = 2.15e9 elements (8.6 GB): row offsets past 2^31
    in every epilogue, 132k output tiles, a ragged last tile column, K shorter
    than one slice.  Integer inputs, so the sampled entries -- both sides of
    the row where the offset crosses 2^31, the last row and column, and
    random ones -- are bit-exact against the oracle.  'planned' takes the
    A^T pass the planner picks here, 'staged' reads A as stored, 'tf32x3' is
    the tensor-core mode."""
    import torch
    M, N, K = 131072, 16400, 24
    assert M * N > 2**31
    A, B = workloads.operands(M, N, K, dist="int4", seed=61)
    if path == "staged":
        tune(transpose_a=0)
    plan = sg.gemm_plan(M, N, K, K, N, N, 0, 0, 0)
    if path == "planned":
        assert plan.transpose_a == 1
    if path == "staged":
        assert plan.transpose_a == 0
    dev = torch.device("cuda", 0)
    Ad = torch.from_numpy(A).to(dev)
    Bd = torch.from_numpy(B).to(dev)
    Cd = torch.full((M * N,), float("nan"), dtype=torch.float32, device=dev)
    try:
        st = torch.cuda.current_stream().cuda_stream
        fn = sg.sgemm_tf32x3_ptr if path == "tf32x3" else sg.sgemm_ptr
        fn(M, N, K, 1.0, Ad.data_ptr(), K, Bd.data_ptr(), N, 0.0, Cd.data_ptr(), N, st)
        torch.cuda.synchronize()
        cross = (2**31) // N                      # the row where i * N passes 2^31
        rows = np.array([0, cross - 1, cross, cross + 1, M - 1], dtype=np.int64)
        ii = np.repeat(rows, 6)
        jj = np.tile(np.array([0, 1, 127, N // 2, N - 2, N - 1], dtype=np.int64), len(rows))
        ri, rj = workloads.sample_indices(M, N, 4000, seed=62)
        ii = np.concatenate([ii, ri])
        jj = np.concatenate([jj, rj])
        got = Cd[torch.from_numpy(ii * N + jj).to(dev)].cpu().numpy()
        last = Cd[(M - 1) * N:].cpu().numpy()
    finally:
        del Cd
        torch.cuda.empty_cache()
    ref = oracle.sgemm_entries(M, N, K, 1.0, A, B, 0.0, None, ii, jj, lda=K, ldb=N)
    assert np.array_equal(got, ref)
    ref_last = oracle.sgemm_rows(M, N, K, 1.0, A, B, 0.0, None, np.array([M - 1]), lda=K, ldb=N)
    assert np.array_equal(last, ref_last.ravel())


def test_transposed_plan_falls_back_when_the_workspace_is_capped(sg, tune):
    """When the workspace for the transposed copy of A cannot be had (here a
    1 MiB cap stands in for a failed allocation), sgemm runs the plan that
    reads A as stored; the tensor mode, which has no such fallback, reports
    SGEMM_ERR_ALLOC and leaves C alone."""
    torch = _torch()
    p = workloads.make(2048, 2048, 512, dist="int4", seed=71, alpha=1.5, beta=0.5,
                       c0_dist="int4")
    assert sg.gemm_plan_for_sms(p.M, p.N, p.K, p.lda, p.ldb, p.ldc).transpose_a == 1
    tune(workspace_limit_mib=1)
    stream = torch.cuda.Stream()     # a stream the library holds no workspace for yet
    A = torch.from_numpy(p.A).cuda()
    B = torch.from_numpy(p.B).cuda()
    C = torch.from_numpy(p.C0).cuda()
    with torch.cuda.stream(stream):
        sg.sgemm_ptr(p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta,
                     C.data_ptr(), p.ldc, stream.cuda_stream)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy()[:, :p.N], oracle.problem(p))
    C2 = torch.from_numpy(p.C0).cuda()
    with pytest.raises(sg.SgemmError) as e:
        sg.sgemm_tf32x3_ptr(p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb,
                            p.beta, C2.data_ptr(), p.ldc, stream.cuda_stream)
    assert e.value.status == 6
    torch.cuda.synchronize()
    assert np.array_equal(C2.cpu().numpy(), p.C0)


@pytest.mark.parametrize("M,N,K,lds,dist", [
    (2048, 1024, 512, None, "uniform"),
    (2046, 1030, 515, (516, 1032, 1036), "uniform"),     # bounds-checked tiles
    (1024, 1536, 768, None, "int4"),
    (1000, 1100, 37, (40, 1104, 1100), "int4"),
])
def test_sixteen_by_eight_kernel(sg, tune, M, N, K, lds, dist):
    """The 16 x 8 per-thread kernel on transposed-A plans (forced)."""
    tune(kernel=2, transpose_a=1, split_k=1, tile=128, schedule=0)
    lda, ldb, ldc = lds if lds else (None, None, None)
    p = workloads.make(M, N, K, dist=dist, seed=67, lda=lda, ldb=ldb, ldc=ldc,
                       alpha=1.5 if dist == "int4" else 0.75, beta=0.5,
                       c0_dist="int4" if dist == "int4" else "uniform")
    plan = sg.gemm_plan_for_sms(p.M, p.N, p.K, p.lda, p.ldb, p.ldc)
    assert plan.transpose_a == 1 and plan.kernel == 2 and plan.bk == 32
    run_and_check(sg, p, exact=dist == "int4")


@pytest.mark.parametrize("M,N,K,lds,beta,dist", [
    (256, 256, 256, None, 0.0, "uniform"),
    (256, 256, 256, None, 0.5, "int4"),
    (100, 70, 33, (35, 70, 71), 1.25, "uniform"),      # unaligned: 4-byte copies
    (31, 33, 1, None, 0.0, "int4"),
    (1000, 900, 256, (257, 903, 901), -0.5, "uniform"),
    (64, 2000, 96, None, 0.0, "int4"),
    (513, 7, 255, None, 2.0, "int4"),
])
def test_small_problem_kernel(sg, tune, M, N, K, lds, beta, dist):
    """The small-problem kernel (forced where the planner would not pick it):
    edges, unaligned operands, beta, exact integers, C's padding untouched."""
    tune(schedule=2)
    lda, ldb, ldc = lds if lds else (None, None, None)
    p = workloads.make(M, N, K, dist=dist, seed=M + N + K, alpha=1.5 if dist == "int4" else 0.75,
                       beta=beta, lda=lda, ldb=ldb, ldc=ldc,
                       c0_dist=("int4" if dist == "int4" else "uniform") if beta else None)
    assert sg.gemm_plan_for_sms(p.M, p.N, p.K, p.lda, p.ldb, p.ldc).schedule == 2
    run_and_check(sg, p, exact=dist == "int4", c_offset=1 if lds else 0)
