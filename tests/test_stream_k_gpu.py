"""GPU parity of the persistent stream-K schedule against the oracle.

Every case forces the stream-K kernel (tuning knob schedule = 1) and varies
what decides its work split: the tile (64 or 128), the fewest K slices a CTA
run may hold (1 and 3 make many CTAs share each tile, so the fixed-order
reduction sums up to 16 contributors), alignment (16-byte and 4-byte
copies), the operand layouts, batches and the fused epilogue.  Tolerances as
everywhere: bit-exact on integer-valued inputs, normalised error <= 1e-6
otherwise; every result is also checked for writes outside C's logical block.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads
from test_ex_gpu import LAYOUTS, ExProblem
from test_parity_gpu import DeviceProblem, run_and_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sg():
    import torch
    import dense_fp32_matrix_06_gb300 as pkg
    pkg.build()
    assert torch.cuda.is_available()
    pkg.load_library()
    return pkg


WORKLOADS = ["square256", "square1024ab", "ragged", "gpt2_qkv", "gpt2_mlp_down"]


@pytest.mark.parametrize("tile", [64, 128])
@pytest.mark.parametrize("min_slices", [None, 1, 3])
@pytest.mark.parametrize("name", WORKLOADS)
def test_configured_workloads(sg, tune, name, tile, min_slices):
    tune(schedule=1, tile=tile, sk_min_slices=min_slices)
    p = workloads.workload(name)
    plan = sg.gemm_plan_for_sms(p.M, p.N, p.K, p.lda, p.ldb, p.ldc)
    assert plan.schedule == 1 and plan.bm == tile
    run_and_check(sg, p)
    q = workloads.workload(name, dist="int4")
    run_and_check(sg, q, exact=True)


@pytest.mark.parametrize("seed", range(16))
def test_shape_fuzz(sg, tune, seed):
    rng = np.random.default_rng(2000 + seed)
    M, N, K = (int(x) for x in rng.integers(1, 400, size=3))
    lda = K + int(rng.integers(0, 6))
    ldb = N + int(rng.integers(0, 6))
    ldc = N + int(rng.integers(0, 6))
    beta = 0.0 if seed % 2 == 0 else float(rng.uniform(-2, 2))
    alpha = float(rng.uniform(-2, 2))
    dist = "int4" if seed % 3 == 0 else "uniform"
    if dist == "int4":
        alpha, beta = 1.5, (0.5 if beta else 0.0)
    tune(schedule=1, tile=(64, 128)[seed % 2], sk_min_slices=(1, 2, None, 5)[seed % 4])
    p = workloads.make(M, N, K, dist=dist, seed=seed, alpha=alpha, beta=beta, lda=lda,
                       ldb=ldb, ldc=ldc, c0_dist=dist if beta else None)
    offs = dict(a_offset=int(seed % 4 == 1), b_offset=int(seed % 5 == 2),
                c_offset=int(seed % 7 == 3))
    run_and_check(sg, p, exact=(dist == "int4"), **offs)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (1, 513, 17), (129, 1, 300), (127, 129, 15),
                                   (3, 5, 4096), (64, 64, 20000), (2500, 2000, 40)])
def test_edge_shapes(sg, tune, M, N, K):
    tune(schedule=1)
    run_and_check(sg, workloads.make(M, N, K, seed=M + N + K))
    run_and_check(sg, workloads.make(M, N, K, dist="int4", seed=M + N + K), exact=True)


def test_whole_k_rounds_then_stream_k(sg, tune):
    """Grids of more than two waves: whole-K rounds first, stream-K after."""
    tune(schedule=1, tile=128)
    p = workloads.make(2560, 4096, 96, dist="int4", seed=81, alpha=1.5, beta=0.5,
                       c0_dist="int4")
    plan = sg.gemm_plan_for_sms(p.M, p.N, p.K, p.lda, p.ldb, p.ldc)
    assert plan.dp_rounds >= 1 and plan.sk_iters > 0
    run_and_check(sg, p, exact=True)


def test_runs_are_bit_identical_and_workspace_reusable(sg, tune):
    """The fix-up order is fixed, so repeated runs agree bit for bit; and
    plans of other shapes that reuse the same workspace right after, over
    whatever partials the previous call left there, are right too."""
    tune(schedule=1, tile=128, sk_min_slices=2)
    p = workloads.workload("square1024ab")
    outs = []
    for _ in range(3):
        d = DeviceProblem(p)
        d.run(sg)
        outs.append(d.result()[0])
        run_and_check(sg, workloads.make(300, 200, 900, seed=5, dist="int4"), exact=True)
    assert all(np.array_equal(outs[0].view(np.uint32), o.view(np.uint32)) for o in outs[1:])


@pytest.mark.parametrize("op_a,op_b", LAYOUTS)
@pytest.mark.parametrize("tile", [64, 128])
def test_layouts_batches_and_epilogue(sg, tune, op_a, op_b, tile):
    tune(schedule=1, tile=tile, sk_min_slices=3)
    p = ExProblem(op_a, op_b, 150, 130, 270, 3, seed=91, alpha=0.75, beta=0.5)
    p.check(p.run(sg), exact=False)
    q = ExProblem(op_a, op_b, 256, 256, 128, 2, seed=92, dist="int4", alpha=1.5, beta=0.5,
                  bias=True, pad=0)
    q.check(q.run(sg), exact=True)
    r = ExProblem(op_a, op_b, 200, 96, 300, 2, seed=93, bias=True, act=1, shared_b=True)
    r.check(r.run(sg), exact=False)


def test_attention_shapes(sg, tune):
    """GPT-2 attention products: Q K^T (op N/T, 64 deep) and P V (N = 64)."""
    tune(schedule=1)
    qk = ExProblem(0, 1, 1024, 1024, 64, 2, seed=94, pad=0)
    qk.check(qk.run(sg), exact=False)
    pv = ExProblem(0, 0, 1024, 64, 1024, 2, seed=95, dist="int4", pad=0)
    pv.check(pv.run(sg), exact=True)


def test_noalloc_runs_stream_k_plans(sg, tune):
    """sgemm_noalloc runs stream-K plans in its own scratch, twice in a row,
    over the partials the previous call left there."""
    import torch
    tune(schedule=1, sk_min_slices=2)
    p = workloads.workload("square1024ab", dist="int4")
    A = torch.from_numpy(p.A).cuda()
    B = torch.from_numpy(p.B).cuda()
    ref = oracle.problem(p)
    for _ in range(2):
        C = torch.from_numpy(p.C0).cuda()
        sg.sgemm_noalloc_ptr(p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb,
                             p.beta, C.data_ptr(), p.ldc, torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert np.array_equal(C.cpu().numpy()[:, :p.N], ref)


@pytest.mark.parametrize("M,N,K,lds,dist", [
    (1024, 1024, 1024, None, "uniform"),
    (2046, 1030, 515, (516, 1032, 1036), "uniform"),     # bounds-checked tiles
    (1024, 1536, 768, None, "int4"),
    (256, 256, 4096, None, "int4"),                      # few tiles: long stream-K runs
])
def test_transposed_a_then_stream_k(sg, tune, M, N, K, lds, dist):
    """A transposed first, then the stream-K kernel with both operands
    copied directly (K slices of 32, three pages)."""
    tune(schedule=1, tile=128, transpose_a=1)
    lda, ldb, ldc = lds if lds else (None, None, None)
    p = workloads.make(M, N, K, dist=dist, seed=97, lda=lda, ldb=ldb, ldc=ldc,
                       alpha=1.5 if dist == "int4" else 0.75, beta=0.5,
                       c0_dist="int4" if dist == "int4" else "uniform")
    plan = sg.gemm_plan_for_sms(p.M, p.N, p.K, p.lda, p.ldb, p.ldc)
    assert plan.transpose_a == 1 and plan.schedule == 1 and plan.bk == 32
    run_and_check(sg, p, exact=dist == "int4")


@pytest.mark.parametrize("transpose_a", [0, 1])
def test_stream_k_plan_with_caller_workspace(sg, tune, transpose_a):
    """gemm_plan + sgemm_with_plan on a stream-K plan, with a caller-owned
    workspace that starts as garbage, used for three calls in a row."""
    import torch
    tune(schedule=1, tile=128, transpose_a=transpose_a, sk_min_slices=2)
    p = workloads.make(1024, 1280, 1536, dist="int4", seed=98, alpha=1.5, beta=0.5,
                       c0_dist="int4")
    A = torch.from_numpy(p.A).cuda()
    B = torch.from_numpy(p.B).cuda()
    plan = sg.gemm_plan(p.M, p.N, p.K, p.lda, p.ldb, p.ldc, A.data_ptr(), B.data_ptr(),
                        A.data_ptr())
    assert plan.schedule == 1 and plan.transpose_a == transpose_a and plan.sk_iters > 0
    ws = torch.full((plan.workspace_bytes,), 0xFF, dtype=torch.uint8, device="cuda")
    ref = oracle.problem(p)
    for _ in range(3):
        C = torch.from_numpy(p.C0).cuda()
        sg.sgemm_with_plan_ptr(plan, p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(),
                               p.ldb, p.beta, C.data_ptr(), p.ldc, ws.data_ptr(),
                               plan.workspace_bytes, torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert np.array_equal(C.cpu().numpy()[:, :p.N], ref)
    # stream-K takes no tickets: the counter block is never written
    assert bool((ws[:sg.WORKSPACE_COUNTER_BYTES] == 0xFF).all())
