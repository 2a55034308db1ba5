"""sgemm_noalloc: the GEMM for callers that must not allocate device memory.

Some callers cannot let a library call cudaMalloc -- for example a plugin
inside a framework that reserved the GPU's memory up front, or a latency-bound
loop where an allocation could stall the device.  sgemm_noalloc serves them by
taking its split-K scratch from a fixed buffer inside the library.

These tests call it through the C ABI, twice in a row on the same inputs (the
second call finds in the shared buffer whatever the first one left), and
check each result against the CPU oracle: bit-exact on integer-valued inputs,
within the normalised 1e-6 bound otherwise.  Each call must also equal, bit
for bit, sgemm's result under the same plan (sgemm with the transposed-A copy
turned off, which is the only plan sgemm_noalloc runs).  A shape that needs
more scratch than the buffer holds is refused before anything runs.

The file name sorts after every other test file on purpose: pytest collects
files in name order, so a run that stops at the first failure (-x) has
already run every other test by the time it gets here.  The tests here pass
on their own in a fresh process as well.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

TOL_FFMA = 1e-6


@pytest.fixture(scope="module")
def sg():
    import torch
    import dense_fp32_matrix_06_gb300 as pkg
    pkg.build()
    assert torch.cuda.is_available()
    pkg.load_library()
    return pkg


def _device_problem(p):
    import torch
    A = torch.from_numpy(p.A).cuda()
    B = torch.from_numpy(p.B).cuda()
    C0 = torch.from_numpy(p.C0).cuda()
    return A, B, C0


def _check_against_oracle(p, got, ref, exact, what):
    if exact:
        assert np.array_equal(got, ref), f"{what}: not bit-exact on integer inputs"
    else:
        C0 = p.C0[:, :p.N] if p.beta != 0 else None
        err = oracle.normalised_error(got, ref, p.K, p.A[:, :p.K], p.B[:, :p.N], p.beta, C0)
        assert err <= TOL_FFMA, f"{what}: normalised error {err:.3e}"


def _two_calls(sg, tune, p, exact, expect_split=None):
    import torch
    A, B, C0 = _device_problem(p)
    stream = torch.cuda.current_stream().cuda_stream
    # the plan sgemm_noalloc runs: sgemm's, without the transposed copy of A
    tune(transpose_a=0)
    plan = sg.gemm_plan(p.M, p.N, p.K, p.lda, p.ldb, p.ldc, A.data_ptr(), B.data_ptr(),
                        C0.data_ptr())
    assert plan.transpose_a == 0
    assert plan.workspace_bytes <= sg.NOALLOC_SCRATCH_BYTES
    if expect_split is not None:
        assert expect_split(plan), sg.GemmPlan.as_dict(plan)

    C_ref = C0.clone()
    sg.sgemm_ptr(p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta,
                 C_ref.data_ptr(), p.ldc, stream)
    torch.cuda.synchronize()
    same_plan = C_ref.cpu().numpy()

    ref = oracle.problem(p)
    for call in range(2):
        C = C0.clone()
        sg.sgemm_noalloc_ptr(p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb,
                             p.beta, C.data_ptr(), p.ldc, stream)
        torch.cuda.synchronize()
        got_full = C.cpu().numpy()
        _check_against_oracle(p, got_full[:, :p.N], ref, exact, f"{p.name} call {call}")
        # bit for bit what sgemm gives under the same plan
        assert np.array_equal(got_full.view(np.uint32), same_plan.view(np.uint32)), \
            f"{p.name} call {call}: differs from sgemm under the same plan"
        # columns past N (the padding of each row) stay untouched
        assert np.array_equal(got_full[:, p.N:].view(np.uint32),
                              p.C0[:, p.N:].view(np.uint32))


@pytest.mark.parametrize("name", ["long_k", "square1024ab", "gpt2_mlp_down", "ragged",
                                  "square256"])
def test_noalloc_matches_oracle_on_two_calls(sg, tune, name):
    _two_calls(sg, tune, workloads.workload(name), exact=False)


@pytest.mark.parametrize("name", ["square1024ab", "long_k", "ragged"])
def test_noalloc_bit_exact_on_integer_inputs(sg, tune, name):
    p = workloads.workload(name, dist="int4")   # C0 (when read) is integer-valued too
    _two_calls(sg, tune, p, exact=True)


def test_noalloc_tail_split(sg, tune):
    """Only the tiles of the last partial wave cut along K: their partial
    tiles sit at the start of the buffer's partial area."""
    tune(tail_split=4)
    p = workloads.make(2560, 2048, 1024, dist="int4", seed=51, alpha=1.5, beta=0.5,
                       c0_dist="int4", name="tail_int4")
    _two_calls(sg, tune, p, exact=True,
               expect_split=lambda q: q.tail_split == 4 and q.tail_start < q.tiles_m * q.tiles_n)
    q = workloads.make(2560, 2048, 1040, seed=52, alpha=0.75, beta=0.5, c0_dist="uniform",
                       name="tail_float")
    _two_calls(sg, tune, q, exact=False, expect_split=lambda r: r.tail_split == 4)


def test_noalloc_refuses_shapes_beyond_its_scratch(sg, tune):
    import torch
    tune(split_k=32)
    M, N, K = 2048, 2048, 8192
    plan = sg.gemm_plan(M, N, K, K, N, N)
    assert plan.workspace_bytes > sg.NOALLOC_SCRATCH_BYTES
    A = torch.zeros((M, K), device="cuda")
    B = torch.zeros((K, N), device="cuda")
    C = torch.full((M, N), 7.0, device="cuda")
    with pytest.raises(sg.SgemmError) as e:
        sg.sgemm_noalloc_ptr(M, N, K, 1.0, A.data_ptr(), K, B.data_ptr(), N, 0.0, C.data_ptr(),
                             N, torch.cuda.current_stream().cuda_stream)
    assert e.value.status == 7   # SGEMM_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert bool((C == 7.0).all())
