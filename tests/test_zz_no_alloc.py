"""sgemm_noalloc: the GEMM for callers that must not allocate device memory.

Some callers cannot let a library call cudaMalloc -- for example a plugin
inside a framework that reserved the GPU's memory up front, or a latency-bound
loop where an allocation could stall the device.  sgemm_noalloc serves them by
taking its split-K scratch from a fixed buffer inside the library.

These tests call it through the C ABI and compare it with sgemm on two calls
in a row (the second call sees the scratch the first one left behind), and
check that a shape needing more scratch than the buffer holds is refused
before anything runs.  The file is named to be collected last.
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


@pytest.mark.parametrize("name", ["long_k", "square1024ab", "gpt2_mlp_down", "ragged",
                                  "square256"])
def test_noalloc_matches_sgemm_on_two_calls(sg, name):
    import torch
    p = workloads.workload(name)
    A, B, C0 = _device_problem(p)
    stream = torch.cuda.current_stream().cuda_stream
    # sgemm_noalloc never plans a transposed copy of A (it would need M x K
    # floats of scratch), so its split-K scratch is that of the plan without it
    import os
    old = os.environ.get("SGEMM_FORCE_TRANSPOSE_A")
    os.environ["SGEMM_FORCE_TRANSPOSE_A"] = "0"
    try:
        plan = sg.gemm_plan(p.M, p.N, p.K, p.lda, p.ldb, p.ldc, A.data_ptr(), B.data_ptr(),
                            C0.data_ptr())
    finally:
        if old is None:
            del os.environ["SGEMM_FORCE_TRANSPOSE_A"]
        else:
            os.environ["SGEMM_FORCE_TRANSPOSE_A"] = old
    assert plan.transpose_a == 0
    assert plan.workspace_bytes <= sg.NOALLOC_SCRATCH_BYTES

    C_ref = C0.clone()
    sg.sgemm_ptr(p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta,
                 C_ref.data_ptr(), p.ldc, stream)
    torch.cuda.synchronize()
    ref = C_ref.cpu().numpy()[:, :p.N]

    A_log, B_log = p.A[:, :p.K], p.B[:, :p.N]
    C0_log = p.C0[:, :p.N] if p.beta != 0 else None
    for call in range(2):
        C = C0.clone()
        sg.sgemm_noalloc_ptr(p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb,
                             p.beta, C.data_ptr(), p.ldc, stream)
        torch.cuda.synchronize()
        got_full = C.cpu().numpy()
        got = got_full[:, :p.N]
        err = oracle.normalised_error(got, ref, p.K, A_log, B_log, p.beta, C0_log)
        assert err <= TOL_FFMA, f"{name} call {call}: normalised error {err:.3e}"
        # columns past N (the padding of each row) stay untouched
        assert np.array_equal(got_full[:, p.N:].view(np.uint32),
                              p.C0[:, p.N:].view(np.uint32))


def test_noalloc_refuses_shapes_beyond_its_scratch(sg, monkeypatch):
    import torch
    monkeypatch.setenv("SGEMM_FORCE_SPLIT", "32")
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
