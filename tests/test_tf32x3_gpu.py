"""GPU parity of the 3xTF32 tensor-core mode (sgemm_tf32x3) against the oracle.

Tolerance for this mode: max|C - C_oracle| / (K*max|A|*max|B| + |beta|*max|C0|)
<= 1e-5; bit-exact on integer-valued inputs (their TF32 low parts are zero and
every partial sum is an integer below 2^24).  Also: the bounded device-side
waits expire cleanly when the operand loads are withheld.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

TOL_TF32X3 = 1e-5
SENTINEL = np.float32(-12345.5)


@pytest.fixture(scope="module")
def sg():
    import torch
    import dense_fp32_matrix_06_gb300 as pkg
    pkg.build()
    assert torch.cuda.is_available()
    pkg.load_library()
    return pkg


def run(sg, p, a_offset=0, c_offset=0):
    """Run the mode on a workloads.Problem; returns (logical C, whole C buffer, C buffer before)."""
    import torch
    dev = torch.device("cuda")
    a_buf = torch.from_numpy(np.concatenate([np.zeros(a_offset, np.float32), p.A.ravel()])).to(dev)
    b_buf = torch.from_numpy(p.B.ravel().copy()).to(dev)
    guard = 32 + c_offset
    c_host = np.full(guard + p.C0.size + 32, SENTINEL, np.float32)
    c_host[guard:guard + p.C0.size] = p.C0.ravel()
    c_buf = torch.from_numpy(c_host.copy()).to(dev)
    stream = torch.cuda.current_stream().cuda_stream
    sg.sgemm_tf32x3_ptr(p.M, p.N, p.K, p.alpha, a_buf.data_ptr() + 4 * a_offset, p.lda,
                        b_buf.data_ptr(), p.ldb, p.beta, c_buf.data_ptr() + 4 * guard, p.ldc,
                        stream)
    assert sg.device_status(stream) == 0
    buf = c_buf.cpu().numpy()
    C = buf[guard:guard + p.C0.size].reshape(p.C0.shape)
    # nothing outside the logical M x N block changed
    mask = np.ones(p.C0.shape, bool)
    mask[:, :p.N] = False
    assert np.array_equal(C[mask].view(np.uint32), p.C0[mask].view(np.uint32))
    assert np.array_equal(buf[:guard].view(np.uint32), c_host[:guard].view(np.uint32))
    tail = guard + p.C0.size
    assert np.array_equal(buf[tail:].view(np.uint32), c_host[tail:].view(np.uint32))
    return C[:, :p.N].copy()


def check(p, C, exact):
    ref = oracle.problem(p)
    if exact:
        assert np.array_equal(C, ref), f"{p.name}: not bit-exact"
    else:
        C0 = p.C0[:, :p.N] if p.beta != 0 else None
        err = oracle.normalised_error(C, ref, p.K, p.A[:, :p.K], p.B[:, :p.N], p.beta, C0)
        assert err <= TOL_TF32X3, f"{p.name}: normalised error {err:.3e}"


SMALL = ["square256", "square256_int", "square1024ab", "ragged", "gpt2_qkv", "gpt2_mlp_up",
         "gpt2_mlp_down"]


@pytest.mark.parametrize("name", SMALL)
def test_workload_parity(sg, name):
    p = workloads.workload(name)
    check(p, run(sg, p), exact=p.meta["dist"] == "int4")


@pytest.mark.parametrize("name", SMALL)
def test_workload_integer_copy_bit_exact(sg, name):
    M, N, K, _, seed, alpha, beta, _ = workloads.WORKLOADS[name]
    p = workloads.make(M, N, K, dist="int4", seed=seed, alpha=alpha, beta=beta, c0_dist="int4")
    check(p, run(sg, p), exact=True)


@pytest.mark.parametrize("seed", range(12))
def test_shape_fuzz(sg, seed):
    rng = np.random.default_rng(2000 + seed)
    M, N, K = (int(x) for x in rng.integers(1, 400, size=3))
    lda = K + int(rng.integers(0, 5))
    ldb = N + int(rng.integers(0, 5))
    ldc = N + int(rng.integers(0, 5))
    beta = 0.0 if seed % 2 == 0 else float(rng.uniform(-2, 2))
    dist = "int4" if seed % 3 == 0 else "uniform"
    alpha = 1.5 if dist == "int4" else float(rng.uniform(-2, 2))
    if dist == "int4" and beta:
        beta = 0.5
    p = workloads.make(M, N, K, dist=dist, seed=seed, alpha=alpha, beta=beta, lda=lda, ldb=ldb,
                       ldc=ldc, c0_dist=dist if beta else None)
    check(p, run(sg, p, a_offset=seed % 2, c_offset=seed % 3), exact=dist == "int4")


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (1, 300, 33), (257, 1, 64), (128, 256, 32),
                                   (129, 257, 31), (64, 64, 4096)])
def test_edge_shapes(sg, M, N, K):
    check(workloads.make(M, N, K, seed=M + N + K),
          run(sg, workloads.make(M, N, K, seed=M + N + K)), exact=False)
    q = workloads.make(M, N, K, dist="int4", seed=M + N + K + 1)
    check(q, run(sg, q), exact=True)


def test_beta_zero_alpha_zero_k_zero(sg):
    p = workloads.make(200, 150, 70, seed=21)        # C0 is NaN; beta = 0 must not read it
    C = run(sg, p)
    assert np.all(np.isfinite(C))
    check(p, C, exact=False)
    q = workloads.make(130, 140, 50, seed=22, beta=0.75, c0_dist="uniform")
    q.A[:, :q.K] = np.nan
    q.alpha = 0.0
    assert np.array_equal(run(sg, q), oracle.problem(q))
    r = workloads.make(64, 96, 0, seed=23, beta=-0.5, c0_dist="uniform")
    assert np.array_equal(run(sg, r), oracle.problem(r))


@pytest.mark.parametrize("split", ["2", "3", "5", "16"])
def test_forced_split(sg, tune, split):
    tune(tf32x3_split=split)
    p = workloads.make(300, 520, 1000, seed=31, beta=0.5, c0_dist="uniform", alpha=0.75)
    check(p, run(sg, p), exact=False)
    q = workloads.make(256, 256, 320, dist="int4", seed=32, alpha=1.5, beta=0.5, c0_dist="int4")
    check(q, run(sg, q), exact=True)        # 10 K blocks: split 16 leaves empty ranges


@pytest.mark.parametrize("fuse", ["0", "1"])
@pytest.mark.parametrize("name", ["square1024ab", "ragged", "gpt2_mlp_down", "long_k",
                                  "square256_int"])
def test_both_splits_of_a(sg, tune, name, fuse):
    """A split in the kernel (default when its stride allows TMA) or by a pre-pass
    (SGEMM_TF32X3_FUSE_A=0)."""
    tune(tf32x3_fuse_a=fuse)
    p = workloads.workload(name)
    check(p, run(sg, p), exact=p.meta["dist"] == "int4")
    q = workloads.make(200, 300, 72, dist="int4", seed=81, alpha=1.5, beta=0.5, c0_dist="int4")
    check(q, run(sg, q), exact=True)


def test_prepass_split_bounded_waits(sg, tune):
    """The same bounded-wait check on the pre-pass kernel."""
    import torch
    tune(tf32x3_fuse_a="0")
    M, N, K = 256, 512, 128
    A = torch.ones((M, K), device="cuda")
    B = torch.ones((K, N), device="cuda")
    C = torch.full((M, N), 3.0, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = sg.tf32x3_stall_selftest(M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N,
                                  20000, stream)
    assert rc == 5
    assert bool((C == 3.0).all())
    assert sg.device_status(stream) == 0


@pytest.mark.parametrize("tail", ["0", "2", "3"])
def test_tail_split(sg, tune, tail):
    """Only the last, partly filled wave of tiles cut along K (2048 x 2560: 160
    tiles of 128 x 256, 8 of them past the first wave on 152 SMs)."""
    tune(tf32x3_tail=tail)
    p = workloads.make(2048, 2560, 1000, seed=91, alpha=0.75, beta=0.5, c0_dist="uniform")
    check(p, run(sg, p), exact=False)
    q = workloads.make(2048, 2560, 800, dist="int4", seed=92, alpha=1.5, beta=0.5,
                       c0_dist="int4")
    check(q, run(sg, q), exact=True)


def test_split_plans_for_small_grids(sg):
    # these run with more K ranges than tiles; parity at full size
    for name in ("long_k", "gpt2_mlp_down", "square1024ab"):
        p = workloads.workload(name)
        check(p, run(sg, p), exact=False)


def test_deterministic(sg):
    p = workloads.workload("long_k")
    first = run(sg, p)
    for _ in range(2):
        assert np.array_equal(run(sg, p).view(np.uint32), first.view(np.uint32))


@pytest.mark.parametrize("name", ["square8192", "skinny_k64", "long_k", "square2048"])
@pytest.mark.parametrize("dist", ["uniform", "int4"])
def test_large_sampled(sg, name, dist):
    import torch
    p = workloads.workload(name, dist=None if dist == "uniform" else dist)
    A = torch.from_numpy(p.A).cuda()
    B = torch.from_numpy(p.B).cuda()
    C = torch.full((p.M, p.ldc), float("nan"), device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    sg.sgemm_tf32x3_ptr(p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb,
                        p.beta, C.data_ptr(), p.ldc, stream)
    assert sg.device_status(stream) == 0
    Ch = C.cpu().numpy()
    ii, jj = workloads.sample_indices(p.M, p.N, 3000, seed=9)
    ref = oracle.sgemm_entries(p.M, p.N, p.K, p.alpha, p.A, p.B, p.beta, p.C0, ii, jj,
                               lda=p.lda, ldb=p.ldb, ldc0=p.ldc)
    rows = np.array([0, p.M // 3, p.M - 1], np.int64)
    ref_rows = oracle.sgemm_rows(p.M, p.N, p.K, p.alpha, p.A, p.B, p.beta, p.C0, rows,
                                 lda=p.lda, ldb=p.ldb, ldc0=p.ldc)
    assert np.all(np.isfinite(Ch[:, :p.N]))
    if dist == "int4":
        assert np.array_equal(Ch[ii, jj], ref)
        assert np.array_equal(Ch[rows, :p.N], ref_rows)
    else:
        den = p.K * float(np.abs(p.A[:, :p.K]).max()) * float(np.abs(p.B[:, :p.N]).max())
        assert float(np.abs(Ch[ii, jj].astype(np.float64) - ref).max()) / den <= TOL_TF32X3
        assert float(np.abs(Ch[rows, :p.N].astype(np.float64) - ref_rows).max()) / den \
            <= TOL_TF32X3


def test_split_k_after_tensor_mode_on_the_same_stream(sg):
    """Both modes use the library's per-stream workspace; the tensor mode must
    leave the split-K tile counters zero."""
    import torch
    stream = torch.cuda.current_stream().cuda_stream
    p = workloads.workload("long_k")           # FFMA plan whose tiles share K ranges
    A = torch.from_numpy(p.A).cuda()
    B = torch.from_numpy(p.B).cuda()
    C = torch.full((p.M, p.N), float("nan"), device="cuda")
    plan = sg.gemm_plan(p.M, p.N, p.K, p.lda, p.ldb, p.ldc, A.data_ptr(), B.data_ptr(),
                        C.data_ptr())
    assert plan.split_k > 1 or plan.sk_iters > 0

    def ffma():
        sg.sgemm_ptr(p.M, p.N, p.K, 1.0, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, 0.0,
                     C.data_ptr(), p.N, stream)

    ffma()                                     # grows the workspace first
    run(sg, workloads.workload("square1024ab"))   # tensor mode reuses it (16 MB)
    C.fill_(float("nan"))
    ffma()                                     # counters must still be zero
    torch.cuda.synchronize()
    Ch = C.cpu().numpy()
    assert np.all(np.isfinite(Ch))
    ii, jj = workloads.sample_indices(p.M, p.N, 2000, seed=3)
    ref = oracle.sgemm_entries(p.M, p.N, p.K, 1.0, p.A, p.B, 0.0, None, ii, jj, lda=p.lda,
                               ldb=p.ldb)
    den = p.K * float(np.abs(p.A).max()) * float(np.abs(p.B).max())
    assert float(np.abs(Ch[ii, jj].astype(np.float64) - ref).max()) / den <= 1e-6


def test_bounded_waits_expire_cleanly(sg):
    """The operand loads are withheld, so every wait runs out after 20 ms: the
    call reports SGEMM_ERR_TIMEOUT, C is untouched, and the context stays
    usable for the next (normal) call."""
    import torch
    M, N, K = 256, 512, 128
    A = torch.ones((M, K), device="cuda")
    B = torch.ones((K, N), device="cuda")
    C = torch.full((M, N), 3.0, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = sg.tf32x3_stall_selftest(M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N,
                                  20000, stream)
    assert rc == 5   # SGEMM_ERR_TIMEOUT
    assert bool((C == 3.0).all())
    assert sg.device_status(stream) == 0   # the record was cleared
    sg.sgemm_tf32x3_ptr(M, N, K, 1.0, A.data_ptr(), K, B.data_ptr(), N, 0.0, C.data_ptr(), N,
                        stream)
    assert sg.device_status(stream) == 0
    assert bool((C == float(K)).all())


@pytest.mark.parametrize("fuse", ["0", "1"])
@pytest.mark.parametrize("M,N,K", [(1024, 768, 3072), (300, 520, 1000), (128, 256, 32),
                                   (1, 33, 7), (1024, 1024, 16384)])
def test_packed_b_reused_for_two_a(sg, tune, M, N, K, fuse):
    import torch
    tune(tf32x3_fuse_a=fuse)
    stream = torch.cuda.current_stream().cuda_stream
    lda = (K + 3) // 4 * 4          # the packed call needs a 16-byte row stride for A
    p1 = workloads.make(M, N, K, seed=71, beta=0.5, c0_dist="uniform", alpha=1.25, lda=lda)
    p2 = workloads.make(M, N, K, seed=72, lda=lda)
    B = torch.from_numpy(p1.B).cuda()
    nbytes = sg.tf32x3_packed_b_bytes(K, N)
    assert nbytes >= 2 * N * K * 4
    packed = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    sg.tf32x3_pack_b_ptr(K, N, B.data_ptr(), p1.ldb, packed.data_ptr(), nbytes, stream)
    for p in (p1, p2):
        p.B = p1.B                       # both products use the packed B
        A = torch.from_numpy(p.A).cuda()
        C = torch.from_numpy(p.C0).cuda()
        sg.sgemm_tf32x3_packed_ptr(p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, packed.data_ptr(),
                                   p.beta, C.data_ptr(), p.ldc, stream)
        assert sg.device_status(stream) == 0
        check(p, C.cpu().numpy()[:, :p.N], exact=False)


def test_packed_b_integer_exact_and_errors(sg):
    import torch
    stream = torch.cuda.current_stream().cuda_stream
    p = workloads.make(257, 300, 96, dist="int4", seed=73, alpha=1.5, beta=0.5, c0_dist="int4")
    B = torch.from_numpy(p.B).cuda()
    nbytes = sg.tf32x3_packed_b_bytes(p.K, p.N)
    packed = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    sg.tf32x3_pack_b_ptr(p.K, p.N, B.data_ptr(), p.ldb, packed.data_ptr(), nbytes, stream)
    A = torch.from_numpy(p.A).cuda()
    C = torch.from_numpy(p.C0).cuda()
    sg.sgemm_tf32x3_packed_ptr(p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, packed.data_ptr(),
                               p.beta, C.data_ptr(), p.ldc, stream)
    check(p, C.cpu().numpy()[:, :p.N], exact=True)
    with pytest.raises(sg.SgemmError) as e:        # A not 16-byte aligned
        sg.sgemm_tf32x3_packed_ptr(p.M, p.N, p.K, 1.0, A.data_ptr() + 4, p.lda, packed.data_ptr(),
                                   0.0, C.data_ptr(), p.ldc, stream)
    assert e.value.status == 2
    with pytest.raises(sg.SgemmError) as e:        # packed buffer too small
        sg.tf32x3_pack_b_ptr(p.K, p.N, B.data_ptr(), p.ldb, packed.data_ptr(), nbytes - 4, stream)
    assert e.value.status == 7
    assert sg.tf32x3_packed_b_bytes(0, 5) == 0


def test_torch_api(sg):
    import torch
    p = workloads.make(300, 200, 150, seed=41, lda=160, ldb=210)
    A = torch.from_numpy(p.A).cuda()[:, :p.K]
    B = torch.from_numpy(p.B).cuda()[:, :p.N]
    C = sg.sgemm_tf32x3(A, B)
    torch.cuda.synchronize()
    check(p, C.cpu().numpy(), exact=False)
    with pytest.raises(ValueError):
        sg.sgemm_tf32x3(A, B[:-1])


@pytest.mark.parametrize("fuse", ["0", "1"])
@pytest.mark.parametrize("split", [None, "3"])
@pytest.mark.parametrize("M,N,K,dist", [
    (1024, 2304, 768, "gpt2"), (1023, 777, 513, "uniform"), (300, 260, 1000, "int4"),
    (129, 257, 31, "uniform"), (1024, 768, 3072, "int4"),
])
def test_narrow_tiles(sg, tune, M, N, K, dist, split, fuse):
    """128-wide tensor tiles (forced): A split in the kernel and by a pre-pass,
    with and without split-K."""
    tune(tf32x3_bn=128, tf32x3_split=split, tf32x3_fuse_a=fuse)
    p = workloads.make(M, N, K, dist=dist, seed=M + K, alpha=1.5 if dist == "int4" else 0.75,
                       beta=0.5, c0_dist="int4" if dist == "int4" else "uniform")
    check(p, run(sg, p, c_offset=1), exact=dist == "int4")


@pytest.mark.parametrize("fuse", ["1", "0"])
def test_non_finite_inputs(sg, tune, fuse):
    """The split cannot carry an infinity: x_hi = inf leaves x_lo = tf32(inf - inf)
    = NaN, and even with x_lo = 0 the term x_hi * y_lo is inf * 0 wherever y is
    exact in TF32.  So the tensor mode returns NaN where fp32 gives +-inf -- a
    non-finite value, never a finite one -- and NaN exactly where fp32 gives
    NaN; entries no special value reaches keep the mode's tolerance."""
    import dataclasses
    tune(tf32x3_fuse_a=fuse)
    p = workloads.make(300, 260, 1000, seed=72, beta=0.5, c0_dist="uniform")
    A = p.A.copy()
    B = p.B.copy()
    A[5, 17] = np.inf
    A[9, 3] = -np.inf
    A[40, 60] = np.nan
    B[100, 7] = np.nan
    p = dataclasses.replace(p, A=A, B=B)
    C = run(sg, p)
    ref = oracle.problem(p)
    assert np.isinf(ref[5]).any() and np.isinf(ref[9]).any() and np.isnan(ref[40]).all()
    assert np.all(np.isnan(C[np.isnan(ref)]))
    assert not np.isfinite(C[np.isinf(ref)]).any()
    fin = np.isfinite(ref)
    assert np.isfinite(C[fin]).all()
    keep = np.ones(p.M, bool)
    keep[[5, 9, 40]] = False
    cols = np.ones(p.N, bool)
    cols[7] = False
    sub = np.ix_(keep, cols)
    Af = np.where(np.isfinite(A[:, :p.K]), A[:, :p.K], 0)
    Bf = np.where(np.isfinite(B[:, :p.N]), B[:, :p.N], 0)
    den = p.K * float(np.abs(Af).max()) * float(np.abs(Bf).max()) + 0.5 * float(
        np.abs(p.C0[:, :p.N]).max())
    assert float(np.abs(C[sub].astype(np.float64) - ref[sub]).max()) / den <= TOL_TF32X3
