"""GPU parity of sgemm_ex (batched, transposed views, fused bias/GELU) against
the oracle's general form.

Tolerance: max|C - C_oracle| / (K*max|op(A)|*max|op(B)| + |beta|*max|C0| +
max|bias|) <= 1e-6 (one fp32 rounding for the bias add and a few ulp for the
GELU sit far inside it); integer inputs without GELU are bit-exact.
"""
from __future__ import annotations

import itertools

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

TOL = 1e-6
SENTINEL = np.float32(-4321.25)


@pytest.fixture(scope="module")
def sg():
    import torch
    import dense_fp32_matrix_06_gb300 as pkg
    pkg.build()
    assert torch.cuda.is_available()
    pkg.load_library()
    return pkg


class ExProblem:
    def __init__(self, op_a, op_b, M, N, K, batch, *, seed, dist="uniform", alpha=1.0, beta=0.0,
                 bias=False, act=0, pad=3, shared_b=False, aligned=False):
        rng = np.random.default_rng(seed)
        draw = (lambda s: rng.integers(-4, 5, s).astype(np.float32)) if dist == "int4" else \
            (lambda s: rng.uniform(-1, 1, s).astype(np.float32))
        self.op_a, self.op_b, self.M, self.N, self.K, self.batch = op_a, op_b, M, N, K, batch
        self.alpha, self.beta, self.act = alpha, beta, act
        ra, ca = (K, M) if op_a else (M, K)
        rb, cb = (N, K) if op_b else (K, N)
        if aligned:   # every row and batch starts on 16 bytes (the vector paths)
            up = lambda x: (x + 3) // 4 * 4
            self.lda, self.ldb, self.ldc = up(ca) + pad, up(cb) + pad, up(N) + pad
            self.sa = ra * self.lda
            self.sb = 0 if shared_b else rb * self.ldb
            self.sc = M * self.ldc
        else:
            self.lda, self.ldb, self.ldc = ca + pad, cb + pad, N + pad
            self.sa = ra * self.lda + 5
            self.sb = 0 if shared_b else rb * self.ldb + 7
            self.sc = M * self.ldc + 2
        self.A = np.full(self.sa * batch + 8, SENTINEL, np.float32)
        self.B = np.full(max(self.sb * batch, rb * self.ldb) + 8, SENTINEL, np.float32)
        self.C0 = np.full(self.sc * batch + 8, SENTINEL, np.float32)
        for b in range(batch):
            self.A[b * self.sa:b * self.sa + ra * self.lda].reshape(ra, self.lda)[:, :ca] = draw((ra, ca))
            if not shared_b or b == 0:
                self.B[b * self.sb:b * self.sb + rb * self.ldb].reshape(rb, self.ldb)[:, :cb] = draw((rb, cb))
            self.C0[b * self.sc:b * self.sc + M * self.ldc].reshape(M, self.ldc)[:, :N] = \
                draw((M, N)) if beta != 0 else np.nan
        self.bias = draw((N,)) if bias else None

    def views(self):
        """(op(A) logical values, op(B), C0) stacked over batches, for the error scale."""
        a, b, c = [], [], []
        ra, ca = (self.K, self.M) if self.op_a else (self.M, self.K)
        rb, cb = (self.N, self.K) if self.op_b else (self.K, self.N)
        for i in range(self.batch):
            a.append(self.A[i * self.sa:i * self.sa + ra * self.lda].reshape(ra, self.lda)[:, :ca])
            b.append(self.B[i * self.sb:i * self.sb + rb * self.ldb].reshape(rb, self.ldb)[:, :cb])
            c.append(self.C0[i * self.sc:i * self.sc + self.M * self.ldc].reshape(self.M, self.ldc)[:, :self.N])
        return np.stack(a), np.stack(b), np.stack(c)

    def oracle(self):
        return oracle.sgemm_ex(self.op_a, self.op_b, self.M, self.N, self.K, self.alpha, self.A,
                               self.lda, self.sa, self.B, self.ldb, self.sb, self.beta, self.C0,
                               self.ldc, self.sc, self.batch, self.bias, self.act)

    def run(self, sg):
        import torch
        dev = torch.device("cuda")
        A = torch.from_numpy(self.A).to(dev)
        B = torch.from_numpy(self.B).to(dev)
        C = torch.from_numpy(self.C0.copy()).to(dev)
        bias = torch.from_numpy(self.bias).to(dev) if self.bias is not None else None
        sg.sgemm_ex_ptr(self.op_a, self.op_b, self.M, self.N, self.K, self.alpha, A.data_ptr(),
                        self.lda, self.sa, B.data_ptr(), self.ldb, self.sb, self.beta,
                        C.data_ptr(), self.ldc, self.sc, self.batch,
                        bias.data_ptr() if bias is not None else 0, self.act,
                        torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        buf = C.cpu().numpy()
        out = np.stack([buf[b * self.sc:b * self.sc + self.M * self.ldc]
                        .reshape(self.M, self.ldc)[:, :self.N] for b in range(self.batch)])
        # everything but the logical blocks is untouched
        mask = np.ones(buf.shape, bool)
        for b in range(self.batch):
            blk = mask[b * self.sc:b * self.sc + self.M * self.ldc].reshape(self.M, self.ldc)
            blk[:, :self.N] = False
        assert np.array_equal(buf[mask].view(np.uint32), self.C0[mask].view(np.uint32))
        return out

    def check(self, got, exact):
        ref = self.oracle()
        if exact:
            assert np.array_equal(got, ref)
            return
        a, b, c = self.views()
        den = 0.0
        if self.alpha != 0 and self.K > 0:      # A and B are not read otherwise
            den = self.K * float(np.abs(a).max(initial=0)) * float(np.abs(b).max(initial=0))
        if self.beta:
            den += abs(self.beta) * float(np.abs(c).max())
        if self.bias is not None:
            den += float(np.abs(self.bias).max())
        err = float(np.abs(got.astype(np.float64) - ref).max()) / den
        assert err <= TOL, f"normalised error {err:.3e}"
        assert np.all(np.isfinite(got))


LAYOUTS = list(itertools.product((0, 1), (0, 1)))


@pytest.mark.parametrize("op_a,op_b", LAYOUTS)
@pytest.mark.parametrize("shape", [(150, 130, 70), (256, 256, 128), (1, 257, 33)])
@pytest.mark.parametrize("batch", [1, 3])
def test_layouts_and_batches(sg, op_a, op_b, shape, batch):
    M, N, K = shape
    p = ExProblem(op_a, op_b, M, N, K, batch, seed=M + N + K + batch, alpha=0.75, beta=0.5,
                  pad=0 if shape == (256, 256, 128) else 3)
    p.check(p.run(sg), exact=False)
    q = ExProblem(op_a, op_b, M, N, K, batch, seed=7 + batch, dist="int4", alpha=1.5, beta=0.5,
                  bias=True, pad=0 if shape == (256, 256, 128) else 3)
    q.check(q.run(sg), exact=True)


@pytest.mark.parametrize("op_a,op_b", LAYOUTS)
@pytest.mark.parametrize("tile", ["64", "128"])
def test_layouts_on_both_tiles(sg, tune, op_a, op_b, tile):
    tune(tile=tile)
    p = ExProblem(op_a, op_b, 200, 136, 100, 2, seed=30, alpha=0.5, beta=-1.0, bias=True, act=1)
    p.check(p.run(sg), exact=False)
    q = ExProblem(op_a, op_b, 128, 192, 64, 3, seed=31, dist="int4", alpha=1.5, beta=0.5,
                  bias=True, pad=0)
    q.check(q.run(sg), exact=True)


@pytest.mark.parametrize("op_a,op_b", LAYOUTS)
def test_bias_and_gelu(sg, op_a, op_b):
    p = ExProblem(op_a, op_b, 200, 190, 96, 2, seed=11, bias=True, act=1, alpha=1.0)
    p.check(p.run(sg), exact=False)
    q = ExProblem(op_a, op_b, 128, 256, 64, 1, seed=12, bias=True, act=1, beta=1.0, pad=0)
    q.check(q.run(sg), exact=False)


def test_shared_operand_and_split_k(sg):
    # B shared by every batch (stride 0); 2 x 4 tiles with a long K -> split-K
    p = ExProblem(0, 0, 256, 512, 4096, 2, seed=13, shared_b=True, pad=0)
    p.check(p.run(sg), exact=False)
    q = ExProblem(0, 1, 256, 256, 4096, 3, seed=14, dist="int4", pad=0, bias=True)
    q.check(q.run(sg), exact=True)


def test_gpt2_attention_scores_and_values(sg):
    # per-head Q K^T / sqrt(64): 12 heads, seq 1024, head dim 64 (op_b = T)
    p = ExProblem(0, 1, 1024, 1024, 64, 12, seed=15, alpha=0.125, pad=0)
    p.check(p.run(sg), exact=False)
    # per-head P V: (1024 x 1024) x (1024 x 64)
    q = ExProblem(0, 0, 1024, 64, 1024, 12, seed=16, pad=0)
    q.check(q.run(sg), exact=False)


def test_gpt2_mlp_up_with_bias_and_gelu(sg):
    p = ExProblem(0, 0, 1024, 3072, 768, 1, seed=17, bias=True, act=1, pad=0)
    p.check(p.run(sg), exact=False)


def test_k_zero_and_alpha_zero_apply_the_epilogue(sg):
    p = ExProblem(0, 0, 70, 90, 0, 2, seed=18, beta=0.5, bias=True, act=1)
    p.check(p.run(sg), exact=False)
    q = ExProblem(1, 1, 70, 90, 20, 2, seed=19, beta=-1.0, bias=True)
    q.alpha = 0.0
    q.A[:] = np.nan
    q.check(q.run(sg), exact=False)


def test_invalid_arguments(sg):
    import torch
    x = torch.zeros(4096, device="cuda")
    ptr = x.data_ptr()
    bad = [
        dict(op_a=2), dict(op_b=-1), dict(act=5), dict(lda=3), dict(ldb=3), dict(ldc=3),
        dict(batch=2, stride_c=8),     # outputs of the two batches would overlap
        dict(stride_a=-1),
    ]
    for kw in bad:
        args = dict(op_a=0, op_b=0, M=8, N=8, K=8, alpha=1.0, A=ptr, lda=8, stride_a=0, B=ptr,
                    ldb=8, stride_b=0, beta=0.0, C=ptr, ldc=8, stride_c=64, batch=1, bias=0,
                    act=0)
        args.update(kw)
        with pytest.raises(sg.SgemmError) as e:
            sg.sgemm_ex_ptr(**args)
        assert e.value.status == 1, kw


def test_torch_matmul_api(sg):
    import torch
    torch.manual_seed(0)
    A = torch.rand(3, 64, 40, device="cuda") - 0.5
    B = torch.rand(50, 40, device="cuda") - 0.5       # shared, read transposed
    bias = torch.rand(50, device="cuda") - 0.5
    C = sg.matmul(A, B, bias=bias, activation="gelu_tanh", trans_b=True)
    torch.cuda.synchronize()
    ref = oracle.sgemm_ex(0, 1, 64, 50, 40, 1.0, A.cpu().numpy(), 40, 64 * 40, B.cpu().numpy(),
                          40, 0, 0.0, None, 50, 64 * 50, 3, bias.cpu().numpy(), 1)
    assert C.shape == (3, 64, 50)
    assert float((C.cpu() - torch.from_numpy(ref)).abs().max()) <= 1e-6 * (40 * 0.25 + 0.5)


@pytest.mark.parametrize("op_a,op_b", LAYOUTS)
@pytest.mark.parametrize("batch,shared_b", [(1, False), (3, False), (2, True)])
def test_transposed_copies_first(sg, tune, op_a, op_b, batch, shared_b):
    """Operands whose rows run along K copied transposed into the workspace
    (forced here), then the product with both operands copied directly --
    batched, with a shared B, bias and GELU, ragged and exact."""
    tune(transpose_a=1, tile=128, schedule=0)
    p = ExProblem(op_a, op_b, 300, 260, 530, batch, seed=61 + batch, alpha=0.75, beta=0.5,
                  bias=True, act=1, pad=4, shared_b=shared_b, aligned=True)
    p.check(p.run(sg), exact=False)
    q = ExProblem(op_a, op_b, 256, 384, 256, batch, seed=71 + batch, dist="int4", alpha=1.5,
                  beta=0.5, bias=True, pad=0, shared_b=shared_b, aligned=True)
    q.check(q.run(sg), exact=True)
    r = ExProblem(op_a, op_b, 128, 129, 1001, batch, seed=81 + batch, pad=4, shared_b=shared_b,
                  aligned=True)
    tune(split_k=3)   # split-K on the copies too
    r.check(r.run(sg), exact=False)


@pytest.mark.parametrize("op_a,op_b", LAYOUTS)
@pytest.mark.parametrize("batch,bias,act", [(1, False, 0), (2, True, 1)])
def test_transposed_copies_packed_issue_bit_identical(sg, tune, op_a, op_b, batch, bias, act):
    """The direct-copy product issues its FMAs packed by default (plain and
    with batches, bias and GELU); scalar issue (tuning knob kernel = 0) gives
    the same C bit for bit, and both match the oracle."""
    tune(transpose_a=1, tile=128, schedule=0)
    p = ExProblem(op_a, op_b, 300, 260, 530, batch, seed=95, alpha=0.75, beta=0.5, bias=bias,
                  act=act, pad=4, aligned=True)
    outs = []
    for kernel in (None, 0):
        tune(kernel=kernel)
        out = p.run(sg)
        p.check(out, exact=False)
        outs.append(out)
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


@pytest.mark.parametrize("op_a,op_b", LAYOUTS)
def test_sixteen_by_eight_kernel_ex(sg, tune, op_a, op_b):
    """sgemm_ex's direct-copy plans on the 16 x 8 per-thread kernel (forced),
    batched with bias and GELU, and exact on integers."""
    tune(kernel=2, transpose_a=1, split_k=1, tile=128, schedule=0)
    p = ExProblem(op_a, op_b, 300, 260, 530, 2, seed=91, alpha=0.75, beta=0.5, bias=True,
                  act=1, pad=4, aligned=True)
    p.check(p.run(sg), exact=False)
    q = ExProblem(op_a, op_b, 256, 384, 256, 3, seed=92, dist="int4", alpha=1.5, beta=0.5,
                  bias=True, pad=0, aligned=True, shared_b=True)
    q.check(q.run(sg), exact=True)
