"""Host-side tests of the C ABI (no GPU work): the library builds, loads and
exports every symbol include/sgemm.h declares; argument checks reject bad
input before anything would be launched; the planner's choices."""
from __future__ import annotations

import ctypes
import sys
import os
import re
import subprocess

import pytest

import dense_fp32_matrix_06_gb300 as sg
from dense_fp32_matrix_06_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sgemm.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return sg.load_library()


def declared_functions() -> list[str]:
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(sg.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", sg.LIB_PATH], check=True,
                         capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_build_targets_sm103a_only():
    flags = _build.ARCH_FLAGS
    assert flags == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert "--use_fast_math" not in _build.NVCC_FLAGS
    # subnormals are kept (no flush to zero, IEEE division and square root),
    # so results follow the IEEE oracle at the bottom of the range too
    for f in ("-ftz=true", "--ftz=true", "-prec-div=false", "-prec-sqrt=false", "-fmad=false"):
        assert f not in _build.NVCC_FLAGS


def test_status_strings(lib):
    for code, name in sg.STATUS_NAMES.items():
        assert sg.status_string(code).startswith(name)
    assert sg.status_string(99) == "SGEMM_ERR_UNKNOWN"


BAD_SHAPES = [
    # M, N, K, lda, ldb, ldc
    (-1, 4, 4, 4, 4, 4),
    (4, -1, 4, 4, 4, 4),
    (4, 4, -1, 4, 4, 4),
    (4, 4, 8, 7, 4, 4),    # lda < K
    (4, 8, 4, 4, 7, 8),    # ldb < N
    (4, 8, 4, 4, 8, 7),    # ldc < N
    (4, 4, 0, 0, 4, 4),    # lda < 1
]


@pytest.mark.parametrize("shape", BAD_SHAPES)
def test_invalid_sizes_rejected_before_any_launch(lib, shape):
    M, N, K, lda, ldb, ldc = shape
    assert lib.sgemm(M, N, K, 1.0, 16, lda, 16, ldb, 0.0, 16, ldc, None) == 1
    plan = sg.GemmPlan()
    assert lib.gemm_plan_for_sms(M, N, K, lda, ldb, ldc, None, None, None, 152,
                                 ctypes.byref(plan)) == 1
    assert lib.sgemm_with_plan(ctypes.byref(plan), M, N, K, 1.0, 16, lda, 16, ldb, 0.0, 16,
                               ldc, None, 0, None) == 1


def test_null_pointers_rejected(lib):
    assert lib.sgemm(4, 4, 4, 1.0, None, 4, 16, 4, 0.0, 16, 4, None) == 1
    assert lib.sgemm(4, 4, 4, 1.0, 16, 4, None, 4, 0.0, 16, 4, None) == 1
    assert lib.sgemm(4, 4, 4, 1.0, 16, 4, 16, 4, 0.0, None, 4, None) == 1
    assert lib.gemm_plan_for_sms(4, 4, 4, 4, 4, 4, None, None, None, 152, None) == 1
    assert lib.gemm_plan_for_sms(4, 4, 4, 4, 4, 4, None, None, None, 0,
                                 ctypes.byref(sg.GemmPlan())) == 1
    assert lib.sgemm_ffma_probe(0, 1, 1, 16, None) == 1
    assert lib.sgemm_ffma_probe(1, 1, 1, None, None) == 1


def test_empty_output_is_a_no_op_without_a_device(lib):
    # M == 0 or N == 0: nothing to do, succeeds before touching the device
    assert lib.sgemm(0, 5, 3, 1.0, None, 3, None, 5, 0.0, None, 5, None) == 0
    assert lib.sgemm(5, 0, 3, 1.0, None, 3, None, 1, 0.0, None, 1, None) == 0


def test_device_calls_report_unsupported_without_a_gpu(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    plan = sg.GemmPlan()
    assert lib.gemm_plan(64, 64, 64, 64, 64, 64, None, None, None, ctypes.byref(plan)) == 3


def plan(M, N, K, lda=None, ldb=None, ldc=None, A=0, B=0, C=0, sms=152):
    return sg.gemm_plan_for_sms(M, N, K, lda or max(K, 1), ldb or max(N, 1), ldc or max(N, 1),
                                A, B, C, sm_count=sms)


def test_plan_full_tiles_take_the_unchecked_vector_path(lib):
    p = plan(8192, 8192, 8192)
    # K slices of 32: after the transpose both operands are row copies
    assert (p.bm, p.bn, p.bk, p.threads) == (128, 128, 32, 256)
    assert p.tiles_m == 64 and p.tiles_n == 64
    assert p.vec == 1 and p.edge == 0
    assert p.split_k == 1 and p.tail_split == 1 and p.tail_start == 4096
    assert p.grid_ctas == 4096
    # A is transposed into the workspace first (K x M after the counter block)
    assert p.transpose_a == 1 and p.a_t_ld == 8192
    assert p.workspace_bytes == sg.WORKSPACE_COUNTER_BYTES + 8192 * 8192 * 4


def test_plan_transpose_choice(lib, tune):
    assert plan(4096, 4096, 4096).transpose_a == 1
    assert plan(2048, 2048, 2048).transpose_a == 1        # 256 tiles, more than one per SM
    assert plan(1024, 2304, 768).transpose_a == 1         # 144 tiles (>= 0.45 of a wave)
    assert plan(1024, 1024, 16384).transpose_a == 1       # long K
    assert plan(8192, 8192, 64).transpose_a == 1          # K = 64 on 13 waves
    assert plan(2048, 2048, 64).transpose_a == 0          # K = 64 on under 8 waves
    assert plan(1024, 1024, 1024).transpose_a == 0        # 64 tiles, K = 1024
    assert plan(4096, 512, 4096).transpose_a == 0         # N < 768
    # A's own alignment does not matter (its copy is aligned); B's and C's do
    q = plan(4096, 4096, 4096, A=4100)
    assert q.transpose_a == 1 and q.vec == 1
    q = plan(4096, 4096, 4095, lda=4095)
    assert q.transpose_a == 1 and q.vec == 1 and q.a_t_ld == 4096
    assert plan(4096, 4096, 4096, B=4100).transpose_a == 0
    assert plan(4096, 4095, 4096, ldb=4095, ldc=4095).transpose_a == 0
    tune(transpose_a="0")
    q = plan(8192, 8192, 8192)
    assert q.transpose_a == 0 and q.workspace_bytes == 0 and q.bk == 16
    tune(transpose_a="1")
    r = plan(1023 * 2, 4096, 515, lda=516)
    assert r.transpose_a == 1 and r.a_t_ld == 2048 and r.edge == 1 and r.bk == 32
    assert r.workspace_bytes == sg.WORKSPACE_COUNTER_BYTES + (515 * 2048 * 4 + 255) // 256 * 256


@pytest.mark.parametrize("M,N,K,family", [
    # one wave of 128-wide tiles is S = 304 resident CTAs on 152 SMs
    (1024, 1024, 1024, "none"),        # 64 tiles (< 0.3 S), K = 1024: split-K, no pass
    (1536, 1024, 1024, "grid"),        # 96 tiles (>= 0.3 S), K = 1024
    (2560, 1024, 1024, "stream_k"),    # 160 tiles: just over one CTA per SM
    (2560, 1024, 4096, "stream_k"),
    (256, 2048, 2048, "none"),         # 32 tiles (< 0.15 S), K = 2048
    (512, 2048, 2048, "grid"),         # 64 tiles, K = 2048
    (1280, 2048, 768, "grid"),         # 160 tiles, K = 768: the grid (stream-K needs K >= 1024)
    (1536, 2048, 2048, "grid"),        # 192 tiles (> 1.25 sms)
    (1792, 2048, 2048, "grid"),        # 224 tiles
    (2048, 2048, 2048, "grid"),        # 256 tiles
    (4480, 1024, 2048, "grid"),        # 280 tiles
    (1024, 2304, 768, "grid"),         # 144 tiles, K = 768
    (1024, 3072, 768, "grid"),         # 192 tiles, K = 768
    (1024, 768, 3072, "grid"),         # 48 tiles, N = 768, K = 3072
    (768, 1024, 768, "none"),          # 48 tiles, K = 768 (< 0.45 S)
    (1024, 1024, 16384, "grid"),       # 64 tiles, long K: split along K after the pass
    (4096, 4096, 4096, "grid"),        # several waves
    (8192, 8192, 64, "grid"),          # 13 waves of K = 64
    (2048, 512, 4096, "none"),         # N < 768: the pass costs too much
])
def test_plan_transpose_family_bands(lib, tune, M, N, K, family):
    """Below one wave, the pass over A and the schedule after it follow the
    bands measured on GB300 (tile count as a fraction of a wave, and K).  The
    bands are a property of 128-wide plans: the tile knob pins that (and
    leaves out the balance rule, tested below)."""
    tune(tile=128)
    p = plan(M, N, K)
    got = "none" if not p.transpose_a else ("stream_k" if p.schedule == 1 else "grid")
    assert got == family
    if p.transpose_a:
        assert p.bk == 32 and p.stages == 3


def test_plan_issue_form(lib, tune):
    """Packed FMA issue on A^T plans and on split-K plans without the pass;
    scalar issue on other plans; the knob overrides."""
    assert plan(8192, 8192, 8192).kernel == 1            # A^T grid
    assert plan(2560, 1024, 2048).kernel == 1            # A^T + stream-K
    assert plan(1024, 1024, 1024).kernel == 1            # split-K, no pass
    assert plan(2048, 2048, 64).kernel == 0              # unsplit 128-wide grid, no pass
    assert plan(1023, 777, 513, lda=513, ldb=777, ldc=777).kernel == 1   # 64-wide tiles
    tune(kernel=0)
    assert plan(8192, 8192, 8192).kernel == 0
    assert plan(1024, 1024, 1024).kernel == 0
    tune(kernel=2)
    assert plan(8192, 8192, 8192).kernel == 2


def test_plan_tail_split_is_opt_in(lib, tune):
    tune(tail_split="2")
    p = plan(8192, 8192, 8192)
    # 4096 tiles over 304 resident slots: 13 full waves + 144 tiles, which
    # are the ones split in two along K
    assert p.split_k == 1
    assert p.tail_start == 4096 - 144 and p.tail_split == 2 and p.tail_k_per_split == 4096
    assert p.grid_ctas == 4096 - 144 + 2 * 144
    assert p.workspace_bytes == sg.WORKSPACE_COUNTER_BYTES + 144 * 2 * 128 * 128 * 4
    assert p.edge == 0
    q = plan(2048, 2048, 2048)                              # 256 tiles: less than a wave
    assert q.tail_split == 1 and q.tail_start == q.tiles_m * q.tiles_n
    r = plan(1000, 1000, 100)                               # short K: nothing to split
    assert r.tail_split == 1 or r.tail_k_per_split >= 16
    tune(tail_split="0")
    t = plan(8192, 8192, 8192)
    assert t.tail_split == 1 and t.grid_ctas == 4096


def test_plan_ragged_shape_takes_the_checked_scalar_path(lib):
    p = plan(1023, 777, 513, lda=513, ldb=777, ldc=777)
    assert p.vec == 0 and p.edge == 1
    # 8 x 7 = 56 tiles of 128 would fill under half of 152 SMs: 64-wide tiles
    assert (p.bm, p.bn, p.bk, p.threads) == (64, 64, 8, 64)
    assert p.tiles_m == 16 and p.tiles_n == 13


def test_plan_tile_choice(lib, tune):
    tune(schedule=0)   # the tiled kernels (small problems have their own kernel)
    assert plan(8192, 8192, 8192).bm == 128
    assert plan(1024, 2304, 768).bm == 128        # 144 tiles of 128
    assert plan(1024, 768, 3072).bm == 128        # 48 tiles of 128, but K is long
    assert plan(1024, 1024, 16384).bm == 128
    assert plan(1023, 777, 513).bm == 64          # 56 tiles, short K
    assert plan(1024, 64, 1024).bm == 64          # a 128-wide tile would be half padding
    assert plan(256, 256, 256).bm == 64
    assert plan(256, 256, 256, sms=4).bm == 128   # a small GPU is filled by 4 tiles
    tune(tile="128")
    assert plan(256, 256, 256).bm == 128
    tune(tile="64")
    q = plan(8192, 8192, 8192)
    assert q.bm == 64 and q.tiles_m == 128 and q.threads == 64 and q.edge == 0


def test_plan_misaligned_pointer_disables_vector_loads(lib):
    assert plan(256, 256, 256, A=4096).vec == 1
    assert plan(256, 256, 256, A=4100).vec == 0
    assert plan(256, 256, 256, C=4104).vec == 0


def test_plan_split_k_fills_the_gpu_when_tiles_are_few(lib, tune):
    tune(schedule=0)   # one CTA per (tile, K range); the stream-K plans have their own tests
    tune(tile="128")
    tune(transpose_a="0")   # split-K bookkeeping only
    p = plan(1024, 1024, 16384)          # 64 tiles, long K
    assert p.split_k > 1
    assert p.k_per_split % p.bk == 0
    assert (16384 + p.k_per_split - 1) // p.k_per_split == p.split_k
    assert p.grid_ctas == 64 * p.split_k
    assert p.tail_split == 1 and p.tail_start == 64
    assert p.workspace_bytes == sg.WORKSPACE_COUNTER_BYTES + 64 * p.split_k * 128 * 128 * 4
    # MLP-down: 48 tiles, K = 3072
    assert plan(1024, 768, 3072).split_k > 1
    tune(tile="64")
    q = plan(1024, 1024, 16384)          # 64-wide tiles: 256 of them, still split along K
    tiles = q.tiles_m * q.tiles_n
    assert q.bm == 64 and tiles == 256 and q.split_k > 1
    assert q.workspace_bytes == sg.WORKSPACE_COUNTER_BYTES + tiles * q.split_k * 64 * 64 * 4
    # a full wave of tiles is never split
    assert plan(8192, 8192, 8192).split_k == 1
    assert plan(4096, 4096, 4096).split_k == 1
    # short K is never split below 8 slices per partition
    q = plan(256, 256, 200)
    assert q.split_k == 1


def test_plan_depends_on_sm_count(lib):
    small = plan(2048, 2048, 2048, sms=8)
    big = plan(2048, 2048, 2048, sms=152)
    assert small.split_k == 1
    assert big.split_k >= 1


def test_sgemm_with_plan_rejects_mismatched_plan_and_small_workspace(lib, tune):
    tune(tile="128")
    tune(schedule=0)
    p = plan(1024, 1024, 16384)
    assert p.split_k > 1
    # workspace too small -> SGEMM_ERR_WORKSPACE (checked before the device)
    rc = lib.sgemm_with_plan(ctypes.byref(p), 1024, 1024, 16384, 1.0, 4096, 16384, 4096, 1024,
                             0.0, 4096, 1024, 4096, 16, None)
    assert rc == 7
    # plan made for another shape -> SGEMM_ERR_INVALID_ARG
    rc = lib.sgemm_with_plan(ctypes.byref(p), 1024, 1024, 8192, 1.0, 4096, 8192, 4096, 1024,
                             0.0, 4096, 1024, 4096, p.workspace_bytes, None)
    assert rc == 1
    # a vector plan used with a misaligned pointer -> SGEMM_ERR_INVALID_ARG
    q = plan(512, 512, 512)
    rc = lib.sgemm_with_plan(ctypes.byref(q), 512, 512, 512, 1.0, 4100, 512, 4096, 512, 0.0,
                             4096, 512, None, 0, None)
    assert rc == 1


def test_forced_split_override(lib, tune):
    tune(tile="128")
    tune(split_k="4")
    p = plan(512, 512, 1024)
    assert p.split_k == 4 and p.k_per_split == 256
    tune(split_k="1")
    assert plan(1024, 1024, 16384).split_k == 1


def test_forced_kernel_override(lib, tune):
    tune(schedule=0)
    tune(tile="128")
    tune(kernel="0")
    assert plan(256, 256, 256).kernel == 0
    tune(kernel="1")
    assert plan(256, 256, 256).kernel == 1


def test_tuning_knobs_round_trip_and_range_checks(lib, tune):
    for knob in sg.TUNING_KNOBS:
        assert sg.get_tuning(knob) is None or isinstance(sg.get_tuning(knob), int)
    tune(tile=64, split_k=3, transpose_a=0)
    assert sg.get_tuning("tile") == 64 and sg.get_tuning("split_k") == 3
    assert plan(8192, 8192, 8192).bm == 64
    tune(tile=None)
    assert sg.get_tuning("tile") is None and plan(8192, 8192, 8192).bm == 128
    # out-of-range values and unknown knobs are refused, the knob is unchanged
    for knob, bad in (("tile", 96), ("split_k", 0), ("split_k", 33), ("kernel", 3),
                      ("transpose_a", 5), ("workspace_limit_mib", -3)):
        before = sg.get_tuning(knob)
        assert lib.sgemm_set_tuning(sg.TUNING_KNOBS[knob], bad) == 1
        assert sg.get_tuning(knob) == before
    assert lib.sgemm_set_tuning(len(sg.TUNING_KNOBS), 1) == 1
    assert lib.sgemm_set_tuning(-1, 1) == 1
    assert lib.sgemm_get_tuning(len(sg.TUNING_KNOBS)) == -2


def test_tuning_env_is_read_once_at_load(lib):
    """The environment seeds the knobs when the library loads; changing it
    afterwards changes no plan (the call path never reads it)."""
    code = (
        "import os, sys; sys.path.insert(0, %r)\n"
        "import dense_fp32_matrix_06_gb300 as sg\n"
        "sg.load_library()\n"
        "a = sg.gemm_plan_for_sms(8192, 8192, 8192, 8192, 8192, 8192).bm\n"
        "os.environ['SGEMM_FORCE_TILE'] = '128'\n"
        "b = sg.gemm_plan_for_sms(8192, 8192, 8192, 8192, 8192, 8192).bm\n"
        "print(a, b, sg.get_tuning('tile'), sg.get_tuning('split_k'))\n" % ROOT)
    env = dict(os.environ, SGEMM_FORCE_TILE="64", SGEMM_FORCE_SPLIT="banana")
    out = subprocess.run([sys.executable, "-c", code], env=env, check=True,
                         capture_output=True, text=True).stdout.split()
    assert out == ["64", "64", "64", "None"]


def test_plan_schedule_choice(lib, tune):
    """Persistent stream-K where it measured faster: tiny grids of 64-wide
    tiles, and (after the A^T pass) partial waves of 128-wide tiles with long
    enough K; one CTA per (tile, K range) elsewhere."""
    p = plan(256, 256, 256)          # 2^24 multiply-adds: the small-problem kernel
    assert p.schedule == 2 and p.bm == 32 and p.bk == 256 and p.threads == 256
    assert p.grid_ctas == 64 and p.workspace_bytes == 0
    p = plan(64, 64, 1000)           # K too long for it: 64-wide stream-K
    assert p.schedule == 1 and p.bm == 64 and p.bk == 8 and p.stages == 4
    q = plan(1024, 1024, 16384)      # 64 tiles, K = 16384: A transposed, then split-K
    assert q.schedule == 0 and q.transpose_a == 1 and q.bk == 32 and q.split_k > 1
    r = plan(2560, 1024, 2048)       # 160 tiles, just over one per SM: A^T, then stream-K
    assert r.schedule == 1 and r.transpose_a == 1
    for shape in [(1024, 1024, 1024), (1023, 777, 513), (1024, 2304, 768), (2048, 2048, 2048),
                  (4096, 4096, 4096), (8192, 8192, 8192), (8192, 8192, 64)]:
        assert plan(*shape).schedule == 0, shape
    tune(schedule=0)
    assert plan(256, 256, 256).schedule == 0
    tune(schedule=1)
    assert plan(8192, 8192, 8192).schedule == 1
    tune(schedule=2)
    assert plan(2000, 3000, 256).schedule == 2       # forced where K allows
    assert plan(2000, 3000, 257).schedule == 0


def test_small_problem_plan_checks(lib, tune):
    p = plan(100, 70, 33, lda=35, ldb=70, ldc=71)
    assert p.schedule == 2 and p.vec == 0 and p.bk == 64 and p.tiles_m == 4 and p.tiles_n == 3
    q = plan(256, 256, 256)
    # a tampered plan is refused before the device is touched
    for field, value in (("bk", 128), ("grid_ctas", 65), ("threads", 128), ("workspace_bytes", 64)):
        r = sg.GemmPlan.from_buffer_copy(q)
        setattr(r, field, value)
        assert lib.sgemm_with_plan(ctypes.byref(r), 256, 256, 256, 1.0, 4096, 256, 4096, 256, 0.0,
                                   4096, 256, None, 0, None) == 1, field
    # a plan for another K
    assert lib.sgemm_with_plan(ctypes.byref(q), 256, 256, 200, 1.0, 4096, 256, 4096, 256, 0.0,
                               4096, 256, None, 0, None) == 1


def test_stream_k_plan_round_trips_through_sgemm_with_plan_checks(lib, tune):
    """A stream-K plan is accepted by sgemm_with_plan's plan check (failing
    only later, on the missing device) and a tampered one is refused."""
    tune(schedule=1, tile=128, transpose_a=0)
    p = plan(1024, 1024, 1024)
    assert p.schedule == 1 and p.sk_iters > 0
    # workspace too small -> SGEMM_ERR_WORKSPACE before the device is touched
    rc = lib.sgemm_with_plan(ctypes.byref(p), 1024, 1024, 1024, 1.0, 4096, 1024, 4096, 1024,
                             0.0, 4096, 1024, 4096, 16, None)
    assert rc == 7
    for field, value in (("grid_ctas", p.sk_iters + 1), ("dp_rounds", 1), ("stages", 3),
                         ("sk_iters", p.sk_iters - 1), ("bk", 32)):
        q = sg.GemmPlan.from_buffer_copy(p)
        setattr(q, field, value)
        rc = lib.sgemm_with_plan(ctypes.byref(q), 1024, 1024, 1024, 1.0, 4096, 1024, 4096,
                                 1024, 0.0, 4096, 1024, 4096, 1 << 30, None)
        assert rc == 1, field


@pytest.mark.parametrize("M,N,K,bm,split", [
    # 128-wide split grids of 256 CTAs (one CTA on 48 SMs, two on 104) move to
    # 64-wide tiles in exact K ranges, about 13.5 CTAs a SM
    (1024, 1024, 1024, 64, 8),
    (512, 2048, 2048, 64, 8),      # (was the A^T pass in 4 ranges)
    (1024, 512, 2048, 64, 16),
    (896, 1536, 1024, 64, 8),      # 252 CTAs
    (640, 2048, 1536, 64, 6),      # 240 CTAs; 6 ranges of 256 divide K exactly
    # grids already near two CTAs a SM keep 128-wide tiles
    (768, 1024, 1024, 128, 6),     # 288 CTAs
    (896, 896, 1536, 128, 6),      # 294 CTAs
])
def test_plan_balanced_small_tiles(lib, M, N, K, bm, split):
    p = plan(M, N, K)
    assert (p.bm, p.split_k) == (bm, split)
    if bm == 64:
        assert p.transpose_a == 0 and p.schedule == 0 and p.edge == 0
        assert p.kernel == 1                         # packed issue
        assert p.k_per_split * split == K and p.k_per_split >= 128
        assert p.grid_ctas == (M // 64) * (N // 64) * split


def test_plan_balanced_small_tiles_needs_aligned_operands_and_no_knobs(lib, tune):
    assert plan(1024, 1024, 1024).bm == 64
    # A's rows not 16-byte aligned: the plan is the one measured for that case
    assert plan(1024, 1024, 1024, lda=1025).bm == 128
    tune(split_k=4)
    assert plan(1024, 1024, 1024).bm == 128
    tune(split_k=None, schedule=0)
    assert plan(1024, 1024, 1024).bm == 128


def _plan_grid():
    shapes = []
    for M in (1, 7, 64, 100, 256, 513, 1024, 1536, 2048, 4096, 8192):
        for N in (1, 64, 200, 768, 1024, 2304, 8192):
            for K in (1, 16, 64, 100, 256, 300, 768, 1024, 2047, 4096, 16384):
                shapes.append((M, N, K))
    return shapes


@pytest.mark.parametrize("sms", [152, 132, 80, 8])
def test_every_planner_output_passes_the_plan_check(lib, sms):
    """The planner and the check sgemm_with_plan applies must agree: every plan
    gemm_plan_for_sms returns, over 847 shapes, three layouts (tight, padded,
    unaligned leading dimensions), a misaligned A and four GPU sizes, passes
    gemm_plan_check for the same arguments."""
    bad = []
    for (M, N, K) in _plan_grid():
        for lda, ldb, ldc, a in ((K, N, N, 0), (K + 4, N + 8, N + 4, 0),
                                 (K + 1, N + 3, N + 1, 0), (K, N, N, 4)):
            p = sg.gemm_plan_for_sms(M, N, K, lda, ldb, ldc, a, 0, 0, sm_count=sms)
            if not sg.gemm_plan_check(p, M, N, K, lda, ldb, ldc, a, 0, 0):
                bad.append((M, N, K, lda, ldb, ldc, a))
    assert not bad, f"{len(bad)} planner outputs rejected, e.g. {bad[:5]}"


def test_plan_check_rejects_edited_plans(lib):
    M = N = K = 2048
    base = plan(M, N, K)
    assert sg.gemm_plan_check(base, M, N, K, K, N, N)
    edits = {
        "split_k": base.split_k + 1, "grid_ctas": base.grid_ctas + 1,
        "workspace_bytes": base.workspace_bytes - 1, "bm": 96, "bk": base.bk * 2,
        "stages": 4, "tiles_m": base.tiles_m + 1, "kernel": 7, "schedule": 5,
    }
    for field, value in edits.items():
        q = sg.GemmPlan.from_buffer_copy(base)
        setattr(q, field, value)
        assert not sg.gemm_plan_check(q, M, N, K, K, N, N), field
    # the same plan for other sizes, or for unaligned B and C
    assert not sg.gemm_plan_check(base, M + 128, N, K, K, N, N)
    assert not sg.gemm_plan_check(base, M, N, K, K, N + 1, N + 1)
    # edge-free plans need whole tiles
    assert base.edge == 0
    assert not sg.gemm_plan_check(base, M - 1, N, K, K, N, N)


def test_balance_rule_invariants_over_the_grid(lib, tune):
    """Wherever the planner's 128-wide plan is an unevenly loaded split grid
    (between sms and 1.75 sms CTAs, operands aligned) and the balance rule
    takes it, the replacement is 64-wide tiles in exact K ranges of at least
    128, at least one full wave of small CTAs; everywhere else the plan is the
    one the planner makes with the rule left out (the tile knob at 128 leaves
    it out, so compare only shapes whose plan is 128-wide either way)."""
    sms = 152
    changed = 0
    for (M, N, K) in _plan_grid():
        p = plan(M, N, K, sms=sms)
        if p.bm != 64 or p.split_k < 2 or p.schedule != 0:
            continue
        # 64-wide by the tile choice itself (padding >= 40 %, or a small grid with
        # K <= 768), not by the rule
        tiles128 = -(-M // 128) * -(-N // 128)
        if M * N < 0.6 * tiles128 * 128 * 128 or (2 * tiles128 < sms and K <= 768):
            continue
        tune(tile=128)
        base = plan(M, N, K, sms=sms)
        tune(tile=None)
        if base.bm != 128 or base.split_k < 2 or base.schedule != 0 or base.tail_split != 1:
            continue
        if not (sms < base.grid_ctas <= 1.75 * sms):
            continue
        changed += 1
        assert K % (8 * p.split_k) == 0 and p.k_per_split == K // p.split_k >= 128
        assert p.grid_ctas >= 8 * sms and p.transpose_a == 0 and p.kernel == 1
        assert p.edge == (0 if M % 64 == 0 and N % 64 == 0 else 1)
    assert changed >= 10
