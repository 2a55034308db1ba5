"""Host logic of bench.py, on CPU: the max-over-ranks reduction under a real
world-size-2 gloo process group, throughput arithmetic, clock-sample parsing,
and the reference arm's JSON line."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, _ = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    t = bench.max_over_ranks(1.5 + rank, dist)
    v = bench.throughput(1e12, 10, w, t)
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"t": t, "v": v}, f)
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r in res:
        assert r["t"] == 2.5                      # the slowest rank's time, on every rank
        assert r["v"] == pytest.approx(1e12 * 10 * 2 / 2.5 / 1e12)   # whole-job TFLOP/s


def test_single_process_needs_no_group():
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(3.0, None) == 3.0
    assert bench.throughput(2e12, 5, 1, 1.0) == pytest.approx(10.0)


def test_clock_summary():
    rows = [
        ["GPU-abc", "2070", "2070", "900", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"],
        ["GPU-abc", "1980", "2070", "1300", "0x4", "Not Active", "Not Active", "Not Active", "Active"],
        ["GPU-xyz", "300", "2070", "90", "0x0", "Active", "Not Active", "Not Active", "Not Active"],
    ]
    s = bench.summarize_clocks(rows, "abc")
    assert s["sm_mhz"] == pytest.approx(2025.0)
    assert s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert bench.summarize_clocks([], None)["sm_mhz"] is None


def test_reference_arm_json_line():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "square256", "--steps", "2", "--warmup", "1",
                          "--ref-seconds", "2"], capture_output=True, text=True, env=env,
                         timeout=300, check=True).stdout
    lines = [l for l in out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 2
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["value"] > 0


def test_reference_arm_other_ranks_print_nothing():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", OMP_NUM_THREADS="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "square256", "--steps", "1", "--warmup", "1"],
                         capture_output=True, text=True, env=env, timeout=120, check=True).stdout
    assert out.strip() == ""


def test_per_workload_roofline_arithmetic():
    import workloads
    p = workloads.workload("square1024ab")
    # A, B read once; C read (beta != 0) and written
    assert bench.algorithmic_bytes(p) == 4 * (1024 * 1024 * 4)
    q = workloads.workload("skinny_k64")
    assert bench.algorithmic_bytes(q) == 4 * (8192 * 64 * 2 + 8192 * 8192)
    # 8192^2 x 64 at 80 TFLOP/s and 6.8 TB/s: 107 us of FMAs, 40 us of HBM
    r = bench.roofline_entry(q.flops, bench.algorithmic_bytes(q), 214.7e-6, 80.0, 6800.0)
    assert r["bound"] == "alu"
    assert r["frac"] == pytest.approx(q.flops / 80e12 / 214.7e-6, rel=1e-3)
    assert r["hbm_gbs"] == pytest.approx(bench.algorithmic_bytes(q) / 214.7e-6 / 1e9, rel=1e-3)
    # at the tensor mode's effective peak the same shape is bound by HBM
    t = bench.roofline_entry(q.flops, bench.algorithmic_bytes(q), 50e-6, 316.0, 6800.0)
    assert t["bound"] == "hbm"
    assert t["frac"] == pytest.approx(bench.algorithmic_bytes(q) / 6800e9 / 50e-6, rel=1e-3)


def test_traffic_hash_ignores_comments_not_code():
    """The DRAM traffic figures are tied to the kernel's code: a comment or
    layout edit keeps the hash, any change of a token outside comments, or
    inside a string literal, changes it."""
    src = 'int f(int x) { // twice\n  return 2 * x; /* done */ }\nconst char *s = "a // b";\n'
    same = 'int f(int x) {\n    return 2 * x;   // doubled\n}\nconst char *s = "a // b";\n'
    other = 'int f(int x) { return 3 * x; }\nconst char *s = "a // b";\n'
    lit = 'int f(int x) { return 2 * x; }\nconst char *s = "a // c";\n'
    assert bench.code_tokens(src) == bench.code_tokens(same)
    assert bench.code_tokens(src) != bench.code_tokens(other)
    assert bench.code_tokens(src) != bench.code_tokens(lit)
    assert "twice" not in bench.code_tokens(src) and '"a // b"' in bench.code_tokens(src)
    assert len(bench.source_hash()) == 16


@pytest.mark.parametrize("dist", ["uniform", "normal", "int4"])
def test_operands_draw_what_make_draws(dist):
    """workloads.operands (A and B alone, for outputs too large to hold on the
    host) draws the same seeded values, padding included, as workloads.make."""
    import numpy as np
    import workloads
    p = workloads.make(37, 53, 29, dist=dist, seed=9, lda=31, ldb=57)
    A, B = workloads.operands(37, 53, 29, dist=dist, seed=9, lda=31, ldb=57)
    assert A.dtype == np.float32 and B.dtype == np.float32
    assert np.array_equal(A, p.A) and np.array_equal(B, p.B)
