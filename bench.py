"""SGEMM throughput on GB300: C = alpha*A*B + beta*C, fp32, through the C ABI.

One "step" is one SGEMM of the benchmark workload (default: M = N = K = 8192,
A and B uniform[-1,1) from seed 4, alpha = 1, beta = 0) with its inputs already
resident in HBM.  The inputs (768 MiB) are larger than the 129 MB L2, so no
flush is needed between steps.

Prints ONE JSON line (rank 0):
  value      TFLOP/s (2*M*N*K per GEMM) over all ranks, device-timed
  e2e        the same metric with host buffers: pinned host->device copies of
             A and B, the GEMM and the device->host copy of C inside the timed
             region, every step
  roofline   the dominant kernel against the fp32 FMA peak of the chip
             (SMs x 128 FMA/clk x 2 FLOP x max SM clock)
  cpu_baseline  the CPU oracle timed on a bounded sample of the same workload

`--impl reference` times the CPU oracle (the only reference this method has)
on the same workload, metric and unit, each step a bounded sample of rows.

Launch: python bench.py [--gpus N --steps K --warmup W]; for N > 1 under
torch.distributed.run, each rank runs an independent replica of the
workload (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "SGEMM TFLOP/s (2MNK/t) at M=N=K=8192 fp32; % of GB300 FP32 FFMA peak"
UNIT = "TFLOP/s"
FMA_PER_SM_PER_CLK = 128      # fp32 FMA lanes per SM (4 sub-partitions x 32)
L2_BYTES = 129 * 1000 * 1000
# the headline product (kernel template, the translation unit that builds
# its packed A^T instantiation, the argument structs) and the transpose pass
KERNEL_SOURCES = [os.path.join(ROOT, "dense_fp32_matrix_06_gb300", "csrc", f)
                  for f in ("ffma_kernel.cuh", "ffma_gemm_tn_packed.cu", "ffma_gemm.cu",
                            "sgemm_internal.h")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def describe(p: workloads.Problem) -> str:
    d = p.meta.get("dist")
    return (f"{p.name}: SGEMM M={p.M} N={p.N} K={p.K} fp32 row-major, lda={p.lda} ldb={p.ldb} "
            f"ldc={p.ldc}, A,B {d} seed {p.meta.get('seed')}, alpha={p.alpha:g}, beta={p.beta:g}")


# --------------------------------------------------------------------------
# distributed plumbing (host logic; tested on CPU with gloo)
# --------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(value: float, dist, device=None) -> float:
    """Max of a float over all ranks (the slowest rank's time)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64,
                     device=device if (device is not None and dist.get_backend() == "nccl")
                     else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput(flops_per_step: float, steps: int, world: int, seconds: float) -> float:
    """Whole-job TFLOP/s: every rank did `steps` GEMMs in at most `seconds`."""
    if seconds <= 0:
        return float("nan")
    return flops_per_step * steps * world / seconds / 1e12


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

CLOCK_FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, interval_ms: int = 200):
        self.interval_ms = interval_ms
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.interval_ms)], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, uuid: str | None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                rows.append(parts)
        os.unlink(self.path)
        return summarize_clocks(rows, uuid)


def summarize_clocks(rows, uuid):
    if uuid:
        mine = [r for r in rows if r[0].replace("GPU-", "") == uuid.replace("GPU-", "")]
        rows = mine or rows
    sm, smax, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for r in rows:
        try:
            sm.append(float(r[1]))
            smax.append(float(r[2]))
        except ValueError:
            continue
        for name, v in zip(names, r[5:9]):
            if v.strip().lower() == "active":
                reasons.add(name)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
    # samples under load: within the top half of the observed range
    lo = max(sm) * 0.5
    loaded = [x for x in sm if x >= lo] or sm
    return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
            "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# the CPU oracle as a timed baseline (bounded sample of rows)
# --------------------------------------------------------------------------

def oracle_rows_rate(p: workloads.Problem, rows: int, seed: int = 0):
    """Time the oracle on `rows` seeded rows of C; returns (seconds, flops, threads)."""
    import oracle
    rng = np.random.default_rng(seed)
    idx = rng.choice(p.M, size=min(rows, p.M), replace=False).astype(np.int64)
    t0 = time.perf_counter()
    oracle.sgemm_rows(p.M, p.N, p.K, p.alpha, p.A, p.B, p.beta, p.C0, idx, lda=p.lda,
                      ldb=p.ldb, ldc0=p.ldc)
    dt = time.perf_counter() - t0
    return dt, 2.0 * len(idx) * p.N * p.K, oracle.max_threads()


def calibrate_rows(p: workloads.Problem, target_s: float) -> int:
    """Rows of C the oracle finishes in about `target_s` seconds on all cores."""
    import oracle
    threads = oracle.max_threads()
    dt, _, _ = oracle_rows_rate(p, threads, seed=99)
    per_batch = max(dt, 1e-3)
    batches = max(1, int(target_s / per_batch))
    return min(p.M, batches * threads)


def cpu_baseline(p: workloads.Problem, target_s: float = 15.0) -> dict:
    rows = calibrate_rows(p, target_s)
    dt, flops, threads = oracle_rows_rate(p, rows, seed=1)
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{rows} of {p.M} rows of C ({rows}x{p.N}x{p.K} fp64-accumulated "
                      f"multiply-adds, {dt:.1f} s on {threads} OpenMP threads)"}


# --------------------------------------------------------------------------
# arms
# --------------------------------------------------------------------------

def code_tokens(text: str) -> str:
    """C/C++ source with comments removed and whitespace runs collapsed (string
    and character literals kept as written), so that a comment edit leaves it
    unchanged and any edit of the code does not."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
            out.append(" ")
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_hash() -> str:
    """Hash of the FFMA kernel's code (traffic figures are tied to it);
    comments and layout do not enter it."""
    h = hashlib.sha256()
    for path in KERNEL_SOURCES:
        with open(path, encoding="utf-8") as f:
            h.update(code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def committed_traffic(kernel_id: int, workload: str, flops_per_launch: float):
    """DRAM bytes per launch from the committed ncu capture, if it was taken on
    the current kernel source (else None)."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    entry = t.get(f"{workload}/kernel{kernel_id}")
    if not entry or entry.get("source_sha") != source_hash():
        return None
    return entry.get("dram_bytes_per_launch")


def peak_fp32_tflops(sms: int) -> tuple[float, float, str]:
    """fp32 FMA peak = SMs x 128 x 2 x max SM clock."""
    mhz, src = None, None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f)["sm_max_mhz"])
            src = "MEASURED_PEAKS.json sm_max_mhz"
    except (OSError, ValueError, KeyError):
        pass
    if mhz is None:
        try:
            out = subprocess.run(["nvidia-smi", "--query-gpu=clocks.max.sm",
                                  "--format=csv,noheader,nounits"], capture_output=True,
                                 text=True, timeout=30).stdout.split()
            mhz = float(out[0])
            src = "nvidia-smi clocks.max.sm"
        except Exception:
            mhz, src = 2070.0, "nominal 2070 MHz"
    return sms * FMA_PER_SM_PER_CLK * 2 * mhz * 1e6 / 1e12, mhz, src


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")

    import dense_fp32_matrix_06_gb300 as sg
    sg.build()
    sg.load_library()

    p = workloads.workload(args.workload)
    flops = float(p.flops)
    A_h = torch.from_numpy(p.A).pin_memory()
    B_h = torch.from_numpy(p.B).pin_memory()
    A = A_h.to(device)
    B = B_h.to(device)
    C = torch.from_numpy(p.C0).to(device)
    stream = torch.cuda.current_stream(device)
    sh = stream.cuda_stream
    plan = sg.gemm_plan(p.M, p.N, p.K, p.lda, p.ldb, p.ldc, A.data_ptr(), B.data_ptr(),
                        C.data_ptr())
    # one product kernel per GEMM, plus the transpose pass when the plan copies
    # A first, plus the reduction of partial tiles when tiles share K ranges
    shares_k = plan.split_k > 1 or plan.tail_split > 1 or (plan.schedule == 1 and plan.sk_iters > 0)
    launches_per_gemm = 1 + int(plan.transpose_a) + int(shares_k)

    def step():
        sg.sgemm_ptr(p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta,
                     C.data_ptr(), p.ldc, sh)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)

    # ---- device-timed region ----
    sampler = ClockSampler()
    sampler.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(dist, device)
    torch.cuda.synchronize(device)
    t_start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(device)
    barrier(dist, device)
    clocks = sampler.stop(str(getattr(torch.cuda.get_device_properties(device), "uuid", "")) or None)
    elapsed = t_start.elapsed_time(t_end) / 1e3
    per_launch = [a.elapsed_time(b) / 1e3 for a, b in ev]
    elapsed_max = max_over_ranks(elapsed, dist, device)
    value = throughput(flops, args.steps, world, elapsed_max)

    # ---- end-to-end: host buffers, copies inside the timed region ----
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(sg, p, A, B, C, A_h, B_h, stream, device, dist, world, args)

    props = torch.cuda.get_device_properties(device)
    sms = props.multi_processor_count
    peak, mhz, peak_src = peak_fp32_tflops(sms)
    avg_launch = statistics.mean(per_launch)
    achieved = flops / avg_launch / 1e12
    traffic = committed_traffic(plan.kernel, p.name, flops)
    roofline = {"bound": "alu", "achieved": round(achieved, 3), "peak": round(peak, 3),
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                "kernel": (f"ffma_gemm_kernel<128, op(A)=A^T copy, K slice 32, "
                           f"{'packed' if plan.kernel == 1 else 'scalar'} FMA issue> after "
                           "transpose_kernel" if plan.transpose_a else
                           f"ffma_gemm_kernel (plan kernel {plan.kernel})"),
                "timed": "each sgemm call (all of its launches) with CUDA events",
                "peak_source": f"{sms} SMs x {FMA_PER_SM_PER_CLK} FMA/clk x 2 x {mhz:.0f} MHz "
                               f"({peak_src})",
                "algorithmic_flops_per_launch": flops,
                "avg_launch_ms": round(avg_launch * 1e3, 4)}
    if clocks.get("sm_mhz"):
        peak_at_clock = sms * FMA_PER_SM_PER_CLK * 2 * clocks["sm_mhz"] * 1e6 / 1e12
        roofline["frac_at_measured_clock"] = round(achieved / peak_at_clock, 4)

    probe = None
    if not args.no_probe:
        probe = ffma_probe(sg, device, sms)
        roofline["probe_tflops"] = probe["scalar"]
        roofline["frac_vs_probe"] = round(achieved / probe["scalar"], 4)

    tc = None
    if not args.no_tf32x3:
        tc = run_tf32x3(sg, p, A, B, C, stream, args, dist, device)

    extras = None
    per_config = None
    if not args.no_extras and rank == 0:
        extras = run_extras(sg, device, stream)
        per_config = run_configs(sg, device, stream, peak,
                                 probe["scalar"] if probe else None)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(p, target_s=args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(elapsed_max / args.steps * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic (seeded uniform[-1,1) inputs, no dataset)",
            "config": {"workload": describe(p), "M": p.M, "N": p.N, "K": p.K,
                       "l2": f"inputs larger than L2 ({(p.A.nbytes + p.B.nbytes) >> 20} MiB of "
                             f"A+B > 129 MB L2); no flush between steps",
                       "plan": plan.as_dict(),
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "e2e": e2e, "gpu_launches": args.steps * launches_per_gemm,
            "roofline": roofline, "cpu_baseline": cpu, "clocks": clocks,
        }
        if probe:
            line["ffma_probe"] = probe
        if tc:
            line["tf32x3"] = tc
        if extras:
            line["sgemm_ex"] = extras
        if per_config:
            line["workloads"] = per_config
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_e2e(sg, p, A, B, C, A_h, B_h, stream, device, dist, world, args):
    """The metric with host buffers: every step uploads its A and B from pinned
    host memory, runs the GEMM through the binding and downloads its C into
    pinned host memory, all inside the timed region.  Steps are pipelined the
    way a streaming caller would run them: two device buffer sets and three
    streams, so the upload of step i+1 and the download of step i-1 overlap
    the GEMM of step i."""
    import torch
    e_steps = max(3, args.e2e_steps if args.e2e_steps > 0 else args.steps)
    up = torch.cuda.Stream(device)
    down = torch.cuda.Stream(device)
    bufs = [(A, B, C), (torch.empty_like(A), torch.empty_like(B), torch.empty_like(C))]
    C_h = [torch.empty((p.M, p.ldc), dtype=torch.float32).pin_memory() for _ in range(2)]
    ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("up", "gemm", "down")}
    sh = stream.cuda_stream
    if p.beta != 0:
        raise ValueError("the end-to-end leg uploads A and B only (beta must be 0)")

    def run(n, start_event):
        up.wait_event(start_event)
        for i in range(n):
            j = i % 2
            Ad, Bd, Cd = bufs[j]
            if i >= 2:
                up.wait_event(ev["gemm"][j])        # step i-2 is done reading Ad, Bd
            with torch.cuda.stream(up):
                Ad.copy_(A_h, non_blocking=True)
                Bd.copy_(B_h, non_blocking=True)
            ev["up"][j].record(up)
            stream.wait_event(ev["up"][j])
            if i >= 2:
                stream.wait_event(ev["down"][j])    # step i-2's C has left Cd
            sg.sgemm_ptr(p.M, p.N, p.K, p.alpha, Ad.data_ptr(), p.lda, Bd.data_ptr(), p.ldb,
                         p.beta, Cd.data_ptr(), p.ldc, sh)
            ev["gemm"][j].record(stream)
            down.wait_event(ev["gemm"][j])
            with torch.cuda.stream(down):
                C_h[j].copy_(Cd, non_blocking=True)
            ev["down"][j].record(down)
        stream.wait_event(ev["down"][(n - 1) % 2])
        if n >= 2:
            stream.wait_event(ev["down"][(n - 2) % 2])

    warm = torch.cuda.Event()
    warm.record(stream)
    run(2, warm)
    torch.cuda.synchronize(device)

    # the pinned copies alone, one step's worth each, on their own streams:
    # one untimed copy (the first after idle runs slow), then three timed
    def copy_seconds(fn, on):
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(on):
            fn()
            c0.record(on)
            for _ in range(3):
                fn()
            c1.record(on)
        torch.cuda.synchronize(device)
        return c0.elapsed_time(c1) / 3e3

    Ad, Bd, Cd = bufs[0]
    h2d_s = copy_seconds(lambda: (Ad.copy_(A_h, non_blocking=True),
                                  Bd.copy_(B_h, non_blocking=True)), up)
    d2h_s = copy_seconds(lambda: C_h[0].copy_(Cd, non_blocking=True), down)
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    barrier(dist, device)
    s0.record(stream)
    run(e_steps, s0)
    s1.record(stream)
    torch.cuda.synchronize(device)
    e_el = max_over_ranks(s0.elapsed_time(s1) / 1e3, dist, device)
    # the last step's result is the one on the host now; check it is finite
    finite = bool(torch.isfinite(C_h[(e_steps - 1) % 2][:, :p.N]).all())
    h2d_bytes = int(p.A.nbytes + p.B.nbytes)
    d2h_bytes = int(C_h[0].numel() * 4)
    return {"value": throughput(float(p.flops), e_steps, world, e_el), "unit": UNIT,
            "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
            "steps": e_steps, "result_finite": finite,
            "h2d_gbs": round(h2d_bytes / h2d_s / 1e9, 1),
            "d2h_gbs": round(d2h_bytes / d2h_s / 1e9, 1),
            "copy_ms_per_step": round(max(h2d_s, d2h_s) * 1e3, 3),
            "pipelining": "two device buffer sets, three streams: the upload of step i+1 and "
                          "the download of step i-1 overlap the GEMM of step i"}


def tf32_peak_tflops() -> tuple[float, str]:
    """Dense tf32 tensor peak: measured bf16 burst x the nominal tf32:bf16 ratio."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            bf16 = float(json.load(f)["bf16_tflops"])
        src = "MEASURED_PEAKS.json bf16_tflops"
    except (OSError, ValueError, KeyError):
        bf16, src = 1900.0, "fallback 1.9 PFLOP/s bf16"
    return bf16 * 1.1 / 2.25, f"{bf16:.1f} TFLOP/s bf16 ({src}) x 1.1/2.25 nominal tf32:bf16"


def run_tf32x3(sg, p, A, B, C, stream, args, dist, device):
    """The separately reported 3xTF32 tensor-core mode on the same workload."""
    import torch
    sh = stream.cuda_stream
    flops = float(p.flops)

    def call():
        sg.sgemm_tf32x3_ptr(p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb,
                            p.beta, C.data_ptr(), p.ldc, sh)

    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(dist, device)
    e0.record(stream)
    for _ in range(args.steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize(device)
    el = max_over_ranks(e0.elapsed_time(e1) / 1e3, dist, device)
    status = sg.device_status(sh)
    world = dist.get_world_size() if dist is not None else 1
    per_call = el / args.steps

    # B packed once (weights reused), and the opt-in in-kernel split of A
    nb = sg.tf32x3_packed_b_bytes(p.K, p.N)
    packed = torch.empty(nb, dtype=torch.uint8, device=device)
    sg.tf32x3_pack_b_ptr(p.K, p.N, B.data_ptr(), p.ldb, packed.data_ptr(), nb, sh)

    def timed(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(device)
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(n):
            fn()
        a1.record(stream)
        torch.cuda.synchronize(device)
        return a0.elapsed_time(a1) / 1e3 / n

    def packed_call():
        sg.sgemm_tf32x3_packed_ptr(p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, packed.data_ptr(),
                                   p.beta, C.data_ptr(), p.ldc, sh)

    n_var = max(3, min(args.steps, 10))
    t_packed = timed(packed_call, n_var)
    old = os.environ.get("SGEMM_TF32X3_FUSE_A")
    os.environ["SGEMM_TF32X3_FUSE_A"] = "0"
    try:
        t_prepass = timed(call, n_var)
    finally:
        if old is None:
            os.environ.pop("SGEMM_TF32X3_FUSE_A", None)
        else:
            os.environ["SGEMM_TF32X3_FUSE_A"] = old
    variants = {"packed_b": {"value": round(flops / t_packed / 1e12, 3),
                             "note": "B split and transposed once (sgemm_tf32x3_pack_b); A split "
                                     "in the kernel"},
                "prepass_a": {"value": round(flops / t_prepass / 1e12, 3),
                              "note": "A split by a pre-pass instead of in the kernel "
                                      "(SGEMM_TF32X3_FUSE_A=0)"}}
    peak, src = tf32_peak_tflops()
    achieved = 3 * flops / per_call / 1e12
    return {"value": round(throughput(flops, args.steps, world, el), 3), "unit": UNIT,
            "ms_per_step": round(per_call * 1e3, 4),
            # B's split-transpose + the tensor kernel, plus A's pre-pass when A's
            # layout keeps TMA from reading it (16-byte alignment, lda % 4)
            "gpu_launches": (2 if (A.data_ptr() % 16 == 0 and p.lda % 4 == 0) else 3) * args.steps,
            "device_status": status,
            "roofline": {"bound": "tensor", "achieved": round(achieved, 2),
                         "peak": round(peak, 1), "unit": "TFLOP/s",
                         "frac": round(achieved / peak, 4), "traffic": None,
                         "kernel": "tf32x3_fused_kernel<256,2> (+ B split/transpose pass)",
                         "peak_source": src,
                         "note": "achieved = 3 tf32 products x 2MNK over the whole call "
                                 "(B's split pass included)"},
            "variants": variants}


# (name, op_a, op_b, M, N, K, batch, bias, act): batched, transposed and
# fused-epilogue forms on GPT-2-small shapes and a square size
EXTRA_CASES = [
    ("gpt2_attn_qkT_12x1024x1024x64", 0, 1, 1024, 1024, 64, 12, False, 0),
    ("gpt2_attn_pv_12x1024x64x1024", 0, 0, 1024, 64, 1024, 12, False, 0),
    ("gpt2_mlp_up_1024x3072x768", 0, 0, 1024, 3072, 768, 1, False, 0),
    ("gpt2_mlp_up_1024x3072x768_bias_gelu", 0, 0, 1024, 3072, 768, 1, True, 1),
    ("square4096_nn", 0, 0, 4096, 4096, 4096, 1, False, 0),
    ("square4096_nt", 0, 1, 4096, 4096, 4096, 1, False, 0),
    ("square4096_tn", 1, 0, 4096, 4096, 4096, 1, False, 0),
    ("square4096_tt", 1, 1, 4096, 4096, 4096, 1, False, 0),
]


def run_extras(sg, device, stream):
    """TFLOP/s (2MNK*batch / time, CUDA events, median of reps) of sgemm_ex forms;
    cases whose operands and result fit in L2 get it flushed (a 256 MiB write)
    before every timed repetition."""
    import torch
    out = {}
    sh = stream.cuda_stream
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(5)
    for name, op_a, op_b, M, N, K, batch, has_bias, act in EXTRA_CASES:
        ra, ca = (K, M) if op_a else (M, K)
        rb, cb = (N, K) if op_b else (K, N)
        A = torch.rand((batch, ra, ca), device=device, generator=g) * 2 - 1
        B = torch.rand((batch, rb, cb), device=device, generator=g) * 2 - 1
        C = torch.empty((batch, M, N), device=device)
        bias = (torch.rand(N, device=device, generator=g) - 0.5) if has_bias else None

        def call():
            sg.sgemm_ex_ptr(op_a, op_b, M, N, K, 1.0, A.data_ptr(), ca, ra * ca, B.data_ptr(),
                            cb, rb * cb, 0.0, C.data_ptr(), N, M * N, batch,
                            bias.data_ptr() if bias is not None else 0, act, sh)

        for _ in range(3):
            call()
        torch.cuda.synchronize(device)
        flops = 2.0 * M * N * K * batch
        small = 4 * batch * (ra * ca + rb * cb + M * N) < 200 << 20
        reps = max(5, min(50, int(2e11 / flops)))
        ts = []
        for _ in range(reps):
            if small:
                flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call()
            e1.record(stream)
            torch.cuda.synchronize(device)
            ts.append(e0.elapsed_time(e1) / 1e3)
        ts.sort()
        med = ts[len(ts) // 2]
        out[name] = {"tflops": round(flops / med / 1e12, 3), "ms": round(med * 1e3, 4),
                     "op": ("T" if op_a else "N") + ("T" if op_b else "N"), "batch": batch,
                     "bias": has_bias, "act": "gelu_tanh" if act else None,
                     "l2_flushed": small}
        del A, B, C, bias
    return out


def hbm_peak_gbs() -> tuple[float, str]:
    """Measured HBM copy bandwidth (MEASURED_PEAKS.json), else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "MEASURED_PEAKS.json hbm_gbs"
    except (OSError, ValueError, KeyError):
        return 6800.0, "fallback 6.8 TB/s"


def algorithmic_bytes(p: workloads.Problem) -> int:
    """Minimum HBM traffic of one GEMM: read A and B once, write C once, and
    read C once more when beta != 0."""
    return 4 * (p.M * p.K + p.K * p.N + p.M * p.N * (2 if p.beta != 0 else 1))


def roofline_entry(flops: float, nbytes: float, seconds: float, peak_tflops: float,
                   hbm_gbs: float) -> dict:
    """Roofline of one timed call: the bound is the slower of the compute peak
    and HBM bandwidth for the call's algorithmic bytes; frac = that time over
    the measured time."""
    t_alu = flops / (peak_tflops * 1e12)
    t_hbm = nbytes / (hbm_gbs * 1e9)
    return {"bound": "hbm" if t_hbm > t_alu else "alu",
            "frac": round(max(t_alu, t_hbm) / seconds, 4),
            "hbm_gbs": round(nbytes / seconds / 1e9, 1)}


def run_configs(sg, device, stream, peak_tflops: float, probe_tflops: float | None):
    """Every configured workload: TFLOP/s of sgemm and sgemm_tf32x3 (inputs
    resident, CUDA events, 5 warm-ups, then the median and minimum of 20-40
    repetitions; workloads under 200 MB get the L2 flushed between
    repetitions) with each one's roofline fraction, and the CPU oracle on a
    sample of the workload's rows.

    FFMA roofline: the slower of the fp32 FMA peak (`peak_tflops`) and HBM
    bandwidth for the algorithmic bytes.  Tensor mode: the tf32 tensor peak
    over the three products it computes (2MNK of effective work per 3*2MNK of
    tf32 work), or HBM, whichever is slower."""
    import torch
    sh = stream.cuda_stream
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    bw, _ = hbm_peak_gbs()
    tf32_peak, _ = tf32_peak_tflops()
    out = {}
    for name in workloads.WORKLOADS:
        p = workloads.workload(name)
        A = torch.from_numpy(p.A).to(device)
        B = torch.from_numpy(p.B).to(device)
        C = torch.from_numpy(p.C0).to(device)
        small = p.A.nbytes + p.B.nbytes + p.C0.nbytes < 200 << 20
        nbytes = algorithmic_bytes(p)
        res = {"shape": f"{p.M}x{p.N}x{p.K}", "alpha": p.alpha, "beta": p.beta,
               "algorithmic_flops": int(p.flops), "algorithmic_bytes": int(nbytes),
               "flop_per_byte": round(p.flops / nbytes, 1)}
        for mode, fn in (("ffma", sg.sgemm_ptr), ("tf32x3", sg.sgemm_tf32x3_ptr)):
            def call():
                fn(p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta,
                   C.data_ptr(), p.ldc, sh)
            for _ in range(5):
                call()
            torch.cuda.synchronize(device)
            reps = max(20, min(40, int(1e12 / p.flops)))
            ts = []
            for _ in range(reps):
                if small:
                    flush.zero_()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                call()
                e1.record(stream)
                torch.cuda.synchronize(device)
                ts.append(e0.elapsed_time(e1) / 1e3)
            ts.sort()
            med = ts[len(ts) // 2]
            res[mode] = round(p.flops / med / 1e12, 3)
            res[f"{mode}_ms"] = round(med * 1e3, 4)
            res[f"{mode}_ms_min"] = round(ts[0] * 1e3, 4)
            if mode == "ffma":
                r = roofline_entry(p.flops, nbytes, med, peak_tflops, bw)
                res.update(r)
                if probe_tflops:
                    t_probe = max(p.flops / (probe_tflops * 1e12), nbytes / (bw * 1e9))
                    res["frac_vs_probe"] = round(t_probe / med, 4)
            else:
                r = roofline_entry(p.flops, nbytes, med, tf32_peak / 3.0, bw)
                res["tf32x3_bound"] = "hbm" if r["bound"] == "hbm" else "tensor"
                res["tf32x3_frac"] = r["frac"]
        # the CPU oracle on a bounded sample of rows of the same problem
        rows = min(p.M, max(16, int(2e10 / max(2.0 * p.N * p.K, 1.0))))
        dt, oflops, threads = oracle_rows_rate(p, rows, seed=3)
        res["oracle"] = round(oflops / dt / 1e12, 5)
        res["oracle_sample"] = f"{rows} of {p.M} rows, {threads} threads"
        res["l2_flushed"] = small
        out[name] = res
        del A, B, C
    return out


def ffma_probe(sg, device, sms):
    """Attainable fp32 FMA rate (packed and scalar issue), CUDA-event timed."""
    import torch
    out = {}
    ctas = sms * 8
    buf = torch.empty(ctas * 256, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device).cuda_stream
    iters = 20000
    for packed in (True, False):
        sg.ffma_probe(ctas, 100, buf.data_ptr(), packed, stream)
        torch.cuda.synchronize(device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        sg.ffma_probe(ctas, iters, buf.data_ptr(), packed, stream)
        e1.record()
        torch.cuda.synchronize(device)
        dt = e0.elapsed_time(e1) / 1e3
        out["packed" if packed else "scalar"] = round(ctas * 256 * iters * 128 / dt / 1e12, 3)
    return out


def run_reference(args):
    """The CPU oracle on the same workload: each step a bounded sample of rows."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    p = workloads.workload(args.workload)
    total_steps = args.steps + args.warmup
    budget = float(args.ref_seconds)
    import oracle
    threads = oracle.max_threads()
    dt1, _, _ = oracle_rows_rate(p, threads, seed=99)
    per_step = budget / max(total_steps, 1)
    rows = max(1, min(p.M, int(per_step / max(dt1, 1e-3)) * threads)) if per_step > dt1 else \
        max(1, min(threads, int(threads * per_step / max(dt1, 1e-3))))
    for i in range(args.warmup):
        oracle_rows_rate(p, rows, seed=1000 + i)
    times, flops = [], 0.0
    for i in range(args.steps):
        dt, f, _ = oracle_rows_rate(p, rows, seed=i)
        times.append(dt)
        flops = f
    el = sum(times)
    value = flops * args.steps / el / 1e12
    sample = (f"{rows} of {p.M} rows of C per step ({rows}x{p.N}x{p.K} fp64-accumulated "
              f"multiply-adds), {threads} OpenMP threads")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded uniform[-1,1) inputs, no dataset)",
        "config": {"workload": describe(p), "M": p.M, "N": p.N, "K": p.K},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def parse(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="square8192", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=0,
                    help="steps of the end-to-end leg (default: as many as --steps)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=90.0)
    ap.add_argument("--no-probe", action="store_true",
                    help="skip the fp32 FMA probe (the attainable FMA rate)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the batched / transposed / fused-epilogue sgemm_ex cases")
    ap.add_argument("--no-tf32x3", action="store_true",
                    help="skip the separately reported 3xTF32 tensor-core mode")
    return ap.parse_args(argv)


def main(argv=None):
    args = parse(argv)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
