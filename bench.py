"""Benchmark of the FP32 GEMM C = A x B on the 8192^3 N(0,1) workload.

One step = one product through the C ABI (split pre-pass + GEMM kernel [+
split-K reduce]) with A, B and C resident in HBM.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--path auto|tf32x3|ffma|tf32bf16] [--split-k S]

--impl reference times the CPU oracle (the plain fp64 triple loop) on a
bounded row sample of the same workload.  Under torchrun every rank runs the
same product on its own GPU (independent replicas: the product has no
exchange step), and the value is the aggregate over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from shared_memory_tiled_fp32_gb300.workloads import WORKLOADS, make_inputs, row_order  # noqa: E402

METRIC = "FP32 GEMM TFLOP/s at M=N=K=4096/8192 and % of roofline; max rel error"
DEFAULT_WORKLOAD = "sq8192_normal"
# tf32 : bf16 dense tensor rate on this part.  The instruction-rate probes
# (tcgen05 kind::tf32 and kind::f16 issue loops on operands resident in shared
# memory) measure tf32 at exactly half the f16/bf16 rate (1216 vs 2432 tensor
# TFLOP/s), so the measured bf16 GEMM peak is scaled by 1/2.  (The nominal
# datasheet ratio, 1.1/2.25, is lower and would overstate the fraction.)
TF32_OVER_BF16 = 0.5
# GB300 CUDA cores: 152 SMs x 128 fp32 FMA lanes x 2 FLOP per clock
FFMA_FLOP_PER_CLK = 152 * 128 * 2
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0,
                  "hbm_gbs": 6800.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--path", default="auto", choices=["auto", "tf32x3", "ffma", "tiled", "tf32bf16"])
    ap.add_argument("--split-k", type=int, default=0)
    ap.add_argument("--op-a", default="N", choices=["N", "T"], help="A stored transposed (K x M)")
    ap.add_argument("--op-b", default="N", choices=["N", "T"], help="B stored transposed (N x K)")
    ap.add_argument("--alpha", type=float, default=1.0)
    ap.add_argument("--beta", type=float, default=0.0)
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--sustained-s", type=float, default=1.0,
                    help="seconds of back-to-back steps for the sustained line (0: skip)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle baseline (profiling runs)")
    ap.add_argument("--no-probes", action="store_true", help="skip the instruction-mix peak probes")
    ap.add_argument("--no-alt", action="store_true",
                    help="skip the lines of the other math paths (tf32 + bf16, FFMA) on the headline workload")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the 4096^3 measurement reported beside the 8192^3 headline")
    ap.add_argument("--transpose", action="store_true",
                    help="measure the tiled-transpose variants instead of the GEMM")
    ap.add_argument("--transpose-n", type=int, default=16384)
    ap.add_argument("--reduce", action="store_true", help="measure the sum-reduction variants instead")
    ap.add_argument("--reduce-n", type=int, default=2 ** 28)
    ap.add_argument("--all-configs", action="store_true",
                    help="one JSON line per workload and path (step and kernel throughput)")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(values, device):
    """Element-wise maximum of `values` over all ranks (identity when not
    distributed).  The timed region of the slowest rank bounds the job."""
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_tflops(flop_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank runs one product per step."""
    return flop_per_rank * world / (ms_per_step * 1e-3) / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0=None, t1=None):
        """Summary of the samples taken between wall times t0 and t1 (the
        timed region; the nearest sample after t0 if none fell inside)."""
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        chosen = self.lines
        if t0 is not None:
            inside = [x for x in self.lines if t0 <= x[0] <= t1 + 0.12]
            after = [x for x in self.lines if x[0] >= t0]
            chosen = inside or after[:1] or self.lines[-1:]
        for _, ln in chosen:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxs.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sms:
            return None
        return {"sm_mhz": float(np.median(sms)), "sm_max_mhz": max(maxs), "samples": len(sms),
                "reasons": sorted(reasons)}


def kernel_source_fingerprint() -> str:
    """sha256 (first 16 hex digits) of the kernels' source (tg_kernels.cu and
    the headers it compiles with: tg_internal.h, tg_ptx.cuh) without
    comments and blank lines: the counters in a profile summary stay valid
    while the code they were taken on is unchanged."""
    csrc = os.path.join(ROOT, "shared_memory_tiled_fp32_gb300", "csrc")
    src = "".join(open(os.path.join(csrc, f)).read() for f in ("tg_kernels.cu", "tg_internal.h", "tg_ptx.cuh"))
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in src.splitlines()]
    code = "\n".join(ln for ln in lines if ln.strip())
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def traffic_from_profiles(kernel_tag: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel code (else None)."""
    sha = kernel_source_fingerprint()
    prof = os.path.join(ROOT, "profiles", f"{kernel_tag}_{workload}.md")
    if not os.path.exists(prof):
        return None
    text = open(prof).read()
    m_sha = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_b = re.search(r"dram_bytes_per_full_launch:\s*([0-9.eE+]+)", text)
    if not (m_sha and m_b) or m_sha.group(1) != sha:
        return None
    return float(m_b.group(1))


def oracle_rows_timed(A_np, B_np, rows):
    import oracle

    t0 = time.perf_counter()
    ref = oracle.sgemm_rows(A_np, B_np, rows)
    return ref, time.perf_counter() - t0


def cpu_baseline(w, A_np, B_np, target_s):
    """Time the oracle on a seeded row sample sized to ~target_s seconds."""
    import oracle

    rows_all = row_order(w).numpy()  # seeded random order of the output rows
    probe = rows_all[: max(oracle.threads(), 8)]
    _, t_probe = oracle_rows_timed(A_np, B_np, probe)
    per_row = t_probe / len(probe)
    n = int(min(w.M, max(len(probe), target_s / max(per_row, 1e-9))))
    n = max(oracle.threads(), n // oracle.threads() * oracle.threads())
    rows = np.sort(rows_all[:n])
    ref, t = oracle_rows_timed(A_np, B_np, rows)
    value = 2.0 * len(rows) * w.N * w.K / t / 1e12
    return rows, ref, {"value": value, "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
                       "sample": f"{len(rows)} of {w.M} output rows (all {w.N} columns), seeded; "
                                 f"{t:.1f} s of fp64 triple-loop work",
                       "full_matrix_s_extrapolated": 2.0 * w.M * w.N * w.K / (value * 1e12),
                       "single_thread_s": oracle_single_thread()}


def oracle_single_thread(names=("sq256_uniform", "ragged_777x1029x513")):
    """Whole products of the two small workloads on one host thread (each
    well under a second), seconds per product."""
    import oracle

    n0 = oracle.threads()
    out = {}
    try:
        oracle.set_threads(1)
        for name in names:
            w = WORKLOADS[name]
            A, B = make_inputs(w.M, w.N, w.K, w.dist, w.seed)
            A_np, B_np = A.numpy(), B.numpy()
            t0 = time.perf_counter()
            oracle.sgemm(A_np, B_np)
            out[name] = time.perf_counter() - t0
    finally:
        oracle.set_threads(n0)
    return out


def run_reference(args, w, world, rank):
    if rank != 0:
        return
    import oracle

    A, B = make_inputs(w.M, w.N, w.K, w.dist, w.seed)
    A_np, B_np = A.numpy(), B.numpy()
    rows_all = row_order(w).numpy()
    probe = rows_all[: max(oracle.threads(), 8)]
    _, t_probe = oracle_rows_timed(A_np, B_np, probe)
    per_row = t_probe / len(probe)
    # each step: a bounded row sample sized so the whole run takes ~2 minutes
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(max(oracle.threads(), min(w.M, budget / max(per_row, 1e-9))))
    n = max(oracle.threads(), n // oracle.threads() * oracle.threads())
    for s in range(args.warmup):
        oracle_rows_timed(A_np, B_np, np.sort(rows_all[s * n % w.M:][:n]))
    times = []
    for s in range(args.steps):
        _, t = oracle_rows_timed(A_np, B_np, np.sort(rows_all[(s + args.warmup) * n % w.M:][:n]))
        times.append(t)
    t_step = float(np.mean(times))
    value = 2.0 * n * w.N * w.K / t_step / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "dist": w.dist, "seed": w.seed,
                   "step": f"oracle on {n} sampled output rows"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
                         "sample": f"{n} of {w.M} output rows per step (all {w.N} columns)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_transpose(args, world, rank, local):
    """The pages' transpose study on GB300: every variant on an n x n fp32
    matrix (inputs larger than L2), 8 bytes moved per element, against the
    measured copy bandwidth."""
    import shared_memory_tiled_fp32_gb300 as tg
    import oracle

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    n = args.transpose_n
    gen = torch.Generator(device=dev).manual_seed(11)
    X = torch.randn(n, n, device=dev, generator=gen)
    Y = torch.empty(n, n, device=dev)
    peaks, src = load_peaks()
    out = {}
    for name in ("direct", "tile32", "padded", "swizzled"):
        for _ in range(args.warmup):
            tg.transpose(X, Y, variant=name)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record()
        for _ in range(args.steps):
            tg.transpose(X, Y, variant=name)
        e1.record()
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / args.steps
        gbs = 8.0 * n * n / (ms * 1e-3) / 1e9
        out[name] = {"ms": ms, "GB/s": gbs, "frac_of_copy": gbs / peaks["hbm_gbs"]}
    # parity on a sampled block against the oracle's index permutation
    r0 = n // 3
    blk = X[r0:r0 + 256, :512].cpu().numpy()
    ok = bool(np.array_equal(Y[:512, r0:r0 + 256].cpu().numpy(), oracle.transpose(blk)))
    best = max(out, key=lambda k: out[k]["GB/s"])
    line = {"metric": "tiled transpose GB/s (8 bytes per element)", "value": out[best]["GB/s"], "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": out[best]["ms"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": {"workload": f"transpose_{n}x{n}", "best_variant": best,
                                            "l2": "inputs larger than L2"},
            "roofline": {"bound": "hbm", "achieved": out[best]["GB/s"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": out[best]["GB/s"] / peaks["hbm_gbs"], "traffic": None,
                         "peak_source": f"copy bandwidth, {src}"},
            "variants": out, "parity_sample_bitexact": ok}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reduce(args, world, rank, local):
    """The pages' reduction study on GB300: every variant summing n fp32
    values (4 bytes read per value, inputs larger than L2) against the
    measured copy bandwidth."""
    import shared_memory_tiled_fp32_gb300 as tg
    import oracle

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    n = args.reduce_n
    x = torch.randn(n, device=dev, generator=torch.Generator(device=dev).manual_seed(12))
    res = torch.empty(1, device=dev)
    peaks, src = load_peaks()
    out = {}
    for name in ("interleaved", "sequential", "shuffle", "atomic", "fast"):
        for _ in range(args.warmup):
            tg.reduce_sum(x, res, variant=name)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record()
        for _ in range(args.steps):
            tg.reduce_sum(x, res, variant=name)
        e1.record()
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / args.steps
        gbs = 4.0 * n / (ms * 1e-3) / 1e9
        out[name] = {"ms": ms, "GB/s": gbs, "frac_of_copy": gbs / peaks["hbm_gbs"], "sum": float(res.item())}
    ref = float(oracle.reduce_sum(x.cpu().numpy()))
    for v in out.values():
        v["abs_err_vs_oracle"] = abs(v["sum"] - ref)
    best = max(out, key=lambda k: out[k]["GB/s"])
    line = {"metric": "sum reduction GB/s (4 bytes read per value)", "value": out[best]["GB/s"], "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": out[best]["ms"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": {"workload": f"reduce_sum_{n}", "best_variant": best,
                                            "l2": "inputs larger than L2"},
            "roofline": {"bound": "hbm", "achieved": out[best]["GB/s"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": out[best]["GB/s"] / peaks["hbm_gbs"], "traffic": None,
                         "peak_source": f"copy bandwidth, {src}"},
            "variants": out, "oracle_sum": ref, "sum_abs": float(x.abs().sum().item())}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_all_configs(args, local):
    """Step and GEMM-kernel throughput of every workload on each path (the
    tiled path only where the automatic choice would take it)."""
    import shared_memory_tiled_fp32_gb300 as tg

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    for name, w in WORKLOADS.items():
        A, B = (t.to(dev) for t in make_inputs(w.M, w.N, w.K, w.dist, w.seed))
        C = torch.empty(w.M, w.N, device=dev)
        auto = tg.plan(w.M, w.N, w.K, A=A.data_ptr(), B=B.data_ptr(), C=C.data_ptr())["path"]
        for path in ("tf32x3", "tf32bf16", "ffma") + (("tiled",) if auto == "tiled" else ()):
            plan = tg.plan(w.M, w.N, w.K, A=A.data_ptr(), B=B.data_ptr(), C=C.data_ptr(), path=path)
            ws = torch.empty(max(1, plan["workspace_bytes"] // 4 + 64), device=dev)
            steps = max(3, min(args.steps, int(2e12 / w.flop) + 3))
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
            for e0, e1 in evs:
                e0.record(stream)
                e1.record(stream)
            for _ in range(args.warmup):
                tg.matmul(A, B, out=C, path=path, workspace=ws, stream=stream)
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            s0.record(stream)
            for i in range(steps):
                tg.matmul(A, B, out=C, path=path, workspace=ws, main_begin=evs[i][0], main_end=evs[i][1],
                          stream=stream)
            s1.record(stream)
            torch.cuda.synchronize(dev)
            ms = s0.elapsed_time(s1) / steps
            kms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
            print(json.dumps({"workload": name, "path": path, "M": w.M, "N": w.N, "K": w.K, "steps": steps,
                              "ms_per_step": ms, "tflops": w.flop / (ms * 1e-3) / 1e12, "kernel_ms": kms,
                              "kernel_tflops": w.flop / (kms * 1e-3) / 1e12,
                              "plan": {k: plan[k] for k in ("pair", "split_k", "units", "grid", "tail_units",
                                                            "tail_lanes", "launches")}}), flush=True)
        del A, B, C


def main():
    args = parse()
    world, rank, local = dist_env()
    w = WORKLOADS[args.workload]
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    if args.all_configs:
        if rank == 0:
            run_all_configs(args, local)
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    if args.reduce:
        run_reduce(args, world, rank, local)
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    if args.transpose:
        run_transpose(args, world, rank, local)
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    if args.impl == "reference":
        run_reference(args, w, world, rank)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    import shared_memory_tiled_fp32_gb300 as tg

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    tg.lib()
    A, B = make_inputs(w.M, w.N, w.K, w.dist, w.seed)
    Ad, Bd = A.to(dev), B.to(dev)
    Cd = torch.empty(w.M, w.N, device=dev)
    stream = torch.cuda.current_stream(dev)
    general = args.op_a == "T" or args.op_b == "T" or args.alpha != 1.0 or args.beta != 0.0
    trans_a, trans_b = args.op_a == "T", args.op_b == "T"
    # the general form's operands as stored (transposed copies of the same data)
    As = Ad.t().contiguous() if trans_a else Ad
    Bs = Bd.t().contiguous() if trans_b else Bd
    if args.beta != 0.0:
        Cd.normal_(generator=torch.Generator(device=dev).manual_seed(w.seed + 77))
    plan = tg.plan_general(trans_a, trans_b, w.M, w.N, w.K, As.stride(0), Bs.stride(0), Cd.stride(0),
                           A=As.data_ptr(), B=Bs.data_ptr(), C=Cd.data_ptr(), path=args.path,
                           split_k=args.split_k)
    ws = torch.empty(max(1, plan["workspace_bytes"] // 4 + 64), device=dev)

    def step(ev0=None, ev1=None):
        if general:
            tg.matmul_general(As, Bs, Cd, trans_a=trans_a, trans_b=trans_b, alpha=args.alpha, beta=args.beta,
                              path=args.path, split_k=args.split_k, workspace=ws, stream=stream,
                              main_begin=ev0, main_end=ev1)
        else:
            tg.matmul(Ad, Bd, out=Cd, path=args.path, split_k=args.split_k, workspace=ws,
                      main_begin=ev0, main_end=ev1, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if tg.sync_status() != 0:
        raise RuntimeError("a kernel reported a timeout during warm-up")

    # per-step events around the main GEMM kernel (recorded once to create them)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for e0, e1 in evs:
        e0.record(stream)
        e1.record(stream)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    t_start.record(stream)
    for i in range(args.steps):
        step(*evs[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop(wall0, wall1)
    elapsed_ms = t_start.elapsed_time(t_end)
    main_ms = float(np.mean([e0.elapsed_time(e1) for e0, e1 in evs]))
    elapsed_ms, main_ms = max_over_ranks([elapsed_ms, main_ms], dev)
    status = tg.sync_status()
    if status != 0:
        raise RuntimeError(f"a kernel reported status {status} in the timed region")
    ms_per_step = elapsed_ms / args.steps
    value = job_tflops(w.flop, world, ms_per_step)

    # Sustained: the same step back to back for about --sustained-s seconds,
    # without the per-kernel events (which separate the call's launches), so
    # the part runs into its power limit as a long job does; a short timed
    # region (the default 20 steps, ~60 ms at 8192^3) measures the burst rate.
    sustained_line = None
    if args.sustained_s > 0:
        n_sus = max(args.steps, int(args.sustained_s / max(ms_per_step * 1e-3, 1e-6)))
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sampler2 = ClockSampler(local)
        sampler2.start()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        w0 = time.time()
        s0.record(stream)
        for _ in range(n_sus):
            step()
        s1.record(stream)
        torch.cuda.synchronize(dev)
        w1 = time.time()
        if world > 1:
            torch.distributed.barrier()
        sus_clocks = sampler2.stop(w0, w1)
        (sus_ms,) = max_over_ranks([s0.elapsed_time(s1)], dev)
        if tg.sync_status() != 0:
            raise RuntimeError("a kernel reported a timeout in the sustained region")
        sustained_line = {"value": job_tflops(w.flop, world, sus_ms / n_sus), "unit": "TFLOP/s",
                          "steps": n_sus, "ms_per_step": sus_ms / n_sus, "seconds": sus_ms * 1e-3,
                          "clocks": sus_clocks}

    # end to end through the host-buffer entry point (pinned memory; the
    # untransposed product, which is what that entry point computes)
    e2e_s = None
    if args.e2e_steps > 0 and not general:
        Ap, Bp = A.pin_memory(), B.pin_memory()
        Cp = torch.empty(w.M, w.N).pin_memory()
        tg.sgemm_host(Ap, Bp, Cp, path=args.path, split_k=args.split_k)
        e2e_times = []
        for _ in range(args.e2e_steps):
            t0 = time.perf_counter()
            tg.sgemm_host(Ap, Bp, Cp, path=args.path, split_k=args.split_k)
            e2e_times.append(time.perf_counter() - t0)
        e2e_s = float(np.mean(e2e_times))

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    # ceilings of the instruction mixes on this GPU: the rate of each path's
    # own issue pattern with operands resident in shared memory (a second
    # roofline, beside the one from the measured GEMM peak)
    probes = None
    if not args.no_probes:
        probes = {"tf32_mma_tensor_tflops": tg.binding.probe_tf32_mma_tflops(use_collector=False),
                  "tf32_mma_tensor_tflops_collector": tg.binding.probe_tf32_mma_tflops(use_collector=True),
                  "f16_mma_tensor_tflops": tg.binding.probe_f16_mma_tflops(),
                  "ffma_tflops": tg.binding.probe_ffma_tflops(),
                  "note": "tcgen05 kind::tf32 / kind::f16 M128 N256 issue loops with operands resident in "
                          "shared memory; 16 independent FMA chains per thread"}

    def probe_peak(path):
        """Useful-FLOP ceiling of a path from the probes (None without them)."""
        if probes is None:
            return None
        tf32p, f16p = probes["tf32_mma_tensor_tflops"], probes["f16_mma_tensor_tflops"]
        if path == "tf32x3":
            return tf32p / 3.0
        if path == "tf32bf16":
            return 1.0 / (1.0 / tf32p + 2.0 / f16p)
        return probes["ffma_tflops"]

    peaks, peak_src = load_peaks()
    timed_region_s = elapsed_ms * 1e-3
    sustained = timed_region_s >= 1.0
    math_tflops = 2.0 * w.M * w.N * w.K / (main_ms * 1e-3) / 1e12
    if plan["path"] == "tf32x3":
        bf16 = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
        peak = bf16 * TF32_OVER_BF16 / 3.0
        bound = "tensor"
        peak_note = (f"tf32 dense = {'sustained' if sustained else 'burst'} bf16 of {peak_src} "
                     f"({bf16} TFLOP/s) x 1/2 (the probes' tf32:f16 rate); three tf32 products per "
                     f"useful FMA -> / 3.  The bf16 figure is a cuBLAS GEMM result, not the tensor "
                     f"issue ceiling: see frac_vs_probe")
        kernel_tag = "tf32x3_gemm"
    elif plan["path"] == "tf32bf16":
        # per useful multiply-add: one tf32 product (hi x hi) and two bf16
        # products (hi x lo, lo x hi)
        bf16 = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
        tf32 = bf16 * TF32_OVER_BF16
        peak = 1.0 / (1.0 / tf32 + 2.0 / bf16)
        bound = "tensor"
        peak_note = (f"{'sustained' if sustained else 'burst'} bf16 of {peak_src} ({bf16} TFLOP/s), tf32 = bf16 x "
                     f"1/2; one tf32 and two bf16 products per useful FMA -> 1 / (1/tf32 + 2/bf16)")
        kernel_tag = "tf32bf16_gemm"
    else:
        peak = FFMA_FLOP_PER_CLK * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        bound = "alu"
        peak_note = "152 SMs x 128 FMA lanes x 2 FLOP x max SM clock"
        kernel_tag = "ffma_gemm"
    traffic = traffic_from_profiles(kernel_tag, w.name)
    if sustained_line is not None and plan["path"] in ("tf32x3", "tf32bf16"):
        # the whole step (pre-pass and reduce included) against the sustained
        # peak of the same derivation as the roofline's
        bf16s = peaks["bf16_tflops_sustained"]
        tf32s = bf16s * TF32_OVER_BF16
        ps = tf32s / 3.0 if plan["path"] == "tf32x3" else 1.0 / (1.0 / tf32s + 2.0 / bf16s)
        sustained_line["peak_sustained"] = ps
        sustained_line["step_frac_of_peak"] = sustained_line["value"] / world / ps

    # correctness and the CPU baseline on the same seeded row sample (one
    # GPU only: with N ranks the others have left, and the baseline is a
    # single-process figure)
    cpu = None
    max_rel = None
    if not args.no_cpu and not general and world == 1:
        rows, ref, cpu = cpu_baseline(w, A.numpy(), B.numpy(), args.cpu_seconds)
        got = Cd[torch.from_numpy(rows).to(dev)].cpu().numpy().astype(np.float64)
        r64 = ref.astype(np.float64)
        max_rel = float(np.linalg.norm(got - r64) / np.linalg.norm(r64))
        elt = float(np.abs(got - r64).max() / np.abs(r64).max())
        max_rel = {"normwise_rel": max_rel, "max_abs_over_max_ref": elt, "rows_checked": len(rows)}

    # the metric also names 4096^3: measured the same way, reported beside the headline
    secondary = None
    if not args.no_secondary and w.name == DEFAULT_WORKLOAD and not general and world == 1:
        w2 = WORKLOADS["sq4096_uniform"]
        A2, B2 = (t.to(dev) for t in make_inputs(w2.M, w2.N, w2.K, w2.dist, w2.seed))
        C2 = torch.empty(w2.M, w2.N, device=dev)
        p2 = tg.plan(w2.M, w2.N, w2.K, A=A2.data_ptr(), B=B2.data_ptr(), C=C2.data_ptr(), path=args.path)
        ws2 = torch.empty(max(1, p2["workspace_bytes"] // 4 + 64), device=dev)
        steps2 = max(args.steps, 10)
        ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps2)]
        for e0, e1 in ev2:
            e0.record(stream)
            e1.record(stream)
        for _ in range(args.warmup):
            tg.matmul(A2, B2, out=C2, path=args.path, workspace=ws2, stream=stream)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        s0.record(stream)
        for i in range(steps2):
            tg.matmul(A2, B2, out=C2, path=args.path, workspace=ws2, main_begin=ev2[i][0], main_end=ev2[i][1],
                      stream=stream)
        s1.record(stream)
        torch.cuda.synchronize(dev)
        ms2 = s0.elapsed_time(s1) / steps2
        k2 = float(np.mean([a.elapsed_time(b) for a, b in ev2]))
        secondary = {"workload": w2.name, "value": w2.flop / (ms2 * 1e-3) / 1e12, "unit": "TFLOP/s",
                     "ms_per_step": ms2, "kernel_ms": k2,
                     "kernel_tflops": w2.flop / (k2 * 1e-3) / 1e12,
                     "roofline_frac": w2.flop / (k2 * 1e-3) / 1e12 / peak, "steps": steps2,
                     "l2": "inputs larger than L2 (A+B = 128 MiB)"}
        if probe_peak(plan["path"]):
            secondary["frac_vs_probe"] = w2.flop / (k2 * 1e-3) / 1e12 / probe_peak(plan["path"])
        del A2, B2, C2, ws2

    # the other math paths on the same inputs, one line each: the opt-in tf32 +
    # bf16 cross-product path and the FFMA path, with throughput, the fraction
    # of their own peak and their error on the oracle's rows
    def other_path(path, peak_p, peak_source):
        pa = tg.plan(w.M, w.N, w.K, A=Ad.data_ptr(), B=Bd.data_ptr(), C=Cd.data_ptr(), path=path)
        wsa = torch.empty(max(1, pa["workspace_bytes"] // 4 + 64), device=dev)
        stepsa = max(args.steps, 10)
        eva = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(stepsa)]
        for e0, e1 in eva:
            e0.record(stream)
            e1.record(stream)
        for _ in range(args.warmup):
            tg.matmul(Ad, Bd, out=Cd, path=path, workspace=wsa, stream=stream)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        s0.record(stream)
        for i in range(stepsa):
            tg.matmul(Ad, Bd, out=Cd, path=path, workspace=wsa, main_begin=eva[i][0], main_end=eva[i][1],
                      stream=stream)
        s1.record(stream)
        torch.cuda.synchronize(dev)
        if tg.sync_status() != 0:
            raise RuntimeError(f"a kernel reported a timeout on the {path} path")
        msa = s0.elapsed_time(s1) / stepsa
        ka = float(np.mean([a.elapsed_time(b) for a, b in eva]))
        out = {"path": path, "value": w.flop / (msa * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": msa,
               "kernel_ms": ka, "kernel_tflops": w.flop / (ka * 1e-3) / 1e12,
               "roofline_frac": w.flop / (ka * 1e-3) / 1e12 / peak_p, "peak": peak_p, "steps": stepsa,
               "peak_source": peak_source}
        pp = probe_peak(path)
        if pp:
            out["peak_probe"] = pp
            out["frac_vs_probe"] = w.flop / (ka * 1e-3) / 1e12 / pp
        if cpu is not None:
            got = Cd[torch.from_numpy(rows).to(dev)].cpu().numpy().astype(np.float64)
            r64 = ref.astype(np.float64)
            out["max_rel_error"] = {"normwise_rel": float(np.linalg.norm(got - r64) / np.linalg.norm(r64)),
                                    "max_abs_over_max_ref": float(np.abs(got - r64).max() / np.abs(r64).max()),
                                    "rows_checked": len(rows)}
        return out

    alt = ffma_line = None
    if not args.no_alt and args.path == "auto" and w.name == DEFAULT_WORKLOAD and not general and world == 1:
        bf16 = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
        alt = other_path("tf32bf16", 1.0 / (1.0 / (bf16 * TF32_OVER_BF16) + 2.0 / bf16),
                         "1 / (1/tf32 + 2/bf16), tf32 = bf16 x 1/2, bf16 as the main line")
        ffma_line = other_path("ffma", FFMA_FLOP_PER_CLK * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12,
                               "152 SMs x 128 FMA lanes x 2 FLOP x max SM clock (CUDA-core fp32 peak)")

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "dist": w.dist, "seed": w.seed,
                   "path": plan["path"], "split_k": plan["split_k"], "grid": plan["grid"],
                   "tile": [plan["block_m"], plan["block_n"], plan["block_k"]],
                   "l2": "inputs larger than L2 (A+B = %d MiB, pre-pass copies %d MiB)"
                         % (4 * (w.M * w.K + w.K * w.N) >> 20, plan["workspace_bytes"] >> 20),
                   "parallelism": f"replicas x{world}",
                   **({"op_a": args.op_a, "op_b": args.op_b, "alpha": args.alpha, "beta": args.beta}
                      if general else {})},
        "roofline": {"bound": bound, "achieved": math_tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": math_tflops / peak, "traffic": traffic, "peak_source": peak_note,
                     "kernel": kernel_tag, "kernel_ms": main_ms,
                     **({"peak_probe": probe_peak(plan["path"]),
                         "frac_vs_probe": math_tflops / probe_peak(plan["path"])}
                        if probe_peak(plan["path"]) else {})},
        "cpu_baseline": cpu,
        "e2e": None if e2e_s is None else {
            "value": w.flop / e2e_s / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": 4 * (w.M * w.K + w.K * w.N), "d2h_bytes_per_step": 4 * w.M * w.N,
            "ms_per_step": e2e_s * 1e3},
        "gpu_launches": plan["launches"] * args.steps,
        "max_rel_error": max_rel,
        "clocks": clocks,
        "sustained": sustained_line,
        "probes": probes,
        "secondary": secondary,
        "alt_path": alt,
        "ffma_path": ffma_line,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
