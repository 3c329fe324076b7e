#!/usr/bin/env python
"""Throughput of the exact residue GEMM, one process per GPU.

A step is one call of the whole path (device planner, residue split, per-prime
tensor-core GEMM, balanced Garner) on one synthetic problem already resident in
HBM.  The default workload is the exact int64 product M = N = K = 4096 with
entries uniform in [-2^23, 2^23) (seed 5), the square product the per-prime
GEMM stage's tensor-core fraction is quoted on.  The metric is effective
2*M*N*K / time, in TOPS (10^12 integer operations per second).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on host cores

For N > 1 the script runs under torch.distributed.run; every rank solves its
own full-size problem (weak scaling, no collective on the data path) and rank
0 prints one JSON line with the whole-job throughput.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "exact int GEMM effective TOPS (2·M·N·K/s) & % of INT8 tensor-core roofline"
UNIT = "TOPS"
L2_FLUSH_BYTES = 512 << 20  # larger than the 129 MB L2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="exact24_4096")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip e2e, cpu baseline, the tensor-rate probes and the secondary workloads")
    ap.add_argument("--solve", type=int, default=0, metavar="N",
                    help="instead, time the exact solve of an N x N system with 24-bit entries")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except OSError:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def workload_description(w):
    if w.kind == "int":
        return f"int64 uniform in [{w.lo}, {w.hi})"
    if w.kind == "limbs":
        return f"signed {64 * w.limbs}-bit integers as {w.limbs} int64 limbs, uniform"
    if w.kind == "normal32":
        return "float32 i.i.d. standard normal (the float64 draw rounded)"
    if w.kind == "interval":
        return "float64 intervals: midpoints standard normal, radii uniform in [0, 2^-20) x |midpoint|"
    return "float64 i.i.d. standard normal"


def workload_dtype(w):
    return {"normal": "f64", "interval": "f64", "normal32": "f32"}.get(w.kind, "int64")


# ---------------------------------------------------------------------------
# the reference arm: the CPU oracle, timed on host cores
# ---------------------------------------------------------------------------


def oracle_call(w, A, B, rows):
    import oracle

    if w.kind == "int":
        return oracle.matmul_i64(A, B, lc=1 if w.out_limbs == 1 else w.out_limbs, rows=rows)
    if w.kind == "limbs":
        return oracle.matmul_limbs(A, B, w.out_limbs, rows=rows)
    if w.kind == "normal32":
        return oracle.enclose_f32(A, B, rows=rows)
    if w.kind == "interval":
        return oracle.interval(A[0], A[1], B[0], B[1], rows=rows)
    return oracle.enclose_f64(A, B, rows=rows)


def time_oracle(w, A, B, target_s):
    """Time the oracle on a growing row sample until one run takes about target_s; when even
    the whole problem is quicker, repeat whole passes until they add up to target_s.
    Returns (rows per run, runs, seconds per run)."""
    import numpy as np

    rows = 1
    while True:
        sel = np.arange(rows, dtype=np.int64)
        t0 = time.perf_counter()
        oracle_call(w, A, B, sel)
        dt = time.perf_counter() - t0
        if dt >= target_s:
            return rows, 1, dt
        if rows >= w.M:
            break
        grow = int(rows * min(8.0, max(1.5, target_s / max(dt, 1e-3))))
        rows = min(w.M, max(rows + 1, grow))
    runs = max(1, min(1000, int(target_s / max(dt, 1e-6))))
    t0 = time.perf_counter()
    for _ in range(runs):
        oracle_call(w, A, B, None)
    return rows, runs, (time.perf_counter() - t0) / runs


def cpu_baseline(w, A, B, target_s=12.0):
    import oracle

    rows, runs, dt = time_oracle(w, A, B, target_s)
    value = 2.0 * rows * w.N * w.K / dt / 1e12
    what = (f"{rows} of {w.M} output rows of {w.name} ({rows * w.N * w.K:.3g} MACs), {dt:.2f} s" if runs == 1 else
            f"the whole of {w.name} ({rows * w.N * w.K:.3g} MACs), {runs} passes of {dt:.3f} s")
    return {"value": value, "unit": UNIT, "cores": oracle.threads_used(), "kind": "oracle",
            "sample": f"{what}, C schoolbook with OpenMP on {os.cpu_count()} host cores"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from workloads import WORKLOADS

    w = WORKLOADS[args.workload]
    A, B = w.generate()
    rows, _, dt = time_oracle(w, A, B, 2.0)  # size one step to about two seconds (or one whole pass)
    import numpy as np

    sel = np.arange(rows, dtype=np.int64) if rows < w.M else None
    for _ in range(args.warmup):
        oracle_call(w, A, B, sel)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_call(w, A, B, sel)
        times.append(time.perf_counter() - t0)
    t = sum(times) / len(times)
    value = 2.0 * rows * w.N * w.K / t / 1e12
    import oracle

    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": workload_dtype(w), "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "entries": workload_description(w),
                   "seed": w.seed, "step": f"{rows} output rows per step (bounded sample)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.threads_used(), "kind": "oracle",
                         "sample": f"{rows} of {w.M} output rows of {w.name} per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------


def gemm_traffic_record(path_src):
    """Per-launch DRAM bytes of the GEMM kernel from the committed ncu summary
    (profiles/residue_gemm_traffic.txt), if it was taken on the current kernel
    source; else None."""
    rec_path = os.path.join(ROOT, "profiles", "residue_gemm_traffic.txt")
    try:
        rec = {}
        with open(rec_path) as f:
            for line in f:
                line = line.strip()
                if line and not line.startswith("#") and "=" in line:
                    k, v = line.split("=", 1)
                    rec[k.strip()] = v.strip()
        with open(path_src, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
        return rec if rec.get("source_sha256") == sha else None
    except OSError:
        return None


# ---------------------------------------------------------------------------
# ranks: one process per GPU; bookkeeping only (the data path has no collective)
# ---------------------------------------------------------------------------


def rank_info():
    """(world, rank, local_rank) from the torch.distributed.run environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_ranks(world):
    """A gloo group for the barrier and the timing reduction (host tensors only)."""
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("gloo")


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's value: the whole job ends when its last rank ends."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(total_ms_max: float, steps: int, macs: int, world: int):
    """(value in TOPS, ms per step): every rank processed `steps` problems of
    `macs` multiply-adds (weak scaling); the job took the slowest rank's time."""
    value = world * steps * 2.0 * macs / (total_ms_max * 1e-3) / 1e12
    return value, total_ms_max / steps


def run_solve(args):
    """Wall time of the exact rational solve (the call synchronises), with its phases, and
    the integer identity A N == d b checked on the result."""
    import numpy as np
    import torch

    import exact_modular_int8_gb300 as rg
    from workloads import solve_system

    n = args.solve
    A, b = solve_system(n)
    dA, db = torch.from_numpy(A).cuda(), torch.from_numpy(b).cuda()
    for _ in range(max(1, args.warmup)):
        rg.solve_integers(dA, db)
    times, infos = [], []
    for _ in range(args.steps):
        info = {}
        t0 = time.perf_counter()
        N, d = rg.solve_integers(dA, db, info=info)
        times.append(time.perf_counter() - t0)
        infos.append(info)
    ok = all(sum(int(A[i, k]) * N[k][0] for k in range(n)) == d * int(b[i, 0]) for i in range(n))
    mean = lambda key: sum(x[key] for x in infos) / len(infos)  # noqa: E731
    line = {"metric": "exact rational solve wall time (A x = b, b one column; numerators and common denominator "
                      "as Python ints)", "value": 1e3 * sum(times) / len(times),
            "unit": "ms", "n_gpus": 1, "steps": args.steps, "warmup": max(1, args.warmup),
            "higher_is_better": False, "dtype": "int64", "data": "synthetic",
            "config": {"workload": f"solve24_{n}", "n": n, "c": 1, "entries": "int64 uniform in [-2^23, 2^23)"},
            "phases_ms": {"inverse": mean("ms_inverse"), "lift": mean("ms_lift"),
                          "reconstruct": mean("ms_reconstruct")},
            "lift_steps": infos[-1]["steps"], "primes": infos[-1]["primes"],
            "denominator_bits": d.bit_length(), "identity_A_N_eq_d_b": ok}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.solve:
        run_solve(args)
        return
    import numpy as np
    import torch

    world, rank, local = rank_info()
    init_ranks(world)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import exact_modular_int8_gb300 as rg
    from workloads import WORKLOADS

    w = WORKLOADS[args.workload]
    A, B = w.generate()
    dA = torch.from_numpy(A).to(dev)
    dB = torch.from_numpy(B).to(dev)
    stream = torch.cuda.current_stream(dev)

    def call(out=None):
        if w.kind == "int":
            return rg.res_gemm_i64(dA, dB, nprimes=w.nprimes, sync=False, out=out)
        if w.kind == "limbs":
            return rg.res_gemm_limbs(dA, dB, w.out_limbs, nprimes=w.nprimes, sync=False, out=out)
        if w.kind == "interval":  # A, B hold (midpoint, radius) stacked
            return rg.interval_gemm(dA[0], dA[1], dB[0], dB[1], sync=False, out=out)
        return rg.enclose_gemm(dA, dB, sync=False, out=out)

    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    out = None
    for _ in range(max(args.warmup, 3)):
        out = call()
    torch.cuda.synchronize(dev)
    st = rg.status()
    if st != rg.RG_OK:
        raise SystemExit(f"warm-up call failed: {rg.strerror(st)}")
    plan = rg.get_plan()
    ref_out = [t.clone() for t in out] if isinstance(out, tuple) else out.clone()

    # the timed steps write one preallocated result (out=), as a caller
    # repeating the product would; a fresh allocation can stall the host
    # while the GPU idles inside the step.  Each step replays the call
    # captured once as a CUDA graph (the same kernels on the same buffers,
    # without the host's per-call path); the eager call is timed beside it.
    replay = graphed(torch, lambda: call(out))
    eager_ms = sum(_time_events(torch, dev, lambda: call(out), args.steps, flush)) / args.steps
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    times = []
    for _ in range(args.steps):
        flush.fill_(1.0)  # evict the inputs from L2 between timed steps
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if replay:
            replay()
        else:
            out = call(out)
        e1.record(stream)
        times.append((e0, e1))
    torch.cuda.synchronize(dev)
    barrier(world)
    clock_info = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in times]
    total_ms = sum(step_ms)
    if rg.status() != rg.RG_OK:
        raise SystemExit("a timed call failed")
    same = all(torch.equal(x, y) for x, y in zip(out, ref_out)) if isinstance(out, tuple) else torch.equal(out, ref_out)
    if not same:
        raise SystemExit("timed results differ from the warm-up result")
    total_ms = max_over_ranks(total_ms, world)
    value, ms_per_step = job_throughput(total_ms, args.steps, w.macs, world)

    # ---- the stages inside the call: the same steps again (L2 flushed before
    # each), with events recorded between the stages on the call's stream
    stage_ev = []
    for _ in range(args.steps):
        flush.fill_(1.0)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        rg.set_stage_events(evs)
        call(out)
        stage_ev.append(evs)
    rg.set_stage_events(None)
    torch.cuda.synchronize(dev)
    stages_ms = {name: sum(e[i].elapsed_time(e[i + 1]) for e in stage_ev) / len(stage_ev)
                 for i, name in enumerate(("plan_and_split", "gemm", "garner"))}

    # ---- dominant kernel: the per-prime tensor-core GEMM.  Its in-call
    # duration (above) is the roofline's denominator; for context it is also
    # timed alone on the residue planes the last call left in the workspace,
    # with L2 flushed before each launch (inputs cold in HBM)
    P = plan["nprimes"]
    peaks, peak_src = load_peaks()
    op = {"int": rg.RG_OP_I64, "limbs": rg.RG_OP_LIMBS, "normal": rg.RG_OP_ENCLOSE, "normal32": rg.RG_OP_ENCLOSE_F32,
          "interval": rg.RG_OP_INTERVAL}[w.kind]
    products = 3 if w.kind == "interval" else 1  # an interval product is three exact products
    la = lb = w.limbs if w.kind == "limbs" else 1
    lc = w.out_limbs if w.kind == "limbs" else 1
    L = rg.workspace_layout(op, w.M, w.N, w.K, la, lb, lc, nprimes=w.nprimes)
    ws = rg.workspace(rg.workspace_bytes(op, w.M, w.N, w.K, la, lb, lc, nprimes=w.nprimes), dev)
    # the alone timing runs the first planes of the workspace as one stage call
    # (an interval call's 3P planes are capped at the 53 the stage accepts)
    Pa = min(P * products, len(rg.primes()))
    ra = ws[L.ra:L.ra + Pa * w.M * L.lda * 2].view(torch.float16).view(Pa, w.M, L.lda)
    rb = ws[L.rb:L.rb + Pa * w.K * L.ldb * 2].view(torch.float16).view(Pa, w.K, L.ldb)
    rc = torch.empty((Pa, w.M, L.ldc), dtype=torch.uint8, device=dev)
    for _ in range(3):
        rg.res_gemm_stage(ra, rb, Pa, w.M, w.N, w.K, RC=rc, sync=False)
    gt = []
    for _ in range(args.steps):
        flush.fill_(1.0)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        rg.res_gemm_stage(ra, rb, Pa, w.M, w.N, w.K, RC=rc, sync=False)
        e1.record(stream)
        gt.append((e0, e1))
    torch.cuda.synchronize(dev)
    gemm_alone_ms = sum(a.elapsed_time(b) for a, b in gt) / len(gt)
    gemm_ms = stages_ms["gemm"]
    gemm_flops = 2.0 * w.macs * P * products
    achieved = gemm_flops / (gemm_ms * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])  # fp16 and bf16 share the nominal dense rate
    traffic = gemm_traffic_record(os.path.join(ROOT, "exact_modular_int8_gb300", "csrc", "gemm_tc.cu"))
    traffic_bytes = None
    if traffic and traffic.get("workload") == w.name:
        traffic_bytes = int(traffic["traffic_bytes_per_launch"])
    kernel = ("residue_gemm_pair_kernel (tcgen05.mma cta_group::2 kind::f16, fp32 TMEM)" if w.M > 128 else
              "residue_gemm_kernel (tcgen05.mma cta_group::1 kind::f16, fp32 TMEM)")
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": traffic_bytes, "kernel": kernel,
                "peak_source": f"{peak_src} bf16 dense burst (MEASURED_PEAKS.json); fp16 nominal rate equals bf16",
                "algorithmic_flops_per_launch": gemm_flops, "avg_launch_ms": gemm_ms,
                "avg_launch": "inside the timed call, events on its stream between the stages",
                "alone_cold_inputs_ms": gemm_alone_ms, "alone_planes": Pa, "primes": P, "products_per_prime": products}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": workload_dtype(w), "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "entries": workload_description(w),
                   "seed": w.seed,
                   "nprimes": f"fixed by the caller: {P}" if w.nprimes else f"planned on the device: {P}",
                   "l2": "flushed between timed steps (512 MiB write outside the timed events)",
                   "launch": ("one CUDA graph replay of the captured call per step" if replay else
                              "one eager call per step")},
        "eager_ms_per_step": eager_ms,
        "roofline": roofline,
        "stages_ms": stages_ms,
        # our kernels per call: split, GEMM and reconstruction, the planner for every kind but int64, the
        # int64 split's plane fix-up pass when its planes are large (16 MiB of A and B residues or more), and
        # the slice sum when the layout lets the GEMM split K
        "gpu_launches": ((3 if w.kind == "int" else 4) + (1 if L.splits > 1 else 0) +
                         (1 if w.kind == "int" and not w.nprimes and (w.M + w.N) * w.K * 2 >= (16 << 20) else 0))
        * args.steps * world,
        "clocks": clock_info,
    }

    if rank == 0 and world == 1 and not args.no_extras:
        line["e2e"] = measure_e2e(rg, w, A, B, args, dev)
        rates = rate_probes(rg, torch, dev)
        line["tensor_rates"] = rates
        int8 = rates.get("mma_sync_s8_tops")
        if int8:
            # the metric's INT8 roofline: the warp-level s8 MMA, the only integer
            # tensor-core instruction on sm_103a; the residue GEMM runs on the fp16
            # pipe instead, so this fraction can exceed 1
            line["roofline"]["int8_peak"] = int8
            line["roofline"]["int8_peak_instruction"] = "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32"
            line["roofline"]["frac_of_int8_peak"] = achieved / int8
        f16 = rates.get("tcgen05_f16_tflops")
        if f16:
            # context: the instruction's own measured rate, from shared-memory operands with no data movement
            line["roofline"]["f16_instruction_peak"] = f16
            line["roofline"]["frac_of_f16_instruction_peak"] = achieved / f16
        line["secondary"] = secondary_workloads(rg, torch, dev, flush, w, dA, dB, out, peak, args)
        line["cpu_baseline"] = cpu_baseline(w, A, B)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def measure_e2e(rg, w, A, B, args, dev):
    """The same call with host buffers: copies in and out inside the timed region."""
    import torch

    hA = torch.from_numpy(A).pin_memory()
    hB = torch.from_numpy(B).pin_memory()
    if w.kind == "int":
        out = torch.empty((w.M, w.N), dtype=torch.int64).pin_memory()
        fn = lambda: rg.res_gemm_i64(hA, hB, nprimes=w.nprimes, out=out)
        d2h = out.numel() * 8
    elif w.kind == "limbs":
        out = torch.empty((w.M, w.N, w.out_limbs), dtype=torch.int64).pin_memory()
        fn = lambda: rg.res_gemm_limbs(hA, hB, w.out_limbs, nprimes=w.nprimes, out=out)
        d2h = out.numel() * 8
    elif w.kind == "interval":
        fn = lambda: rg.interval_gemm(hA[0], hA[1], hB[0], hB[1])
        d2h = 2 * w.M * w.N * 8
    else:
        fn = lambda: rg.enclose_gemm(hA, hB)
        d2h = 2 * w.M * w.N * A.itemsize
    for _ in range(3):
        fn()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fn()  # synchronises: the result is on the host when it returns
    dt = (time.perf_counter() - t0) / args.steps
    return {"value": 2.0 * w.macs / dt / 1e12, "unit": UNIT, "h2d_bytes_per_step": int(A.nbytes + B.nbytes),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": dt * 1e3,
            "api": "exact_modular_int8_gb300 call on pinned host tensors (C ABI with RG_FLAG_HOST; large int64 "
                   "products pipeline A's row blocks and C's over the link)"}


def graphed(torch, fn):
    """fn (one library call on fixed buffers: stream-ordered, no host synchronisation) captured
    once into a CUDA graph after a run on a side stream; returns the graph's replay, or None if
    the capture fails."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(g):
            fn()
    except RuntimeError:
        torch.cuda.synchronize()
        return None
    return g.replay


def _time_events(torch, dev, fn, reps, flush=None):
    """Per-launch milliseconds of fn() over `reps` launches, each bracketed by events on the
    current stream (L2 flushed before each when `flush` is given)."""
    ev = []
    for _ in range(reps):
        if flush is not None:
            flush.fill_(1.0)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        ev.append((e0, e1))
    torch.cuda.synchronize(dev)
    return [a.elapsed_time(b) for a, b in ev]


def rate_probes(rg, torch, dev):
    """Peak rates of the tensor-core instructions a residue product could run on, measured
    here: the warp-level INT8 MMA (the metric's INT8 roofline), tcgen05 kind::f16 (what the
    residue GEMM uses) and kind::f8f6f4 E4M3 (what an FP8 digit split would use); plus the
    INT8 library GEMM (torch._int_mm, 8192^3) for context.  Best of five launches after three
    warm-ups, CUDA events on the launching stream; SM clocks sampled over the probes."""
    out = {}
    clocks = ClockSampler(dev.index)
    clocks.start()
    for key, kind, iters in (("mma_sync_s8_tops", rg.RG_PROBE_MMA_S8, 20000),
                             ("tcgen05_f16_tflops", rg.RG_PROBE_TCGEN05_F16, 8192),
                             ("tcgen05_e4m3_tflops", rg.RG_PROBE_TCGEN05_E4M3, 8192),
                             ("mma_sync_f16_tflops", rg.RG_PROBE_MMA_F16, 20000)):
        ops = [0.0]

        def launch(kind=kind, iters=iters, ops=ops):
            ops[0] = rg.probe_mma_rate(kind, iters)

        for _ in range(3):
            launch()
        ms = _time_events(torch, dev, launch, 5)
        if rg.status() != rg.RG_OK:
            out[key] = None
            continue
        out[key] = ops[0] / (min(ms) * 1e-3) / 1e12
        out[key.rsplit("_", 1)[0] + "_ms"] = min(ms)
    out["clocks"] = clocks.stop()
    if out.get("tcgen05_f16_tflops") and out.get("tcgen05_e4m3_tflops"):
        # an FP8 balanced base-17 digit split needs three E4M3 sub-products per fp16 one
        out["e4m3_over_f16"] = out["tcgen05_e4m3_tflops"] / out["tcgen05_f16_tflops"]
        out["fp8_digit_split_speedup"] = out["e4m3_over_f16"] / 3.0
    try:
        n = 8192
        a = torch.randint(-128, 128, (n, n), dtype=torch.int8, device=dev)
        b = torch.randint(-128, 128, (n, n), dtype=torch.int8, device=dev)
        for _ in range(2):
            torch._int_mm(a, b)
        out["int8_library_tops"] = 2.0 * n**3 / (min(_time_events(torch, dev, lambda: torch._int_mm(a, b), 5)) *
                                                 1e-3) / 1e12
        del a, b
    except Exception:  # noqa: BLE001 - a missing library kernel only removes a context figure
        out["int8_library_tops"] = None
    return out


def _stage_times(rg, torch, dev, flush, fn, reps):
    """Mean per-stage milliseconds (split, GEMM, Garner) of fn() with the stage-event hook."""
    st = []
    for _ in range(reps):
        flush.fill_(1.0)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        rg.set_stage_events(evs)
        fn()
        rg.set_stage_events(None)
        st.append(evs)
    torch.cuda.synchronize(dev)
    return {n: sum(e[i].elapsed_time(e[i + 1]) for e in st) / len(st)
            for i, n in enumerate(("split_ms", "gemm_ms", "garner_ms"))}


def secondary_workloads(rg, torch, dev, flush, w, dA, dB, ref, peak, args):
    """Context figures beside the headline line, each call timed alone with L2 flushed before
    it: the 1024^3 exact product (the latency-bound size), and, for an int64 headline, the same
    call on all 53 primes (batched-prime scaling; its integers must equal the planned call's)."""
    from workloads import WORKLOADS

    res = {}
    reps = max(args.steps, 10)
    if w.name != "exact24_1024":
        s = WORKLOADS["exact24_1024"]
        A, B = s.generate()
        sA, sB = torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev)
        o = rg.res_gemm_i64(sA, sB)
        o_ref = o.clone()
        eager = _time_events(torch, dev, lambda: rg.res_gemm_i64(sA, sB, sync=False, out=o), reps, flush)
        replay = graphed(torch, lambda: rg.res_gemm_i64(sA, sB, sync=False, out=o))
        ms = _time_events(torch, dev, replay, reps, flush) if replay else eager
        stages = _stage_times(rg, torch, dev, flush, lambda: rg.res_gemm_i64(sA, sB, sync=False, out=o), reps)
        P = rg.get_plan()["nprimes"]
        if rg.status() != rg.RG_OK or not torch.equal(o, o_ref):
            raise SystemExit("the replayed 1024^3 product differs from the eager one")
        res["exact24_1024"] = {"call_ms": sum(ms) / len(ms), "call_effective_tops": 2.0 * s.macs / (
            sum(ms) / len(ms) * 1e-3) / 1e12, "call_ms_median": sorted(ms)[len(ms) // 2],
            "call_ms_eager": sum(eager) / len(eager), "launch": "CUDA graph replay" if replay else "eager",
            **stages, "primes": P,
            "gemm_frac_of_fp16_peak": 2.0 * s.macs * P / (stages["gemm_ms"] * 1e-3) / 1e12 / peak}
    if w.kind == "int" and not w.nprimes:
        P53 = len(rg.primes())
        o53 = rg.res_gemm_i64(dA, dB, nprimes=P53)
        if rg.status() != rg.RG_OK or not torch.equal(o53, ref):
            raise SystemExit("the 53-prime call differs from the planned one")
        ms = _time_events(torch, dev, lambda: rg.res_gemm_i64(dA, dB, nprimes=P53, sync=False, out=o53), 3, flush)
        st = _stage_times(rg, torch, dev, flush, lambda: rg.res_gemm_i64(dA, dB, nprimes=P53, sync=False, out=o53), 3)
        tf = 2.0 * w.macs * P53 / (st["gemm_ms"] * 1e-3) / 1e12
        res["all_53_primes"] = {**st, "call_ms": sum(ms) / len(ms), "gemm_tflops": tf, "frac_of_fp16_peak": tf / peak}
    return res


if __name__ == "__main__":
    main()
