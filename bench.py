"""Benchmark of the FP8 block-scaled GEMM on GB300.

One step = one pass of the hot path over the dense workload pair
(4096 x 7168 x 2048 and 4096 x 24576 x 1536, E4M3 with 1x128 / 128x128 fp32
scales, bf16 out): both GEMMs, each launched through the C ABI.  The metric
is TFLOP/s over the step (2*M*N*K per GEMM).  The GEMMs run back to back on
one stream, one CUDA-event pair around the K timed steps; each workload's
inputs rotate over R device copies, with R chosen so that the bytes the other
launches stream through L2 between two uses of a copy exceed twice the L2 size
(so every launch reads inputs that are no longer in L2).  The per-kernel
durations (the roofline's and the per-shape lines') come from a second timed
region per workload: K launches of that GEMM alone, back to back, between one
event pair on its stream (events between launches would serialise them).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

--workload picks another single workload (the other entries of
workloads.WORKLOADS) for measurement runs; the default is the dense pair.
--impl reference times the CPU oracle on the host cores over a bounded sample
of the same workload.  Under torchrun every rank runs the same workload on its
own GPU (independent replicas); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np

import workloads as wl

METRIC = "FP8 block-scaled GEMM TFLOPS (% of GB300 FP8 peak); GB/s at small M"
DEFAULT_PAIR = ["dense_4096x7168x2048", "dense_4096x24576x1536"]
FP8_OVER_BF16 = 2.0      # nominal dense fp8 / bf16 tensor ratio (4.5 / 2.25 PFLOP/s)
HBM_BOUND = {"smallm_64x7168x16384", "smallm_128x7168x16384", "masked_g16_m256_n7168_k2048"}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------------------- ranks

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    if ws <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float, device=None) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, x: float, device=None) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------- peaks

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": pk["hbm_gbs"], "bf16_tflops": pk["bf16_tflops"],
                "bf16_tflops_sustained": pk.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self._reader = threading.Thread(target=self._read, daemon=True)
        self._reader.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if self.t0 and self.t0 - 0.15 <= r[0] <= (self.t1 or 1e30) + 0.15]
        use = inside or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use)}


# ----------------------------------------------------------------------------- GPU arm

class GemmCase:
    """One workload resident on the device, callable through the C ABI."""

    def __init__(self, name, device, dist_rank=0, l2_bytes=0):
        import torch
        from tests import gpu_util as gu
        self.name = name
        t0 = time.time()
        self.p = wl.make(name)
        self.t = gu.dev_tensors(self.p, device)
        self.D = gu.new_d(self.p, device)
        # rotating copies of the inputs: between two uses of one copy the other
        # launches stream more than 2 x L2 through the cache
        in_bytes = sum(v.numel() * v.element_size() for v in self.t.values())
        out_bytes = self.D.numel() * self.D.element_size()
        self.copies = max(2, min(8, -(-2 * l2_bytes // max(1, in_bytes + out_bytes)) + 1)) if l2_bytes else 1
        self.sets = [self.t] + [{k: v.clone() for k, v in self.t.items()} for _ in range(self.copies - 1)]
        self.ws = gu.workspace_for(self.p, device)
        self.flops = self.p.flops()
        self.bytes = self.p.algorithmic_bytes()
        # pinned host copies for the end-to-end measurement; two device input
        # sets (copies 0 and 1) and two outputs let consecutive steps overlap
        self.host = {k: v.cpu().pin_memory() for k, v in self.t.items()}
        self.D_host = [torch.empty(self.D.shape, dtype=self.D.dtype).pin_memory() for _ in range(2)]
        self.D2 = [self.D, torch.empty_like(self.D)]
        self.h2d_bytes = sum(v.numel() * v.element_size() for v in self.host.values())
        self.d2h_bytes = self.D.numel() * self.D.element_size()
        if dist_rank == 0:
            log(f"[bench] {name}: inputs ready in {time.time() - t0:.1f}s")

    def launch(self, stream=None, step=0):
        from tests import gpu_util as gu
        return gu.call(self.p, self.sets[step % self.copies], self.D, workspace=self.ws, stream=stream)

    def e2e_h2d(self, buf):
        """Host -> device copies of the inputs into device set `buf` (0 or 1)."""
        for k, v in self.host.items():
            self.sets[buf][k].copy_(v, non_blocking=True)

    def e2e_gemm(self, buf, stream):
        from tests import gpu_util as gu
        return gu.call(self.p, self.sets[buf], self.D2[buf], workspace=self.ws, stream=stream)

    def e2e_d2h(self, buf):
        """Device -> host copy of output buffer `buf` into pinned memory."""
        self.D_host[buf].copy_(self.D2[buf], non_blocking=True)


def run_ours(args, dist, ws, rank, local):
    import torch
    import fp8_block_scaled_persistent_gb300 as fg

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    fg.library()
    names = DEFAULT_PAIR if args.workload == "dense_pair" else [args.workload]
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    cases = [GemmCase(n, device, rank, l2) for n in names]
    stream = torch.cuda.current_stream(device)

    def step(s, only=None):
        for i, c in enumerate(cases):
            if only is not None and i != only:
                continue
            st = c.launch(stream, s)
            if st != 0:
                raise fg.Fp8GemmError(st, c.name)

    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize()
    fg.check(fg.fp8_gemm_get_device_error(), "warm-up")

    sampler = ClockSampler(local) if rank == 0 and not args.no_clocks else None
    if sampler:
        sampler.start()
    barrier(dist)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_start()
    wall0 = time.time()
    region0 = torch.cuda.Event(enable_timing=True)
    region1 = torch.cuda.Event(enable_timing=True)
    region0.record(stream)
    for s in range(args.steps):
        step(args.warmup + s)
    region1.record(stream)
    torch.cuda.synchronize()
    wall = time.time() - wall0
    if sampler:
        sampler.mark_end()
    barrier(dist)
    clocks = sampler.stop() if sampler else None
    fg.check(fg.fp8_gemm_get_device_error(), "timed steps")

    total_ms = max_over_ranks(dist, region0.elapsed_time(region1), device)

    # per-kernel durations: each workload alone, back to back, one event pair
    per_case_n = max(8, min(args.steps, 400))
    per_case_ms = []
    for i, c in enumerate(cases):
        for s in range(2):
            step(s, only=i)
        e_a = torch.cuda.Event(enable_timing=True)
        e_b = torch.cuda.Event(enable_timing=True)
        e_a.record(stream)
        for s in range(per_case_n):
            step(s, only=i)
        e_b.record(stream)
        torch.cuda.synchronize()
        per_case_ms.append([max_over_ranks(dist, e_a.elapsed_time(e_b), device) / per_case_n])
    fg.check(fg.fp8_gemm_get_device_error(), "per-kernel timing")
    ms_per_step = total_ms / args.steps
    flops_step = sum(c.flops for c in cases)
    bytes_step = sum(c.bytes for c in cases)
    value = sum_over_ranks(dist, flops_step * args.steps, device) / (total_ms / 1e3) / 1e12

    # end-to-end through the C ABI with host buffers (pinned), copies timed.
    # Three streams: inputs in, GEMMs, result out; step s uses device buffer
    # s % 2, so step s+1's inputs travel while step s computes and step s-1's
    # result travels back.  Events keep a buffer from being refilled before
    # its GEMM has read it and an output from being overwritten before it has
    # been copied out.
    e2e_steps = max(4, min(50, args.steps // 20))
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    s_gemm = stream

    def e2e_run(nsteps):
        consumed = [[None, None] for _ in cases]    # GEMM done with input buffer
        copied = [[None, None] for _ in cases]      # output buffer copied out
        for st_i in range(nsteps):
            buf = st_i % 2
            for i, c in enumerate(cases):
                with torch.cuda.stream(s_in):
                    if consumed[i][buf] is not None:
                        s_in.wait_event(consumed[i][buf])
                    c.e2e_h2d(buf)
                    ready = torch.cuda.Event()
                    ready.record(s_in)
                s_gemm.wait_event(ready)
                if copied[i][buf] is not None:
                    s_gemm.wait_event(copied[i][buf])
                rc = c.e2e_gemm(buf, s_gemm)
                if rc != 0:
                    raise fg.Fp8GemmError(rc, c.name)
                done = torch.cuda.Event()
                done.record(s_gemm)
                consumed[i][buf] = done
                with torch.cuda.stream(s_out):
                    s_out.wait_event(done)
                    c.e2e_d2h(buf)
                    out = torch.cuda.Event()
                    out.record(s_out)
                copied[i][buf] = out

    e2e_run(2)
    torch.cuda.synchronize()
    barrier(dist)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_gemm)
    s_in.wait_event(e0)
    e2e_run(e2e_steps)
    s_gemm.wait_stream(s_out)
    e1.record(s_gemm)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(dist, e0.elapsed_time(e1), device)
    e2e_value = sum_over_ranks(dist, flops_step * e2e_steps, device) / (e2e_ms / 1e3) / 1e12

    peaks = load_peaks()
    hbm = args.workload in HBM_BOUND
    # dominant kernel: the case with the largest share of device time
    i_dom = int(np.argmax([sum(x) for x in per_case_ms]))
    dom = cases[i_dom]
    dom_ms = statistics.mean(per_case_ms[i_dom])
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    traffic = load_traffic(dom.name)
    if hbm:
        achieved = dom.bytes / (dom_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                "kernel": f"fp8_gemm_kernel ({dom.name})",
                "peak_source": f"{peaks['source']} HBM copy bandwidth"}
    else:
        achieved = dom.flops / (dom_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": achieved / fp8_peak, "traffic": traffic,
                "kernel": f"fp8_gemm_kernel ({dom.name})",
                "peak_source": f"{peaks['source']} bf16 burst x {FP8_OVER_BF16} (nominal fp8/bf16)"}
    shapes = []
    for i, c in enumerate(cases):
        ms = statistics.mean(per_case_ms[i])
        shapes.append({"workload": c.name, "ms": ms, "tflops": c.flops / (ms / 1e3) / 1e12,
                       "gbs": c.bytes / (ms / 1e3) / 1e9,
                       "frac_fp8_peak": c.flops / (ms / 1e3) / 1e12 / fp8_peak,
                       "frac_hbm": c.bytes / (ms / 1e3) / 1e9 / peaks["hbm_gbs"]})
    out = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": "+".join(names), "accumulate": "f32 per 128-K block, promoted in f32",
                   "output": "bf16", "seed": 0,
                   "l2": "inputs larger than L2: each workload's inputs rotate over "
                         + ", ".join(f"{c.copies}" for c in cases)
                         + " device copies, more than 2 x L2 streamed between two uses of a copy; no flush",
                   "per_kernel_timing": f"{per_case_n} launches of each workload alone, back to back, "
                                        "between one CUDA-event pair on its stream",
                   **({"addend": "fp32 C [M][N], added once (fp8_gemm_nt_accumulate)"}
                      if any(c.p.C is not None for c in cases) else {}),
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "flops_per_step": flops_step, "algorithmic_bytes_per_step": bytes_step},
        "shapes": shapes, "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s",
                "h2d_bytes_per_step": sum(c.h2d_bytes for c in cases),
                "d2h_bytes_per_step": sum(c.d2h_bytes for c in cases), "steps": e2e_steps,
                "overlap": "3 streams (inputs in, GEMMs, result out), double-buffered across steps"},
        "gpu_launches": len(cases) * args.steps,
        "clocks": clocks, "wall_s_timed_region": wall, "impl": "ours",
    }
    return out, cases


def load_traffic(name):
    """DRAM bytes per launch from the committed ncu summary
    (profiles/traffic.txt), or None when it does not describe the current
    kernel."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        parts = line.split("#")[0].split()
        if len(parts) == 2 and parts[0] == name:
            try:
                return float(parts[1])
            except ValueError:
                return None
    return None


# ----------------------------------------------------------------------------- CPU oracle

def oracle_sample(cases_or_names, budget_s: float, threads: int, refs=None):
    """Times the CPU oracle on a bounded sample: for each workload, rows of the
    output (all columns), as many rows as fit the time budget.  Returns
    (TFLOP/s, seconds, description); appends (problem, rows, oracle rows) to
    `refs` when given."""
    import oracle
    probs = []
    for c in cases_or_names:
        p = c.p if hasattr(c, "p") else wl.make(c)
        probs.append(p)
    # calibrate: one row of each
    t0 = time.time()
    for p in probs:
        _run_rows(oracle, p, np.array([0], np.int32), 1)
    per_row = (time.time() - t0) / len(probs)
    rows = max(threads, int(budget_s * threads / max(per_row * len(probs), 1e-6)))
    macs = 0
    t0 = time.time()
    desc = []
    for p in probs:
        r = np.linspace(0, p.M - 1, num=min(rows, p.M)).astype(np.int32)
        ref = _run_rows(oracle, p, r, threads)
        if refs is not None:
            refs.append((p, r, ref))
        macs += len(r) * p.N * p.K
        desc.append(f"{len(r)} rows x {p.N} cols of {p.name}")
    dt = time.time() - t0
    return 2 * macs / dt / 1e12, dt, "; ".join(desc)


def _run_rows(oracle, p, rows, threads):
    if p.kind == "nt":
        return oracle.gemm_nt_rows(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, rows, threads=threads)
    if p.kind == "nt_acc":
        return oracle.gemm_nt_acc_rows(p.A, p.SFA, p.B, p.SFB, p.C, p.M, p.N, p.K, rows, threads=threads)
    if p.kind == "contiguous":
        return oracle.gemm_grouped_contiguous_rows(p.A, p.SFA, p.B, p.SFB, p.m_indices, p.M, p.N,
                                                   p.K, p.G, rows, threads=threads)
    g = int(np.argmax(p.masked_m))
    rows = rows[rows < int(p.masked_m[g])]
    return oracle.gemm_grouped_masked_rows(p.A, p.SFA, p.B, p.SFB, p.masked_m, p.G, p.M, p.N, p.K,
                                           g, rows, threads=threads)


def parity_of(cases, refs):
    """The GPU output the timed launches left in each workload's D against
    the oracle rows of the CPU sample, with the method's tolerance."""
    from tests import gpu_util as gu
    from tests.tolerance import check
    out = {"rows": 0, "elements": 0, "max_err_over_bound": 0.0, "global_diff": 0.0, "ok": True}
    for c, (p, r, ref) in zip(cases, refs):
        d = gu.bits(c.D)
        if p.kind == "masked":
            g = int(np.argmax(p.masked_m))
            r = r[r < int(p.masked_m[g])]
            d = d[g]
        try:
            st = check(d[r], ref, p.name)
        except AssertionError as e:
            out["ok"] = False
            out.setdefault("failures", []).append(str(e))
            continue
        out["rows"] += len(r)
        out["elements"] += st["elements"]
        out["max_err_over_bound"] = max(out["max_err_over_bound"], st["max_err_over_bound"])
        out["global_diff"] = max(out["global_diff"], st["global_diff"])
    return out


def run_reference(args, rank):
    """The oracle on the host cores, each step a bounded sample of the workload."""
    import oracle
    threads = oracle.default_threads()
    names = DEFAULT_PAIR if args.workload == "dense_pair" else [args.workload]
    probs = [wl.make(n) for n in names]
    budget = 90.0 / max(1, args.steps + args.warmup)     # whole run about 1.5 minutes
    # rows per step from a one-row calibration, at least one row per thread... or one row
    t0 = time.time()
    for p in probs:
        _run_rows(oracle, p, np.array([0], np.int32), 1)
    per_row = (time.time() - t0)
    rows = max(1, min(threads, int(budget * threads / max(per_row, 1e-6))))
    rng = np.random.default_rng(0)

    def one_step():
        macs = 0
        for p in probs:
            r = np.sort(rng.choice(p.M, size=rows, replace=False)).astype(np.int32)
            _run_rows(oracle, p, r, min(threads, rows))
            macs += rows * p.N * p.K
        return macs

    for _ in range(args.warmup):
        one_step()
    t0 = time.time()
    macs = 0
    for _ in range(args.steps):
        macs += one_step()
    dt = time.time() - t0
    value = 2 * macs / dt / 1e12
    sample = f"{rows} random rows (all columns) of each of {', '.join(names)} per step"
    return {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "+".join(names), "seed": 0},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": min(threads, rows),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------- main

def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="dense_pair",
                    choices=["dense_pair"] + sorted(wl.WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of CPU oracle work for the cpu_baseline sample")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    ws, rank, local = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank)), flush=True)
        return 0

    dist = init_dist(ws, "nccl")
    out, cases = run_ours(args, dist, ws, rank, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            import oracle
            threads = oracle.default_threads()
            refs = []
            v, dt, sample = oracle_sample(cases, args.cpu_budget, threads, refs)
            out["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                   "sample": sample, "seconds": dt}
            # the measured output itself, on the rows the oracle just computed
            out["parity"] = parity_of(cases, refs)
            # the same oracle on one core, over a smaller row sample; the rate
            # is what the whole workload would take at that pace (extrapolated)
            v1, dt1, sample1 = oracle_sample(cases, max(1.0, args.cpu_budget / 5), 1)
            out["cpu_baseline"]["single_core"] = {
                "value": v1, "unit": "TFLOP/s", "cores": 1, "sample": sample1, "seconds": dt1,
                "full_step_seconds_extrapolated": sum(c.flops for c in cases) / (v1 * 1e12)}
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
