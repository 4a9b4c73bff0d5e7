"""Benchmark of the FP8 block-scaled GEMM on GB300.

One step = one pass of the hot path over the dense workload pair
(4096 x 7168 x 2048 and 4096 x 24576 x 1536, E4M3 with 1x128 / 128x128 fp32
scales, bf16 out): both GEMMs, each launched through the C ABI.  The headline
metric is TFLOP/s over the step (2*M*N*K per GEMM).  The GEMMs run back to
back on one stream, one CUDA-event pair around the K timed steps; each
workload's inputs rotate over R device copies, with R chosen so that the
bytes the other launches stream through L2 between two uses of a copy exceed
twice the L2 size (so every launch reads inputs that are no longer in L2).

Every configuration of the method's evaluation is also measured in the same
run, each in a timed region of its own (``shapes``): the 128 x 256 x 512
latency case, the dense pair, small M (64 and 128 x 7168 x 16384), the
contiguous grouped workload (8 groups, N 4096, K 7168) and the masked one (16
groups of up to 256 rows, N 7168, K 2048).  Each shape is launched at least
200 times back to back over its rotating copies, twice: eagerly through the C
ABI (``ms_eager``) and replayed from one CUDA graph of the same launches
(``ms_graph``: the device time without the host's per-call cost); the
shape's ``ms`` and roofline use the faster of the two batches.  Each shape line carries its roofline (tensor-bound
shapes against the fp8 peak, HBM-bound ones against the copy bandwidth) and
its parity: the output the timed launches left in D against the CPU oracle on
sampled rows (all rows of the small shapes).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--headline-only]

--workload picks another single workload (the other entries of
workloads.WORKLOADS) as the headline; the default is the dense pair.
--impl reference times the CPU oracle on the host cores over a bounded sample
of the same workload.  --gpus N with N > 1 runs N ranks (this script
re-launches itself under torch.distributed.run when it was not started that
way); every rank runs the same workload on its own GPU (independent
replicas), and rank 0 prints one JSON line.
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
# every configuration of the method's evaluation, in the order the shapes
# lines list them
ALL_SHAPES = ["single_128x256x512", "dense_4096x7168x2048", "dense_4096x24576x1536",
              "smallm_64x7168x16384", "smallm_128x7168x16384",
              "contiguous_g8_n4096_k7168", "masked_g16_m256_n7168_k2048",
              # the power-of-two (UE8M0) scale variant on the dense shapes
              "ue8m0_4096x7168x2048", "ue8m0_4096x24576x1536"]
FP8_OVER_BF16 = 2.0      # nominal dense fp8 / bf16 tensor ratio (4.5 / 2.25 PFLOP/s)
FP8_NOMINAL_TFLOPS = 4500.0   # GB300 nominal dense FP8 (no sparsity)
HBM_BOUND = {"smallm_64x7168x16384", "smallm_128x7168x16384", "masked_g16_m256_n7168_k2048"}
LATENCY_BOUND = {"single_128x256x512"}
MIN_SHAPE_LAUNCHES = 200


def bound_of(name):
    if name in LATENCY_BOUND:
        return "latency"
    return "hbm" if name in HBM_BOUND else "tensor"


def kernel_of(name):
    """The library kernel the automatic choice runs for a workload (what the
    launch lists in profiles/ show for it)."""
    if name.startswith("smallm_"):
        return "fp8_gemm_narrow_kernel"
    if name.startswith("ue8m0_"):
        return "fp8_gemm_ue8m0_pair_kernel"
    if name.startswith("dense_") or name.startswith("acc_"):
        return "fp8_gemm_pair_kernel"
    return "fp8_gemm_kernel"


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

    def __init__(self, name, device, dist_rank=0, l2_bytes=0, e2e=False):
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
        self.h2d_bytes = sum(v.numel() * v.element_size() for v in self.t.values())
        self.d2h_bytes = self.D.numel() * self.D.element_size()
        if e2e:
            # pinned host copies for the end-to-end measurement; two device
            # input sets (copies 0 and 1) and two outputs let consecutive
            # steps overlap
            self.host = {k: v.cpu().pin_memory() for k, v in self.t.items()}
            self.D_host = [torch.empty(self.D.shape, dtype=self.D.dtype).pin_memory() for _ in range(2)]
            self.D2 = [self.D, torch.empty_like(self.D)]
        if dist_rank == 0:
            log(f"[bench] {name}: inputs ready in {time.time() - t0:.1f}s ({self.copies} copies)")

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


def _launch_all(fg, case, stream, n, offset=0):
    for s in range(n):
        st = case.launch(stream, offset + s)
        if st != 0:
            raise fg.Fp8GemmError(st, case.name)


def time_shape(fg, case, stream, n, dist, device):
    """Per-launch device time of one workload alone: n launches back to back
    over its rotating copies, (1) eagerly through the C ABI and (2) replayed
    from one CUDA graph that captured the same n launches.  One CUDA-event
    pair on the launching stream around each batch.  Returns (graph ms or
    None, eager ms) per launch, max over ranks."""
    import torch
    _launch_all(fg, case, stream, 3)
    e_a = torch.cuda.Event(enable_timing=True)
    e_b = torch.cuda.Event(enable_timing=True)
    e_a.record(stream)
    _launch_all(fg, case, stream, n)
    e_b.record(stream)
    torch.cuda.synchronize()
    eager = max_over_ranks(dist, e_a.elapsed_time(e_b), device) / n
    fg.check(fg.fp8_gemm_get_device_error(), f"{case.name} eager timing")

    graph_ms = None
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device)
    side.wait_stream(stream)
    with torch.cuda.graph(g, stream=side):
        _launch_all(fg, case, side, n)
    stream.wait_stream(side)
    with torch.cuda.stream(stream):
        g.replay()                       # warm-up replay
        e_a.record(stream)
        g.replay()
        e_b.record(stream)
    torch.cuda.synchronize()
    graph_ms = max_over_ranks(dist, e_a.elapsed_time(e_b), device) / n
    fg.check(fg.fp8_gemm_get_device_error(), f"{case.name} graph timing")
    del g
    return graph_ms, eager


def roofline_entry(case, ms, peaks):
    """The shape's position against its roofline.  t_roof is the slower of
    the FLOPs at the fp8 tensor peak and the algorithmic bytes at the copy
    bandwidth; frac_roofline = t_roof / t."""
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    tflops = case.flops / (ms / 1e3) / 1e12
    gbs = case.bytes / (ms / 1e3) / 1e9
    t_roof = max(case.flops / (fp8_peak * 1e12), case.bytes / (peaks["hbm_gbs"] * 1e9))
    bound = bound_of(case.name)
    e = {"workload": case.name, "bound": bound, "ms": ms, "us": ms * 1e3, "tflops": tflops, "gbs": gbs,
         "frac_roofline": t_roof / (ms / 1e3), "frac_fp8_peak": tflops / fp8_peak,
         "frac_fp8_nominal": tflops / FP8_NOMINAL_TFLOPS, "frac_hbm": gbs / peaks["hbm_gbs"],
         "flops": case.flops, "algorithmic_bytes": case.bytes, "traffic": load_traffic(case.name)}
    if bound == "hbm":
        e.update(achieved=gbs, peak=peaks["hbm_gbs"], unit="GB/s", frac=gbs / peaks["hbm_gbs"])
    elif bound == "tensor":
        e.update(achieved=tflops, peak=fp8_peak, unit="TFLOP/s", frac=tflops / fp8_peak)
    else:
        e.update(achieved=ms * 1e3, peak=None, unit="us", frac=None)
    if case.p.kind == "contiguous":
        e["sum_m"] = int(case.p.M)
    if case.p.kind == "masked":
        e["sum_m"] = int(np.clip(case.p.masked_m, 0, case.p.M).sum())
    return e


def run_ours(args, dist, ws, rank, local):
    import torch
    import fp8_block_scaled_persistent_gb300 as fg

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py (--impl ours) needs a CUDA device")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    fg.library()
    headline = DEFAULT_PAIR if args.workload == "dense_pair" else [args.workload]
    if args.headline_only or args.workload != "dense_pair":
        shape_names = list(headline)
    else:
        shape_names = list(ALL_SHAPES)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    by_name = {}
    for n in dict.fromkeys(headline + shape_names):
        by_name[n] = GemmCase(n, device, rank, l2, e2e=n in headline)
    cases = [by_name[n] for n in headline]
    stream = torch.cuda.current_stream(device)

    def step(s):
        for c in cases:
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
    barrier(dist)
    fg.check(fg.fp8_gemm_get_device_error(), "timed steps")
    total_ms = max_over_ranks(dist, region0.elapsed_time(region1), device)

    # per-shape device times: each workload alone, at least MIN_SHAPE_LAUNCHES
    # launches back to back (eager, and replayed from a CUDA graph)
    per_n = max(args.shape_launches, min(args.steps, 2000))
    timed = {}
    for n in shape_names:
        timed[n] = time_shape(fg, by_name[n], stream, per_n, dist, device)
    if sampler:
        sampler.mark_end()
    clocks = sampler.stop() if sampler else None

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
    fg.check(fg.fp8_gemm_get_device_error(), "end-to-end steps")

    peaks = load_peaks()
    shapes = []
    for n in shape_names:
        graph_ms, eager_ms = timed[n]
        # the faster of the two batches of the same launches: the graph
        # removes the host's per-call cost from short kernels; long kernels
        # are device-bound either way
        use_graph = graph_ms is not None and graph_ms <= eager_ms
        e = roofline_entry(by_name[n], graph_ms if use_graph else eager_ms, peaks)
        e["ms_eager"] = eager_ms
        e["ms_graph"] = graph_ms
        e["launches"] = per_n
        e["timing"] = "CUDA graph replay" if use_graph else "eager"
        shapes.append(e)
    # the dominant kernel of the headline step: the case with the largest
    # share of device time, its per-launch time from its own timed region
    head = [e for e in shapes if e["workload"] in headline] or \
        [roofline_entry(c, ms_per_step, peaks) for c in cases]
    dom = max(head, key=lambda e: e["ms"])
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    roof = {"bound": dom["bound"], "achieved": dom["achieved"], "peak": dom["peak"], "unit": dom["unit"],
            "frac": dom["frac"], "traffic": dom["traffic"], "kernel": f"{kernel_of(dom['workload'])} ({dom['workload']})",
            "ms_per_launch": dom["ms"],
            "peak_source": (f"{peaks['source']} HBM copy bandwidth" if dom["bound"] == "hbm" else
                            f"{peaks['source']} bf16 burst x {FP8_OVER_BF16} (nominal fp8/bf16)")}
    if dom["bound"] == "tensor":
        roof["frac_fp8_nominal"] = dom["frac_fp8_nominal"]
    out = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": "+".join(headline), "accumulate": "f32 per 128-K block, promoted in f32",
                   "output": "bf16", "seed": 0,
                   "l2": "inputs larger than L2: each workload's inputs rotate over "
                         + ", ".join(f"{by_name[n].copies}" for n in headline)
                         + " device copies, more than 2 x L2 streamed between two uses of a copy; no flush",
                   "per_shape_timing": f"{per_n} launches of each workload alone, back to back over its "
                                       "rotating copies, between one CUDA-event pair on its stream: replayed "
                                       "from one CUDA graph (ms_graph) and eagerly through the C ABI "
                                       "(ms_eager); ms is the faster of the two",
                   **({"addend": "fp32 C [M][N], added once (fp8_gemm_nt_accumulate)"}
                      if any(c.p.C is not None for c in cases) else {}),
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "flops_per_step": flops_step, "algorithmic_bytes_per_step": bytes_step,
                   "fp8_peak_tflops": fp8_peak, "hbm_peak_gbs": peaks["hbm_gbs"]},
        "shapes": shapes, "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s",
                "h2d_bytes_per_step": sum(c.h2d_bytes for c in cases),
                "d2h_bytes_per_step": sum(c.d2h_bytes for c in cases), "steps": e2e_steps,
                "overlap": "3 streams (inputs in, GEMMs, result out), double-buffered across steps"},
        "gpu_launches": len(cases) * args.steps,
        "clocks": clocks, "wall_s_timed_region": wall, "impl": "ours",
    }
    return out, cases, [by_name[n] for n in shape_names]


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
    """The GPU output the timed launches left in each headline workload's D
    against the oracle rows of the CPU sample, with the method's tolerance."""
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


def parity_rows(p, extra=24, seed=0):
    """Rows of D to compare for one workload, as (group or None, rows):
    every row of a problem of at most 256 rows; otherwise the first and last
    rows, the rows on both sides of the first 128-row block boundaries and of
    the last one, and `extra` random rows.  Contiguous: also the first and
    last row of every group and the rows on both sides of every group
    boundary.  Masked: per live group, its first and last valid row, the rows
    on both sides of the 128-row boundary when the count crosses it, and a
    few random valid rows."""
    rng = np.random.default_rng(seed)
    if p.kind == "masked":
        out = []
        for g in range(p.G):
            c = int(min(max(int(p.masked_m[g]), 0), p.M))
            if c == 0:
                continue
            rows = {0, c - 1} | ({127, 128} if c > 128 else set())
            rows |= set(int(x) for x in rng.integers(0, c, size=min(3, c)))
            out.append((g, np.array(sorted(r for r in rows if r < c), np.int32)))
        return out
    if p.M <= 256:
        return [(None, np.arange(p.M, dtype=np.int32))]
    must = {0, 1, 127, 128, 255, 256, p.M - 129, p.M - 128, p.M - 1}
    if p.kind == "contiguous":
        lay = np.asarray(p.m_indices)
        edges = np.flatnonzero(np.diff(lay)) + 1          # first row of each later group
        for e in edges:
            must |= {int(e) - 1, int(e)}
    must |= set(int(x) for x in rng.integers(0, p.M, size=extra))
    return [(None, np.array(sorted(r for r in must if 0 <= r < p.M), np.int32))]


def shape_parity(case, threads):
    """The output the timed launches left in the workload's D against the
    oracle on parity_rows, within the method's tolerance; for the masked
    layout also that every row at or past a group's count still holds the
    sentinel the buffer was filled with."""
    import oracle
    from tests import gpu_util as gu
    from tests.tolerance import check
    p = case.p
    d = gu.bits(case.D)
    out = {"rows": 0, "elements": 0, "max_err_over_bound": 0.0, "global_diff": 0.0, "ok": True}
    try:
        for g, rows in parity_rows(p):
            if p.kind == "masked":
                ref = oracle.gemm_grouped_masked_rows(p.A, p.SFA, p.B, p.SFB, p.masked_m, p.G, p.M, p.N, p.K,
                                                      g, rows, threads=threads)
                got = d[g][rows]
            elif p.kind == "contiguous":
                ref = oracle.gemm_grouped_contiguous_rows(p.A, p.SFA, p.B, p.SFB, p.m_indices, p.M, p.N, p.K,
                                                          p.G, rows, threads=threads)
                got = d[rows]
            elif p.kind == "nt_ue8m0":
                ref = oracle.gemm_nt_ue8m0_rows(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, rows, threads=threads)
                got = d[rows]
            elif p.kind == "nt_acc":
                ref = oracle.gemm_nt_acc_rows(p.A, p.SFA, p.B, p.SFB, p.C, p.M, p.N, p.K, rows,
                                              threads=threads)
                got = d[rows]
            else:
                ref = oracle.gemm_nt_rows(p.A, p.SFA, p.B, p.SFB, p.M, p.N, p.K, rows, threads=threads)
                got = d[rows]
            st = check(got, ref, f"{p.name} group {g}" if g is not None else p.name)
            out["rows"] += len(rows)
            out["elements"] += st["elements"]
            out["max_err_over_bound"] = max(out["max_err_over_bound"], st["max_err_over_bound"])
            out["global_diff"] = max(out["global_diff"], st["global_diff"])
        if p.kind == "masked":
            untouched = 0
            for g in range(p.G):
                c = int(min(max(int(p.masked_m[g]), 0), p.M))
                tail = d[g][c:]
                assert (tail == gu.SENTINEL).all(), f"{p.name}: group {g} rows past its count were written"
                untouched += tail.shape[0]
            out["untouched_rows_checked"] = untouched
    except AssertionError as e:
        out["ok"] = False
        out["failure"] = str(e)
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

def relaunch_under_torchrun(argv, n):
    """Runs this script as n ranks under torch.distributed.run on this node
    (127.0.0.1 rendezvous, a free port) and returns its exit status."""
    import socket
    sock = socket.socket()
    sock.bind(("127.0.0.1", 0))
    port = sock.getsockname()[1]
    sock.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__), *argv]
    log(f"[bench] --gpus {n}: launching {n} ranks under torch.distributed.run")
    return subprocess.call(cmd)


def main(argv=None):
    argv = list(sys.argv[1:] if argv is None else argv)
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="dense_pair",
                    choices=["dense_pair"] + sorted(wl.WORKLOADS))
    ap.add_argument("--headline-only", action="store_true",
                    help="time only the headline workload(s), not every configuration")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of CPU oracle work for the cpu_baseline sample")
    ap.add_argument("--shape-launches", type=int, default=MIN_SHAPE_LAUNCHES,
                    help="launches per shape in the per-shape timing (profiling runs use a few)")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")

    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        return relaunch_under_torchrun(argv, args.gpus)
    ws, rank, local = dist_env()
    if ws != args.gpus:
        log(f"[bench] --gpus {args.gpus} does not match WORLD_SIZE={ws}")
        return 2
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank)), flush=True)
        return 0

    dist = init_dist(ws, "nccl")
    out, cases, shape_cases = run_ours(args, dist, ws, rank, local)
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
            # every shape's own output against the oracle
            for e, c in zip(out["shapes"], shape_cases):
                e["parity"] = shape_parity(c, threads)
            out["parity"]["shapes_ok"] = all(e["parity"]["ok"] for e in out["shapes"])
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
