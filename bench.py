"""Benchmark of the attention forward pass on GB300 (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one attention forward (the whole hot path) over one batch of seeded
synthetic input. The default workload is the long-sequence causal one
(B=2 H=16 N=8192 d=128, bf16), whose Q, K, V (201 MB) exceed the 129 MB L2,
so no flush is needed between steps. FLOPs are counted as 4*B*H*N^2*d, halved
under causal masking.

Under torchrun each rank runs an independent replica on its own GPU (the work
units share nothing), so the value is the total FLOPs of all ranks over the
slowest rank's time ("weak" scaling).

On one GPU the line also carries two records outside the timed region:
``per_config`` (forward and backward TFLOP/s on each of the five measured
workloads, each timed by the same rule: L2 flushed before every launch when
the inputs fit in it, back to back otherwise; workloads that fit in L2 are
also timed back to back over rotating cold copies of their inputs, which
leaves out the per-launch event pair's fixed cost) and ``sustained`` (the default
workload back to back for about 1.5 s with the SM clock sampled, reported
against the measured sustained peak as well).

--impl reference times the fp64 CPU oracle on this machine's host cores on a
bounded sample of the same workload (the pages ship no runnable code; the
oracle is the reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s on 1 GB300 (bf16) and fraction of dense BF16 peak"
UNIT = "TFLOP/s"
KERNEL_SOURCES = ("blocked_online_softmax_gb300/csrc/attn_fwd_sm103.cu",
                  "blocked_online_softmax_gb300/csrc/sm103_ptx.cuh")
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="causal_b2h16n8192d128")
    ap.add_argument("--dtype", choices=("bf16", "fp16"), default="bf16",
                    help="element type of q, k, v, o for --op attention (the host-buffer e2e leg is bf16 only)")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target oracle sample time")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload record (every measured workload, forward and backward)")
    ap.add_argument("--sustained-seconds", type=float, default=1.5,
                    help="length of the back-to-back sustained leg on the default workload (0 = skip)")
    ap.add_argument("--op", choices=("attention", "softmax", "backward"), default="attention",
                    help="attention (the default hot path), the fused row softmax (a memory-bound workload), "
                         "or the attention backward pass")
    ap.add_argument("--softmax-shape", default="32768x4096", help="rows x cols of the --op softmax matrix (fp32)")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The slowest rank's value (the job's time is set by its last replica)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step: float, steps: int, world: int, seconds: float) -> float:
    """Whole-job TFLOP/s: every rank runs its own replica of the workload (weak scaling)."""
    return flops_per_step * steps * world / seconds / 1e12


def code_without_comments(text: str) -> str:
    """C/C++/CUDA source with its comments and blank lines removed and each line
    stripped (these sources hold no comment markers inside string literals)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    lines = (re.sub(r"//.*", "", ln).strip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_source_hash() -> str:
    """Hash of the attention kernel's code (the counters in profiles/ are tied to
    it); comments do not enter it, so a comment-only edit keeps the counters."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            code = code_without_comments(f.read())
        h.update(os.path.basename(rel).encode() + b"\0" + code.encode())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"bf16_tflops": FALLBACK_BF16_TFLOPS}, "fallback"


def recorded_traffic(workload_name: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current kernel."""
    path = os.path.join(ROOT, "profiles", f"attn_fwd_{workload_name}_traffic.txt")
    try:
        fields = {}
        with open(path) as f:
            for line in f:
                if ":" in line:
                    key, val = line.split(":", 1)
                    fields[key.strip()] = val.strip()
        if fields.get("kernel_source_sha") != kernel_source_hash():
            return None
        return float(fields["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        self.t0 = time.time()

    def mark(self):
        self.t_start = time.time()

    def stop(self):
        self.t_end = time.time()
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                        rows.append(parts)
            os.unlink(self.path)
        except OSError:
            pass
        return self.summarise(rows)

    @staticmethod
    def summarise(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        smax = max(float(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, val in zip(names, r[5:9]) if val.lower() == "active"})
        # samples taken while the kernel ran (the GPU at least half-way up its clock range)
        loaded = [s for s in sm if s >= 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows if _isnum(r[3]))
                if any(_isnum(r[3]) for r in rows) else None}


def _isnum(s):
    try:
        float(s)
        return True
    except ValueError:
        return False


def oracle_rows_flops(w, rows):
    """FLOPs of the sampled rows by the same rule as the metric: 4*d per visited (row, key) pair."""
    import numpy as np
    i = np.asarray(rows) % w.N
    keys = (i + 1) if w.causal else np.full_like(i, w.N)
    return float(4.0 * w.d * keys.sum())


def time_oracle(w, q, k, v, target_seconds):
    """Time the oracle as it stands on evenly spaced rows of head 0, about target_seconds long."""
    import numpy as np

    import oracle
    oracle.build()
    cores = oracle.max_threads()
    probe = np.arange(0, w.N, max(1, w.N // 64), dtype=np.int64)
    t0 = time.perf_counter()
    oracle.attention(q, k, v, w.scale, w.causal, rows=probe)
    dt = max(time.perf_counter() - t0, 1e-6)
    per_flop = dt / oracle_rows_flops(w, probe)
    head_flops = oracle_rows_flops(w, np.arange(w.N))
    if head_flops * per_flop < 4.0 * target_seconds:
        # a few rows overstate the cost per FLOP (thread start-up, uneven rows):
        # re-estimate on one whole head when that is cheap
        t0 = time.perf_counter()
        oracle.attention(q, k, v, w.scale, w.causal, rows=np.arange(w.N, dtype=np.int64))
        per_flop = max(time.perf_counter() - t0, 1e-6) / head_flops
    # grow the sample to about target_seconds; whole heads first, then strided rows of one head
    n_heads = int(max(0, min(w.B * w.H, target_seconds / (per_flop * head_flops))))
    if n_heads >= 1:
        rows = np.arange(n_heads * w.N, dtype=np.int64)
        desc = f"{n_heads} whole head(s) of {w.B * w.H} ({n_heads * w.N} query rows)"
    else:
        stride = max(1, int(math.ceil(head_flops * per_flop / max(target_seconds, 1e-3))))
        rows = np.arange(0, w.N, stride, dtype=np.int64)
        desc = f"every {stride}th query row of head 0 ({rows.size} rows)"
    t0 = time.perf_counter()
    oracle.attention(q, k, v, w.scale, w.causal, rows=rows)
    dt = time.perf_counter() - t0
    flops = oracle_rows_flops(w, rows)
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{desc}; fp64 C oracle, three-pass softmax over materialised score rows; "
                      f"{dt:.2f} s", "seconds": dt, "host_cpus": len(os.sched_getaffinity(0))}


def run_reference(args, w):
    """The reference arm: the fp64 oracle on the host cores, bounded per-step samples."""
    import numpy as np

    import oracle
    from blocked_online_softmax_gb300.workloads import workload_qkv
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    oracle.build()
    cores = oracle.max_threads()
    q, k, v = workload_qkv(w)
    budget = 120.0 / max(1, args.steps + args.warmup)         # seconds per step
    probe = np.arange(0, w.N, max(1, w.N // 32), dtype=np.int64)
    t0 = time.perf_counter()
    oracle.attention(q, k, v, w.scale, w.causal, rows=probe)
    per_flop = (time.perf_counter() - t0) / oracle_rows_flops(w, probe)
    head_flops = oracle_rows_flops(w, np.arange(w.N))
    stride = max(1, int(math.ceil(head_flops * per_flop / budget)))
    rows = np.arange(0, w.N, stride, dtype=np.int64)
    flops = oracle_rows_flops(w, rows)
    for _ in range(args.warmup):
        oracle.attention(q, k, v, w.scale, w.causal, rows=rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attention(q, k, v, w.scale, w.causal, rows=rows)
    dt = time.perf_counter() - t0
    value = flops * args.steps / dt / 1e12
    sample = (f"per step: every {stride}th query row of head 0 ({rows.size} rows) of {w.name}; "
              f"fp64 C oracle on {cores} threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w):
    in_bytes = 3 * w.B * w.H * w.N * w.d * 2
    return {"workload": w.describe(), "name": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
            "causal": w.causal, "scale": w.scale, "logit_mult": w.logit_mult,
            "flops_per_step": w.flops, "parallelism": "replicas (one per GPU)",
            "l2": f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB > 129 MB), no flush"
            if in_bytes > 129e6 else "L2 flushed between steps, outside the timed launches"}


def time_forward_launches(w, dev, launches, q=None, k=None, v=None):
    """Mean device time of one forward launch on workload w, by the bench's rule:
    inputs larger than L2 run back to back between two events; inputs that fit
    get a 256 MB write before every launch and an event pair around each launch."""
    import torch

    import blocked_online_softmax_gb300 as bos
    from blocked_online_softmax_gb300.workloads import workload_qkv
    if q is None:
        q, k, v = (t.to(dev) for t in workload_qkv(w))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    in_bytes = 3 * q.numel() * 2
    flush = torch.empty(int(256e6) // 4, dtype=torch.float32, device=dev) if in_bytes <= 129e6 else None
    launch = lambda: bos.attn_fwd(q, k, v, o, lse, w.B, w.H, w.N, w.d, w.scale, w.causal, stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            if flush is not None:
                flush.zero_()
            launch()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(launches)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for s_ev, e_ev in ev:
            if flush is not None:
                flush.zero_()
                s_ev.record(stream)
            launch()
            if flush is not None:
                e_ev.record(stream)
        t1.record(stream)
    torch.cuda.synchronize(dev)
    if flush is not None:
        ms = statistics.fmean(s_ev.elapsed_time(e_ev) for s_ev, e_ev in ev)
        mode = "CUDA events around each launch, L2 flushed before each"
    else:
        ms = t0.elapsed_time(t1) / launches
        mode = "back-to-back launches between two CUDA events (inputs larger than L2)"
    return ms, mode


def time_backward_steps(w, dev, steps):
    """Mean device time of one attn_bwd call (three launches) on workload w, with the
    forward's timing rule (L2 flushed before each step when the step's inputs fit)."""
    import torch

    import blocked_online_softmax_gb300 as bos
    from blocked_online_softmax_gb300.workloads import workload_qkv
    q_h, k_h, v_h = workload_qkv(w)
    do_h = torch.randn(q_h.shape, generator=torch.Generator().manual_seed(99)).to(torch.bfloat16)
    q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
    o, lse = bos.attention(q, k, v, scale=w.scale, causal=w.causal)
    nbytes = bos.attn_bwd_workspace_bytes(w.B, w.H, w.N, w.d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    stream = torch.cuda.current_stream(dev)
    in_bytes = 5 * q.numel() * 2
    flush = torch.empty(int(256e6) // 4, dtype=torch.float32, device=dev) if in_bytes <= 129e6 else None
    step = lambda: bos.attn_bwd(q, k, v, o, do, lse, None, dq, dk, dv, ws, nbytes, w.B, w.H, w.N, w.d, w.scale,
                                w.causal, stream)
    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s_ev, e_ev in ev:
        if flush is not None:
            flush.zero_()
            s_ev.record(stream)
        step()
        if flush is not None:
            e_ev.record(stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if flush is not None:
        return statistics.fmean(s_ev.elapsed_time(e_ev) for s_ev, e_ev in ev), \
            "CUDA events around each step, L2 flushed before each"
    return t0.elapsed_time(t1) / steps, "back-to-back steps between two CUDA events (inputs larger than L2)"


def time_forward_rotating(w, dev, launches):
    """Mean device time of one forward launch on workload w, back to back over
    rotating copies of the inputs whose total exceeds the 129 MB L2 (so each
    launch still reads cold inputs), with no event or flush between launches:
    the launch's own time without the fixed cost of the per-launch event pair."""
    import torch

    import blocked_online_softmax_gb300 as bos
    from blocked_online_softmax_gb300.workloads import workload_qkv
    base = workload_qkv(w)
    in_bytes = 3 * base[0].numel() * 2
    ncopy = max(2, int(math.ceil(260e6 / in_bytes)) + 1)
    copies = []
    for _ in range(ncopy):
        q, k, v = (t.to(dev) for t in base)
        copies.append((q, k, v, torch.empty_like(q), torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)))
    stream = torch.cuda.Stream(device=dev)
    run = lambda i: bos.attn_fwd(*copies[i % ncopy], w.B, w.H, w.N, w.d, w.scale, w.causal, stream)
    with torch.cuda.stream(stream):
        for i in range(2 * ncopy):
            run(i)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for i in range(launches):
            run(i)
        t1.record(stream)
    torch.cuda.synchronize(dev)
    return t0.elapsed_time(t1) / launches, ncopy


def per_config_record(dev, peak, peak_sus, launches=30, bwd_steps=10):
    """Forward and backward on every measured workload (the five of the survey's
    measurement table), each by the bench's timing rule."""
    from blocked_online_softmax_gb300.workloads import WORKLOADS
    out = []
    for w in WORKLOADS:
        ms, mode = time_forward_launches(w, dev, launches)
        tf = w.flops / (ms / 1e3) / 1e12
        rec = {"name": w.name, "workload": w.describe(), "fwd_tflops": tf, "fwd_frac": tf / peak,
               "fwd_frac_of_sustained": tf / peak_sus, "fwd_mean_launch_ms": ms, "fwd_launches": launches,
               "fwd_timing": mode}
        if 3 * w.B * w.H * w.N * w.d * 2 <= 129e6:
            # inputs that fit in L2: also back to back over rotating cold copies,
            # which leaves out the per-launch event pair's fixed cost
            rms, ncopy = time_forward_rotating(w, dev, 2 * launches)
            rtf = w.flops / (rms / 1e3) / 1e12
            rec.update({"fwd_rotating_tflops": rtf, "fwd_rotating_frac": rtf / peak,
                        "fwd_rotating_mean_launch_ms": rms,
                        "fwd_rotating_timing": f"back-to-back launches between two CUDA events over {ncopy} "
                                               "rotating input copies (more than L2 in all)"})
        bms, bmode = time_backward_steps(w, dev, bwd_steps)
        btf = 2.5 * w.flops / (bms / 1e3) / 1e12
        rec.update({"bwd_tflops": btf, "bwd_frac": btf / peak, "bwd_mean_step_ms": bms,
                    "bwd_over_fwd_latency": bms / ms, "bwd_steps": bwd_steps, "bwd_timing": bmode,
                    "bwd_flops_counted": "2.5x the forward's (five N^2 d products)"})
        out.append(rec)
    return out


def sustained_record(w, dev, seconds, peak, peak_sus, q, k, v):
    """The default workload back to back for about `seconds`, clocks sampled throughout."""
    ms_probe, _ = time_forward_launches(w, dev, 5, q, k, v)
    launches = max(10, int(seconds * 1e3 / max(ms_probe, 1e-3)))
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    sampler.mark()
    ms, mode = time_forward_launches(w, dev, launches, q, k, v)
    clocks = sampler.stop()
    tf = w.flops / (ms / 1e3) / 1e12
    mhz = clocks.get("sm_mhz")
    return {"workload": w.name, "launches": launches, "seconds": ms * launches / 1e3, "tflops": tf,
            "frac": tf / peak, "frac_of_sustained": tf / peak_sus, "mean_launch_ms": ms, "timing": mode,
            "clocks": clocks,
            "launch_kcycles_at_median_sm_clock": (ms * mhz) if mhz else None}


def run_ours(args, w):
    import torch

    import blocked_online_softmax_gb300 as bos
    from blocked_online_softmax_gb300 import _build
    from blocked_online_softmax_gb300.workloads import workload_qkv

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    _build.build()
    bos.load_library()

    f16 = args.dtype == "fp16"
    if f16:
        from blocked_online_softmax_gb300.workloads import make_qkv
        q_h, k_h, v_h = make_qkv(w.B, w.H, w.N, w.d, w.seed, w.logit_mult, dtype=torch.float16)
    else:
        q_h, k_h, v_h = workload_qkv(w)
    q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def launch():
        if f16:
            bos.attn_fwd_ex(q, k, v, o, lse, w.B, w.H, w.N, w.d, None, None, None, None, w.scale, w.causal,
                            bos.ATTN_DTYPE_F16, stream)
        else:
            bos.attn_fwd(q, k, v, o, lse, w.B, w.H, w.N, w.d, w.scale, w.causal, stream)
    in_bytes = 3 * q.numel() * 2
    flush = None
    if in_bytes <= 129e6:
        flush = torch.empty(int(256e6) // 4, dtype=torch.float32, device=dev)

    def step():
        if flush is not None:
            flush.zero_()
        launch()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(local_rank)
    sampler.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.mark()
    # Inputs larger than L2: the K launches run back to back between two events
    # (per-launch events in between would also stop a launch's set-up from
    # overlapping the previous one). Inputs that fit in L2: an L2 flush runs
    # before every launch and per-launch events keep it out of the launch time.
    with torch.cuda.stream(stream):
        t_begin.record(stream)
        for i in range(args.steps):
            if flush is not None:
                flush.zero_()
                starts[i].record(stream)
            launch()
            if flush is not None:
                ends[i].record(stream)
        t_end.record(stream)
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop()
    total_ms = t_begin.elapsed_time(t_end)
    if flush is not None:
        # the flushes run between the timed launches: the steps' time is the
        # sum of the per-launch event pairs
        launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        total_ms = sum(launch_ms)
    else:
        launch_ms = [total_ms / args.steps]
    total_ms = max_over_ranks(total_ms, dist, dev)
    value = job_throughput(w.flops, args.steps, world, total_ms / 1e3)

    # end to end through the host-buffer entry point (pinned host memory)
    e2e_value, e2e_steps = None, 0
    if not args.no_e2e and not f16:
        qp, kp, vp = (t.pin_memory() for t in (q_h, k_h, v_h))
        op = torch.empty_like(q_h).pin_memory()
        lp = torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()
        e2e_steps = max(1, min(args.steps, 200))
        bos.attn_fwd_host(qp, kp, vp, op, lp, w.B, w.H, w.N, w.d, w.scale, w.causal, stream)
        if dist is not None:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            bos.attn_fwd_host(qp, kp, vp, op, lp, w.B, w.H, w.N, w.d, w.scale, w.causal, stream)
        e2e_s = time.perf_counter() - t0
        e2e_s = max_over_ranks(e2e_s, dist, dev)
        e2e_value = job_throughput(w.flops, e2e_steps, world, e2e_s)

    peaks, peaks_kind = measured_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    avg_launch_ms = statistics.fmean(launch_ms)
    achieved = w.flops / (avg_launch_ms / 1e3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                "frac": achieved / peak, "traffic": None if f16 else recorded_traffic(w.name),
                "peak_kind": f"{peaks_kind} dense bf16 burst (cuBLAS)",
                "kernel": "attn_fwd", "mean_launch_ms": avg_launch_ms,
                "launch_timing": ("K back-to-back launches between two CUDA events" if flush is None
                                  else "CUDA events around each launch, L2 flushed before each"),
                "algorithmic_bytes": 8.0 * w.B * w.H * w.N * w.d + 4.0 * w.B * w.H * w.N,
                "frac_of_sustained": achieved / float(peaks.get("bf16_tflops_sustained", peak))}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = time_oracle(w, *((t.double() if f16 else t) for t in (q_h, k_h, v_h)), args.cpu_seconds)

    per_config, sustained = None, None
    peak_sus = float(peaks.get("bf16_tflops_sustained", peak))
    if rank == 0 and world == 1 and not f16:
        if not args.no_per_config:
            per_config = per_config_record(dev, peak, peak_sus)
        if args.sustained_seconds > 0:
            sustained = sustained_record(w, dev, args.sustained_seconds, peak, peak_sus, q, k, v)

    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return 0
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16" if f16 else "bf16", "data": "synthetic",
            "config": workload_config(w),
            "frac_of_peak": value / world / peak,
            "roofline": roofline, "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "steps": e2e_steps,
                    "h2d_bytes_per_step": int(in_bytes),
                    "d2h_bytes_per_step": int(o.numel() * 2 + lse.numel() * 4),
                    "api": "attn_fwd_host (pinned host buffers; copies, kernel, copies back, sync)"},
            "gpu_launches": args.steps, "clocks": clocks,
            "kernel_source_sha": kernel_source_hash(),
            "per_config": per_config, "sustained": sustained}
    print(json.dumps(line), flush=True)
    return 0


SOFTMAX_SOURCES = ("blocked_online_softmax_gb300/csrc/softmax_rows.cu",)


def run_softmax(args):
    """The fused row softmax on one GPU: GB/s against the measured HBM copy bandwidth.

    Algorithmic bytes: one read and one write of the fp32 matrix (rows that fit
    on chip), or two reads and one write (the online two-pass path). The matrix
    is larger than L2, so the K launches run back to back between two events.
    """
    import torch

    import blocked_online_softmax_gb300 as bos
    rows, cols = (int(v) for v in args.softmax_shape.lower().split("x"))
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = torch.Generator().manual_seed(11)
    x_h = torch.randn(rows, cols, generator=g)
    x = x_h.to(dev)
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream()
    passes = 2 if cols <= 16384 else 3
    nbytes = float(passes) * rows * cols * 4
    for _ in range(max(3, args.warmup)):
        bos.softmax_rows_fwd(x, y, rows, cols, cols, cols, stream)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(0)
    sampler.start()
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    sampler.mark()
    t_begin.record(stream)
    for _ in range(args.steps):
        bos.softmax_rows_fwd(x, y, rows, cols, cols, cols, stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    total_ms = t_begin.elapsed_time(t_end)
    gbs = nbytes * args.steps / (total_ms / 1e3) / 1e9
    peaks, peaks_kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))
    h = hashlib.sha256()
    for rel in SOFTMAX_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    traffic = None
    try:   # the committed capture of a smaller matrix, scaled by the element count
        fields = {}
        with open(os.path.join(ROOT, "profiles", "softmax_rows_16384x4096_traffic.txt")) as f:
            for ln in f:
                if ":" in ln:
                    key, val = ln.split(":", 1)
                    fields[key.strip()] = val.strip()
        if fields.get("kernel_source_sha") == h.hexdigest()[:16] and int(fields["cols"]) == cols:
            traffic = float(fields["dram_bytes_per_launch"]) * rows / int(fields["rows"])
    except (OSError, KeyError, ValueError):
        traffic = None
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        oracle.build()
        xs = x_h.numpy()
        t0 = time.perf_counter()
        done = 0
        while time.perf_counter() - t0 < min(args.cpu_seconds, 10.0) and done < rows:
            oracle.softmax_rows(xs[done:done + 64])
            done += 64
        dt = time.perf_counter() - t0
        cpu = {"value": 2.0 * done * cols * 4 / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"first {done} rows of the same matrix; fp64 three-pass softmax per row; {dt:.2f} s"}
    line = {"metric": "fused row softmax GB/s on 1 GB300 (fp32)", "value": gbs, "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"row softmax fp32 {rows}x{cols}", "rows": rows, "cols": cols,
                       "l2": f"matrix {rows * cols * 4 / 1e6:.0f} MB read + written per step (> 129 MB L2), no flush"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "traffic": traffic, "peak_kind": f"{peaks_kind} copy bandwidth",
                         "kernel": "softmax_rows_fwd", "algorithmic_bytes": nbytes,
                         "mean_launch_ms": total_ms / args.steps},
            "cpu_baseline": cpu, "e2e": None, "gpu_launches": args.steps, "clocks": clocks,
            "kernel_source_sha": h.hexdigest()[:16]}
    print(json.dumps(line), flush=True)
    return 0


def run_backward(args, w):
    """The attention backward pass (attn_bwd) on one GPU, on the chosen workload.

    FLOPs counted: five 2*N*N*d products per (batch, head) (S, dP, dV, dK, dQ),
    i.e. 10*B*H*N^2*d, halved under causal masking (2.5x the forward count). The
    timed step is the whole backward call (D preprocess, key-block kernel, dQ
    cast); the forward outputs it needs are computed once before timing.
    """
    import torch

    import blocked_online_softmax_gb300 as bos
    from blocked_online_softmax_gb300.workloads import workload_qkv
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    q_h, k_h, v_h = workload_qkv(w)
    g = torch.Generator().manual_seed(99)
    do_h = torch.randn(q_h.shape, generator=g).to(torch.bfloat16)
    q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
    o, lse = bos.attention(q, k, v, scale=w.scale, causal=w.causal)
    nbytes = bos.attn_bwd_workspace_bytes(w.B, w.H, w.N, w.d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    stream = torch.cuda.current_stream()
    step = lambda: bos.attn_bwd(q, k, v, o, do, lse, None, dq, dk, dv, ws, nbytes, w.B, w.H, w.N, w.d, w.scale,
                                w.causal, stream)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(0)
    sampler.start()
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler.mark()
    t_begin.record(stream)
    for _ in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    total_ms = t_begin.elapsed_time(t_end)
    flops = 2.5 * w.flops
    tf = flops * args.steps / (total_ms / 1e3) / 1e12
    peaks, peaks_kind = measured_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    line = {"metric": "attention bwd TFLOP/s on 1 GB300 (bf16)", "value": tf, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.describe().replace("attention fwd", "attention bwd"), "name": w.name, "B": w.B, "H": w.H, "N": w.N,
                       "d": w.d, "causal": w.causal, "flops_per_step": flops,
                       "l2": "inputs larger than L2, no flush" if 5 * w.B * w.H * w.N * w.d * 2 > 129e6
                       else "inputs fit in L2, no flush"},
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": UNIT, "frac": tf / peak,
                         "traffic": None, "peak_kind": f"{peaks_kind} dense bf16 burst (cuBLAS)",
                         "kernel": "attn_bwd (3 kernels per step)", "mean_launch_ms": total_ms / args.steps},
            "cpu_baseline": None, "e2e": None, "gpu_launches": 3 * args.steps, "clocks": clocks,
            "kernel_source_sha": kernel_source_hash()}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.op == "softmax":
        return run_softmax(args)
    from blocked_online_softmax_gb300.workloads import BY_NAME
    if args.workload not in BY_NAME:
        raise SystemExit(f"unknown workload {args.workload}; choose from {sorted(BY_NAME)}")
    w = BY_NAME[args.workload]
    if args.op == "backward":
        return run_backward(args, w)
    if args.impl == "ours":
        args.warmup = max(3, args.warmup)          # at least 3 untimed warm-up steps
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
