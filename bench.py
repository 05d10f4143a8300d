#!/usr/bin/env python3
"""Benchmark: fused RNN-T loss + gradient on GB300, logit elements per second.

One step = one ``rnnt_loss_fused`` call (offsets/schedule, row pass, alpha/beta
DP, gradient pass, loss check) over the whole BPE-ASR workload: B=16,
T_b ~ U[300, 500], U_b ~ U[50, 100], V=1024, float16 logits ~ N(0, 1.5),
blank=-1, no clamp, in-kernel log-softmax, reduction "sum" (about 4.9e8
logit elements, 1 GB).  Inputs are resident in HBM before timing; L2 is
flushed (512 MiB write) between timed steps and the inputs alone exceed L2.

Prints one JSON line.  ``value`` = logit elements/s over all ranks
(weak scaling: each rank runs its own copy of the workload, no collective on
the data path); ``roofline`` describes the dominant kernel against the
measured HBM copy bandwidth; ``e2e`` times the public Python API with the
step's inputs copied from pinned host memory and the loss copied back;
``cpu_baseline`` times the float64 oracle on the host cores on a bounded
sub-batch.  ``--impl reference`` times that oracle alone (the reference arm).
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "RNN-T loss+grad logit elements/s (fwd+bwd, 1 GB300); % of HBM roofline"
UNIT = "logit elements/s"
FALLBACK_HBM_GBS = 6800.0
REF_BUDGET_S = 120.0    # host time of the reference arm's warm-up and timed steps
STAGES = ("prepare", "row_pass", "alpha_beta_dp", "combine", "grad_pass", "finalize")
KERNEL_FILE = os.path.join(ROOT, "rnn_transducer_loss_gb300", "csrc", "rnnt_gb300.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.txt")


def dist_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    """The maximum of a per-rank scalar over all ranks (identity on one rank).

    The GPU arm passes its CUDA device (NCCL); the multi-rank CPU tests pass
    "cpu" with a gloo process group."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, ms: float, world: int) -> float:
    """Whole-job units/s: every rank processes units_per_rank units (weak
    scaling, one replica per rank) within the slowest rank's ms."""
    return world * units_per_rank / (ms / 1e3)


def load_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    with open(KERNEL_FILE, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches this kernel source."""
    try:
        lines = open(TRAFFIC_FILE).read().splitlines()
    except OSError:
        return None
    kv = dict(l.split("=", 1) for l in lines if "=" in l and not l.startswith("#"))
    if kv.get("source_sha256_16") != kernel_source_hash() or kv.get("workload") != workload:
        return None
    v = kv.get(f"{kernel}.dram_bytes_per_launch")
    return float(v) if v else None


CLOCK_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


def parse_clock_lines(lines):
    """Samples of `nvidia-smi --query-gpu=timestamp,index,clocks.sm,clocks.max.sm,
    power.draw,clocks_event_reasons.active,<the four CLOCK_REASONS>` lines
    (csv, noheader, nounits): [(datetime, sm MHz, max MHz, {active reasons})].
    Lines that do not parse are skipped."""
    import datetime as dt
    out = []
    for line in lines:
        f = [x.strip() for x in line.split(",")]
        if len(f) < 10:
            continue
        try:
            sm, smax = float(f[2]), float(f[3])
        except ValueError:
            continue
        ts = None   # a timestamp in another format leaves the sample untimed
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                ts = dt.datetime.strptime(f[0], fmt)
                break
            except ValueError:
                pass
        out.append((ts, sm, smax, {n for n, v in zip(CLOCK_REASONS, f[6:10])
                                   if v.lower() == "active"}))
    return out


def summarize_clocks(samples, begin, end, loaded_begin=None):
    """The clocks line of the bench: samples taken inside [begin, end] (the
    timed region), or inside [loaded_begin, end] when the timed steps follow a
    pre-roll of the same steps that keeps the GPU under the same load (a short
    timed region holds few 20 ms samples); ``samples_timed`` counts the
    samples inside the timed region itself.  With no sample in the window,
    the three samples nearest to the timed region, and the line says so."""
    out = {}
    w0 = loaded_begin if loaded_begin is not None else begin
    if any(x[0] is None for x in samples):
        inside = list(samples)
        out["note"] = "samples without a readable timestamp: all samples"
    else:
        inside = [x for x in samples if w0 <= x[0] <= end]
        out["samples_timed"] = sum(1 for x in samples if begin <= x[0] <= end)
        if loaded_begin is not None:
            out["window_s"] = round((end - w0).total_seconds(), 3)
            out["window"] = "pre-roll of the same steps, then the timed steps"
    if not inside and samples:
        mid = begin + (end - begin) / 2
        inside = sorted(samples, key=lambda x: abs((x[0] - mid).total_seconds()))[:3]
        out["note"] = "no sample inside the timed region; the 3 nearest samples"
    if not inside:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
    reasons = set().union(*(x[3] for x in inside))
    out.update({"sm_mhz": statistics.median(x[1] for x in inside),
                "sm_max_mhz": max(x[2] for x in inside), "reasons": sorted(reasons),
                "samples": len(inside)})
    return out


class ClockSampler:
    """nvidia-smi clock/throttle samples every 20 ms around the timed region;
    mark() records the region's start and end on the same wall clock."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.window = {}

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", str(self.gpu)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def mark(self, which: str):
        import datetime as dt
        self.window[which] = dt.datetime.now()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        try:
            with open(self.path) as f:
                samples = parse_clock_lines(f)
            os.unlink(self.path)
            return summarize_clocks(samples, self.window["begin"], self.window["end"],
                                    self.window.get("loaded"))
        except Exception as e:   # the clocks line must never stop the bench
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [f"sampler error: {e}"]}


def oracle_sample_run(wl, n_samples: int):
    """Float64 oracle loss+grad over the first n_samples samples; returns (elements, seconds)."""
    import numpy as np
    import oracle
    n = min(n_samples, wl.cfg.B)
    r1 = int(wl.offsets[n])
    t = wl.logits[:r1]
    x = (t.float() if str(t.dtype) == "torch.bfloat16" else t).cpu().numpy()   # exact widening
    t0 = time.perf_counter()
    oracle.rnnt_loss(x, wl.targets[:n], wl.T[:n], wl.U[:n], blank=wl.cfg.blank,
                     clamp=wl.cfg.clamp, reduction=wl.cfg.reduction,
                     fused_log_softmax=wl.cfg.fused)
    dt = time.perf_counter() - t0
    del x
    _ = np  # numpy is the oracle's array type
    return r1 * wl.cfg.V, dt


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine() or "unknown"


def oracle_rate(workload: str, budget_s: float) -> dict:
    """Oracle loss+grad rate on a whole workload, repeated for about budget_s."""
    from rnn_transducer_loss_gb300 import workloads as W
    import oracle
    wl = W.make(workload, "cpu")
    el, dt = oracle_sample_run(wl, wl.cfg.B)
    tot_el, tot_t, reps = el, dt, 1
    while tot_t + dt < budget_s and reps < 50:
        e2, t2 = oracle_sample_run(wl, wl.cfg.B)
        tot_el, tot_t, reps = tot_el + e2, tot_t + t2, reps + 1
    return {"value": tot_el / tot_t, "unit": UNIT, "cores": oracle.num_threads(),
            "sample": f"whole {workload} workload ({el} logit elements) x {reps} runs, "
                      f"{tot_t:.1f} s"}


def oracle_one_thread(workload: str = "char_asr", budget_s: float = 3.0):
    """The oracle on one host thread (OMP_NUM_THREADS=1 in a child process)."""
    code = ("import json, bench; print(json.dumps(bench.oracle_rate(%r, %r)))"
            % (workload, budget_s))
    env = dict(os.environ, OMP_NUM_THREADS="1")
    try:
        out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env,
                             capture_output=True, text=True, timeout=300)
        return json.loads(out.stdout.strip().splitlines()[-1])
    except Exception as e:   # the baseline must never stop the bench
        return {"error": f"{type(e).__name__}: {e}"}


def cpu_baseline(wl, budget_s: float = 15.0):
    import oracle
    cores = oracle.num_threads()
    n = max(1, min(wl.cfg.B, cores))
    el, dt = oracle_sample_run(wl, n)
    total_el, total_t, reps = el, dt, 1
    while total_t + dt < budget_s and reps < 40:
        e2, t2 = oracle_sample_run(wl, n)
        total_el += e2
        total_t += t2
        reps += 1
    return {"value": total_el / total_t, "unit": UNIT, "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"first {n} of {wl.cfg.B} samples ({el} logit elements) x {reps} runs, "
                      f"float64 loss+grad, OpenMP over samples, {total_t:.1f} s",
            "one_thread_char_asr": oracle_one_thread("char_asr")}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    from rnn_transducer_loss_gb300 import workloads as W
    oracle.build()
    wl = W.make(args.workload, "cpu")
    cores = oracle.num_threads()
    n = max(1, min(wl.cfg.B, args.ref_samples or cores))
    # Bounded: size each step's sample so that the warm-up and timed steps
    # together take about REF_BUDGET_S of host time (the rate does not depend
    # on the sample's size).
    _, t1 = oracle_sample_run(wl, n)
    per_step = REF_BUDGET_S / max(1, args.steps + args.warmup)
    if t1 > per_step and n > 1:
        n = max(1, int(n * per_step / t1))
    for _ in range(args.warmup):
        oracle_sample_run(wl, n)
    times, el = [], 0
    for _ in range(args.steps):
        el, dt = oracle_sample_run(wl, n)
        times.append(dt)
    ms = 1e3 * statistics.mean(times)
    value = el / (ms / 1e3)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl, args, l2="host run"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "cpu_model": cpu_model(),
                         "sample": f"first {n} of {wl.cfg.B} samples per step ({el} logit "
                                   f"elements), float64 loss+grad"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(wl, args, l2):
    c = wl.cfg
    out = {"workload": c.name, "B": c.B, "V": c.V, "rows": wl.rows, "elements": wl.elements,
           "logit_dtype": c.dtype, "T_range": list(c.T_range), "U_range": list(c.U_range),
           "blank": c.blank, "clamp": c.clamp, "fused_log_softmax": c.fused,
           "reduction": c.reduction, "seed": c.seed, "l2": l2,
           "parallelism": f"replicas x{args.gpus}" if args.gpus > 1 else "single GPU"}
    if getattr(args, "padded", False):
        out["layout"] = (f"padded (B, max_T, max_U+1, V) = ({c.B}, {int(wl.T.max())}, "
                         f"{int(wl.U.max()) + 1}, {c.V})")
    if getattr(args, "fastemit", 0.0):
        out["fastemit_lambda"] = args.fastemit
    if getattr(args, "big_blanks", ""):
        out["big_blank_durations"] = [int(v) for v in args.big_blanks.split(",")]
    if getattr(args, "sigma", 0.0):
        out["sigma"] = args.sigma
    if getattr(args, "inplace", False):
        out["inplace"] = True
    if getattr(args, "logits", "normal") != "normal":
        out["logits"] = "constant (every logit 0)"
    return out


def make_workload(args, device):
    """The named workload, optionally cut to its first samples or stored in another dtype."""
    from dataclasses import replace
    from rnn_transducer_loss_gb300 import workloads as W
    cfg = W.CONFIGS[args.workload]
    if args.dtype and args.dtype != cfg.dtype:
        cfg = replace(cfg, name=f"{cfg.name}_{args.dtype}", dtype=args.dtype)
    wl = W.make(cfg, device)
    return W.subset(wl, args.samples) if args.samples else wl


def algorithmic_bytes(fused: bool, elements: int, rows: int, out_elements: int,
                      esize: int) -> int:
    """Bytes the method must move per call.  In-kernel log-softmax: one read
    of every lattice logit and one write of every gradient element.  Without
    it only the blank and label log-probabilities of a row are read (2
    elements per row) and every gradient element is written."""
    if fused:
        return elements * esize + out_elements * esize
    return out_elements * esize + 2 * rows * esize


def kernel_roofline(kernel: str, bytes_per_launch: float, kernel_ms: float, step_ms: float,
                    peak: float, peak_kind: str, traffic):
    """Roofline record of the dominant kernel; refused (frac None) when its time
    exceeds the whole step's, which no kernel of the step can do."""
    rec = {"bound": "hbm", "kernel": kernel, "unit": "GB/s", "peak": peak,
           "peak_kind": f"{peak_kind} (hbm_gbs, copy bandwidth)",
           "algorithmic_bytes_per_launch": bytes_per_launch, "kernel_ms": kernel_ms,
           "traffic": traffic}
    if not (kernel_ms > 0) or kernel_ms > step_ms * 1.0001:
        rec.update(achieved=None, frac=None,
                   note=f"kernel time {kernel_ms:.4f} ms exceeds the step's {step_ms:.4f} ms: "
                        "not reported")
        return rec
    ach = bytes_per_launch / (kernel_ms / 1e3) / 1e9
    rec.update(achieved=ach, frac=ach / peak)
    return rec


def dp_latency(trace_rec, T, U):
    """ns per anti-diagonal of the alpha/beta recursions from a task trace:
    per sample, the recursion task's duration / (T_b + U_b)."""
    import numpy as np
    m = trace_rec["kind"] == 1
    if not m.any():
        return None
    b = trace_rec["sample"][m]
    dur_ns = (trace_rec["end_us"][m] - trace_rec["start_us"][m]) * 1e3
    per = dur_ns / (T[b].astype(np.float64) + U[b])
    longest = int(np.argmax(T[b].astype(np.int64) + U[b]))
    return {"median_ns": float(np.median(per)), "max_ns": float(per.max()),
            "min_ns": float(per.min()), "samples": int(m.sum()),
            "longest_lattice": {"T": int(T[b[longest]]), "U": int(U[b[longest]]),
                                "us": float(dur_ns[longest] / 1e3),
                                "ns_per_diagonal": float(per[longest])}}


def run_gpu(args, rank, world, local_rank):
    import numpy as np
    import torch
    import torch.distributed as dist
    from rnn_transducer_loss_gb300 import _native as N
    from rnn_transducer_loss_gb300 import build as B
    from rnn_transducer_loss_gb300 import trace as TR
    from rnn_transducer_loss_gb300 import workloads as W
    from rnn_transducer_loss_gb300.functional import _DT, rnnt_loss_forward

    B.build()
    N.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    wl = make_workload(args, dev)
    cfg = wl.cfg
    if args.logits == "constant":
        wl.logits.zero_()   # every alignment equally likely: the widest posterior band
    rows, V = wl.rows, cfg.V
    dt = _DT[wl.logits.dtype]
    esize = wl.logits.element_size()
    # Options of rnnt_loss_fused_ex: the padded layout and the FastEmit weight.
    x_in = wl.logits
    padded = None
    if args.padded:
        x_in = W.to_padded(wl)
        padded = (x_in.shape[1], x_in.shape[2] - 1)
    in_rows = x_in.numel() // V
    # Multi-blank: big blanks take the outputs below the standard blank (V-1);
    # the workload's labels are folded below them.
    durs = [int(v) for v in args.big_blanks.split(",")] if args.big_blanks else []
    blank_id = cfg.blank + V if cfg.blank < 0 else cfg.blank
    big = [(blank_id - 1 - i, d) for i, d in enumerate(durs)]
    if big:
        if blank_id != V - 1:
            raise SystemExit("--big-blanks needs a workload whose blank is the last output")
        wl.targets[:] = wl.targets % (V - 1 - len(big))
    mb_opts = dict(big_blanks=big, sigma=args.sigma) if (big or args.sigma) else {}
    ex_opts = dict(fastemit_lambda=args.fastemit, padded=padded, **mb_opts)
    use_ex = padded is not None or args.fastemit > 0 or bool(mb_opts)
    targets = torch.as_tensor(wl.targets, device=dev)
    Tl = torch.as_tensor(wl.T, device=dev)
    Ul = torch.as_tensor(wl.U, device=dev)
    nbytes = (N.rnnt_workspace_size_ex(cfg.B, in_rows, V, dt, **mb_opts) if mb_opts
              else N.rnnt_workspace_size(cfg.B, in_rows, V, dt))
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    loss = torch.empty(cfg.B, dtype=torch.float32, device=dev)
    red = torch.empty((), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    # In place: the gradient overwrites the logits; every step first restores
    # them from a pristine copy (a 1 GB copy, which also evicts L2).
    pristine = x_in.clone() if args.inplace else None
    grad = x_in if args.inplace else torch.empty_like(x_in)
    plan = N.rnnt_plan(cfg.B, in_rows, V, dt, targets.shape[1], cfg.fused, True,
                       **(ex_opts if use_ex else {}))
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(128 << 20, dtype=torch.float32, device=dev)

    def flush_l2():
        if args.inplace:
            x_in.copy_(pristine)
            return
        # Write 512 MiB (evicts everything), then read 512 MiB of another buffer so
        # the dirty flush lines are written back here, outside the timed region.
        flush.zero_()
        flush_rd.sum()
    stream = torch.cuda.current_stream(dev)
    red_code = N.REDUCTIONS[cfg.reduction]

    def make_events():
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
        for e in ev:
            e.record(stream)
        return ev

    def step(ev, stages=True):
        # Timed steps record only the first and last event (each extra event
        # record is a few microseconds of stream work); stage breakdowns all 7.
        if use_ex:
            # rnnt_loss_fused_ex records no stage events: time the whole call.
            ev[0].record(stream)
            rc = N.rnnt_loss_fused_ex(
                x_in.data_ptr(), dt, in_rows, V, targets.data_ptr(), targets.shape[1],
                Tl.data_ptr(), Ul.data_ptr(), cfg.B, cfg.blank, cfg.clamp, cfg.fused, red_code,
                loss.data_ptr(), red.data_ptr(), grad.data_ptr(), ws.data_ptr(), nbytes,
                status.data_ptr(), stream.cuda_stream, **ex_opts)
            for e in ev[1:]:
                e.record(stream)
            if rc != N.RNNT_OK:
                raise N.RNNTError(rc, "rnnt_loss_fused_ex")
            return
        handles = [e.cuda_event if (stages or i in (0, 6)) else None for i, e in enumerate(ev)]
        rc = N.rnnt_loss_fused_staged(
            x_in.data_ptr(), dt, rows, V, targets.data_ptr(), targets.shape[1],
            Tl.data_ptr(), Ul.data_ptr(), cfg.B, cfg.blank, cfg.clamp, cfg.fused, red_code,
            loss.data_ptr(), red.data_ptr(), grad.data_ptr(), ws.data_ptr(), nbytes,
            status.data_ptr(), stream.cuda_stream, handles)
        if rc != N.RNNT_OK:
            raise N.RNNTError(rc, "rnnt_loss_fused_staged")

    if args.trace:
        # Task timeline of the call (after two warm calls).
        ev = make_events()
        for _ in range(2):
            flush_l2()
            step(ev)
        flush_l2()
        rec = TR.traced(lambda: step(ev))
        print(json.dumps({"trace": TR.summary(rec),
                          "dp_ns_per_diagonal": dp_latency(rec, wl.T, wl.U)}), flush=True)
        return

    if args.profile_steps:
        # Profiling mode (for ncu): run the path a fixed number of times, report nothing.
        ev = make_events()
        for _ in range(args.profile_steps):
            flush_l2()
            step(ev)
        torch.cuda.synchronize()
        if int(status.item()) != N.RNNT_OK:
            raise N.RNNTError(int(status.item()), "profile run")
        if world > 1:
            dist.destroy_process_group()
        return

    warm_ev = make_events()
    warmup = max(3, args.warmup)
    for _ in range(warmup):
        flush_l2()
        step(warm_ev)
    torch.cuda.synchronize()
    if int(status.item()) != N.RNNT_OK:
        raise N.RNNTError(int(status.item()), "bench warm-up")

    evs = [make_events() for _ in range(args.steps)]
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    # Pre-roll: the same steps for about half a second right before the timed
    # ones, so that the clock samples (every 20 ms) see the GPU under this load
    # even when the timed region itself is short.  Not timed.
    clocks.mark("loaded")
    tp = time.perf_counter()
    while time.perf_counter() - tp < 0.5:
        for _ in range(10):
            flush_l2()
            step(warm_ev, stages=False)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark("begin")
    t0 = time.perf_counter()
    for k in range(args.steps):
        flush_l2()
        step(evs[k], stages=False)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    clocks.mark("end")
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    step_ms = [ev[0].elapsed_time(ev[6]) for ev in evs]
    ms = max_over_ranks(statistics.mean(step_ms), world, dev)
    value = job_throughput(wl.elements, ms, world)

    peak, peak_kind = load_peak()
    step_bytes = algorithmic_bytes(cfg.fused, wl.elements, rows, x_in.numel(), esize)
    stage_ms = None
    if use_ex or plan["persistent"]:
        # The library reports that one kernel runs the whole call (or, for the
        # options, the call is timed as a whole): its time is the timed steps'.
        kname = ("persistent_main" if (plan["persistent"] and plan["launches"] == 1)
                 else "call")
        roof = kernel_roofline(kname, step_bytes, ms, ms, peak, peak_kind,
                               recorded_traffic(kname, cfg.name))
    else:
        # Per-stage kernels: the median of 20 untimed steps that record every
        # stage boundary, and the dominant stage.
        bevs = [make_events() for _ in range(20)]
        for ev in bevs:
            flush_l2()
            step(ev)
        torch.cuda.synchronize()
        stage_ms = {s_: statistics.median(ev[i].elapsed_time(ev[i + 1]) for ev in bevs)
                    for i, s_ in enumerate(STAGES)}
        kernel_bytes = {
            "row_pass": wl.elements * esize if cfg.fused else 2 * rows * esize,
            "grad_pass": (2 * wl.elements * esize if cfg.fused
                          else wl.elements * esize + 2 * rows * esize)}
        dom = max(("row_pass", "alpha_beta_dp", "grad_pass"), key=lambda k: stage_ms[k])
        if dom == "alpha_beta_dp":
            roof = {"bound": "latency", "kernel": dom, "achieved": None, "peak": None,
                    "unit": "GB/s", "frac": None, "traffic": None,
                    "kernel_ms": stage_ms[dom],
                    "note": "the DP is bound by T+U dependent anti-diagonal steps"}
        else:
            roof = kernel_roofline(dom, kernel_bytes[dom], stage_ms[dom], ms, peak, peak_kind,
                                   recorded_traffic(dom, cfg.name))
    step_ach = step_bytes / (ms / 1e3) / 1e9

    # Recursion latency per anti-diagonal, from one traced call (not timed).
    flush_l2()
    rec = TR.traced(lambda: step(make_events()))
    dpl = dp_latency(rec, wl.T, wl.U)
    # Rows the gradient pass had to re-read: those whose gradient is not all zero.
    if not args.inplace:
        nz = int((grad.reshape(in_rows, V) != 0).any(dim=1).sum())
        reread = {"rows_nonzero": nz, "rows": in_rows, "frac": nz / in_rows}
    else:
        reread = None

    # End to end through the public API: pinned host inputs -> device, loss -> host.
    h_logits = (pristine if args.inplace else x_in).cpu().pin_memory()
    h_targets = targets.cpu().pin_memory()
    h_T, h_U = Tl.cpu().pin_memory(), Ul.cpu().pin_memory()
    d_logits = torch.empty_like(x_in)
    d_targets, d_T, d_U = torch.empty_like(targets), torch.empty_like(Tl), torch.empty_like(Ul)
    h_loss = torch.empty(cfg.B, dtype=torch.float32).pin_memory()
    h_red = torch.empty((), dtype=torch.float32).pin_memory()

    def e2e_step():
        d_logits.copy_(h_logits, non_blocking=True)
        d_targets.copy_(h_targets, non_blocking=True)
        d_T.copy_(h_T, non_blocking=True)
        d_U.copy_(h_U, non_blocking=True)
        l, r, g, _ = rnnt_loss_forward(d_logits, d_targets, d_T, d_U, cfg.blank, cfg.clamp,
                                       cfg.reduction, cfg.fused, check=False,
                                       inplace_grad=args.inplace,
                                       fastemit_lambda=args.fastemit, **mb_opts)
        h_loss.copy_(l, non_blocking=True)
        h_red.copy_(r, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for _ in range(max(3, min(args.steps, 10))):
        flush_l2()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms.append(a.elapsed_time(b))
    e2e_t = max_over_ranks(statistics.mean(e2e_ms), world, dev)
    h2d = (h_logits.numel() * h_logits.element_size() + h_targets.numel() * 4
           + h_T.numel() * 4 + h_U.numel() * 4)
    d2h = h_loss.numel() * 4 + 4

    l2 = ("restored from a pristine copy before each step (1 GB copy, evicts L2)"
          if args.inplace else
          "flushed between steps (512 MiB write, then 512 MiB read of another buffer); "
          "inputs 1 GB > L2")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "storage_dtype": cfg.dtype,
        "data": f"synthetic (seeded; shapes and value distribution of the {cfg.name} workload"
                + (", constant logits" if args.logits == "constant" else "") + ")",
        "config": config_of(wl, args, l2=l2),
        "roofline": roof,
        "step_roofline": {"bound": "hbm", "achieved": step_ach, "peak": peak, "unit": "GB/s",
                          "frac": step_ach / peak, "algorithmic_bytes": step_bytes,
                          "note": ("whole call: one logit read + one grad write per element"
                                   if cfg.fused else "whole call: one grad write per element "
                                   "+ the blank and label log-probabilities of each row")},
        "design_roofline_2r1w": {"frac_ceiling": 2 / 3,
                                 "note": "if every row were re-read by the gradient pass"},
        "grad_rows_reread": reread,
        "dp_ns_per_diagonal": dpl,
        "plan": plan,
        "e2e": {"value": job_throughput(wl.elements, e2e_t, world), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_t},
        "gpu_launches": plan["launches"] * args.steps,
        "clocks": clk,
        "wall_ms_timed_region": wall * 1e3,
        "kernel_source_sha256_16": kernel_source_hash(),
    }
    if stage_ms is not None:
        line["stages_ms_median"] = stage_ms
    del h_logits, d_logits
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--workload", default="bpe_asr")
    ap.add_argument("--dtype", choices=("f32", "f16", "bf16"), default=None,
                    help="store the workload's logits in another dtype")
    ap.add_argument("--padded", action="store_true",
                    help="time the padded (B, max_T, max_U+1, V) layout (rnnt_loss_fused_ex)")
    ap.add_argument("--fastemit", type=float, default=0.0,
                    help="FastEmit weight (rnnt_loss_fused_ex)")
    ap.add_argument("--big-blanks", default="",
                    help="multi-blank durations, e.g. 2,4,8 (rnnt_loss_fused_ex)")
    ap.add_argument("--sigma", type=float, default=0.0,
                    help="multi-blank logit under-normalisation")
    ap.add_argument("--ref-samples", type=int, default=0,
                    help="samples per reference step (default: host core count)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--samples", type=int, default=0,
                    help="keep only the first N samples of the workload (profiling)")
    ap.add_argument("--trace", action="store_true",
                    help="print the persistent kernel's task timeline and exit")
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="run the path N times and exit without timing (for ncu)")
    ap.add_argument("--inplace", action="store_true",
                    help="gradient written over the logits (grad == logits)")
    ap.add_argument("--logits", choices=("normal", "constant"), default="normal",
                    help="constant: every logit 0 (all alignments equally likely)")
    args = ap.parse_args(argv)
    rank, world, local_rank = dist_info()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
