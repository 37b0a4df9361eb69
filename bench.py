"""Benchmark of batched speculative-sampling verification on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config 4] [--op verify|sample|filtered|lmhead|tree]
                    [--per-config 5,1,2,3]

A step is one verification call over one batch of the workload (all accept
tests, first-rejection scans and correction / bonus draws of every sequence).
The default workload is the largest one by bytes: B=256 sequences, k=8 draft
positions, V=151936, fp32 logits, per-sequence temperature from
{0, 0.5, 1.0, 1.3} (2.6 GB of logits per step, far larger than the 129 MB L2,
so no L2 flush is needed between steps).  Inputs are synthetic (seeded numpy,
see speculative_decoding_verification_65_gb300/synth.py).

The verify run also measures the other workloads in the same process and
reports them under `per_config`: workload 5 at full size (one call per step)
and workloads 1-3 under CUDA graph replay (they are launch-bound), each with
its roofline, stage times, clocks and oracle baseline.

Metric: verified draft positions per second (B*k / step time), summed over
ranks.  Under torchrun every rank verifies its own batch of B sequences
(weak scaling: sequences are independent, so there is no collective on the
data path; one scalar all-reduce takes the max time over ranks).

`--op filtered` benchmarks top-k / top-p filtered verification on the same
workloads (default workload 5, top-k 50, top-p 0.9), the draft tokens drawn
from the filtered draft distribution.

`--op sample` benchmarks the batched sampler instead (one token per row from
softmax(logits / T), the draft model's step before verification): a step is
one spec_sample call over the draft rows of a workload (default workload 5:
4096 rows of V=128256 bf16, 1.05 GB), metric sampled tokens per second.

`--op tree` benchmarks tree verification (several candidate continuations
per sequence): a step is one spec_verify_tree call over 512 trees of 29
nodes (4 first-level candidates, 2 below each, then two single
continuations) over V=128256 bf16, T from {0, 0.7, 1}; metric verified tree
candidates per second (B*(N-1) / step time).  Its roofline counts the bytes
the walk must read once: the rows of the nodes it visits.

Prints one JSON line on rank 0.
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

import numpy as np  # noqa: E402

METRIC = "verified draft positions/sec"
UNIT = "positions/s"
CSRC = os.path.join(ROOT, "speculative_decoding_verification_65_gb300", "csrc")
# the sources each timed kernel is built from (keys of profiles/traffic.json)
KERNEL_SRCS = {
    "stats_kernel": [os.path.join(CSRC, "spec_verify.cu"), os.path.join(CSRC, "device_common.cuh")],
    "chunk_kernel": [os.path.join(CSRC, "spec_sample.cu"), os.path.join(CSRC, "device_common.cuh")],
    "wfilter_kernel": [os.path.join(CSRC, "spec_verify.cu"), os.path.join(CSRC, "device_common.cuh")],
    "gemm_kernel": [os.path.join(CSRC, "spec_lmhead.cu"), os.path.join(CSRC, "device_common.cuh")],
    "tree_kernel": [os.path.join(CSRC, "spec_tree.cu"), os.path.join(CSRC, "device_common.cuh")],
}
SAMPLE_METRIC = "sampled tokens/sec"
SAMPLE_UNIT = "tokens/s"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(x: float, world: int, device=None) -> float:
    """The maximum of a scalar over all ranks (the step time every rank waits
    for); a no-op on one rank.  Works on nccl (device tensor) and gloo (host
    tensor) process groups."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units_per_rank: int, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time (weak scaling: every rank has its own batch)."""
    return world * units_per_rank * steps / max_seconds


def read_probe_gbs(dev, reps: int = 20, nbytes: int = 4 << 30):
    """Read bandwidth of the library's streaming read probe over a buffer far
    larger than L2 (CUDA events on the launch stream, after warm-up)."""
    import torch
    import speculative_decoding_verification_65_gb300 as sv
    buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    sink = torch.empty(sv.spec_bench_read_sink_words(), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        sv.spec_bench_read(buf, sink, stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        sv.spec_bench_read(buf, sink, stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    gbs = nbytes * reps / (e0.elapsed_time(e1) / 1e3) / 1e9
    del buf, sink
    torch.cuda.empty_cache()
    return gbs


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def kernel_source_hash(kernel: str = "stats_kernel") -> str:
    h = hashlib.sha256()
    for path in KERNEL_SRCS[kernel]:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str = "stats_kernel"):
    """DRAM bytes per launch from an ncu capture, if it was taken on the
    current kernel sources (profiles/traffic.json)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(workload)
    if not ent or ent.get("kernel") != kernel or ent.get("kernel_sha") != kernel_source_hash(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
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
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


def make_workload(cfg: int, rank: int, batch=None):
    from speculative_decoding_verification_65_gb300 import synth
    return synth.make_config(cfg, B=batch, seed_offset=100 * rank)


def time_oracle(case, budget_s: float, threads: int):
    """Oracle throughput on a bounded sample: chunks of `threads` sequences
    until the time budget is spent or the batch is done."""
    import oracle
    done, t_used = 0, 0.0
    chunk = max(threads, 1)
    while done < case.B and t_used < budget_s:
        idx = np.arange(done, min(case.B, done + chunk))
        sub = case.subset(idx)
        t0 = time.perf_counter()
        oracle.verify(sub.target, sub.draft, sub.tokens, sub.u_accept, sub.u_resample,
                      sub.temperature, nthreads=threads, want_trace=False)
        t_used += time.perf_counter() - t0
        done += len(idx)
    return done * case.k / t_used, done, t_used


def oracle_alpha(case, n_seq: int):
    """Analytic acceptance of the workload: alpha_i = sum_x min(p_i, q_i)
    = 1 - sum_x max(0, p_i - q_i), averaged over the drafted positions of the
    first `n_seq` sampling sequences (fp64, the oracle's softmax and residual).
    Returns (mean, positions)."""
    import oracle
    from speculative_decoding_verification_65_gb300 import synth
    vals = []
    for b in np.flatnonzero(case.temperature > 0)[:n_seq]:
        T = float(case.temperature[b])
        for i in range(case.k):
            p = oracle.softmax(synth.decode(case.target[b, i]), T)
            q = oracle.softmax(synth.decode(case.draft[b, i]), T)
            vals.append(1.0 - oracle.residual(p, q)[1])
    return (float(np.mean(vals)) if vals else None), len(vals)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from speculative_decoding_verification_65_gb300 import synth
    case = make_workload(args.config, 0, args.batch)
    cores = host_cores()
    # each step verifies a bounded sample of the batch on all host cores
    per_step = min(case.B, max(cores, 16))
    import oracle
    oracle.build()
    sub = case.subset(np.arange(per_step))
    for _ in range(args.warmup):
        oracle.verify(sub.target, sub.draft, sub.tokens, sub.u_accept, sub.u_resample,
                      sub.temperature, nthreads=cores, want_trace=False)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.verify(sub.target, sub.draft, sub.tokens, sub.u_accept, sub.u_resample,
                      sub.temperature, nthreads=cores, want_trace=False)
    dt = time.perf_counter() - t0
    value = per_step * case.k * args.steps / dt
    sample = f"first {per_step} of {case.B} sequences per step, {synth.CONFIG_NAMES[args.config]}"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": synth.CONFIG_NAMES[args.config], "B": per_step, "k": case.k,
                   "V": case.V, "input_dtype": case.dtype,
                   "what": "fp64 CPU oracle (plain C, threads over sequences)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def nvtx_range(name):
    """An NVTX range around the timed calls, so a profiler can select them."""
    import contextlib

    import torch
    try:
        rng = torch.cuda.nvtx.range(name)
    except (AttributeError, RuntimeError):
        rng = contextlib.nullcontext()
    return rng


def measure_verify(case, dev, steps: int, warmup: int, graph: bool, barrier=lambda: None,
                   min_staged_s: float = 0.0):
    """Times `steps` whole spec_verify calls on one batch (CUDA events on the
    launch stream; a barrier and a device synchronise on both sides), then
    per-stage durations over further calls with stage events (at least
    `min_staged_s` seconds of them, so the clock sampler sees the same work).
    Returns the measurements and the staged loop's clock record."""
    import torch

    import speculative_decoding_verification_65_gb300 as sv
    from speculative_decoding_verification_65_gb300 import synth

    B, k, V = case.B, case.k, case.V
    d = sv.to_device(case, dev)
    dt_code = sv.SPEC_F32 if case.dtype == synth.F32 else sv.SPEC_BF16
    stream = torch.cuda.current_stream(dev)
    ws = sv.workspace(B, k, V, dt_code, dev, stream)
    out_t = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    out_n = torch.empty((B,), dtype=torch.int32, device=dev)

    def step(events=None):
        if events is None:
            sv.spec_verify(**d, out_tokens=out_t, out_num_accepted=out_n, ws=ws, stream=stream)
        else:
            sv.spec_verify_timed(**d, out_tokens=out_t, out_num_accepted=out_n, ws=ws,
                                 stage_events=events, stream=stream)

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    if sv.spec_verify_read_status(ws) != sv.SPEC_DEV_OK:
        raise RuntimeError("device status nonzero after warm-up")

    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    g, per_graph = None, 1
    if graph:
        # a batch of whole calls captured into one CUDA graph and replayed:
        # for launch-bound sizes this removes the host's launch cost per call
        per_graph = min(steps, 50)
        while steps % per_graph:
            per_graph -= 1
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(per_graph):
                sv.spec_verify(**d, out_tokens=out_t, out_num_accepted=out_n, ws=ws)
        g.replay()
        torch.cuda.synchronize(dev)
    barrier()
    torch.cuda.synchronize(dev)
    # the timed region: K whole verification calls, as a user issues them
    with ClockSampler(dev.index) as clk_timed, nvtx_range("spec_verify timed region"):
        t0.record(stream)
        if g is not None:
            for _ in range(steps // per_graph):
                g.replay()
        else:
            for _ in range(steps):
                step()
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier()
    total_ms = t0.elapsed_time(t1)
    del g

    # per-stage durations: further calls, each with an event before it and one
    # after each stage (statistics, accept scan, draw tiles, final search,
    # exact draws) on the launch stream; stage events keep the kernels plainly
    # ordered.  Run for at least min_staged_s so that the clock sampler, which
    # polls every 50 ms, sees the same work under load.
    per_step_s = max(total_ms / steps / 1e3, 1e-6)
    n_staged = max(steps, int(min_staged_s / per_step_s) + 1)
    n_staged = min(n_staged, 20000)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_staged)]
    stages = [[torch.cuda.Event(enable_timing=True) for _ in range(sv.SPEC_STAGES)]
              for _ in range(n_staged)]
    for ev in [e for row in stages for e in row]:
        ev.record(stream)  # creates the underlying CUDA events
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clk_staged:
        for i in range(n_staged):
            starts[i].record(stream)
            step(stages[i])
        torch.cuda.synchronize(dev)
    kern_ms = [s_.elapsed_time(e[0]) for s_, e in zip(starts, stages)]  # statistics kernel
    stage_ms = [statistics.mean(
        (starts[i] if j == 0 else stages[i][j - 1]).elapsed_time(stages[i][j])
        for i in range(n_staged)) for j in range(sv.SPEC_STAGES)]
    status = sv.spec_verify_read_status(ws)
    n_host = out_n.cpu().numpy()  # the last call's accept counts
    ok_rows = n_host >= 0
    acceptance = {"mean_accepted": float(n_host[ok_rows].mean()) if ok_rows.any() else None,
                  "error_sequences": int((~ok_rows).sum()), "sequences": int(B)}
    staged_median = statistics.median(s_.elapsed_time(e[-1]) for s_, e in zip(starts, stages))
    del d, ws, out_t, out_n
    torch.cuda.empty_cache()
    return dict(total_ms=total_ms, per_graph=per_graph, kern_ms=kern_ms, stage_ms=stage_ms,
                n_staged=n_staged, status=status, acceptance=acceptance,
                staged_median=staged_median, clocks_timed=clk_timed.summary(),
                clocks_staged=clk_staged.summary())


def stage_dict(stage_ms):
    return {"stats": stage_ms[0], "scan": stage_ms[1], "draw": stage_ms[2],
            "final": stage_ms[3], "exact_draws": stage_ms[4]}


def merged_clocks(m):
    """The timed region's clock record; where it holds no sample (a region
    shorter than the 50 ms poll), the staged loop's (the same calls, under
    load, right after it), said so."""
    c = dict(m["clocks_timed"])
    if c.get("sm_mhz") is None:
        st = dict(m["clocks_staged"])
        st["source"] = (f"staged-timing loop right after the timed region "
                        f"({m['n_staged']} calls of the same work)")
        return st
    c["source"] = "timed region"
    return c


def roofline_of(kern_ms, alg_bytes, peak, peak_src, workload, read_gbs=None):
    kern_avg_s = statistics.mean(kern_ms) / 1e3
    achieved = alg_bytes / kern_avg_s / 1e9
    r = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
         "frac": achieved / peak, "traffic": recorded_traffic(workload),
         "peak_source": f"{peak_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
         if peak_src == "measured" else "fallback 6.8 TB/s",
         "kernel": "stats_kernel (row statistics, the HBM-bound stage)",
         "kernel_timing": "CUDA events after each stage, further steps",
         "kernel_ms_avg": kern_avg_s * 1e3, "kernel_ms_min": min(kern_ms),
         "frac_of_nominal_8TBs": achieved / 8000.0}
    if read_gbs:
        r["read_probe_gbs"] = read_gbs
        r["frac_of_read_probe"] = achieved / read_gbs
    return r


def per_config_block(args, dev, peak, peak_src):
    """Workload 5 at full size (one call per step) and workloads 1-3 under
    CUDA graph replay (launch-bound sizes), measured in the same process as
    the headline, each with its roofline, stage times and oracle baseline."""
    from speculative_decoding_verification_65_gb300 import synth

    out = {}
    for cfg in args.per_config:
        if cfg == args.config:
            continue
        case = make_workload(cfg, 0, None)
        graph = cfg in (1, 2, 3)
        steps = max(args.steps, 200) if graph else max(args.steps, 100)
        m = measure_verify(case, dev, steps, args.warmup, graph, min_staged_s=0.3)
        alg_bytes = synth.algorithmic_bytes(case)
        ms = m["total_ms"] / steps
        workload = synth.CONFIG_NAMES[cfg]
        entry = {
            "workload": workload, "B": case.B, "k": case.k, "V": case.V,
            "input_dtype": case.dtype, "steps": steps, "ms_per_step": ms,
            "value": case.B * case.k / (ms / 1e3), "unit": UNIT,
            "launch": f"CUDA graph replay of {m['per_graph']} calls" if graph
            else "one library call per step",
            "algorithmic_bytes_per_step": alg_bytes,
            "roofline": roofline_of(m["kern_ms"], alg_bytes, peak, peak_src, workload),
            "stage_ms": stage_dict(m["stage_ms"]),
            "ms_per_step_median_staged": m["staged_median"],
            "clocks": merged_clocks(m), "acceptance": m["acceptance"],
            "device_status": m["status"],
        }
        if not args.no_cpu_baseline:
            cores = host_cores()
            v, n_seq, used = time_oracle(case, min(args.cpu_budget, 4.0), cores)
            entry["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                     "sample": f"{n_seq} of {case.B} sequences of {workload}, "
                                               f"{used:.1f} s on {cores} threads"}
        out[f"cfg{cfg}"] = entry
        del case
    return out


def run_ours(args):
    import torch

    import speculative_decoding_verification_65_gb300 as sv
    from speculative_decoding_verification_65_gb300 import synth

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    case = make_workload(args.config, rank, args.batch)
    B, k, V = case.B, case.k, case.V
    dt_code = sv.SPEC_F32 if case.dtype == synth.F32 else sv.SPEC_BF16
    stream = torch.cuda.current_stream(dev)
    alg_bytes = synth.algorithmic_bytes(case)
    m = measure_verify(case, dev, args.steps, args.warmup, args.graph, barrier,
                       min_staged_s=0.5)
    total_ms = reduce_max(m["total_ms"], world, dev)
    ms_per_step = total_ms / args.steps
    value = aggregate_rate(B * k, args.steps, world, total_ms / 1e3)
    kern_ms, stage_ms = m["kern_ms"], m["stage_ms"]

    # end to end through the public API on host buffers (pinned), every step
    # copies the inputs in and the results out
    pin = lambda a: torch.from_numpy(a).pin_memory()
    if case.dtype == synth.BF16:
        h_t = pin(case.target.view(np.int16)).view(torch.bfloat16)
        h_d = pin(case.draft.view(np.int16)).view(torch.bfloat16)
    else:
        h_t, h_d = pin(case.target), pin(case.draft)
    h_g, h_ua, h_ur, h_T = pin(case.tokens), pin(case.u_accept), pin(case.u_resample), \
        pin(case.temperature)
    h_ot = torch.empty((B, k + 1), dtype=torch.int32).pin_memory()
    h_on = torch.empty((B,), dtype=torch.int32).pin_memory()
    arena = torch.empty(sv.spec_verify_host_arena_size(B, k, V, dt_code), dtype=torch.uint8,
                        device=dev)
    e2e_steps = max(1, min(args.steps, 20))
    sv.spec_verify_host(h_t, h_d, h_g, h_ua, h_ur, h_T, arena, h_ot, h_on, stream=stream)
    barrier()
    e0 = time.perf_counter()
    for _ in range(e2e_steps):
        sv.spec_verify_host(h_t, h_d, h_g, h_ua, h_ur, h_T, arena, h_ot, h_on, stream=stream)
    e2e_s = reduce_max(time.perf_counter() - e0, world, dev)
    e2e_value = aggregate_rate(B * k, e2e_steps, world, e2e_s)
    # the draft rows of greedy sequences stay on the host (never read)
    h2d = sum(int(x.numel() * x.element_size()) for x in (h_t, h_g, h_ua, h_ur, h_T)) + \
        int(np.count_nonzero(case.temperature != 0)) * k * V * h_d.element_size()
    d2h = int(h_ot.numel() * 4 + h_on.numel() * 4)
    del arena
    torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    peaks, peak_src = measured_peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))
    workload = synth.CONFIG_NAMES[args.config] if args.batch is None else case.name
    read_gbs = None if args.no_read_probe else read_probe_gbs(dev)
    acceptance = m["acceptance"]
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cores = host_cores()
        v, n_seq, used = time_oracle(case, args.cpu_budget, cores)
        v1, n1, used1 = time_oracle(case, args.cpu_budget / 4, 1)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{n_seq} of {B} sequences of {workload}, {used:.1f} s on {cores} threads",
               "value_1thread": v1,
               "sample_1thread": f"{n1} sequences, {used1:.1f} s on 1 thread"}
        a, n_pos = oracle_alpha(case, 16)
        acceptance["oracle_alpha"] = a
        acceptance["oracle_alpha_sample"] = f"{n_pos} drafted positions of the first 16 sampling sequences"
    roof = roofline_of(kern_ms, alg_bytes, peak, peak_src, workload, read_gbs)
    roof["step_GBps"] = alg_bytes / (ms_per_step / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload, "B_per_gpu": B, "k": k, "V": V,
                   "input_dtype": case.dtype, "global_batch": B * world,
                   "algorithmic_bytes_per_step": alg_bytes,
                   "l2": "inputs larger than L2 (no flush)" if alg_bytes > (129 << 20)
                   else "inputs smaller than L2 (no flush; launch-bound size)",
                   "launch": f"CUDA graph replay of {m['per_graph']} calls" if args.graph
                   else "one library call per step", "parallelism": f"dp{world}"},
        "gpu_launches": (sv.SPEC_STAGES + 1) * args.steps,
        "roofline": roof,
        "stage_ms": stage_dict(stage_ms),
        "stage_calls": m["n_staged"],
        "ms_per_step_median_staged": m["staged_median"],
        "clocks": merged_clocks(m),
        "clocks_timed_region": m["clocks_timed"],
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "cpu_baseline": cpu,
        "acceptance": acceptance,
        "device_status": m["status"],
    }
    if world == 1 and args.batch is None and args.per_config:
        line["per_config"] = per_config_block(args, dev, peak, peak_src)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------ filtered

def filtered_draft_tokens(draft, temperature, top_k: int, top_p: float, seed: int):
    """Input generation: draft tokens g_i drawn from the top-k / top-p filtered
    draft distribution (greedy sequences: the draft argmax), on the GPU with
    torch (ranking by logit with ties in index order, as the filter reads)."""
    import torch
    B, k, V = draft.shape
    gen = torch.Generator(device=draft.device)
    gen.manual_seed(seed)
    toks = torch.empty((B, k), dtype=torch.int32, device=draft.device)
    for b0 in range(0, B, 64):
        d = draft[b0:b0 + 64].float()
        T = temperature[b0:b0 + 64].view(-1, 1, 1)
        vals, idx = torch.sort(d, dim=-1, descending=True, stable=True)
        greedy = (T == 0).view(-1)
        z = (vals - vals[..., :1]) / torch.where(T > 0, T, torch.ones_like(T))
        w = torch.exp(z)
        K = top_k if 0 < top_k < V else V
        w[..., K:] = 0.0
        if top_p < 1.0:
            tot = w.sum(-1, keepdim=True)
            before = torch.cumsum(w, -1) - w
            w = torch.where(before < top_p * tot, w, torch.zeros_like(w))
        pick = torch.multinomial(w.view(-1, V), 1, generator=gen).view(d.shape[0], k)
        g = torch.gather(idx, -1, pick.unsqueeze(-1)).squeeze(-1)
        g[greedy] = idx[greedy][..., 0]
        toks[b0:b0 + 64] = g.to(torch.int32)
    return toks


def run_reference_filtered(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    import torch
    oracle.build()
    case = make_workload(args.config, 0, args.batch)
    cores = host_cores()
    per_step = min(case.B, max(cores, 16))
    sub = case.subset(np.arange(per_step))
    # tokens from the filtered draft distribution (generated on the CPU here)
    d = torch.from_numpy(synth_decode(sub.draft))
    sub.tokens = filtered_draft_tokens(d, torch.from_numpy(sub.temperature), args.top_k,
                                       args.top_p, 1234).numpy()
    tk = np.full(per_step, args.top_k, np.int32)
    tp = np.full(per_step, args.top_p)
    run = lambda: oracle.verify_filtered(sub.target, sub.draft, sub.tokens, sub.u_accept,
                                         sub.u_resample, sub.temperature, tk, tp,
                                         nthreads=cores, want_trace=False)
    for _ in range(args.warmup):
        run()
    # bounded by the CPU budget (steps of the filtered oracle sort every row)
    t0 = time.perf_counter()
    steps = 0
    while steps < args.steps and (steps == 0 or time.perf_counter() - t0 < args.cpu_budget):
        run()
        steps += 1
    dt = time.perf_counter() - t0
    args.steps = steps
    value = per_step * case.k * steps / dt
    from speculative_decoding_verification_65_gb300 import synth
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": synth.CONFIG_NAMES[args.config], "B": per_step, "k": case.k,
                   "V": case.V, "top_k": args.top_k, "top_p": args.top_p,
                   "what": "fp64 CPU oracle, filtered (plain C, threads over sequences)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"first {per_step} of {case.B} sequences per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def synth_decode(a):
    from speculative_decoding_verification_65_gb300 import synth
    return synth.decode(a)


def run_ours_filtered(args):
    import torch

    import speculative_decoding_verification_65_gb300 as sv
    from speculative_decoding_verification_65_gb300 import synth

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    case = make_workload(args.config, rank, args.batch)
    B, k, V = case.B, case.k, case.V
    d = sv.to_device(case, dev)
    d["tokens"] = filtered_draft_tokens(d["draft"], d["temperature"], args.top_k, args.top_p,
                                        1234 + rank)
    top_k = torch.full((B,), args.top_k, dtype=torch.int32, device=dev)
    top_p = torch.full((B,), args.top_p, dtype=torch.float32, device=dev)
    dt_code = sv.SPEC_F32 if case.dtype == synth.F32 else sv.SPEC_BF16
    stream = torch.cuda.current_stream(dev)
    # the binding's default workspace has room for the group maxima (top-k rows
    # cut from them); the smaller one sends every row through the streaming
    # filter, timed too
    ws = sv.filtered_workspace(B, k, V, dt_code, dev, stream)
    ws_stream = torch.zeros(sv.spec_verify_workspace_size(B, k, V, dt_code), dtype=torch.uint8,
                            device=dev)
    out_t = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    out_n = torch.empty((B,), dtype=torch.int32, device=dev)
    alg_bytes = synth.algorithmic_bytes(case)

    def step(events=None, w=None):
        w = ws if w is None else w
        if events is None:
            sv.spec_verify_filtered(**d, top_k=top_k, top_p=top_p, out_tokens=out_t,
                                    out_num_accepted=out_n, ws=w, stream=stream)
        else:
            sv.spec_verify_filtered_timed(**d, top_k=top_k, top_p=top_p, out_tokens=out_t,
                                          out_num_accepted=out_n, ws=w, stage_events=events,
                                          stream=stream)

    def measure(w):
        """K timed calls (one event pair, clocks sampled), then K calls with an
        event after each stage: (ms for K calls, mean ms per stage, clocks)."""
        for _ in range(max(args.warmup, 3)):
            step(w=w)
        torch.cuda.synchronize(dev)
        if sv.spec_verify_read_status(w) != sv.SPEC_DEV_OK:
            raise RuntimeError("device status nonzero after warm-up")
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize(dev)
        with ClockSampler(local) as clk, nvtx_range("spec_verify_filtered timed region"):
            t0.record(stream)
            for _ in range(args.steps):
                step(w=w)
            t1.record(stream)
            torch.cuda.synchronize(dev)
        barrier()
        tot = reduce_max(t0.elapsed_time(t1), world, dev)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        stages = [[torch.cuda.Event(enable_timing=True) for _ in range(sv.SPEC_FILTERED_STAGES)]
                  for _ in range(args.steps)]
        for ev in [e for row in stages for e in row]:
            ev.record(stream)
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            starts[i].record(stream)
            step(stages[i], w=w)
        torch.cuda.synchronize(dev)
        sm = [statistics.mean(
            (starts[i] if j == 0 else stages[i][j - 1]).elapsed_time(stages[i][j])
            for i in range(args.steps)) for j in range(sv.SPEC_FILTERED_STAGES)]
        return tot, sm, clk.summary()

    stream_ms, stream_stage_ms, stream_clk = measure(ws_stream)
    stream_out = (out_t.clone(), out_n.clone())
    total_ms, stage_ms, clocks = measure(ws)
    same_as_streaming = bool(torch.equal(stream_out[0], out_t) and torch.equal(stream_out[1], out_n))
    n_err = int((out_n < 0).sum().item())
    ms_per_step = total_ms / args.steps
    value = aggregate_rate(B * k, args.steps, world, total_ms / 1e3)
    status = sv.spec_verify_read_status(ws)

    # end to end: pinned host inputs copied in, the call, the outputs copied back
    pin = lambda t: t.cpu().pin_memory()
    host = {n: pin(t) for n, t in d.items()}
    h_k, h_p = pin(top_k), pin(top_p)
    h_ot = torch.empty((B, k + 1), dtype=torch.int32).pin_memory()
    h_on = torch.empty((B,), dtype=torch.int32).pin_memory()
    e2e_steps = max(1, min(args.steps, 20))
    barrier()
    e0 = time.perf_counter()
    for _ in range(e2e_steps):
        dd = {n: t.to(dev, non_blocking=True) for n, t in host.items()}
        tk, tp = h_k.to(dev, non_blocking=True), h_p.to(dev, non_blocking=True)
        sv.spec_verify_filtered(**dd, top_k=tk, top_p=tp, out_tokens=out_t,
                                out_num_accepted=out_n, ws=ws, stream=stream)
        h_ot.copy_(out_t, non_blocking=True)
        h_on.copy_(out_n, non_blocking=True)
        torch.cuda.synchronize(dev)
    e2e_s = reduce_max(time.perf_counter() - e0, world, dev)
    e2e_value = aggregate_rate(B * k, e2e_steps, world, e2e_s)
    h2d = sum(int(t.numel() * t.element_size()) for t in host.values()) + 8 * B
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    peaks, peak_src = measured_peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))
    # the streaming filter's algorithmic bytes are one read of every row it
    # filters (all 2k+1 rows of a sampled sequence whose filters are on;
    # greedy sequences are not read)
    filt_on = (args.top_k > 0 and args.top_k < V) or args.top_p < 1.0
    n_sampled = int(np.sum(case.temperature > 0)) if filt_on else 0
    filt_bytes = n_sampled * (2 * k + 1) * V * (2 if case.dtype == "bf16" else 4)
    stream_achieved = filt_bytes / (stream_stage_ms[1] / 1e3) / 1e9
    achieved = alg_bytes / (stage_ms[0] / 1e3) / 1e9  # the statistics kernel
    workload = synth.CONFIG_NAMES[args.config] if args.batch is None else case.name
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload, "B_per_gpu": B, "k": k, "V": V,
                   "input_dtype": case.dtype, "top_k": args.top_k, "top_p": args.top_p,
                   "draft_tokens": "drawn from the filtered draft distribution",
                   "error_sequences": n_err, "algorithmic_bytes_per_step": alg_bytes,
                   "l2": "inputs larger than L2 (no flush)", "parallelism": f"dp{world}"},
        "gpu_launches": (sv.SPEC_FILTERED_STAGES + 3) * args.steps,  # nine kernels a call
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": recorded_traffic(f"{workload}_top{args.top_k}_p{args.top_p}",
                                                 "stats_kernel"),
                     "peak_source": f"{peak_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "kernel": "stats_kernel (one read of every logit, with the group maxima "
                               "of the top-k cut)",
                     "kernel_timing": "CUDA events after each kernel, K further steps",
                     "step_GBps": alg_bytes / (ms_per_step / 1e3) / 1e9},
        "stage_ms": {"stats": stage_ms[0], "filter": stage_ms[1], "scan": stage_ms[2],
                     "draw": stage_ms[3], "final": stage_ms[4], "exact_draws": stage_ms[5]},
        "streaming_filter": {
            "what": "the same calls with a workspace without room for group maxima: every "
                    "row cut by the streaming window filter (wfilter_kernel, then "
                    "filter_kernel for the rows it flags)",
            "ms_per_step": stream_ms / args.steps, "same_outputs": same_as_streaming,
            "stage_ms": {"stats": stream_stage_ms[0], "filter": stream_stage_ms[1],
                         "scan": stream_stage_ms[2], "draw": stream_stage_ms[3],
                         "final": stream_stage_ms[4], "exact_draws": stream_stage_ms[5]},
            "roofline": {"bound": "hbm", "achieved": stream_achieved, "peak": peak,
                         "unit": "GB/s", "frac": stream_achieved / peak,
                         "algorithmic_bytes_per_launch": filt_bytes,
                         "traffic": recorded_traffic(
                             f"{workload}_top{args.top_k}_p{args.top_p}_streaming",
                             "wfilter_kernel")},
            "clocks": stream_clk},
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": int(B * (k + 2) * 4), "steps": e2e_steps,
                "path": "torch copies of pinned host tensors around spec_verify_filtered"},
        "cpu_baseline": None,
        "device_status": status,
    }
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        cores = host_cores()
        sub = case.subset(np.arange(min(B, max(cores, 16))))
        sub.tokens = d["tokens"][:sub.B].cpu().numpy()
        tk_n = np.full(sub.B, args.top_k, np.int32)
        tp_n = np.full(sub.B, args.top_p)
        c0 = time.perf_counter()
        oracle.verify_filtered(sub.target, sub.draft, sub.tokens, sub.u_accept, sub.u_resample,
                               sub.temperature, tk_n, tp_n, nthreads=cores, want_trace=False)
        used = time.perf_counter() - c0
        line["cpu_baseline"] = {"value": sub.B * k / used, "unit": UNIT, "cores": cores,
                                "kind": "oracle",
                                "sample": f"{sub.B} of {B} sequences, {used:.1f} s on {cores} threads"}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------ sampling

def make_sample_workload(cfg: int, rank: int, batch=None):
    from speculative_decoding_verification_65_gb300 import synth
    return synth.make_sample_config(cfg, B=batch, seed_offset=100 * rank)


def time_oracle_sample(sc, budget_s: float, threads: int):
    """Oracle sampling throughput on a bounded sample: blocks of rows until the
    time budget is spent or every row is done."""
    import oracle
    done, t_used = 0, 0.0
    block = max(4 * threads, 64)
    while done < sc.R and t_used < budget_s:
        sl = slice(done, min(sc.R, done + block))
        t0 = time.perf_counter()
        oracle.sample(sc.logits[sl], sc.u[sl], sc.temperature[sl], nthreads=threads,
                      want_trace=False)
        t_used += time.perf_counter() - t0
        done = sl.stop
    return done / t_used, done, t_used


def sample_workload_name(args, sc):
    return sc.name if args.batch is None else f"{sc.name} (B={args.batch} of workload {args.config})"


def run_reference_sample(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    sc = make_sample_workload(args.config, 0, args.batch)
    cores = host_cores()
    per_step = min(sc.R, max(4 * cores, 64))
    sl = slice(0, per_step)
    run = lambda: oracle.sample(sc.logits[sl], sc.u[sl], sc.temperature[sl], nthreads=cores,
                                want_trace=False)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    value = per_step * args.steps / dt
    line = {
        "impl": "reference", "metric": SAMPLE_METRIC, "value": value, "unit": SAMPLE_UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": sample_workload_name(args, sc), "R": per_step, "V": sc.V,
                   "input_dtype": sc.dtype,
                   "what": "fp64 CPU oracle (plain C, threads over rows)"},
        "cpu_baseline": {"value": value, "unit": SAMPLE_UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"first {per_step} of {sc.R} rows per step"},
        "e2e": {"value": value, "unit": SAMPLE_UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours_sample(args):
    import torch

    import speculative_decoding_verification_65_gb300 as sv
    from speculative_decoding_verification_65_gb300 import synth

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def max_over_ranks(x):
        return reduce_max(x, world, dev)

    sc = make_sample_workload(args.config, rank, args.batch)
    R, V = sc.R, sc.V
    d = sv.sample_to_device(sc, dev)
    dt_code = sv.SPEC_F32 if sc.dtype == synth.F32 else sv.SPEC_BF16
    stream = torch.cuda.current_stream(dev)
    ws = sv.sample_workspace(R, V, dt_code, dev, stream)
    out = torch.empty((R,), dtype=torch.int32, device=dev)
    alg_bytes = synth.sample_bytes(sc)

    def step(events=None):
        if events is None:
            sv.spec_sample(**d, out=out, ws=ws, stream=stream)
        else:
            sv.spec_sample_timed(**d, out=out, ws=ws, stage_events=events, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    if sv.spec_verify_read_status(ws) != sv.SPEC_DEV_OK:
        raise RuntimeError("device status nonzero after warm-up")

    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:  # the timed region: K whole sampling calls
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier()
    total_ms = max_over_ranks(t0.elapsed_time(t1))

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    stages = [[torch.cuda.Event(enable_timing=True) for _ in range(sv.SPEC_SAMPLE_STAGES)]
              for _ in range(args.steps)]
    for ev in [e for row in stages for e in row]:
        ev.record(stream)
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        starts[i].record(stream)
        step(stages[i])
    torch.cuda.synchronize(dev)
    kern_ms = [s.elapsed_time(e[0]) for s, e in zip(starts, stages)]
    pick_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in stages)
    exact_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in stages)
    ms_per_step = total_ms / args.steps
    value = aggregate_rate(R, args.steps, world, total_ms / 1e3)
    status = sv.spec_verify_read_status(ws)

    # end to end through the C ABI on pinned host buffers
    if sc.dtype == synth.BF16:
        h_l = torch.from_numpy(sc.logits.view(np.int16)).pin_memory().view(torch.bfloat16)
    else:
        h_l = torch.from_numpy(sc.logits).pin_memory()
    h_u = torch.from_numpy(sc.u).pin_memory()
    h_T = torch.from_numpy(sc.temperature).pin_memory()
    h_o = torch.empty((R,), dtype=torch.int32).pin_memory()
    del d
    torch.cuda.empty_cache()
    arena = torch.empty(sv.spec_sample_host_arena_size(R, V, dt_code), dtype=torch.uint8,
                        device=dev)
    e2e_steps = max(1, min(args.steps, 20))
    sv.spec_sample_host(h_l, h_u, h_T, arena, h_o, stream=stream)
    barrier()
    e0 = time.perf_counter()
    for _ in range(e2e_steps):
        sv.spec_sample_host(h_l, h_u, h_T, arena, h_o, stream=stream)
    e2e_s = max_over_ranks(time.perf_counter() - e0)
    e2e_value = aggregate_rate(R, e2e_steps, world, e2e_s)
    h2d = sum(int(x.numel() * x.element_size()) for x in (h_l, h_u, h_T))

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    peaks, peak_src = measured_peaks()
    kern_avg_s = statistics.mean(kern_ms) / 1e3
    achieved = alg_bytes / kern_avg_s / 1e9
    peak = float(peaks.get("hbm_gbs", 6800.0))
    workload = sample_workload_name(args, sc)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cores = host_cores()
        v, n_rows, used = time_oracle_sample(sc, args.cpu_budget, cores)
        cpu = {"value": v, "unit": SAMPLE_UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{n_rows} of {R} rows of {workload}, {used:.1f} s on {cores} threads"}
    line = {
        "metric": SAMPLE_METRIC, "value": value, "unit": SAMPLE_UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload, "R_per_gpu": R, "V": V, "input_dtype": sc.dtype,
                   "algorithmic_bytes_per_step": alg_bytes,
                   "l2": "inputs larger than L2 (no flush)", "parallelism": f"dp{world}"},
        "gpu_launches": sv.SPEC_SAMPLE_STAGES * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": recorded_traffic(workload, "chunk_kernel"),
                     "peak_source": f"{peak_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "kernel": "chunk_kernel (the one read of the logits)",
                     "kernel_timing": "CUDA events after each kernel, K further steps",
                     "kernel_ms_avg": kern_avg_s * 1e3, "kernel_ms_min": min(kern_ms),
                     "frac_of_nominal_8TBs": achieved / 8000.0,
                     "step_GBps": alg_bytes / (ms_per_step / 1e3) / 1e9},
        "stage_ms": {"chunk": kern_avg_s * 1e3, "pick": pick_ms, "exact_draws": exact_ms},
        "clocks": clk.summary(),
        "e2e": {"value": e2e_value, "unit": SAMPLE_UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": R * 4, "steps": e2e_steps},
        "cpu_baseline": cpu,
        "device_status": status,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------ LM-head-fused verification

LMHEAD_SHAPE = dict(B=1024, k=4, V=128256, d=4096)  # workload 5's shape, d of an 8B-class model


def lmhead_inputs(B, k, V, d, seed, device):
    """Input generation for the fused workload with torch on `device`: target
    hidden states h ~ N(0, 1), LM head W ~ N(0, (2.5 / sqrt d)^2), both bf16;
    a draft model sharing W that sees h + N(0, 0.3^2) gives the draft logits
    (bf16, computed by torch); draft tokens sampled from them at T = 1;
    uniforms in [0, 1)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    hidden = torch.randn((B, k + 1, d), generator=g, device=device).to(torch.bfloat16)
    W = torch.empty((V, d), dtype=torch.bfloat16, device=device)
    for r0 in range(0, V, 16384):  # in slices: no 2 GB fp32 temporary
        r1 = min(V, r0 + 16384)
        W[r0:r1] = (torch.randn((r1 - r0, d), generator=g, device=device)
                    * (2.5 / d ** 0.5)).to(torch.bfloat16)
    hd = (hidden[:, :k].float()
          + 0.3 * torch.randn((B, k, d), generator=g, device=device)).to(torch.bfloat16)
    draft = torch.empty((B, k, V), dtype=torch.bfloat16, device=device)
    for b0 in range(0, B, 64):
        b1 = min(B, b0 + 64)
        mm = hd[b0:b1].reshape(-1, d).float() @ W.float().T if device == "cpu" else \
            hd[b0:b1].reshape(-1, d) @ W.T
        draft[b0:b1] = mm.reshape(b1 - b0, k, V).to(torch.bfloat16)
    temperature = torch.ones((B,), dtype=torch.float32, device=device)
    u_accept = torch.rand((B, k), generator=g, device=device)
    u_resample = torch.rand((B,), generator=g, device=device)
    tokens = filtered_draft_tokens(draft, temperature, 0, 1.0, seed + 1)
    return dict(hidden=hidden, lm_head=W, draft=draft, tokens=tokens, u_accept=u_accept,
                u_resample=u_resample, temperature=temperature)


def lmhead_name(B, k, V, d):
    return f"lmhead_B{B}_k{k}_V{V}_d{d}_bf16"


def _bits(t):
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def run_ours_lmhead(args):
    import torch

    import speculative_decoding_verification_65_gb300 as sv

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    sh = dict(LMHEAD_SHAPE)
    if args.batch is not None:
        sh["B"] = args.batch
    B, k, V, d = sh["B"], sh["k"], sh["V"], sh["d"]
    x = lmhead_inputs(B, k, V, d, 4321 + rank, dev)
    stream = torch.cuda.current_stream(dev)
    ws = sv.lmhead_workspace(B, k, V, d, sv.SPEC_BF16, dev)
    out_t = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    out_n = torch.empty((B,), dtype=torch.int32, device=dev)

    def step(events=None):
        if events is None:
            sv.spec_verify_lmhead(**x, out_tokens=out_t, out_num_accepted=out_n, ws=ws,
                                  stream=stream)
        else:
            sv.spec_verify_lmhead_timed(**x, out_tokens=out_t, out_num_accepted=out_n, ws=ws,
                                        stage_events=events, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    if sv.spec_verify_read_status(ws) != sv.SPEC_DEV_OK:
        raise RuntimeError("device status nonzero after warm-up")
    n_err = int((out_n < 0).sum().item())
    acc_mean = float(out_n[out_n >= 0].float().mean().item())
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize(dev)
    total_ms = reduce_max(t0.elapsed_time(t1), world, dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    stages = [[torch.cuda.Event(enable_timing=True) for _ in range(sv.SPEC_LMHEAD_STAGES)]
              for _ in range(args.steps)]
    for ev in [e for row in stages for e in row]:
        ev.record(stream)
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        starts[i].record(stream)
        step(stages[i])
    torch.cuda.synchronize(dev)
    stage_ms = [statistics.mean(
        (starts[i] if j == 0 else stages[i][j - 1]).elapsed_time(stages[i][j])
        for i in range(args.steps)) for j in range(sv.SPEC_LMHEAD_STAGES)]
    ms_per_step = total_ms / args.steps
    value = aggregate_rate(B * k, args.steps, world, total_ms / 1e3)
    status = sv.spec_verify_read_status(ws)
    # end to end: the step's inputs (hidden states, draft logits, tokens,
    # uniforms, temperatures) copied in from pinned host memory each step, the
    # outputs copied back; the LM head is a model weight and stays resident
    host = {n: t.cpu().pin_memory() for n, t in x.items() if n != "lm_head"}
    h_ot = torch.empty((B, k + 1), dtype=torch.int32).pin_memory()
    h_on = torch.empty((B,), dtype=torch.int32).pin_memory()
    e2e_steps = max(1, min(args.steps, 10))
    e0 = time.perf_counter()
    for _ in range(e2e_steps):
        dd = {n: t.to(dev, non_blocking=True) for n, t in host.items()}
        sv.spec_verify_lmhead(**dd, lm_head=x["lm_head"], out_tokens=out_t,
                              out_num_accepted=out_n, ws=ws, stream=stream)
        h_ot.copy_(out_t, non_blocking=True)
        h_on.copy_(out_n, non_blocking=True)
        torch.cuda.synchronize(dev)
    e2e_s = reduce_max(time.perf_counter() - e0, world, dev)
    h2d = sum(int(t.numel() * t.element_size()) for t in host.values())
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    peaks, peak_src = measured_peaks()
    flops = 2 * B * (k + 1) * V * d
    tflops = flops / (stage_ms[1] / 1e3) / 1e12
    # the burst peak while the timed region kept the SM clock at its maximum
    # (no power cap reached), the sustained one once the clock came down
    cs = clk.summary()
    at_max = (cs.get("sm_mhz") is not None and cs.get("sm_max_mhz")
              and cs["sm_mhz"] >= 0.95 * cs["sm_max_mhz"])
    which = "bf16_tflops" if at_max else "bf16_tflops_sustained"
    peak = float(peaks.get(which, 1900.0 if at_max else 1700.0))
    draw_flops = 2 * B * V * d
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (random weights and hidden states, see DESIGN)",
        "config": {"workload": lmhead_name(B, k, V, d), "B_per_gpu": B, "k": k, "V": V, "d": d,
                   "draft_dtype": "bf16", "temperature": 1.0, "error_sequences": n_err,
                   "mean_accepted": acc_mean, "gemm_flops_per_step": flops + draw_flops,
                   "l2": "the 1 GB LM head and 1 GB of draft logits per step exceed L2",
                   "parallelism": f"dp{world}"},
        "gpu_launches": sv.SPEC_LMHEAD_STAGES * args.steps,
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": tflops / peak,
                     "traffic": recorded_traffic(lmhead_name(B, k, V, d), "gemm_kernel"),
                     "peak_source": (f"measured cuBLAS bf16 (MEASURED_PEAKS.json {which}; "
                                     f"SM clock median {cs.get('sm_mhz')} MHz)")
                     if peak_src == "measured" else f"fallback for {which}",
                     "kernel": "gemm_kernel<STATS> (h W^T on tcgen05, statistics epilogue)",
                     "flops_per_launch": flops,
                     "kernel_timing": "CUDA events after each kernel, K further steps",
                     "draw_gemm_tflops": draw_flops / (stage_ms[3] / 1e3) / 1e12},
        "stage_ms": {"draft_records": stage_ms[0], "stats_gemm": stage_ms[1],
                     "scan": stage_ms[2], "draw_gemm": stage_ms[3], "final": stage_ms[4]},
        "clocks": cs,
        "e2e": {"value": aggregate_rate(B * k, e2e_steps, world, e2e_s), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": int(B * (k + 2) * 4),
                "steps": e2e_steps,
                "path": "torch copies of pinned host tensors around spec_verify_lmhead"},
        "cpu_baseline": None,
        "device_status": status,
    }
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        cores = host_cores()
        bs = min(B, 8)
        W = _bits(x["lm_head"])
        sub = [_bits(x["hidden"][:bs]), W, _bits(x["draft"][:bs])]
        rest = [x[n][:bs].cpu().numpy() for n in ("tokens", "u_accept", "u_resample",
                                                  "temperature")]
        c0 = time.perf_counter()
        oracle.verify_lmhead(*sub, *rest, nthreads=cores, want_trace=False)
        used = time.perf_counter() - c0
        line["cpu_baseline"] = {"value": bs * k / used, "unit": UNIT, "cores": cores,
                                "kind": "oracle",
                                "sample": f"{bs} of {B} sequences (fp64 LM head product and "
                                          f"verification), {used:.1f} s"}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference_lmhead(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    sh = dict(LMHEAD_SHAPE)
    B, k, V, d = sh["B"], sh["k"], sh["V"], sh["d"]
    per_step = 4
    x = lmhead_inputs(per_step, k, V, d, 4321, "cpu")
    cores = host_cores()
    args_np = [_bits(x["hidden"]), _bits(x["lm_head"]), _bits(x["draft"])] + \
        [x[n].numpy() for n in ("tokens", "u_accept", "u_resample", "temperature")]
    run = lambda: oracle.verify_lmhead(*args_np, nthreads=cores, want_trace=False)
    for _ in range(args.warmup):
        run()
    # each step takes about a second on 16 cores: stop at the CPU budget
    t0 = time.perf_counter()
    steps = 0
    while steps < args.steps and (steps == 0 or time.perf_counter() - t0 < args.cpu_budget):
        run()
        steps += 1
    dt = time.perf_counter() - t0
    value = per_step * k * steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": dt / steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": lmhead_name(B, k, V, d), "B": per_step, "k": k, "V": V, "d": d,
                   "what": "fp64 CPU oracle: LM head product (numpy) and verification (C)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} of {B} sequences per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------- tree verification

TREE_METRIC = "verified tree candidates/sec"
TREE_UNIT = "candidates/s"


def make_tree_workload(cfg: int, rank: int, batch=None):
    from speculative_decoding_verification_65_gb300 import synth
    return synth.make_tree_config(cfg, B=batch, seed_offset=100 * rank)


def tree_workload_name(args, tc):
    return tc.name if args.batch is None else \
        f"{tc.name} (B={args.batch} of tree workload {args.tree_config})"


def time_oracle_tree(tc, budget_s: float, threads: int):
    """Oracle throughput (candidates/s) on a bounded sample: blocks of
    sequences until the time budget is spent or every sequence is done."""
    import oracle
    done, t_used = 0, 0.0
    block = max(2 * threads, 32)
    while done < tc.B and t_used < budget_s:
        sub = tc.subset(np.arange(done, min(tc.B, done + block)))
        t0 = time.perf_counter()
        oracle.verify_tree(sub.target, sub.draft, sub.parent, sub.tokens, sub.n_nodes,
                           sub.u_accept, sub.u_resample, sub.temperature, nthreads=threads,
                           want_trace=False)
        t_used += time.perf_counter() - t0
        done += sub.B
    return done * (tc.N - 1) / t_used, done, t_used


def run_reference_tree(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    tc = make_tree_workload(args.tree_config, 0, args.batch)
    cores = host_cores()
    per_step = min(tc.B, max(2 * cores, 32))
    sub = tc.subset(np.arange(per_step))
    run = lambda: oracle.verify_tree(sub.target, sub.draft, sub.parent, sub.tokens, sub.n_nodes,
                                     sub.u_accept, sub.u_resample, sub.temperature,
                                     nthreads=cores, want_trace=False)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    value = per_step * (tc.N - 1) * args.steps / dt
    line = {
        "impl": "reference", "metric": TREE_METRIC, "value": value, "unit": TREE_UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": tree_workload_name(args, tc), "B": per_step, "N": tc.N,
                   "V": tc.V, "input_dtype": tc.dtype,
                   "what": "fp64 CPU oracle (plain C, threads over sequences)"},
        "cpu_baseline": {"value": value, "unit": TREE_UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"first {per_step} of {tc.B} trees per step"},
        "e2e": {"value": value, "unit": TREE_UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours_tree(args):
    import torch

    import speculative_decoding_verification_65_gb300 as sv
    from speculative_decoding_verification_65_gb300 import synth

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    tc = make_tree_workload(args.tree_config, rank, args.batch)
    B, N, V = tc.B, tc.N, tc.V
    d = sv.tree_to_device(tc, dev)
    stream = torch.cuda.current_stream(dev)
    ot = torch.empty((B, N), dtype=torch.int32, device=dev)
    on = torch.empty((B, N), dtype=torch.int32, device=dev)
    na = torch.empty((B,), dtype=torch.int32, device=dev)

    def step():
        sv.spec_verify_tree(**d, out_tokens=ot, out_nodes=on, out_num_accepted=na, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    nodes_h, n_h = on.cpu().numpy(), na.cpu().numpy()
    alg_bytes = synth.tree_bytes(tc, nodes_h, n_h)
    emitted = int(np.sum(n_h[n_h >= 0] + 1))

    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk, nvtx_range("spec_verify_tree timed region"):
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier()
    total_ms = reduce_max(t0.elapsed_time(t1), world, dev)
    ms_per_step = total_ms / args.steps
    value = aggregate_rate(B * (N - 1), args.steps, world, total_ms / 1e3)

    # one event pair around each call: the kernel's own duration
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps)]
    for a, b in pairs:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize(dev)
    kern_ms = [a.elapsed_time(b) for a, b in pairs]

    # end to end: pinned host inputs copied in, outputs copied back, every step
    def pinned(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).pin_memory().view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    host = dict(target=pinned(tc.target), draft=pinned(tc.draft), parent=pinned(tc.parent),
                tokens=pinned(tc.tokens), n_nodes=pinned(tc.n_nodes),
                u_accept=pinned(tc.u_accept), u_resample=pinned(tc.u_resample),
                temperature=pinned(tc.temperature))
    h_out = [torch.empty_like(x, device="cpu").pin_memory() for x in (ot, on, na)]

    def e2e_step():
        for k_, v in host.items():
            d[k_].copy_(v, non_blocking=True)
        step()
        for h, g in zip(h_out, (ot, on, na)):
            h.copy_(g, non_blocking=True)
        torch.cuda.synchronize(dev)
    e2e_step()
    e2e_steps = max(1, min(args.steps, 5))
    barrier()
    e0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = reduce_max(time.perf_counter() - e0, world, dev)
    e2e_value = aggregate_rate(B * (N - 1), e2e_steps, world, e2e_s)
    h2d = sum(int(x.numel() * x.element_size()) for x in host.values())
    d2h = sum(int(x.numel() * x.element_size()) for x in h_out)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    peaks, peak_src = measured_peaks()
    kern_avg_s = statistics.mean(kern_ms) / 1e3
    achieved = alg_bytes / kern_avg_s / 1e9
    peak = float(peaks.get("hbm_gbs", 6800.0))
    workload = tree_workload_name(args, tc)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cores = host_cores()
        v, n_seq, used = time_oracle_tree(tc, args.cpu_budget, cores)
        cpu = {"value": v, "unit": TREE_UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{n_seq} of {B} trees of {workload}, {used:.1f} s on {cores} threads"}
    line = {
        "metric": TREE_METRIC, "value": value, "unit": TREE_UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload, "B_per_gpu": B, "N": N, "V": V,
                   "input_dtype": tc.dtype, "branching": list(tc.meta.get("branching", [])),
                   "algorithmic_bytes_per_step": alg_bytes,
                   "emitted_tokens_per_step": emitted,
                   "l2": "rows read per step far larger than L2 (no flush)",
                   "parallelism": f"dp{world}"},
        "emitted_tokens_per_s": emitted * args.steps * world / (total_ms / 1e3),
        "mean_accepted": float(np.mean(n_h[n_h >= 0])),
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": recorded_traffic(workload, "tree_kernel"),
                     "peak_source": f"{peak_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "kernel": "tree_kernel (the whole step)",
                     "kernel_timing": "CUDA events around each call, K further steps",
                     "kernel_ms_avg": kern_avg_s * 1e3, "kernel_ms_min": min(kern_ms),
                     "frac_of_nominal_8TBs": achieved / 8000.0},
        "clocks": clk.summary(),
        "e2e": {"value": e2e_value, "unit": TREE_UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=None, choices=[1, 2, 3, 4, 5],
                    help="workload (default 4 for verify, 5 for sample)")
    ap.add_argument("--op", choices=["verify", "sample", "filtered", "lmhead", "tree"],
                    default="verify")
    ap.add_argument("--tree-config", type=int, default=2, choices=[1, 2],
                    help="tree workload of --op tree")
    ap.add_argument("--top-k", type=int, default=50, help="top-k of --op filtered (0: none)")
    ap.add_argument("--top-p", type=float, default=0.9, help="top-p of --op filtered (1: none)")
    ap.add_argument("--batch", type=int, default=None,
                    help="smaller batch of the same recipe (profiling captures only)")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-read-probe", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="time CUDA-graph replays of the verification calls")
    ap.add_argument("--per-config", default="5,1,2,3",
                    help="verify: other workloads measured in the same run and reported "
                         "under per_config (comma list; empty for none)")
    args = ap.parse_args()
    if args.config is None:
        args.config = 4 if args.op == "verify" else 5
    args.per_config = [int(x) for x in args.per_config.split(",") if x.strip()]
    if args.op == "sample":
        if args.impl == "reference":
            run_reference_sample(args)
        else:
            run_ours_sample(args)
    elif args.op == "filtered":
        if args.impl == "reference":
            run_reference_filtered(args)
        else:
            run_ours_filtered(args)
    elif args.op == "lmhead":
        if args.impl == "reference":
            run_reference_lmhead(args)
        else:
            run_ours_lmhead(args)
    elif args.op == "tree":
        if args.impl == "reference":
            run_reference_tree(args)
        else:
            run_ours_tree(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
