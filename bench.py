"""Throughput of the log-linear Mamba-2 forward (T=16384, H=16, d=128, bf16).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

One step = one ll_attn_fwd call over the whole workload (all of the hot path:
intra-chunk attention, chunk states, Fenwick tree, inter-chunk levels).
Inputs are resident in HBM when a timed step starts; L2 is flushed between
steps (a write of 2x the L2 size, outside the timed events).  Each step is
timed with CUDA events on the launching stream; `value` = tokens of all
ranks / max over ranks of the mean step time.  `e2e` times the same call with
the inputs copied from pinned host memory and the output copied back, all
inside the timed region.

With torchrun (N > 1) every rank runs the same workload on its own GPU with
no collective in the data path (weak scaling); a barrier brackets the timed
region.  `--impl reference` times the float64 CPU oracle instead (rank 0
only), on a bounded sample of query rows per step.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "log-linear Mamba-2 fwd tokens/s at T=16K,H=16,d=128; % of roofline"
PROFILES = os.path.join(ROOT, "profiles")


# ----------------------------------------------------------------------------
# algorithmic work of one forward (counted per (b, h), times B*H)
# ----------------------------------------------------------------------------
def algorithmic_bytes(cfg) -> int:
    """q, k, v read once, log_alpha and lam (float32) read once, o written once."""
    b_io = 2 if cfg["io"] == "bf16" else 4
    d = cfg["dk"]
    per_bh = cfg["T"] * (3 * d * b_io + 4 + 4 * cfg["L"] + cfg["dv"] * b_io)
    return per_bh * cfg["B"] * cfg["H"]


def algorithmic_flops(cfg) -> int:
    """Causal pairs inside a chunk, chunk states, tree combines and the
    popcount(c) non-empty inter-chunk levels of every chunk c."""
    T, C, d = cfg["T"], cfg["chunk"], cfg["dk"]
    N = T // C
    P = sum(bin(c).count("1") for c in range(N))
    per_bh = 2 * d * T * (C + 1) + 2 * T * d * d + 3 * d * d * N + 2 * d * d * C * P
    return per_bh * cfg["B"] * cfg["H"]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], "measured"
    return 6800.0, 1900.0, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "log_linear_attention_chunked_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(f.encode())
                h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None when there is none or the kernels changed since."""
    path = os.path.join(PROFILES, f"traffic_{workload}.json")
    if not os.path.exists(path):
        return None, None
    with open(path) as f:
        t = json.load(f)
    if t.get("source_hash") != kernel_source_hash():
        return None, t.get("kernel")
    return t.get("dram_bytes_per_launch"), t.get("kernel")


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, p in zip(names, parts[2:]):
                if p.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# oracle timing (CPU baseline / reference arm)
# ----------------------------------------------------------------------------
_W = {}


def _oracle_init(cfg, tag):
    """Worker set-up (untimed): draw one (b, h) slice of the workload."""
    from log_linear_attention_chunked_gb300 import synth
    inp = synth.make_inputs(dict(cfg, B=1, H=1), tag=tag)
    _W["x"] = tuple(synth.to_f64(inp[n][0, 0]) for n in ("q", "k", "v", "log_alpha", "lam"))


def _oracle_rows_worker(rows):
    from oracle import mamba2
    q, k, v, la, lam = _W["x"]
    mamba2.forward_rows(q, k, v, la, lam, rows)
    return len(rows)


def oracle_pool(cores: int, cfg: dict, tag: str = "oracle"):
    """Spawned single-threaded oracle processes, started before any GPU work."""
    import multiprocessing as mp
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    return mp.get_context("spawn").Pool(cores, initializer=_oracle_init, initargs=(cfg, tag))


def oracle_sample(pool, cores, T, rows_total, seed=0):
    """Time the float64 oracle (row-restricted dense form) on `rows_total`
    query rows drawn uniformly from [0, T), split over `cores` processes.
    Returns (rows per second of wall time, rows, seconds)."""
    import numpy as np
    rng = np.random.default_rng(seed)
    per = max(1, rows_total // cores)
    jobs = [sorted(int(x) for x in rng.integers(0, T, per)) for _ in range(cores)]
    t0 = time.perf_counter()
    n = sum(pool.map(_oracle_rows_worker, jobs, chunksize=1))
    wall = time.perf_counter() - t0
    return n / wall, n, wall


# ----------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mamba2_bf16_t16k")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from log_linear_attention_chunked_gb300 import synth
    cfg = dict(synth.WORKLOADS[args.workload])
    config = {"workload": args.workload, "B": cfg["B"], "H": cfg["H"], "T": cfg["T"], "dk": cfg["dk"],
              "dv": cfg["dv"], "chunk": cfg["chunk"], "L": cfg["L"], "io": cfg["io"],
              "l2": "flushed between steps (write of 2x L2)", "parallelism": f"replicas x{world} (b,h) weak"}
    tokens_per_step = cfg["B"] * cfg["H"] * cfg["T"]

    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)

    if args.impl == "reference":
        if rank != 0:
            return
        pool = oracle_pool(cores, cfg)
        # calibrate: size each step so that all steps take about a minute of wall time
        oracle_sample(pool, cores, cfg["T"], cores, seed=998)  # workers finish their set-up
        _, n, wall = oracle_sample(pool, cores, cfg["T"], cores * 16, seed=999)
        row_wall = wall / n
        rows_per_step = max(cores, int(60.0 / max(args.steps, 1) / row_wall) // cores * cores)
        for i in range(args.warmup):
            oracle_sample(pool, cores, cfg["T"], cores, seed=1000 + i)
        times, rows = [], 0
        for i in range(args.steps):
            _, n, wall = oracle_sample(pool, cores, cfg["T"], rows_per_step, seed=i)
            times.append(wall)
            rows += n
        pool.close()
        total = sum(times)
        value = rows / total
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                 "sample": f"{rows_per_step} uniformly drawn query rows per step of the row-restricted "
                                           f"dense float64 form, {cores} single-threaded processes"},
                "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    pool = None
    if rank == 0 and not args.no_cpu_baseline:
        pool = oracle_pool(cores, cfg)  # spawned before the first GPU call

    import torch
    from log_linear_attention_chunked_gb300 import binding

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    binding.lib()

    inp_host = synth.make_inputs(cfg, tag=f"rank{rank}" if rank else "")
    names = ("q", "k", "v", "log_alpha", "lam")
    host = {n: inp_host[n].pin_memory() for n in names}
    g = {n: host[n].to(dev) for n in names}
    Bn, H, T, dk = g["q"].shape
    dv = g["v"].shape[-1]
    shape = binding.make_shape(Bn, H, T, dk, dv, cfg["L"], cfg["chunk"], 0, binding._io(g["q"].dtype))
    ws = binding.alloc_workspace(binding.ll_attn_fwd_workspace_size(shape), dev)
    o = torch.empty(Bn, H, T, dv, dtype=g["q"].dtype, device=dev)
    o_host = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    launches_per_call = binding.ll_attn_fwd_launches(shape)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        binding.ll_attn_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["lam"], cfg["chunk"], o=o, workspace=ws)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    if binding.ll_last_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    time.sleep(0.1)
    barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier()
    clocks = sampler.stop()
    if binding.ll_last_device_error() != 0:
        raise RuntimeError("device error during the timed region")
    step_ms = [a.elapsed_time(b) for a, b in ev]
    mean_ms = sum(step_ms) / len(step_ms)
    if world > 1:
        t = torch.tensor([mean_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        mean_ms = float(t.item())
    value = tokens_per_step * world / (mean_ms * 1e-3)

    # end to end: pinned host inputs -> device -> forward -> host output
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = o_host.numel() * o_host.element_size()
    e2e_steps = max(3, min(args.steps, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(e2e_steps + 2):
        if i == 2:
            barrier()
            torch.cuda.synchronize()
            e0.record(stream)
        for n in names:
            g[n].copy_(host[n], non_blocking=True)
        step()
        o_host.copy_(o, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    if world > 1:
        t = torch.tensor([e2e_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_ms = float(t.item())
    e2e = {"value": tokens_per_step * world / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}

    # roofline of the dominant kernel (one launch per call on the tensor-core path)
    hbm, bf16, src = measured_peaks()
    abytes = algorithmic_bytes(cfg)
    aflops = algorithmic_flops(cfg)
    achieved_gbs = abytes / (mean_ms * 1e-3) / 1e9
    traffic, kname = ncu_traffic(args.workload)
    roofline = {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm, "unit": "GB/s", "frac": achieved_gbs / hbm,
                "traffic": traffic, "peak_source": f"{src} (HBM copy)",
                "algorithmic_bytes_per_launch": abytes, "launches_per_step": launches_per_call,
                "kernel": kname,
                "tensor": {"achieved_tflops": aflops / (mean_ms * 1e-3) / 1e12, "peak_tflops": bf16,
                           "frac": aflops / (mean_ms * 1e-3) / 1e12 / bf16, "algorithmic_flops": aflops}}

    cpu = None
    if pool is not None:
        oracle_sample(pool, cores, cfg["T"], cores, seed=998)  # workers finish their set-up
        _, n, wall = oracle_sample(pool, cores, cfg["T"], cores * 16, seed=999)
        rows_total = max(cores, int(12.0 / (wall / n)))  # about 12 s of wall time on all cores
        tps, n, secs = oracle_sample(pool, cores, cfg["T"], rows_total)
        pool.close()
        cpu = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} uniformly drawn query rows of the row-restricted dense float64 form "
                         f"({secs:.1f} s wall, {cores} single-threaded processes)"}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": cfg["io"] if cfg["io"] != "f32" else "f32", "data": "synthetic",
                "config": config, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
                "gpu_launches": launches_per_call * args.steps,
                "wall_s_timed_region": wall, "step_ms_min": min(step_ms), "step_ms_median": statistics.median(step_ms)}
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
