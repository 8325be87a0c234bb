"""Throughput of the log-linear attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

Default workload: the log-linear Mamba-2 forward at B=1, H=16, T=16384,
d=128, bf16 in / float32 accumulate.  One step = one ll_attn_fwd call over the
whole workload (every step of the hot path: intra-chunk attention, chunk
states, the Fenwick node tree and the inter-chunk levels).  Other workloads:
`decode_b64_t64k` (one ll_attn_decode_step for 64 x 32 heads with 17 stored
levels, positions 65536 onward), `gdn_bf16_t4k` (one ll_gdn_fwd),
`gdn_b_bf16_t4k` (one ll_gdn_fwd_b), `gdn_decode_b64_t64k` (one
ll_gdn_decode_step), `mamba2_cont_bf16_t16k` (one ll_attn_fwd_cont),
`level_decay_bf16_t16k` (one ll_attn_fwd_level_decay) and
`mamba2_bwd_bf16_t16k` (one ll_attn_bwd over the default workload's shape,
with an upstream gradient of o).

A default run (the forward workload, no --workload) also times, in the same
process and on the same GPU, the decode step (`decode_b64_t64k`, 256 steps),
the Gated DeltaNet forward (`gdn_bf16_t4k`) and the forward with one decay
per level (`level_decay_bf16_t16k`), each with its own warm-up, clock
record, roofline and end-to-end figure, under the line's `secondary` key
(`--no-secondary` skips them).

Roofline of a step: the slower of its algorithmic flops at the measured bf16
tensor peak and its algorithmic bytes at the measured HBM copy bandwidth; the
line reports the achieved rate of that resource and its fraction.

Inputs are resident in HBM when a timed step starts.  The forward workloads
flush L2 between steps (a write of 2x the L2 size, outside the timed
events); the decode workload streams 2.3 GB of states, far larger than L2.
Each step is timed with CUDA events on the launching stream; `value` = units
of all ranks / max over ranks of the mean step time.  `e2e` times the same
public call with its inputs copied from pinned host memory and its output
copied back, all inside the timed region.

Under torchrun (N > 1) every rank runs the same workload on its own GPU with
no collective in the data path (weak scaling); a barrier brackets the timed
region.  `--impl reference` times the float64 CPU oracle instead (rank 0
only), on a bounded sample of the workload per step.
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

PROFILES = os.path.join(ROOT, "profiles")
METRICS = {
    "mamba2": "log-linear Mamba-2 fwd tokens/s at T=16K,H=16,d=128; % of roofline",
    "decode": "log-linear Mamba-2 Fenwick decode tokens/s (B=64, H=32, d=128, 17 levels); % of HBM roofline",
    "gdn": "log-linear Gated DeltaNet fwd tokens/s (B=2, H=16, T=4096, d=128)",
    "gdn_b": "log-linear Gated DeltaNet fwd, reading B, tokens/s (B=2, H=16, T=4096, d=128)",
    "mamba2_cont": "log-linear Mamba-2 prefill continuation tokens/s (16K new tokens at 49152, H=16, d=128); "
                   "% of roofline",
    "gdn_decode": "log-linear Gated DeltaNet Fenwick decode tokens/s (B=64, H=32, d=128, 17 levels); "
                  "% of HBM roofline",
    "mamba2_bwd": "log-linear Mamba-2 bwd tokens/s (dq, dk, dv, dlog_alpha, dlam) at T=16K,H=16,d=128",
    "level_decay": "log-linear Mamba-2 fwd with one decay per level, tokens/s at T=16K,H=16,d=128",
}


# ----------------------------------------------------------------------------
# algorithmic work (counted per (b, h), times B*H)
# ----------------------------------------------------------------------------
def algorithmic_bytes(cfg) -> int:
    """Forward: q, k, v read once, log_alpha and lam (float32) read once, o
    written once; plus beta for Gated DeltaNet.  Backward: its inputs (the
    forward's and dout) read once and the five gradients written once."""
    b_io = 2 if cfg["io"] == "bf16" else 4
    if cfg["kind"] == "mamba2_bwd":
        # q, k, v, dout read and dq, dk, dv written (io dtype); log_alpha and
        # lam read and their gradients written (float32)
        dk, dv = cfg["dk"], cfg["dv"]
        per_bh = cfg["T"] * ((2 * dk + 2 * dv) * b_io + (2 * dk + dv) * b_io + 2 * (4 + 4 * cfg["L"]))
        return per_bh * cfg["B"] * cfg["H"]
    per_bh = cfg["T"] * (3 * cfg["dk"] * b_io + 4 + 4 * cfg["L"] + cfg["dv"] * b_io)
    if cfg["kind"] == "level_decay":  # log_alpha has L columns
        per_bh += cfg["T"] * 4 * (cfg["L"] - 1)
    if cfg["kind"] in ("gdn", "gdn_b"):
        per_bh += cfg["T"] * 4
    if cfg["kind"] == "mamba2_cont":  # the prefix states read, the states of t0 + T written (float32)
        t0, t1, d = cfg["t0"], cfg["t0"] + cfg["T"], cfg["dk"]
        per_bh += (bin(t0).count("1") + bin(t1).count("1")) * d * d * 4 + 2 * cfg["Ls"] * 4
    return per_bh * cfg["B"] * cfg["H"]


def algorithmic_flops(cfg) -> int:
    """Forward: causal pairs inside a chunk, chunk states, tree combines and
    the popcount(c) non-empty inter-chunk levels of every chunk c."""
    T, C, d = cfg["T"], cfg["chunk"], cfg["dk"]
    N = T // C
    P = sum(bin(c).count("1") for c in range(N))
    if cfg["kind"] == "mamba2_bwd":  # counted for the tiles the path runs on
        return backward_flops(dict(cfg, chunk=128) if backward_on_tensor_cores(cfg) else cfg)
    if cfg["kind"] == "gdn":
        per_chunk = 10 * C * C * d + (4 * C ** 3) // 3 + 2 * C * d * d
        per_bh = N * per_chunk + P * (6 * C * d * d + 2 * C * C * d)
    elif cfg["kind"] == "gdn_b":
        # per chunk: K K^T (lower half), Tinv, U and W (triangular), S_c; the
        # single-state pass (S W^T and the update, 4 C d^2); then the
        # log-linear Mamba-2 forward on the pseudo-values
        per_chunk = 3 * C * C * d + (2 * C ** 3) // 3 + 2 * C * d * d + 4 * C * d * d
        per_bh = N * per_chunk + 2 * d * T * (C + 1) + 2 * T * d * d + 3 * d * d * N + 2 * d * d * C * P
    else:
        per_bh = 2 * d * T * (C + 1) + 2 * T * d * d + 3 * d * d * N + 2 * d * d * C * P
        if cfg["kind"] == "mamba2_cont":  # every token also reads the prefix levels
            per_bh += 2 * d * d * T * bin(cfg["t0"]).count("1")
    return per_bh * cfg["B"] * cfg["H"]


def backward_flops(cfg) -> int:
    """Backward, per chunk: the causal pairs' scores and dO V^T, then dq, dk, dv
    (10 d flops per pair) and the chunk state; per set bit of a chunk, the
    query side (F^T dO) and its share of the key-side node (4 C d^2); per chunk
    with later queries, the key-side products (4 C d^2) and the node sum; the
    Fenwick tree's combines."""
    T, C, d = cfg["T"], cfg["chunk"], cfg["dk"]
    N = (T + C - 1) // C
    pairs = C * (C + 1) // 2
    per_bh = N * (10 * d * pairs + 2 * C * d * d)
    for c in range(N):
        per_bh += 4 * C * d * d * bin(c).count("1")
        n = 0
        for h in range(31):
            if (c >> h) & 1:
                continue
            e = ((c >> (h + 1)) << (h + 1)) + (1 << h) - 1
            if e + 1 >= N:
                break
            n += 1
        if n:
            per_bh += 4 * C * d * d + 2 * n * d * d
        per_bh += 2 * d * d * ((~c & (c + 1)).bit_length() - 1)  # merges into node c
    return per_bh * cfg["B"] * cfg["H"]


def level_decay_on_tensor_cores(cfg) -> bool:
    """The per-level forward's tensor-core path: bf16, d = 128, whole 128-token
    tiles, at most 16 levels (the CUDA-core kernels take every other shape)."""
    return (cfg["io"] == "bf16" and cfg["dk"] == 128 and cfg["dv"] == 128 and cfg["T"] % 128 == 0
            and cfg["L"] <= 16)


def backward_on_tensor_cores(cfg) -> bool:
    """The backward of bf16 io with d_k = d_v = 128 runs on the tensor cores over
    128-token tiles; every other shape on the CUDA cores."""
    return cfg["io"] == "bf16" and cfg["dk"] == 128 and cfg["dv"] == 128


def gdn_decode_bytes(B, H, d, Ls, t) -> int:
    """One Gated DeltaNet decode step: the popcount(t) non-empty states read
    once; the ones above the carry written back transitioned and the merged
    one written (float32); q, k, v and o (bf16), log_alpha, beta and lam
    (float32)."""
    pc = bin(t).count("1")
    j = ((t + 1) & -(t + 1)).bit_length() - 1  # trailing ones of t
    return B * H * ((2 * pc - j + 1) * d * d * 4 + 3 * d * 2 + 4 * (Ls + 1) + 8 + d * 2)


def decode_bytes(B, H, d, Ls, t) -> int:
    """One decode step: the popcount(t) non-empty states read once and one merged
    state written (float32), q, k, v and o (bf16), log_alpha and lam (float32)."""
    return B * H * ((bin(t).count("1") + 1) * d * d * 4 + 3 * d * 2 + 4 * (Ls + 1) + 4 + d * 2)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p.get("sm_max_mhz", 2070.0), "measured"
    return 6800.0, 1900.0, 2070.0, "fallback"


# the sources each workload's kernels are built from: a traffic figure stays
# valid while these files are unchanged
KERNEL_SOURCES = {
    "mamba2": ("fwd_tc.cu", "level_decay.cuh", "common.cuh", "sm100.cuh"),
    "decode": ("decode.cu", "common.cuh"),
    "gdn_decode": ("gdn_decode.cu", "common.cuh"),
    "gdn": ("gdn_tc.cu", "common.cuh", "sm100.cuh"),             # dominant: the tensor-core level scan
    "gdn_b": ("gdn_tc.cu", "common.cuh", "sm100.cuh"),         # dominant: the tensor-core preparation
    "mamba2_cont": ("fwd_tc.cu", "level_decay.cuh", "common.cuh", "sm100.cuh"),  # dominant: the tensor-core forward
    "mamba2_bwd": ("bwd_tc.cu", "bwd.cuh", "common.cuh", "sm100.cuh"),  # dominant: the query-side kernel
    "level_decay": ("fwd_tc.cu", "level_decay.cuh", "common.cuh", "sm100.cuh"),  # dominant: the tensor-core forward
}


def kernel_source_hash(files) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "log_linear_attention_chunked_gb300", "csrc")
    for f in sorted(files):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None when there is none or its sources changed since."""
    path = os.path.join(PROFILES, f"traffic_{workload}.json")
    if not os.path.exists(path):
        return None, None
    with open(path) as f:
        t = json.load(f)
    if t.get("source_hash") != kernel_source_hash(t.get("source_files", ())):
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
# oracle timing (CPU baseline / reference arm), in spawned single-threaded workers
# ----------------------------------------------------------------------------
_W = {}


def _oracle_init(cfg, tag):
    """Worker set-up (untimed): draw one (b, h) slice of the workload."""
    import numpy as np
    from log_linear_attention_chunked_gb300 import synth
    _W["cfg"] = cfg
    if cfg["kind"] == "decode":
        rng = np.random.default_rng(7)
        d, Ls, S = cfg["dk"], cfg["Ls"], cfg["steps"]
        _W["x"] = (rng.standard_normal((Ls, d, d)) * 0.01, rng.standard_normal((S, d)) / np.sqrt(d),
                   rng.standard_normal((S, d)) / np.sqrt(d), rng.standard_normal((S, d)),
                   -np.log1p(np.exp(rng.standard_normal(S))), np.log1p(np.exp(rng.standard_normal((S, Ls + 1)))))
        return
    if cfg["kind"] == "gdn_decode":
        dec = synth.make_decode_inputs(cfg, B=1, H=1)
        rng = np.random.default_rng(7)
        _W["x"] = (rng.standard_normal((cfg["Ls"], cfg["dv"], cfg["dk"])) * 0.05,) + tuple(
            synth.to_f64(dec[n][:, 0, 0]) for n in ("q", "k", "v", "log_alpha", "beta", "lam"))
        return
    if cfg["kind"] == "mamba2_cont":  # the whole sequence: the oracle has no prefix states
        cfg = dict(cfg, kind="mamba2", T=cfg["t0"] + cfg["T"])
    inp = synth.make_inputs(dict(cfg, B=1, H=1), tag=tag)
    names = ("q", "k", "v", "log_alpha", "lam") + (("beta",) if cfg["kind"] in ("gdn", "gdn_b") else ())
    if cfg["kind"] == "mamba2_bwd":
        names += ("dout",)
    _W["x"] = tuple(synth.to_f64(inp[n][0, 0]) for n in names)


def _oracle_worker(job):
    """One bounded piece of oracle work; returns the number of tokens it covered."""
    cfg = _W["cfg"]
    if cfg["kind"] in ("mamba2", "mamba2_cont"):
        from oracle import mamba2
        q, k, v, la, lam = _W["x"]
        mamba2.forward_rows(q, k, v, la, lam, job)
        return float(len(job))
    if cfg["kind"] == "level_decay":
        from oracle import level_decay
        q, k, v, la, lam = _W["x"]
        level_decay.forward_rows(q, k, v, la, lam, job)
        return float(len(job))
    if cfg["kind"] == "gdn":
        from oracle import gdn
        q, k, v, la, lam, beta = _W["x"]
        gdn.gdn_rows_A(q, k, v, beta, la, lam, job)
        return float(len(job))
    if cfg["kind"] == "mamba2_bwd":  # a token's every gradient: its query row and its key row
        from oracle import backward
        backward.backward_query_rows(*_W["x"], job)
        backward.backward_key_rows(*_W["x"], job)
        return float(len(job))
    if cfg["kind"] == "gdn_b":
        from oracle import gdn
        q, k, v, la, lam, beta = _W["x"]
        for _ in range(job):  # whole (b, h) slices: the pseudo-values couple every row
            gdn.gdn_forward_B(q, k, v, beta, la, lam)
        return float(job * q.shape[0])
    if cfg["kind"] == "gdn_decode":
        from oracle import gdn
        S, q, k, v, la, beta, lam = _W["x"]
        t0 = cfg["T"]
        ne = [((t0 >> i) & 1) == 1 for i in range(S.shape[0])]
        left = job
        while left > 0:
            m = min(left, q.shape[0])
            gdn.gdn_decode_steps(S, ne, t0, q[:m], k[:m], v[:m], beta[:m], la[:m], lam[:m])
            left -= m
        return job / cfg["H"]
    from oracle import decode
    S, q, k, v, la, lam = _W["x"]
    t0 = cfg["T"]
    ne = [((t0 >> i) & 1) == 1 for i in range(S.shape[0])]
    # `job` decode steps, cycling over the drawn step inputs (each pass
    # restarts from the stored states at position T)
    left = job
    while left > 0:
        m = min(left, q.shape[0])
        decode.decode_steps(S, ne, t0, q[:m], k[:m], v[:m], la[:m], lam[:m])
        left -= m
    return job / cfg["H"]  # one (b, h) step is 1/H of a token of a batch row


def oracle_pool(cores: int, cfg: dict, tag: str = "oracle"):
    """Spawned single-threaded oracle processes, started before any GPU work."""
    import multiprocessing as mp
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    return mp.get_context("spawn").Pool(cores, initializer=_oracle_init, initargs=(cfg, tag))


def oracle_jobs(cfg, cores, size, seed):
    import numpy as np
    rng = np.random.default_rng(seed)
    if cfg["kind"] in ("mamba2", "gdn", "mamba2_bwd", "level_decay"):
        return [sorted(int(x) for x in rng.integers(0, cfg["T"], size)) for _ in range(cores)]
    if cfg["kind"] == "mamba2_cont":  # rows of the new tokens, positions t0 .. t0 + T - 1
        return [sorted(int(x) for x in rng.integers(cfg["t0"], cfg["t0"] + cfg["T"], size)) for _ in range(cores)]
    return [size for _ in range(cores)]


def oracle_sample(pool, cfg, cores, size, seed=0):
    """Run `cores` jobs of `size` units in parallel; returns (tokens/s, tokens, seconds)."""
    jobs = oracle_jobs(cfg, cores, size, seed)
    t0 = time.perf_counter()
    n = sum(pool.map(_oracle_worker, jobs, chunksize=1))
    wall = time.perf_counter() - t0
    return n / wall, n, wall


def calibrate(pool, cfg, cores, budget_s):
    """Job size so that one sample takes about `budget_s` seconds of wall time."""
    small = 1 if cfg["kind"] == "gdn_b" else 16
    oracle_sample(pool, cfg, cores, 1, seed=998)  # workers finish their set-up
    _, n, wall = oracle_sample(pool, cfg, cores, small, seed=999)
    return int(min(10 ** 6, max(1, budget_s / (wall / small))))


def sample_desc(cfg, size):
    if cfg["kind"] == "mamba2":
        return f"{size} uniformly drawn query rows per process of the row-restricted dense float64 form"
    if cfg["kind"] == "level_decay":
        return (f"{size} uniformly drawn query rows per process of the row-restricted float64 form with one "
                "decay per level")
    if cfg["kind"] == "mamba2_cont":
        return (f"{size} uniformly drawn rows of the new tokens per process of the row-restricted dense float64 "
                "form over the whole sequence")
    if cfg["kind"] == "gdn":
        return (f"{size} uniformly drawn query rows per process of the row-restricted float64 reading-A form "
                "(each call builds its unit-triangular system)")
    if cfg["kind"] == "gdn_decode":
        return f"{size} float64 Gated DeltaNet decode steps of one (b, h) per process"
    if cfg["kind"] == "mamba2_bwd":
        return (f"{size} uniformly drawn tokens per process of the row-restricted dense float64 gradients "
                "(query row: dq, dlam; key row: dk, dv; both: the token's dc)")
    if cfg["kind"] == "gdn_b":
        return (f"{size} whole (b, h) slices ({cfg['T']} tokens) per process of the dense float64 reading-B "
                "form (one triangular solve per slice)")
    return f"{size} float64 decode steps of one (b, h) per process"


# ----------------------------------------------------------------------------
# multi-rank aggregation (one process per GPU; ranks hold independent replicas)
# ----------------------------------------------------------------------------
def max_over_ranks(x: float, world: int, device=None) -> float:
    """The slowest rank's figure: every rank passes its own, all get the max."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Units of all ranks per second when every rank took (at most) `ms` per step."""
    return units_per_rank * world / (ms * 1e-3)


# ----------------------------------------------------------------------------
# GPU workloads
# ----------------------------------------------------------------------------
def forward_workload(cfg, dev, rank, binding, synth, torch):
    """Forward (Mamba-2 or Gated DeltaNet): device and pinned host inputs, step functions."""
    gdn = cfg["kind"] in ("gdn", "gdn_b")
    reading_b = cfg["kind"] == "gdn_b"
    cont = cfg["kind"] == "mamba2_cont"
    per_level = cfg["kind"] == "level_decay"
    inp_host = synth.make_inputs(cfg, tag=f"rank{rank}" if rank else "")
    names = ("q", "k", "v", "log_alpha", "lam") + (("beta",) if gdn else ())
    host = {n: inp_host[n].pin_memory() for n in names}
    g = {n: host[n].to(dev) for n in names}
    Bn, H, T, dk = g["q"].shape
    dv = g["v"].shape[-1]
    shape = binding.make_shape(Bn, H, T, dk, dv, cfg["L"], cfg["chunk"], 0, binding._io(g["q"].dtype))
    if cont:
        t0, Ls = cfg["t0"], cfg["Ls"]
        shape = binding.make_shape(Bn, H, T, dk, dv, cfg["L"], cfg["chunk"], Ls, binding._io(g["q"].dtype))
        ws = binding.alloc_workspace(binding.ll_attn_fwd_cont_workspace_size(shape, t0), dev)
        gen = torch.Generator(device=dev)
        gen.manual_seed(cfg["seed"] + 17 + rank)
        keep = torch.tensor([float((t0 >> i) & 1) for i in range(Ls)], device=dev)
        st_in = torch.randn(Bn, H, Ls, dv, dk, device=dev, generator=gen) * 0.01 * keep[None, None, :, None, None]
        sc_in = keep.expand(Bn, H, Ls).contiguous()
        st_out, sc_out = torch.empty_like(st_in), torch.empty_like(sc_in)
        launches = 3  # prefix nodes, forward, the export of the states of t0 + T
    elif per_level:
        ws = binding.alloc_workspace(binding.ll_attn_fwd_level_decay_workspace_size(shape), dev)
        launches = binding.ll_attn_fwd_level_decay_launches(shape)
    elif reading_b:
        ws = binding.alloc_workspace(binding.ll_gdn_fwd_b_workspace_size(shape), dev)
        launches = 2 + binding.ll_attn_fwd_launches(shape)
    elif gdn:
        ws = binding.alloc_workspace(binding.ll_gdn_fwd_workspace_size(shape), dev)
        launches = 2
    else:
        ws = binding.alloc_workspace(binding.ll_attn_fwd_workspace_size(shape), dev)
        launches = binding.ll_attn_fwd_launches(shape)
    o = torch.empty(Bn, H, T, dv, dtype=g["q"].dtype, device=dev)
    o_host = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)

    def run(x, out):  # one call of the public API on the current stream
        if cont:
            binding.ll_attn_fwd_cont(t0, st_in, sc_in, x["q"], x["k"], x["v"], x["log_alpha"], x["lam"],
                                     cfg["chunk"], o=out, state_out=st_out, scale_out=sc_out, workspace=ws)
        elif per_level:
            binding.ll_attn_fwd_level_decay(x["q"], x["k"], x["v"], x["log_alpha"], x["lam"], cfg["chunk"], o=out,
                                            workspace=ws)
        elif reading_b:
            binding.ll_gdn_fwd_b(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["lam"], cfg["chunk"], o=out,
                                 workspace=ws)
        elif gdn:
            binding.ll_gdn_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["lam"], cfg["chunk"], o=out,
                               workspace=ws)
        else:
            binding.ll_attn_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["lam"], cfg["chunk"], o=out, workspace=ws)

    def step(i=0):
        run(g, o)

    # End to end: every step uploads its inputs from pinned host memory and
    # reads its output back; two device input sets and two outputs let the
    # upload of step i+1 (one copy stream) and the read-back of step i-1
    # (another) run while step i computes.
    gset = [g, {n: torch.empty_like(g[n]) for n in names}]
    oset = [o, torch.empty_like(o)]
    ohost = [o_host, torch.empty(o.shape, dtype=o.dtype, pin_memory=True)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def e2e_step(i=0):
        b = i & 1
        comp = torch.cuda.current_stream(dev)
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(ev_done[b])  # the call of step i-2 has read this input set
            for n in names:
                gset[b][n].copy_(host[n], non_blocking=True)
            ev_in[b].record(s_in)
        comp.wait_event(ev_in[b])
        if used[b]:
            comp.wait_event(ev_out[b])  # the output of step i-2 is back on the host
        run(gset[b], oset[b])
        ev_done[b].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[b])
            ohost[b].copy_(oset[b], non_blocking=True)
            ev_out[b].record(s_out)
        used[b] = True

    def e2e_begin(ev0):  # the first timed upload starts after the start event
        s_in.wait_event(ev0)

    def e2e_end():  # the current stream waits for the last read-back
        torch.cuda.current_stream(dev).wait_stream(s_out)

    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = o_host.numel() * o_host.element_size()
    return dict(step=step, e2e_step=e2e_step, e2e_begin=e2e_begin, e2e_end=e2e_end, units=Bn * H * T, h2d=h2d,
                d2h=d2h, launches=launches, flush=True, abytes=algorithmic_bytes(cfg), aflops=algorithmic_flops(cfg))


def backward_workload(cfg, dev, rank, binding, synth, torch):
    """Backward: the forward's inputs plus dout resident; one ll_attn_bwd per step."""
    names = ("q", "k", "v", "log_alpha", "lam", "dout")
    inp_host = synth.make_inputs(cfg, tag=f"rank{rank}" if rank else "")
    host = {n: inp_host[n].pin_memory() for n in names}
    g = {n: host[n].to(dev) for n in names}
    Bn, H, T, dk = g["q"].shape
    dv = g["v"].shape[-1]
    shape = binding.make_shape(Bn, H, T, dk, dv, cfg["L"], cfg["chunk"], 0, binding._io(g["q"].dtype))
    ws = binding.alloc_workspace(binding.ll_attn_bwd_workspace_size(shape), dev)
    launches = binding.ll_attn_bwd_launches(shape)
    gnames = ("q", "k", "v", "log_alpha", "lam")

    def new_grads():
        return tuple(torch.empty_like(g[n]) for n in gnames)

    grads = new_grads()

    def run(x, out):
        binding.ll_attn_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["lam"], x["dout"], cfg["chunk"], grads=out,
                            workspace=ws)

    def step(i=0):
        run(g, grads)

    # End to end as for the forward: inputs up on one copy stream, the five
    # gradients down on another, two sets of each
    gset = [g, {n: torch.empty_like(g[n]) for n in names}]
    oset = [grads, new_grads()]
    ohost = [tuple(torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in grads) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def e2e_step(i=0):
        b = i & 1
        comp = torch.cuda.current_stream(dev)
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(ev_done[b])
            for n in names:
                gset[b][n].copy_(host[n], non_blocking=True)
            ev_in[b].record(s_in)
        comp.wait_event(ev_in[b])
        if used[b]:
            comp.wait_event(ev_out[b])
        run(gset[b], oset[b])
        ev_done[b].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[b])
            for hst, dev_grad in zip(ohost[b], oset[b]):
                hst.copy_(dev_grad, non_blocking=True)
            ev_out[b].record(s_out)
        used[b] = True

    def e2e_begin(ev0):
        s_in.wait_event(ev0)

    def e2e_end():
        torch.cuda.current_stream(dev).wait_stream(s_out)

    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = sum(x.numel() * x.element_size() for x in grads)
    return dict(step=step, e2e_step=e2e_step, e2e_begin=e2e_begin, e2e_end=e2e_end, units=Bn * H * T, h2d=h2d,
                d2h=d2h, launches=launches, flush=True, abytes=algorithmic_bytes(cfg), aflops=algorithmic_flops(cfg))


def decode_workload(cfg, dev, rank, binding, synth, torch):
    """Decode: 2.3 GB of level states (random values: the work of a step does not
    depend on them), per-step inputs drawn once, positions 65536 onward."""
    Bn, H, d, Ls, S = cfg["B"], cfg["H"], cfg["dk"], cfg["Ls"], cfg["steps"]
    gdn = cfg["kind"] == "gdn_decode"
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg["seed"] + rank)
    states = torch.randn(Bn, H, Ls, d, d, device=dev, generator=gen) * 0.01
    scales = torch.ones(Bn, H, Ls, device=dev)
    dec = synth.make_decode_inputs(cfg, device="cpu", B=Bn, H=H)
    names = ("q", "k", "v", "log_alpha", "lam") + (("beta",) if gdn else ())
    host = {n: dec[n].pin_memory() for n in names}
    g = {n: host[n].to(dev) for n in names}
    t_host = torch.tensor([[cfg["T"] + i] * Bn for i in range(S)], dtype=torch.int64).pin_memory()
    t_dev = t_host.to(dev)
    o = torch.empty(Bn, H, d, dtype=g["q"].dtype, device=dev)
    o_host = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    pos = [0]

    def call(t, x, out):
        if gdn:
            binding.ll_gdn_decode_step(t, x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["lam"], states,
                                       o=out)
        else:
            binding.ll_attn_decode_step(t, x["q"], x["k"], x["v"], x["log_alpha"], x["lam"], states, scales, o=out)

    def step(i=0):
        s = pos[0] % S
        call(t_dev[s], {n: g[n][s] for n in names}, o)
        pos[0] += 1

    def reset():
        pos[0] = 0
        scales.fill_(1.0)

    # End to end: each step uploads its token inputs and position and reads its
    # output back; two input sets and two outputs let step i+1's upload and
    # step i-1's read-back run on copy streams while step i computes (the
    # steps themselves stay in order on the compute stream: they update the
    # states in place).
    xset = [{n: torch.empty_like(g[n][0]) for n in names} for _ in range(2)]
    tset = [torch.empty_like(t_dev[0]) for _ in range(2)]
    oset = [o, torch.empty_like(o)]
    ohost = [o_host, torch.empty(o.shape, dtype=o.dtype, pin_memory=True)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def e2e_step(i=0):
        s, b = pos[0] % S, i & 1
        comp = torch.cuda.current_stream(dev)
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(ev_done[b])  # the step that last read this input set is done
            for n in names:
                xset[b][n].copy_(host[n][s], non_blocking=True)
            tset[b].copy_(t_host[s], non_blocking=True)
            ev_in[b].record(s_in)
        comp.wait_event(ev_in[b])
        if used[b]:
            comp.wait_event(ev_out[b])  # that step's output is back on the host
        call(tset[b], xset[b], oset[b])
        ev_done[b].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[b])
            ohost[b].copy_(oset[b], non_blocking=True)
            ev_out[b].record(s_out)
        used[b] = True
        pos[0] += 1

    def e2e_begin(ev0):
        s_in.wait_event(ev0)

    def e2e_end():
        torch.cuda.current_stream(dev).wait_stream(s_out)

    h2d = sum(host[n][0].numel() * host[n].element_size() for n in names) + Bn * 8
    d2h = o_host.numel() * o_host.element_size()
    nbytes = gdn_decode_bytes if gdn else decode_bytes
    return dict(step=step, e2e_step=e2e_step, e2e_begin=e2e_begin, e2e_end=e2e_end, reset=reset, units=Bn, h2d=h2d,
                d2h=d2h, launches=1, flush=False, step_bytes=lambda i: nbytes(Bn, H, d, Ls, cfg["T"] + (i % S)))


DEFAULT_WORKLOAD = "mamba2_bf16_t16k"
# timed after the primary in a default run: (workload, steps)
SECONDARY = (("decode_b64_t64k", 256), ("gdn_bf16_t4k", 50), ("level_decay_bf16_t16k", 100))


def workload_config(cfg, name, world):
    """The `config` object of a JSON line: the workload and its sizes."""
    kind = cfg["kind"]
    config = {"workload": name, "B": cfg["B"], "H": cfg["H"], "T": cfg["T"], "dk": cfg["dk"],
              "dv": cfg["dv"], "chunk": cfg["chunk"], "L": cfg["L"], "io": cfg["io"],
              "parallelism": f"replicas x{world} (b,h) weak"}
    if kind in ("decode", "gdn_decode"):
        config.update(Ls=cfg["Ls"], positions=f"{cfg['T']}..{cfg['T'] + cfg['steps'] - 1} cycled",
                      l2="states (2.3 GB) larger than L2, no flush")
    elif kind == "mamba2_cont":
        config.update(t0=cfg["t0"], Ls=cfg["Ls"], l2="flushed between steps (write of 2x L2)",
                      prefix="decode states of position t0 (random values on its set bits), states of t0+T exported")
    else:
        config["l2"] = "flushed between steps (write of 2x L2)"
    return config


# ----------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="default workload only: skip the decode, Gated DeltaNet and per-level-decay blocks")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from log_linear_attention_chunked_gb300 import synth
    cfg = dict(synth.WORKLOADS[args.workload])
    kind = cfg["kind"]
    metric = METRICS[kind]
    config = workload_config(cfg, args.workload, world)

    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)

    if args.impl == "reference":
        if rank != 0:
            return
        pool = oracle_pool(cores, cfg)
        size = calibrate(pool, cfg, cores, budget_s=60.0 / max(args.steps + args.warmup, 1))
        for i in range(args.warmup):
            oracle_sample(pool, cfg, cores, size, seed=1000 + i)
        times, units = [], 0.0
        for i in range(args.steps):
            _, n, wall = oracle_sample(pool, cfg, cores, size, seed=i)
            times.append(wall)
            units += n
        pool.close()
        total = sum(times)
        value = units / total
        line = {"impl": "reference", "metric": metric, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                 "sample": sample_desc(cfg, size) + f", {cores} single-threaded processes"},
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

    r = measure(cfg, args.workload, args.steps, args.warmup, dev, rank, world, binding, synth, torch)

    # the other hot-path steps, timed in the same run on the same GPU (their
    # own inputs, warm-up and clock record); weak scaling like the primary
    secondary = {}
    if args.workload == DEFAULT_WORKLOAD and not args.no_secondary:
        for name, steps in SECONDARY:
            c2 = dict(synth.WORKLOADS[name])
            r2 = measure(c2, name, steps, args.warmup, dev, rank, world, binding, synth, torch)
            secondary[name] = {"metric": METRICS[c2["kind"]], "value": r2["value"], "unit": "tokens/s",
                               "steps": steps, "warmup": args.warmup, "ms_per_step": r2["mean_ms"],
                               "step_ms_median": statistics.median(r2["step_ms"]), "roofline": r2["roofline"],
                               "e2e": r2["e2e"], "clocks": r2["clocks"], "gpu_launches": r2["launches"] * steps,
                               "config": workload_config(c2, name, world)}

    cpu = None
    if pool is not None:
        size = calibrate(pool, cfg, cores, budget_s=12.0)
        tps, n, secs = oracle_sample(pool, cfg, cores, size)
        pool.close()
        cpu = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": sample_desc(cfg, size) + f" ({secs:.1f} s wall, {cores} single-threaded processes)"}

    if rank == 0:
        line = {"metric": metric, "value": r["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": r["mean_ms"], "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": cfg["io"], "data": "synthetic", "config": config,
                "roofline": r["roofline"], "cpu_baseline": cpu, "e2e": r["e2e"], "clocks": r["clocks"],
                "gpu_launches": r["launches"] * args.steps, "wall_s_timed_region": r["wall"],
                "step_ms_min": min(r["step_ms"]), "step_ms_median": statistics.median(r["step_ms"])}
        if secondary:
            line["secondary"] = secondary
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


def roofline_of(cfg, workload, w, mean_ms, dev, torch):
    """Roofline of one step: the slower of its algorithmic flops at the bf16
    tensor peak and its algorithmic bytes at the HBM copy bandwidth; the
    achieved rate of that resource over the measured step time."""
    kind = cfg["kind"]
    hbm, bf16, sm_mhz, src = measured_peaks()
    traffic, kname = ncu_traffic(workload)
    if kind in ("decode", "gdn_decode"):
        abytes = sum(w["step_bytes"](i) for i in range(w["timed_steps"])) / w["timed_steps"]
        achieved = abytes / (mean_ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": traffic, "peak_source": f"{src} (HBM copy)", "algorithmic_bytes_per_launch": abytes,
                "launches_per_step": w["launches"], "kernel": kname}
    abytes, aflops = w["abytes"], w["aflops"]
    if (kind == "mamba2_bwd" and not backward_on_tensor_cores(cfg)) or (
            kind == "level_decay" and not level_decay_on_tensor_cores(cfg)):
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        alu_peak = sms * 128 * 2 * sm_mhz * 1e6 / 1e12  # float32 FMA lanes x clock
        achieved = aflops / (mean_ms * 1e-3) / 1e12
        return {"bound": "alu", "achieved": achieved, "peak": alu_peak, "unit": "TFLOP/s",
                "frac": achieved / alu_peak, "traffic": traffic,
                "peak_source": f"float32 FMA: {sms} SMs x 128 lanes x 2 x {sm_mhz:.0f} MHz ({src} clock)",
                "algorithmic_flops_per_step": aflops, "launches_per_step": w["launches"], "kernel": kname}
    t_hbm = abytes / (hbm * 1e9)
    t_tensor = aflops / (bf16 * 1e12)
    gbs = abytes / (mean_ms * 1e-3) / 1e9
    tfs = aflops / (mean_ms * 1e-3) / 1e12
    other_hbm = {"achieved_gbs": gbs, "peak": hbm, "frac": gbs / hbm, "algorithmic_bytes": abytes}
    other_tensor = {"achieved_tflops": tfs, "peak_tflops": bf16, "frac": tfs / bf16, "algorithmic_flops": aflops}
    if t_tensor > t_hbm:
        return {"bound": "tensor", "achieved": tfs, "peak": bf16, "unit": "TFLOP/s", "frac": tfs / bf16,
                "traffic": traffic, "peak_source": f"{src} (cuBLAS bf16 burst)", "algorithmic_flops_per_step": aflops,
                "launches_per_step": w["launches"], "kernel": kname, "hbm": other_hbm,
                "roof_us": {"tensor": t_tensor * 1e6, "hbm": t_hbm * 1e6}}
    return {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm, "traffic": traffic,
            "peak_source": f"{src} (HBM copy)", "algorithmic_bytes_per_launch": abytes,
            "launches_per_step": w["launches"], "kernel": kname, "tensor": other_tensor,
            "roof_us": {"tensor": t_tensor * 1e6, "hbm": t_hbm * 1e6}}


def measure(cfg, workload, steps, warmup, dev, rank, world, binding, synth, torch):
    """Warm up, then time `steps` steps of one workload (CUDA events on the
    launching stream, clocks sampled meanwhile, barrier + synchronise on both
    sides), then the same number of end-to-end steps through the public call
    with host buffers.  Returns the figures of the JSON line."""
    kind = cfg["kind"]
    if kind in ("decode", "gdn_decode"):
        w = decode_workload(cfg, dev, rank, binding, synth, torch)
    elif kind == "mamba2_bwd":
        w = backward_workload(cfg, dev, rank, binding, synth, torch)
    else:
        w = forward_workload(cfg, dev, rank, binding, synth, torch)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev) if w["flush"] else None
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for i in range(warmup):
        if flush is not None:
            flush.fill_(1.0)
        w["step"](i)
    torch.cuda.synchronize()
    if binding.ll_last_device_error() != 0:
        raise RuntimeError(f"{workload}: device error during warm-up")
    if "reset" in w:
        w["reset"]()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sampler = ClockSampler(dev.index)
    time.sleep(0.1)
    barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(steps):
        if flush is not None:
            flush.fill_(float(i))
        ev[i][0].record(stream)
        w["step"](i)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier()
    clocks = sampler.stop()
    if binding.ll_last_device_error() != 0:
        raise RuntimeError(f"{workload}: device error during the timed region")
    step_ms = [a.elapsed_time(b) for a, b in ev]
    mean_ms = max_over_ranks(sum(step_ms) / len(step_ms), world, dev)
    value = whole_job_rate(w["units"], world, mean_ms)

    # end to end through the public call: host inputs in, host output out
    if "reset" in w:
        w["reset"]()
    e2e_steps = max(3, steps)  # the same number of steps (decode: the same positions) as the timed loop
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(e2e_steps + 2):
        if i == 2:
            barrier()
            torch.cuda.synchronize()
            e0.record(stream)
            if "e2e_begin" in w:
                w["e2e_begin"](e0)
        w["e2e_step"](i)
    if "e2e_end" in w:
        w["e2e_end"]()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)
    e2e = {"value": whole_job_rate(w["units"], world, e2e_ms), "unit": "tokens/s", "h2d_bytes_per_step": w["h2d"],
           "d2h_bytes_per_step": w["d2h"], "ms_per_step": e2e_ms}
    w["timed_steps"] = steps
    roofline = roofline_of(cfg, workload, w, mean_ms, dev, torch)
    out = dict(value=value, mean_ms=mean_ms, step_ms=step_ms, wall=wall, clocks=clocks, e2e=e2e, roofline=roofline,
               launches=w["launches"])
    del w, flush
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


if __name__ == "__main__":
    main()
