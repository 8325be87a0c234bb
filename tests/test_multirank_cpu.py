"""The benchmark's multi-rank path on the CPU: two gloo ranks (one process
each, as under torchrun), replicas of the (b, h) work with no data-path
collective; the timing reduction takes the slowest rank and the figure
counts every rank's units; each rank draws its own inputs."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from log_linear_attention_chunked_gb300 import synth
        own_ms = [0.40, 0.55][rank]                      # rank 1 is the slower one
        ms = bench.max_over_ranks(own_ms, world)
        rate = bench.whole_job_rate(1000.0, world, ms)
        cfg = dict(synth.WORKLOADS["mamba2_fp32_t64"])
        x = synth.make_inputs(cfg, tag=f"rank{rank}" if rank else "")["q"]
        got = [torch.zeros_like(x) for _ in range(world)]
        dist.all_gather(got, x)                          # test-only: compare the ranks' draws
        q.put((rank, ms, rate, bool(torch.equal(got[0], got[1]))))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, rate, same in res:
        assert ms == pytest.approx(0.55)                 # every rank holds the slowest rank's time
        assert rate == pytest.approx(2 * 1000.0 / 0.55e-3)
        assert not same                                  # replicas work on different inputs


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(0.3, 1) == 0.3
    assert bench.whole_job_rate(10.0, 1, 2.0) == pytest.approx(5000.0)
