"""Host logic of bench.py (no GPU): the algorithmic counts behind the
roofline, the tie of a traffic figure to its kernel sources, and the oracle
workers of the CPU baseline and reference arms."""

import json
import os

import numpy as np
import pytest

import bench
from log_linear_attention_chunked_gb300 import synth


def test_forward_counts_match_the_documented_figures():
    cfg = synth.WORKLOADS["mamba2_bf16_t16k"]
    # B*H*T*(3d*2 + 4 + 4L + d*2) bytes
    assert bench.algorithmic_bytes(cfg) == 16 * 16384 * (3 * 128 * 2 + 4 + 4 * 15 + 128 * 2) == 285_212_672
    assert abs(bench.algorithmic_flops(cfg) - 4.75e10) / 4.75e10 < 0.01


def test_backward_counts():
    cfg = synth.WORKLOADS["mamba2_bwd_bf16_t16k"]
    d, L, T = 128, 15, 16384
    # q, k, v, dout read and dq, dk, dv written (seven bf16 tensors of d per token);
    # log_alpha and lam read and their gradients written (float32)
    assert bench.algorithmic_bytes(cfg) == 16 * T * (7 * d * 2 + 2 * (4 + 4 * L)) == 503_316_480
    # the tensor-core path runs 128-token tiles whatever the chunk: the count follows the tiles
    assert bench.backward_on_tensor_cores(cfg)
    assert bench.algorithmic_flops(cfg) == bench.backward_flops(dict(cfg, chunk=128))
    assert not bench.backward_on_tensor_cores(dict(cfg, io="f32"))
    assert bench.algorithmic_flops(dict(cfg, io="f32")) == bench.backward_flops(dict(cfg, io="f32"))


def test_backward_flops_grow_with_the_levels():
    # one chunk: intra and chunk state only; more chunks add the level work
    base = dict(synth.WORKLOADS["mamba2_bwd_bf16_t16k"], B=1, H=1, chunk=64)
    one = bench.backward_flops(dict(base, T=64))
    C, d = 64, 128
    assert one == 10 * d * (C * (C + 1) // 2) + 2 * C * d * d
    two = bench.backward_flops(dict(base, T=128))
    # chunk 1 has bit 0 set (query side, 4 C d^2); chunk 0 has later queries at level 0
    # (key side, 4 C d^2 + the node sum 2 d^2); node 1 merges one child (2 d^2)
    assert two == 2 * one + 4 * C * d * d + (4 * C * d * d + 2 * d * d) + 2 * d * d


def test_traffic_figure_follows_its_sources(tmp_path, monkeypatch):
    files = bench.KERNEL_SOURCES["mamba2"]
    rec = {"kernel": "k", "dram_bytes_per_launch": 123.0, "source_files": list(files),
           "source_hash": bench.kernel_source_hash(files)}
    (tmp_path / "traffic_w.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    assert bench.ncu_traffic("w") == (123.0, "k")
    rec["source_hash"] = "0" * 16  # the sources changed since the capture
    (tmp_path / "traffic_w.json").write_text(json.dumps(rec))
    assert bench.ncu_traffic("w") == (None, "k")
    assert bench.ncu_traffic("absent") == (None, None)


def test_committed_traffic_figures_are_keyed():
    # every committed figure names existing sources and a kernel
    for name in bench.KERNEL_SOURCES:
        for f in bench.KERNEL_SOURCES[name]:
            assert os.path.exists(os.path.join(bench.ROOT, "log_linear_attention_chunked_gb300", "csrc", f)), f


def test_backward_oracle_worker_matches_the_dense_gradients():
    from oracle import backward
    cfg = dict(synth.WORKLOADS["mamba2_bwd_bf16_t16k"], T=96, dk=8, dv=8, L=8, chunk=32)
    bench._oracle_init(cfg, "t")
    rows = [0, 5, 50, 95]
    assert bench._oracle_worker(rows) == float(len(rows))
    q, k, v, la, lam, do = bench._W["x"]
    dq, dk, dv, dla, dlam = backward.backward_dense(q, k, v, la, lam, do)
    rq, rl, _ = backward.backward_query_rows(q, k, v, la, lam, do, rows)
    np.testing.assert_allclose(rq, dq[rows], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(rl, dlam[rows], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
def test_every_workload_has_a_metric_and_a_sample_description(name):
    cfg = synth.WORKLOADS[name]
    assert bench.METRICS[cfg["kind"]]
    assert bench.sample_desc(cfg, 3)


def test_roofline_is_the_slower_of_tensor_and_hbm():
    """The bound of a step is the slower of its flops at the bf16 tensor peak
    and its bytes at the HBM bandwidth: HBM for the 16K-token Mamba-2 forward,
    the tensor cores for the Gated DeltaNet forward."""
    hbm, bf16, _, _ = bench.measured_peaks()
    for name, bound in (("mamba2_bf16_t16k", "hbm"), ("gdn_bf16_t4k", "tensor"), ("mamba2_bwd_bf16_t16k", "hbm")):
        cfg = synth.WORKLOADS[name]
        w = {"abytes": bench.algorithmic_bytes(cfg), "aflops": bench.algorithmic_flops(cfg), "launches": 1}
        r = bench.roofline_of(cfg, name, w, 1.0, None, None)
        assert r["bound"] == bound, name
        if bound == "tensor":
            assert r["peak"] == bf16 and abs(r["achieved"] - w["aflops"] / 1e-3 / 1e12) < 1e-6
        else:
            assert r["peak"] == hbm and abs(r["achieved"] - w["abytes"] / 1e-3 / 1e9) < 1e-6
        assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-12
