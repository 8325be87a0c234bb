"""A bounded device-side wait that expires ends the kernel cleanly.

Every wait of the tensor-core forward on data another CTA publishes (a
Fenwick node's publication word, the mbarriers of its own pipeline) gives up
after a limit, records LL_ERR_TIMEOUT in the device error word and lets the
kernel drain and finish.  Here a test hook withholds the publication of one
node (a word that nothing will ever write) with a 2 ms limit: the call must
return, ll_last_device_error must report the timeout, and the same process
must then run a normal forward to oracle parity (the context is intact).
No GPU fault, trap or unbounded spin is involved.
"""

import time

import pytest
import torch

from oracle import mamba2
from oracle.partition import levels_needed
from log_linear_attention_chunked_gb300 import synth
from tests._parity import TOL_BF16, rel_err

pytestmark = pytest.mark.gpu

LL_ERR_TIMEOUT = 4


@pytest.fixture(scope="module")
def B():
    from log_linear_attention_chunked_gb300 import binding
    binding.lib()
    return binding


def _inputs(T, H, tag):
    cfg = dict(synth.WORKLOADS["mamba2_bf16_t16k"], B=1, H=H, T=T, L=levels_needed(T))
    return synth.make_inputs(cfg, la_mode="slow", tag=tag)


@pytest.mark.parametrize("T,H,node", [(256, 1, 0), (1024, 2, 9)])
def test_withheld_node_times_out_and_context_survives(B, T, H, node):
    dev = torch.device("cuda")
    inp = _inputs(T, H, "timeout")
    g = {n: inp[n].to(dev) for n in ("q", "k", "v", "log_alpha", "lam")}
    assert B.ll_last_device_error() == 0
    t0 = time.perf_counter()
    st = B.ll_test_fwd_withhold_node(g["q"], g["k"], g["v"], g["log_alpha"], g["lam"], 64, node, 2_000_000)
    assert st == 0
    assert B.ll_last_device_error() == LL_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 30.0  # bounded: the waits gave up
    assert B.ll_last_device_error() == 0    # the error word was read and cleared

    # the context is usable: a normal call on fresh buffers passes parity
    o = B.ll_attn_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["lam"], 64)
    assert B.ll_last_device_error() == 0
    f = {n: synth.to_f64(inp[n]) for n in ("q", "k", "v", "log_alpha", "lam")}
    ref = mamba2.forward_dense_bh(f["q"], f["k"], f["v"], f["log_alpha"], f["lam"])
    assert rel_err(o.float().cpu().numpy(), ref) <= TOL_BF16
