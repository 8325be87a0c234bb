"""GPU parity of ll_gdn_fwd_b (Log-Linear Gated DeltaNet, reading B) against
the oracle (oracle.gdn.gdn_forward_B)."""

import numpy as np
import pytest
import torch

from oracle import gdn
from oracle.partition import levels_needed
from log_linear_attention_chunked_gb300 import synth
from tests._parity import TOL_BF16, TOL_F32, Guarded, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from log_linear_attention_chunked_gb300 import binding
    binding.lib()
    return binding


def _cfg(T, Bn=1, H=2, io="bf16", chunk=64, seed=37):
    return dict(synth.WORKLOADS["gdn_bf16_t4k"], B=Bn, H=H, T=T, chunk=chunk, L=levels_needed(T), io=io, seed=seed)


def _run(B, inp, chunk):
    dev = torch.device("cuda")
    g = {n: inp[n].to(dev) for n in ("q", "k", "v", "log_alpha", "beta", "lam")}
    Bn, H, T, dk = g["q"].shape
    dv = g["v"].shape[-1]
    shape = B.make_shape(Bn, H, T, dk, dv, g["lam"].shape[-1], chunk, 0, B._io(g["q"].dtype))
    o = Guarded((Bn, H, T, dv), g["q"].dtype)
    ws = Guarded((B.ll_gdn_fwd_b_workspace_size(shape),), torch.uint8)
    B.ll_gdn_fwd_b(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], g["lam"], chunk, o=o.view, workspace=ws.view)
    assert B.ll_last_device_error() == 0
    assert o.intact() and ws.intact(), "write outside the buffer"
    return o.view.float().cpu().numpy()


def _oracle(inp):
    f = {n: synth.to_f64(inp[n]) for n in ("q", "k", "v", "log_alpha", "beta", "lam")}
    Bn, H = f["q"].shape[:2]
    out = np.zeros(f["v"].shape)
    for b in range(Bn):
        for h in range(H):
            out[b, h] = gdn.gdn_forward_B(f["q"][b, h], f["k"][b, h], f["v"][b, h], f["beta"][b, h],
                                          f["log_alpha"][b, h], f["lam"][b, h])
    return out


@pytest.mark.parametrize("T,io,chunk", [(64, "f32", 64), (384, "f32", 64), (384, "bf16", 64), (1024, "bf16", 128),
                                        (2048, "f32", 64), (4160, "f32", 64), (2048, "bf16", 64)])
def test_matches_oracle(B, T, io, chunk):
    inp = synth.make_inputs(_cfg(T, io=io), tag=f"gb{T}{io}")
    tol = TOL_F32 if io == "f32" else TOL_BF16
    assert rel_err(_run(B, inp, chunk), _oracle(inp)) <= tol


@pytest.mark.parametrize("T,la_mode", [(2048, "zero"), (2048, "slow"), (4096, "slow"), (128, "softplus")])
def test_tensor_core_path_long_state(B, T, la_mode):
    """bf16, d = 128, T a multiple of 128: the tensor-core preparation and
    single-state scan.  alpha = 1 and slow decay keep the gated-delta state
    alive over every chunk, so each chunk's pseudo-values depend on all the
    earlier ones."""
    inp = synth.make_inputs(_cfg(T, io="bf16"), la_mode=la_mode, tag=f"gbtc{T}{la_mode}")
    assert rel_err(_run(B, inp, 64), _oracle(inp)) <= TOL_BF16


def test_tensor_core_path_full_size_heads(B):
    """The benchmark's per-head shape (T=4096, d=128, bf16) at its own decay,
    two heads."""
    cfg = dict(synth.WORKLOADS["gdn_b_bf16_t4k"], B=1, H=2)
    inp = synth.make_inputs(cfg)
    assert rel_err(_run(B, inp, cfg["chunk"]), _oracle(inp)) <= TOL_BF16


def test_differs_from_reading_a(B):
    """The two readings are different operators (same inputs, outputs far apart)."""
    inp = synth.make_inputs(_cfg(512, io="f32"), la_mode="zero", tag="gba")
    dev = torch.device("cuda")
    g = {n: inp[n].to(dev) for n in ("q", "k", "v", "log_alpha", "beta", "lam")}
    a = B.ll_gdn_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], g["lam"], 64).cpu().numpy()
    b = _run(B, inp, 64)
    assert rel_err(b, _oracle(inp)) <= TOL_F32
    assert rel_err(a, b) > 1e-3


def test_unsupported_head_dim_is_refused(B):
    shape = B.make_shape(1, 1, 256, 64, 64, levels_needed(256), 64, 0, 1)
    assert B.ll_gdn_fwd_b_workspace_size(shape) == 0
