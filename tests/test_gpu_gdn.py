"""GPU parity of ll_gdn_fwd (Log-Linear Gated DeltaNet, reading A) against the oracle."""

import numpy as np
import pytest
import torch

from oracle import gdn
from oracle.partition import levels_needed
from log_linear_attention_chunked_gb300 import synth
from tests._parity import TOL_BF16, TOL_F32, Guarded, rel_err

pytestmark = pytest.mark.gpu

# The chunked delta-rule path solves a unit-triangular system per chunk in
# float32; float32 io is held to the float32 tolerance like the other paths.
TOL_GDN_F32 = TOL_F32


@pytest.fixture(scope="module")
def B():
    from log_linear_attention_chunked_gb300 import binding
    binding.lib()
    return binding


def _cfg(T, d=128, Bn=1, H=2, io="bf16", chunk=64, seed=31, dv=None):
    return dict(synth.WORKLOADS["gdn_bf16_t4k"], B=Bn, H=H, T=T, dk=d, dv=dv or d, chunk=chunk, L=levels_needed(T),
                io=io, seed=seed)


def _run(B, inp, chunk):
    dev = torch.device("cuda")
    g = {n: inp[n].to(dev) for n in ("q", "k", "v", "log_alpha", "beta", "lam")}
    Bn, H, T, dk = g["q"].shape
    dv = g["v"].shape[-1]
    shape = B.make_shape(Bn, H, T, dk, dv, g["lam"].shape[-1], chunk, 0, B._io(g["q"].dtype))
    o = Guarded((Bn, H, T, dv), g["q"].dtype)
    ws = Guarded((B.ll_gdn_fwd_workspace_size(shape),), torch.uint8)
    B.ll_gdn_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], g["lam"], chunk, o=o.view, workspace=ws.view)
    assert B.ll_last_device_error() == 0
    assert o.intact() and ws.intact(), "write outside the buffer"
    return o.view.float().cpu().numpy()


def _oracle(inp):
    f = {n: synth.to_f64(inp[n]) for n in ("q", "k", "v", "log_alpha", "beta", "lam")}
    Bn, H = f["q"].shape[:2]
    out = np.zeros(f["v"].shape)
    for b in range(Bn):
        for h in range(H):
            out[b, h] = gdn.gdn_forward_A(f["q"][b, h], f["k"][b, h], f["v"][b, h], f["beta"][b, h],
                                          f["log_alpha"][b, h], f["lam"][b, h])
    return out


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("T,d,chunk", [(16, 16, 16), (64, 16, 16), (256, 32, 32), (512, 64, 64), (384, 128, 64)])
def test_shapes(B, io, T, d, chunk):
    inp = synth.make_inputs(_cfg(T, d=d, io=io), tag=f"g{T}{d}")
    tol = TOL_GDN_F32 if io == "f32" else TOL_BF16
    assert rel_err(_run(B, inp, chunk), _oracle(inp)) <= tol


@pytest.mark.parametrize("T,io", [(2048, "f32"), (4160, "f32"), (8192, "f32"), (8192, "bf16")])
def test_d128_chunk64_heights(B, T, io):
    """d = 128 with 64-token chunks takes the register-tiled scan: up to eight
    heights (T = 8192), and a chunk count that is not a power of two."""
    inp = synth.make_inputs(_cfg(T, io=io), tag=f"gh{T}")
    tol = TOL_GDN_F32 if io == "f32" else TOL_BF16
    assert rel_err(_run(B, inp, 64), _oracle(inp)) <= tol


@pytest.mark.parametrize("la_mode,lam_mode", [("zero", "softplus"), ("slow", "const"), ("slow", "onehot")])
def test_decay_lambda_variants(B, la_mode, lam_mode):
    inp = synth.make_inputs(_cfg(1024, d=64, io="f32"), la_mode=la_mode, lam_mode=lam_mode, lam_level=9,
                            tag="gvar")
    ref = _oracle(inp)
    assert np.abs(ref).max() > 0
    assert rel_err(_run(B, inp, 64), ref) <= TOL_GDN_F32


def test_independent_of_chunk(B):
    inp = synth.make_inputs(_cfg(512, d=32, io="f32"), la_mode="slow", tag="gch")
    ref = _oracle(inp)
    for c in (16, 32, 64, 128):
        assert rel_err(_run(B, inp, c), ref) <= TOL_GDN_F32, c


def test_workload_gdn_t4k_sampled_rows(B):
    """B=2, H=16, T=4096, d=128 at full size; sampled rows of sampled heads."""
    cfg = synth.WORKLOADS["gdn_bf16_t4k"]
    inp = synth.make_inputs(cfg)
    out = _run(B, inp, cfg["chunk"])
    T = cfg["T"]
    rng = np.random.default_rng(1)
    rows = sorted(set([0, 1, 63, 64, 1023, 1024, T - 1] + list(rng.integers(0, T, 9))))
    f = {n: synth.to_f64(inp[n]) for n in ("q", "k", "v", "log_alpha", "beta", "lam")}
    for b, h in [(0, 0), (0, 7), (1, 3), (1, 15)]:
        ref = gdn.gdn_rows_A(f["q"][b, h], f["k"][b, h], f["v"][b, h], f["beta"][b, h], f["log_alpha"][b, h],
                             f["lam"][b, h], rows)
        assert rel_err(out[b, h][rows][None, None], ref[None, None]) <= TOL_BF16, (b, h)


@pytest.mark.parametrize("T,dk,dv,io", [(512, 128, 64, "f32"), (384, 64, 128, "bf16"), (256, 32, 16, "f32")])
def test_key_and_value_dims_differ(B, T, dk, dv, io):
    """dk != dv: the register-tiled scan takes d_k = 128 with any d_v multiple of 16,
    the generic kernels the rest."""
    inp = synth.make_inputs(_cfg(T, d=dk, dv=dv, io=io), tag=f"gdv{T}{dk}{dv}")
    tol = TOL_GDN_F32 if io == "f32" else TOL_BF16
    assert rel_err(_run(B, inp, 64), _oracle(inp)) <= tol


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("la_mode,lam_mode,lvl", [("zero", "softplus", 0), ("slow", "softplus", 0),
                                                  ("slow", "onehot", 9), ("zero", "onehot", 11)])
def test_d128_scan_levels_without_underflow(B, io, la_mode, lam_mode, lvl):
    """The d = 128, 64-token-chunk scan (the workload's kernels) where the
    level states above height 0 carry weight: alpha = 1 or slow decay, so keys
    2048 tokens back still count.  32 chunks give heights 0..4 (levels 7..11);
    the one-hot cases isolate one level (9 = height 2, 11 = height 4) so a
    dropped or misplaced height cannot hide behind the others."""
    T = 2048
    inp = synth.make_inputs(_cfg(T, io=io), la_mode=la_mode, lam_mode=lam_mode, lam_level=lvl,
                            tag=f"g128{la_mode}{lam_mode}")
    ref = _oracle(inp)
    if lam_mode == "onehot":
        # rows whose level-lvl bucket is non-empty carry the whole output
        assert np.abs(ref[:, :, (1 << (lvl - 1)):]).max() > 1e-3
    tol = TOL_GDN_F32 if io == "f32" else TOL_BF16
    assert rel_err(_run(B, inp, 64), ref) <= tol


def test_d128_scan_all_heights_slow_decay_t4096(B):
    """The workload's shape per head (T = 4096, heights 0..5) with slow decay,
    bf16 io: every height of the level scan contributes."""
    inp = synth.make_inputs(_cfg(4096, Bn=1, H=2, io="bf16"), la_mode="slow", tag="g128slow4k")
    assert rel_err(_run(B, inp, 64), _oracle(inp)) <= TOL_BF16
