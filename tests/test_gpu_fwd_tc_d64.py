"""GPU parity of the tensor-core forward at head size 64 (bf16, T a multiple
of 128): the persistent kernel runs its 128-wide tiles with the upper 64
columns zero-filled by the TMA and stores only the first 64 output columns.
Compared element by element with the float64 oracle."""

import numpy as np
import pytest
import torch

from oracle import level_decay as ld
from oracle import mamba2
from oracle.partition import levels_needed
from log_linear_attention_chunked_gb300 import synth
from tests._parity import TOL_BF16, Guarded, rel_err

pytestmark = pytest.mark.gpu

W2K = synth.WORKLOADS["mamba2_bf16_t2k"]  # B=2, H=8, T=2048, d=64


@pytest.fixture(scope="module")
def B():
    from log_linear_attention_chunked_gb300 import binding
    binding.lib()
    return binding


def _cfg(T, Bn=1, H=2, L=None, seed=31, kind="mamba2"):
    return dict(kind=kind, B=Bn, H=H, T=T, dk=64, dv=64, chunk=64, L=L or levels_needed(T), io="bf16",
                seed=seed, shift=0.0)


def _dev(inp):
    dev = torch.device("cuda")
    return {n: inp[n].to(dev) for n in ("q", "k", "v", "log_alpha", "lam")}


def _run(B, inp, Ls=0, expect_launches=None):
    g = _dev(inp)
    Bn, H, T, d = g["q"].shape
    shape = B.make_shape(Bn, H, T, d, d, g["lam"].shape[-1], 64, Ls, B.LL_BF16)
    if expect_launches is not None:
        assert B.ll_attn_fwd_launches(shape) == expect_launches, "tensor-core path not selected"
    o = Guarded((Bn, H, T, d), torch.bfloat16)
    ws = Guarded((B.ll_attn_fwd_workspace_size(shape),), torch.uint8)
    st = sc = None
    if Ls:
        st = Guarded((Bn, H, Ls, d, d), torch.float32)
        sc = Guarded((Bn, H, Ls), torch.float32)
    B.ll_attn_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["lam"], 64, o=o.view, workspace=ws.view,
                  state_out=st.view if st else None, scale_out=sc.view if sc else None)
    assert B.ll_last_device_error() == 0
    for x in (o, ws, st, sc):
        if x is not None:
            assert x.intact(), "write outside the buffer"
    out = o.view.float().cpu().numpy()
    if Ls:
        return out, st.view.cpu().numpy(), sc.view.cpu().numpy()
    return out


def _f64(inp):
    return {n: synth.to_f64(inp[n]) for n in ("q", "k", "v", "log_alpha", "lam")}


def _oracle(inp):
    f = _f64(inp)
    return mamba2.forward_dense_bh(f["q"], f["k"], f["v"], f["log_alpha"], f["lam"])


@pytest.mark.parametrize("T", [128, 256, 1024, 2048])
@pytest.mark.parametrize("la_mode", ["softplus", "zero", "slow"])
def test_tiles_and_levels(B, T, la_mode):
    inp = synth.make_inputs(_cfg(T), la_mode=la_mode, tag=f"d64{T}")
    assert rel_err(_run(B, inp, expect_launches=1), _oracle(inp)) <= TOL_BF16


@pytest.mark.parametrize("lvl", [0, 4, 6, 7, 8, 10, 11])
def test_onehot_levels(B, lvl):
    inp = synth.make_inputs(_cfg(2048), la_mode="slow", lam_mode="onehot", lam_level=lvl, tag="d64oh")
    assert rel_err(_run(B, inp, expect_launches=1), _oracle(inp)) <= TOL_BF16


def test_workload_bf16_t2k(B):
    """The d = 64 workload (B=2, H=8, T=2048) in full, on the tensor cores."""
    inp = synth.make_inputs(W2K)
    assert rel_err(_run(B, inp, expect_launches=1), _oracle(inp)) <= TOL_BF16


def test_state_export(B):
    T, Ls = 1024, 11
    inp = synth.make_inputs(_cfg(T), la_mode="slow", tag="d64st")
    out, st, sc = _run(B, inp, Ls=Ls, expect_launches=2)
    f = _f64(inp)
    assert rel_err(out, _oracle(inp)) <= TOL_BF16
    for h in range(2):
        S, ne = mamba2.states_at(f["k"][0, h], f["v"][0, h], f["log_alpha"][0, h], T, Ls)
        np.testing.assert_array_equal(sc[0, h], ne.astype(np.float32))
        true = st[0, h] * sc[0, h][:, None, None]
        assert rel_err(true[ne][None, None], S[ne][None, None]) <= TOL_BF16


@pytest.mark.parametrize("T", [1000, 2047])
def test_ragged_length(B, T):
    """Whole tiles on the tensor cores, the tail as a continuation."""
    inp = synth.make_inputs(_cfg(T), tag=f"d64r{T}")
    assert rel_err(_run(B, inp), _oracle(inp)) <= TOL_BF16


@pytest.mark.parametrize("t0,T", [(1024, 512), (192, 300)])
def test_continuation(B, t0, T):
    """A segment after a prefix held as decode states (aligned and not)."""
    total = t0 + T
    Ls = total.bit_length()
    cfg = _cfg(total, L=levels_needed(total))
    inp = synth.make_inputs(cfg, la_mode="slow", tag=f"d64c{t0}")
    dev = torch.device("cuda")
    g = _dev(inp)
    st = torch.empty(1, 2, Ls, 64, 64, device=dev)
    sc = torch.empty(1, 2, Ls, device=dev)
    cut = lambda x, a, b: x[:, :, a:b].contiguous()  # noqa: E731
    B.ll_attn_fwd(*(cut(g[n], 0, t0) for n in ("q", "k", "v", "log_alpha", "lam")), 64, state_out=st, scale_out=sc)
    o = B.ll_attn_fwd_cont(t0, st, sc, *(cut(g[n], t0, total) for n in ("q", "k", "v", "log_alpha", "lam")), 64)
    assert B.ll_last_device_error() == 0
    ref = _oracle(inp)[:, :, t0:]
    assert rel_err(o.float().cpu().numpy(), ref) <= TOL_BF16


@pytest.mark.parametrize("T,la", [(1024, "softplus"), (2048, "slow")])
def test_level_decay(B, T, la):
    """The per-level forward's tensor-core mode at head size 64."""
    cfg = _cfg(T, kind="level_decay")
    inp = synth.make_inputs(cfg, la_mode=la, tag=f"d64ld{T}")
    g = _dev(inp)
    shape = B.make_shape(1, 2, T, 64, 64, cfg["L"], 64, 0, B.LL_BF16)
    assert B.ll_attn_fwd_level_decay_launches(shape) == 3, "tensor-core path not selected"
    o = B.ll_attn_fwd_level_decay(g["q"], g["k"], g["v"], g["log_alpha"], g["lam"], 64)
    assert B.ll_last_device_error() == 0
    f = _f64(inp)
    ref = ld.forward_dense_bh(f["q"], f["k"], f["v"], f["log_alpha"], f["lam"])
    assert rel_err(o.float().cpu().numpy(), ref) <= TOL_BF16
