"""GPU parity of ll_gdn_decode_step (log-linear Gated DeltaNet, reading A,
Fenwick-state decoding) against the oracle's step recurrence
(oracle.gdn.gdn_decode_steps, itself pinned to the dense matrix form)."""

import numpy as np
import pytest
import torch

from oracle import gdn
from log_linear_attention_chunked_gb300 import synth
from tests._parity import TOL_BF16, TOL_F32, rel_err

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS["gdn_decode_b64_t64k"]
NAMES = ("q", "k", "v", "log_alpha", "beta", "lam")


@pytest.fixture(scope="module")
def B():
    from log_linear_attention_chunked_gb300 import binding
    binding.lib()
    return binding


def _cfg(Bn, H, d, Ls, n, io, seed):
    return dict(W, B=Bn, H=H, dk=d, dv=d, Ls=Ls, steps=n, io=io, seed=seed)


def _random_states(Bn, H, Ls, d, t0, seed, dv=None):
    """float32 states, N(0, 0.05^2) on the set bits of t0, zero elsewhere."""
    g = torch.Generator().manual_seed(seed)
    st = torch.randn(Bn, H, Ls, dv or d, d, generator=g) * 0.05
    ne = [((t0 >> i) & 1) == 1 for i in range(Ls)]
    st *= torch.tensor(ne, dtype=torch.float32)[None, None, :, None, None]
    return st, ne


def _run(B, dec, st, t0, n):
    dev = torch.device("cuda")
    g = {x: dec[x].to(dev) for x in NAMES}
    st = st.to(dev)
    Bn = st.shape[0]
    outs = []
    for i in range(n):
        t = torch.full((Bn,), t0 + i, dtype=torch.int64, device=dev)
        # one step's slabs, copied so that each starts 16-byte aligned
        x = {nm: g[nm][i].clone() for nm in NAMES}
        outs.append(B.ll_gdn_decode_step(t, x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["lam"], st).float())
    assert B.ll_last_device_error() == 0
    return torch.stack(outs, 0).cpu().numpy(), st.cpu().numpy()  # [n, B, H, d], states


def _check(dec, S0, ne, t0, out, st, heads, tol):
    for b, h in heads:
        f = {x: synth.to_f64(dec[x][:, b, h]) for x in NAMES}
        ref, S, nef = gdn.gdn_decode_steps(S0[b, h].double().numpy(), ne, t0, f["q"], f["k"], f["v"], f["beta"],
                                           f["log_alpha"], f["lam"])
        assert rel_err(out[:, b, h][None, None], ref[None, None]) <= tol, (b, h)
        assert rel_err(st[b, h][nef][None, None], S[nef][None, None]) <= tol, (b, h)


@pytest.mark.parametrize("io,d,n", [("f32", 16, 70), ("f32", 32, 40), ("bf16", 64, 40), ("f32", 128, 33),
                                    ("bf16", 128, 33)])
def test_from_position_zero(B, io, d, n):
    """Every step from an empty state: each output is a row of the dense form."""
    Bn, H = 2, 3
    Ls = n.bit_length() + 1
    dec = synth.make_decode_inputs(_cfg(Bn, H, d, Ls, n, io, 40 + d))
    S0 = torch.zeros(Bn, H, Ls, d, d)
    out, st = _run(B, dec, S0, 0, n)
    heads = [(b, h) for b in range(Bn) for h in range(H)]
    _check(dec, S0, [False] * Ls, 0, out, st, heads, TOL_F32 if io == "f32" else TOL_BF16)


@pytest.mark.parametrize("io,d,t0", [("f32", 64, 1000), ("f32", 128, 4095), ("bf16", 128, 45677)])
def test_from_random_states(B, io, d, t0):
    """Stored states on the set bits of t0 (4095: twelve of them merge at once)."""
    Bn, H, n = 2, 2, 20
    Ls = (t0 + n).bit_length() + 1
    dec = synth.make_decode_inputs(_cfg(Bn, H, d, Ls, n, io, 50 + t0 % 97))
    S0, ne = _random_states(Bn, H, Ls, d, t0, seed=t0)
    out, st = _run(B, dec, S0, t0, n)
    _check(dec, S0, ne, t0, out, st, [(b, h) for b in range(Bn) for h in range(H)],
           TOL_F32 if io == "f32" else TOL_BF16)


def test_full_batch_sampled(B):
    """The benchmark's launch: 64 x 32 heads, 17 level slots, position 65536
    onward, random states on the set bits (a 65536-token prefix for 2048 heads
    would take the float64 oracle hours); 8 steps, sampled heads."""
    Bn, H, d, Ls, t0, n = W["B"], W["H"], W["dk"], W["Ls"], W["T"], 8
    dec = synth.make_decode_inputs(dict(W), steps=n)
    S0, ne = _random_states(Bn, H, Ls, d, t0, seed=5)
    out, st = _run(B, dec, S0, t0, n)
    _check(dec, S0, ne, t0, out, st, [(0, 0), (13, 7), (31, 16), (63, 31)], TOL_BF16)


def test_rejects_position_beyond_levels(B):
    dev = torch.device("cuda")
    Bn, H, d, Ls = 2, 1, 16, 4
    st = torch.zeros(Bn, H, Ls, d, d, device=dev)
    z = torch.zeros(Bn, H, d, device=dev)
    ones = torch.ones(Bn, H, Ls + 1, device=dev)
    zh = torch.zeros(Bn, H, device=dev)
    t = torch.tensor([3, 15], dtype=torch.int64, device=dev)  # 15 + 1 = 2^4: no slot to carry into
    B.ll_gdn_decode_step(t, z, z, z, zh, zh, ones, st)
    assert B.ll_last_device_error() == 6
    assert B.ll_last_device_error() == 0  # cleared; the context is still usable
    t = torch.tensor([3, 4], dtype=torch.int64, device=dev)
    B.ll_gdn_decode_step(t, z, z, z, zh, zh, ones, st)
    assert B.ll_last_device_error() == 0


@pytest.mark.parametrize("io,dk,dv", [("f32", 64, 128), ("bf16", 128, 32), ("f32", 16, 64)])
def test_key_and_value_dims_differ(B, io, dk, dv):
    Bn, H, n, t0 = 2, 2, 12, 77
    Ls = (t0 + n).bit_length() + 1
    cfg = dict(W, B=Bn, H=H, dk=dk, dv=dv, Ls=Ls, steps=n, io=io, seed=71)
    dec = synth.make_decode_inputs(cfg)
    S0, ne = _random_states(Bn, H, Ls, dk, t0, seed=9, dv=dv)
    out, st = _run(B, dec, S0, t0, n)
    _check(dec, S0, ne, t0, out, st, [(b, h) for b in range(Bn) for h in range(H)],
           TOL_F32 if io == "f32" else TOL_BF16)
