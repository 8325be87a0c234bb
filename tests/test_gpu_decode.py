"""GPU parity of ll_attn_decode_step (Fenwick-state decoding) against the oracle.

A prefix is run through ll_attn_fwd with state export, then single-token
steps continue from it; every step's output is compared with the dense
definition's row for that position, and the final states with the bucket
sums of the oracle.
"""

import numpy as np
import pytest
import torch

from oracle import mamba2
from oracle.partition import levels_needed
from log_linear_attention_chunked_gb300 import synth
from tests._parity import TOL_BF16, TOL_F32, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from log_linear_attention_chunked_gb300 import binding
    binding.lib()
    return binding


def _sequence(io, Bn, H, d, P, n, seed_tag):
    T = P + n
    Ls = (T + 1).bit_length()
    cfg = dict(kind="mamba2", B=Bn, H=H, T=T, dk=d, dv=d, chunk=16, L=Ls + 1, io=io, seed=11, shift=0.0)
    return synth.make_inputs(cfg, tag=seed_tag), Ls


def _prefix_and_steps(B, inp, P, n, Ls, chunk, sample=None):
    dev = torch.device("cuda")
    q, k, v = (inp[x].to(dev) for x in ("q", "k", "v"))
    la, lam = inp["log_alpha"].to(dev), inp["lam"].to(dev)
    Bn, H, T, d = q.shape
    st = torch.empty(Bn, H, Ls, d, d, device=dev)
    sc = torch.empty(Bn, H, Ls, device=dev)
    B.ll_attn_fwd(q[:, :, :P].contiguous(), k[:, :, :P].contiguous(), v[:, :, :P].contiguous(),
                  la[:, :, :P].contiguous(), lam[:, :, :P].contiguous(), chunk, state_out=st, scale_out=sc)
    outs = []
    for i in range(n):
        t = torch.full((Bn,), P + i, dtype=torch.int64, device=dev)
        o = B.ll_attn_decode_step(t, q[:, :, P + i].contiguous(), k[:, :, P + i].contiguous(),
                                  v[:, :, P + i].contiguous(), la[:, :, P + i].contiguous(),
                                  lam[:, :, P + i].contiguous(), st, sc)
        outs.append(o.float())
    assert B.ll_last_device_error() == 0
    return torch.stack(outs, 2).cpu().numpy(), st.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("io,d,P,n,chunk", [("f32", 32, 192, 70, 16), ("bf16", 64, 256, 64, 64),
                                            ("f32", 16, 16, 50, 16), ("bf16", 128, 512, 40, 128)])
def test_decode_matches_dense_rows(B, io, d, P, n, chunk):
    inp, Ls = _sequence(io, 2, 3, d, P, n, f"dec{io}{d}")
    out, st, sc = _prefix_and_steps(B, inp, P, n, Ls, chunk)
    f = {x: synth.to_f64(inp[x]) for x in ("q", "k", "v", "log_alpha", "lam")}
    tol = TOL_F32 if io == "f32" else TOL_BF16
    for b in range(2):
        for h in range(3):
            ref = mamba2.forward_rows(f["q"][b, h], f["k"][b, h], f["v"][b, h], f["log_alpha"][b, h],
                                      f["lam"][b, h], range(P, P + n))
            assert rel_err(out[b, h][None, None], ref[None, None]) <= tol, (b, h)
            S, ne = mamba2.states_at(f["k"][b, h], f["v"][b, h], f["log_alpha"][b, h], P + n, Ls)
            true = st[b, h] * sc[b, h][:, None, None]
            assert rel_err(true[ne][None, None], S[ne][None, None]) <= tol


def test_decode_rejects_position_beyond_levels(B):
    dev = torch.device("cuda")
    Bn, H, d, Ls = 2, 2, 16, 4
    z = torch.zeros(Bn, H, d, device=dev)
    st = torch.zeros(Bn, H, Ls, d, d, device=dev)
    sc = torch.zeros(Bn, H, Ls, device=dev)
    t = torch.tensor([3, 15], dtype=torch.int64, device=dev)  # 15 + 1 = 2^4: no slot to carry into
    B.ll_attn_decode_step(t, z, z, z, torch.zeros(Bn, H, device=dev), torch.ones(Bn, H, Ls + 1, device=dev), st, sc)
    assert B.ll_last_device_error() == 6
    assert B.ll_last_device_error() == 0  # cleared; the context is still usable
    t = torch.tensor([3, 4], dtype=torch.int64, device=dev)
    B.ll_attn_decode_step(t, z, z, z, torch.zeros(Bn, H, device=dev), torch.ones(Bn, H, Ls + 1, device=dev), st, sc)
    assert B.ll_last_device_error() == 0


def test_decode_long_prefix_sampled(B):
    """Prefix of 65536 tokens then 256 steps (B and H reduced so the float64
    oracle stays quick); sampled heads are checked row by row."""
    P, n, d = 65536, 256, 128
    Bn, H = 2, 2
    Ls = 17
    cfg = dict(W_DECODE)
    cfg.update(B=Bn, H=H)
    inp = synth.make_inputs(dict(cfg, T=P + n, L=Ls + 1))
    out, st, sc = _prefix_and_steps(B, inp, P, n, Ls, 64)
    f = {x: synth.to_f64(inp[x]) for x in ("q", "k", "v", "log_alpha", "lam")}
    for b in range(Bn):
        for h in range(H):
            ref = mamba2.forward_rows(f["q"][b, h], f["k"][b, h], f["v"][b, h], f["log_alpha"][b, h],
                                      f["lam"][b, h], range(P, P + n))
            assert rel_err(out[b, h][None, None], ref[None, None]) <= TOL_BF16


W_DECODE = synth.WORKLOADS["decode_b64_t64k"]


def test_decode_full_batch_sampled(B):
    """The benchmark's decode launch: 64 x 32 heads, 17 level slots, position
    65536 onward.  The states of the non-empty levels are drawn at random (a
    65536-token prefix for all 2048 heads would take the float64 oracle
    hours); 8 steps run on the GPU and sampled heads are checked against the
    oracle's step recurrence started from the same states."""
    from oracle import decode
    dev = torch.device("cuda")
    cfg = dict(W_DECODE)
    Bn, H, d, Ls, t0, n = cfg["B"], cfg["H"], cfg["dk"], cfg["Ls"], cfg["T"], 8
    ne = [((t0 >> i) & 1) == 1 for i in range(Ls)]
    gen = torch.Generator(device=dev)
    gen.manual_seed(5)
    st = torch.randn(Bn, H, Ls, d, d, device=dev, generator=gen) * 0.05
    keep = torch.tensor(ne, device=dev)
    st *= keep[None, None, :, None, None].float()
    sc = keep.float().expand(Bn, H, Ls).contiguous()
    pairs = [(0, 0), (13, 7), (31, 16), (63, 31)]
    S0 = {pr: st[pr[0], pr[1]].double().cpu().numpy() for pr in pairs}
    dec = synth.make_decode_inputs(cfg, device="cpu", steps=n)
    g = {x: dec[x].to(dev) for x in ("q", "k", "v", "log_alpha", "lam")}
    outs = []
    for i in range(n):
        t = torch.full((Bn,), t0 + i, dtype=torch.int64, device=dev)
        outs.append(B.ll_attn_decode_step(t, g["q"][i], g["k"][i], g["v"][i], g["log_alpha"][i], g["lam"][i],
                                          st, sc).float())
    assert B.ll_last_device_error() == 0
    out = torch.stack(outs, 0).cpu().numpy()  # [n, B, H, d]
    for b, h in pairs:
        f = {x: synth.to_f64(dec[x][:, b, h]) for x in ("q", "k", "v", "log_alpha", "lam")}
        ref, S, nef = decode.decode_steps(S0[(b, h)], ne, t0, f["q"], f["k"], f["v"], f["log_alpha"], f["lam"])
        assert rel_err(out[:, b, h][None, None], ref[None, None]) <= TOL_BF16, (b, h)
        true = (st[b, h] * sc[b, h][:, None, None]).double().cpu().numpy()
        assert rel_err(true[nef][None, None], S[nef][None, None]) <= TOL_BF16, (b, h)
