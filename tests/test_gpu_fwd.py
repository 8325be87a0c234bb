"""GPU parity of ll_attn_fwd (log-linear Mamba-2 forward) against the float64 oracle."""

import numpy as np
import pytest
import torch

from oracle import mamba2
from oracle.partition import levels_needed
from log_linear_attention_chunked_gb300 import synth
from tests._parity import TOL_BF16, TOL_F32, Guarded, rel_err

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture(scope="module")
def B():
    from log_linear_attention_chunked_gb300 import binding
    binding.lib()
    return binding


def _cfg(base, **kw):
    c = dict(W[base])
    c.update(kw)
    return c


def _run(B, inp, chunk, guard=False, Ls=0):
    dev = torch.device("cuda")
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    la, lam = inp["log_alpha"].to(dev), inp["lam"].to(dev)
    Bn, H, T, dk = q.shape
    dv = v.shape[-1]
    shape = B.make_shape(Bn, H, T, dk, dv, lam.shape[-1], chunk, Ls, B._io(q.dtype))
    ws_n = B.ll_attn_fwd_workspace_size(shape)
    o = Guarded((Bn, H, T, dv), q.dtype)
    ws = Guarded((ws_n,), torch.uint8)
    st = sc = None
    if Ls:
        st = Guarded((Bn, H, Ls, dv, dk), torch.float32)
        sc = Guarded((Bn, H, Ls), torch.float32)
    B.ll_attn_fwd(q, k, v, la, lam, chunk, o=o.view, workspace=ws.view,
                  state_out=st.view if st else None, scale_out=sc.view if sc else None)
    assert B.ll_last_device_error() == 0
    for g in (o, ws, st, sc):
        if g is not None:
            assert g.intact(), "write outside the buffer"
    out = o.view.float().cpu().numpy()
    if Ls:
        return out, st.view.cpu().numpy(), sc.view.cpu().numpy()
    return out


def _oracle(inp):
    f = {n: synth.to_f64(inp[n]) for n in ("q", "k", "v", "log_alpha", "lam")}
    return mamba2.forward_dense_bh(f["q"], f["k"], f["v"], f["log_alpha"], f["lam"])


def test_workload_fp32_t64(B):
    cfg = W["mamba2_fp32_t64"]
    inp = synth.make_inputs(cfg)
    out = _run(B, inp, cfg["chunk"])
    assert rel_err(out, _oracle(inp)) <= TOL_F32


def test_workload_bf16_t2k(B):
    cfg = W["mamba2_bf16_t2k"]
    inp = synth.make_inputs(cfg)
    out = _run(B, inp, cfg["chunk"])
    assert rel_err(out, _oracle(inp)) <= TOL_BF16


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("la_mode,lam_mode", [("zero", "softplus"), ("slow", "softplus"), ("softplus", "const"),
                                              ("zero", "const"), ("slow", "onehot")])
def test_decay_and_lambda_variants(B, io, la_mode, lam_mode):
    cfg = _cfg("mamba2_fp32_t64", io=io, T=512, dk=32, dv=32, L=levels_needed(512), H=2, chunk=32)
    for lvl in ([0, 3, 6, 9] if lam_mode == "onehot" else [0]):
        inp = synth.make_inputs(cfg, la_mode=la_mode, lam_mode=lam_mode, lam_level=lvl, tag=f"{la_mode}{lam_mode}")
        out = _run(B, inp, cfg["chunk"])
        tol = TOL_F32 if io == "f32" else TOL_BF16
        assert rel_err(out, _oracle(inp)) <= tol, (la_mode, lam_mode, lvl)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_independent_of_chunk(B, io):
    cfg = _cfg("mamba2_fp32_t64", io=io, T=1024, dk=64, dv=64, L=levels_needed(1024), B=1, H=2, la_mode=None)
    inp = synth.make_inputs(cfg, la_mode="slow", tag="chunks")
    ref = _oracle(inp)
    tol = TOL_F32 if io == "f32" else TOL_BF16
    outs = [_run(B, inp, c) for c in (16, 32, 64, 128)]
    for o in outs:
        assert rel_err(o, ref) <= tol


@pytest.mark.parametrize("T,chunk,dk,dv,io", [
    (16, 16, 16, 16, "f32"),     # single chunk (T == C)
    (32, 16, 16, 16, "f32"),     # two chunks
    (48, 16, 32, 16, "f32"),     # dk != dv, N = 3 (ragged Fenwick tail)
    (96, 32, 16, 64, "bf16"),    # dk < dv
    (1, 16, 16, 16, "f32"),      # T = 1: one partial chunk of one row
    (37, 16, 16, 16, "f32"),     # ragged: two full chunks and 5 rows
    (100, 64, 32, 32, "bf16"),   # ragged: one full chunk and 36 rows
    (208, 16, 128, 128, "f32"),  # N = 13 chunks of a wide head
    (384, 128, 64, 64, "bf16"),  # chunk 128
    (300, 128, 128, 128, "bf16"),  # bf16 d = 128 with T not a multiple of 128: CUDA-core path
])
def test_shapes_and_edges(B, T, chunk, dk, dv, io):
    cfg = _cfg("mamba2_fp32_t64", io=io, T=T, dk=dk, dv=dv, L=levels_needed(T), B=2, H=3)
    inp = synth.make_inputs(cfg, tag=f"shape{T}{dk}{dv}")
    out = _run(B, inp, chunk)
    tol = TOL_F32 if io == "f32" else TOL_BF16
    assert rel_err(out, _oracle(inp)) <= tol


@pytest.mark.parametrize("io,T,chunk", [("f32", 208, 16), ("bf16", 512, 64), ("f32", 1024, 64),
                                        ("f32", 77, 16), ("f32", 1000, 64), ("bf16", 383, 128), ("f32", 5, 16)])
def test_state_export(B, io, T, chunk):
    """Decode states of position T (ragged T included: the levels up to
    log2(chunk) then come from the partial last chunk)."""
    cfg = _cfg("mamba2_fp32_t64", io=io, T=T, dk=32, dv=16, L=levels_needed(T), B=1, H=2)
    inp = synth.make_inputs(cfg, tag="export")
    Ls = T.bit_length() + 1
    out, st, sc = _run(B, inp, chunk, Ls=Ls)
    f = {n: synth.to_f64(inp[n]) for n in ("k", "v", "log_alpha")}
    tol = TOL_F32 if io == "f32" else TOL_BF16
    for b in range(1):
        for h in range(2):
            S, ne = mamba2.states_at(f["k"][b, h], f["v"][b, h], f["log_alpha"][b, h], T, Ls)
            assert list(sc[b, h] > 0) == list(ne)
            assert rel_err(st[b, h][None, None] * sc[b, h][None, None, :, None, None], S[None, None]) <= tol
            assert np.all(st[b, h][~ne] == 0)
    assert rel_err(out, _oracle(inp)) <= tol


def test_workload_bf16_t16k_sampled_rows(B):
    """The T=16384, H=16, d=128 workload at full size, checked on sampled rows."""
    cfg = W["mamba2_bf16_t16k"]
    inp = synth.make_inputs(cfg)
    out = _run(B, inp, cfg["chunk"])
    T = cfg["T"]
    rng = np.random.default_rng(0)
    rows = sorted(set([0, 1, 63, 64, 127, 128, 4095, 4096, 8191, 8192, T - 2, T - 1] +
                      list(rng.integers(0, T, 20))))
    f = {n: synth.to_f64(inp[n]) for n in ("q", "k", "v", "log_alpha", "lam")}
    for h in range(cfg["H"]):
        ref = mamba2.forward_rows(f["q"][0, h], f["k"][0, h], f["v"][0, h], f["log_alpha"][0, h], f["lam"][0, h], rows)
        assert rel_err(out[0, h][rows][None, None], ref[None, None]) <= TOL_BF16, h


def test_launch_errors_are_reported(B):
    cfg = _cfg("mamba2_fp32_t64")
    inp = synth.make_inputs(cfg)
    dev = torch.device("cuda")
    q = inp["q"].to(dev)
    with pytest.raises(B.LLError) as e:
        B.ll_attn_fwd(q, q, inp["v"].to(dev), inp["log_alpha"].to(dev), inp["lam"].to(dev)[..., :5].contiguous(), 16)
    assert e.value.status == 1  # too few lambda levels
