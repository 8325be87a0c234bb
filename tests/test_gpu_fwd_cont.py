"""GPU parity of ll_attn_fwd_cont (prefill continuation) against the oracle:
the outputs of the new tokens are rows of the dense definition over the whole
sequence, and the exported states are the oracle's level states of t0 + T."""

import numpy as np
import pytest
import torch

from oracle import mamba2
from oracle.partition import levels_needed
from log_linear_attention_chunked_gb300 import synth
from tests._parity import TOL_BF16, TOL_F32, Guarded, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from log_linear_attention_chunked_gb300 import binding
    binding.lib()
    return binding


def _inputs(io, d, T, t0, seed_tag, Bn=1, H=2, la_mode="softplus"):
    t1 = t0 + T
    Ls = max(t1.bit_length(), 1)
    cfg = dict(kind="mamba2", B=Bn, H=H, T=t1, dk=d, dv=d, chunk=16, L=levels_needed(t1), io=io, seed=61,
               shift=2.0 if la_mode == "softplus" else 0.0)
    return synth.make_inputs(cfg, tag=seed_tag, la_mode=la_mode), Ls


def _prefix_states(f, t0, Ls):
    Bn, H = f["q"].shape[:2]
    d = f["v"].shape[-1]
    S = np.zeros((Bn, H, Ls, d, f["k"].shape[-1]))
    for b in range(Bn):
        for h in range(H):
            S[b, h], _ = mamba2.states_at(f["k"][b, h], f["v"][b, h], f["log_alpha"][b, h], t0, Ls)
    return S


def _cont(B, inp, t0, T, Ls, chunk, S0, sc0):
    dev = torch.device("cuda")
    g = {n: inp[n][:, :, t0:].contiguous().to(dev) for n in ("q", "k", "v", "log_alpha", "lam")}
    Bn, H = g["q"].shape[:2]
    d = g["v"].shape[-1]
    st_in = torch.tensor(S0, dtype=torch.float32, device=dev)
    sc_in = torch.tensor(sc0, dtype=torch.float32, device=dev)
    st_out = Guarded((Bn, H, Ls, d, d), torch.float32)
    sc_out = Guarded((Bn, H, Ls), torch.float32)
    o = Guarded((Bn, H, T, d), g["q"].dtype)
    shape = B.make_shape(Bn, H, T, d, d, g["lam"].shape[-1], chunk, Ls, B._io(g["q"].dtype))
    ws = Guarded((B.ll_attn_fwd_cont_workspace_size(shape, t0),), torch.uint8)
    B.ll_attn_fwd_cont(t0, st_in, sc_in, g["q"], g["k"], g["v"], g["log_alpha"], g["lam"], chunk, o=o.view,
                       state_out=st_out.view, scale_out=sc_out.view, workspace=ws.view)
    assert B.ll_last_device_error() == 0
    assert o.intact() and st_out.intact() and sc_out.intact() and ws.intact(), "write outside a buffer"
    return (o.view.float().cpu().numpy(), st_out.view.cpu().numpy(), sc_out.view.cpu().numpy())


@pytest.mark.parametrize("io,d,T,t0,chunk", [
    ("f32", 16, 64, 320, 16),      # T = P: the segment closes its block and carries
    ("f32", 32, 192, 512, 32),     # T < P
    ("f32", 32, 256, 768, 32),     # T = P, the prefix bucket of 512 keeps its level
    ("f32", 64, 128, 1024, 64),
    ("f32", 32, 128, 0, 32),       # no prefix
    ("bf16", 64, 256, 1792, 64),   # three prefix buckets
    ("f32", 32, 100, 128, 32),       # ragged segment: a partial last chunk (P = 128 > T)
    ("bf16", 64, 37, 192, 16),       # ragged, P = 64
    ("bf16", 128, 512, 1536, 128),   # from here on the tensor-core path (bf16, d = 128)
    ("bf16", 128, 128, 128, 64),     # prefix bucket at the first tile level
    ("bf16", 128, 256, 768, 64),     # two prefix buckets, the segment closes its block
    ("bf16", 128, 384, 3584, 64),    # T < P, three prefix buckets
    ("bf16", 128, 1024, 3072, 128),  # eight tiles per head
])
def test_matches_dense_rows(B, io, d, T, t0, chunk):
    inp, Ls = _inputs(io, d, T, t0, f"c{io}{d}{T}{t0}")
    f = {n: synth.to_f64(inp[n]) for n in ("q", "k", "v", "log_alpha", "lam")}
    S0 = _prefix_states(f, t0, Ls)
    sc0 = np.array([[[1.0 if (t0 >> i) & 1 else 0.0 for i in range(Ls)]] * S0.shape[1]] * S0.shape[0])
    out, st, sc = _cont(B, inp, t0, T, Ls, chunk, S0, sc0)
    tol = TOL_F32 if io == "f32" else TOL_BF16
    full = mamba2.forward_dense_bh(f["q"], f["k"], f["v"], f["log_alpha"], f["lam"])
    assert rel_err(out, full[:, :, t0:]) <= tol
    t1 = t0 + T
    want = _prefix_states(f, t1, Ls)
    ne = [(t1 >> i) & 1 == 1 for i in range(Ls)]
    assert list(sc[0, 0] != 0) == ne
    true = st * sc[..., None, None]
    assert rel_err(true[:, :, ne], want[:, :, ne]) <= tol


def test_chained_segments_from_the_forward_export(B):
    """Prefix of 1024 tokens by ll_attn_fwd with state export, then two
    256-token continuations, each from the previous one's states; float32."""
    dev = torch.device("cuda")
    d, t0, T = 32, 1024, 256
    inp, Ls = _inputs("f32", d, 2 * T, t0, "chain", la_mode="slow")
    g = {n: inp[n].to(dev) for n in ("q", "k", "v", "log_alpha", "lam")}
    Bn, H = g["q"].shape[:2]
    st = torch.empty(Bn, H, Ls, d, d, device=dev)
    sc = torch.empty(Bn, H, Ls, device=dev)
    cut = lambda x, a, b: x[:, :, a:b].contiguous()
    B.ll_attn_fwd(*(cut(g[n], 0, t0) for n in ("q", "k", "v", "log_alpha", "lam")), 32, state_out=st, scale_out=sc)
    outs = []
    for seg in range(2):
        a = t0 + seg * T
        st2, sc2 = torch.empty_like(st), torch.empty_like(sc)
        outs.append(B.ll_attn_fwd_cont(a, st, sc, *(cut(g[n], a, a + T) for n in ("q", "k", "v", "log_alpha", "lam")),
                                       32, state_out=st2, scale_out=sc2).cpu().numpy())
        st, sc = st2, sc2
    assert B.ll_last_device_error() == 0
    f = {n: synth.to_f64(inp[n]) for n in ("q", "k", "v", "log_alpha", "lam")}
    full = mamba2.forward_dense_bh(f["q"], f["k"], f["v"], f["log_alpha"], f["lam"])
    assert rel_err(np.concatenate(outs, 2), full[:, :, t0:]) <= TOL_F32


def test_pieces_of_an_unaligned_start():
    # the host-side split of a segment into aligned single-block pieces
    from log_linear_attention_chunked_gb300 import binding
    binding.lib()
    shape = binding.make_shape(1, 1, 256, 32, 32, 12, 32, 11, 0)
    assert binding.ll_attn_fwd_cont_workspace_size(shape, 768) > 0
    assert binding.ll_attn_fwd_cont_workspace_size(shape, 640) > 0   # 640 = 5 x 128: pieces 128 then 128


@pytest.mark.parametrize("io,d,T,t0,chunk", [
    ("f32", 32, 256, 640, 32),       # 640 is not a multiple of 256: pieces 128 + 128
    ("f32", 16, 100, 37, 16),        # an odd start: pieces 1, 2, 8, 16, ... and a ragged remainder
    ("bf16", 64, 300, 192, 64),      # pieces 64, 128 (ragged remainder 108)
    ("bf16", 128, 1024, 384, 64),    # tensor-core pieces 128, 512, then 384 at 1024
    ("bf16", 128, 1000, 3200, 128),  # tensor-core pieces and a ragged remainder on the CUDA cores
])
def test_unaligned_start_matches_dense_rows(B, io, d, T, t0, chunk):
    """A continuation whose start is not a multiple of the smallest power of
    two >= T runs as aligned pieces chained through their decode states; the
    outputs and the states of t0 + T must still match the dense definition."""
    inp, Ls = _inputs(io, d, T, t0, f"u{io}{d}{T}{t0}", la_mode="slow")
    f = {n: synth.to_f64(inp[n]) for n in ("q", "k", "v", "log_alpha", "lam")}
    S0 = _prefix_states(f, t0, Ls)
    sc0 = np.array([[[1.0 if (t0 >> i) & 1 else 0.0 for i in range(Ls)]] * S0.shape[1]] * S0.shape[0])
    out, st, sc = _cont(B, inp, t0, T, Ls, chunk, S0, sc0)
    tol = TOL_F32 if io == "f32" else TOL_BF16
    full = mamba2.forward_dense_bh(f["q"], f["k"], f["v"], f["log_alpha"], f["lam"])
    assert rel_err(out, full[:, :, t0:]) <= tol
    t1 = t0 + T
    want = _prefix_states(f, t1, Ls)
    ne = [(t1 >> i) & 1 == 1 for i in range(Ls)]
    assert list(sc[0, 0] != 0) == ne
    true = st * sc[..., None, None]
    assert rel_err(true[:, :, ne], want[:, :, ne]) <= tol


def test_chained_segments_tensor_cores(B):
    """bf16, d = 128: a 1024-token prefix by ll_attn_fwd (tensor cores, with
    state export), then two 512-token continuations on the tensor-core path."""
    dev = torch.device("cuda")
    d, t0, T = 128, 1024, 512
    inp, Ls = _inputs("bf16", d, 2 * T, t0, "chaintc")
    g = {n: inp[n].to(dev) for n in ("q", "k", "v", "log_alpha", "lam")}
    Bn, H = g["q"].shape[:2]
    st = torch.empty(Bn, H, Ls, d, d, device=dev)
    sc = torch.empty(Bn, H, Ls, device=dev)
    cut = lambda x, a, b: x[:, :, a:b].contiguous()
    B.ll_attn_fwd(*(cut(g[n], 0, t0) for n in ("q", "k", "v", "log_alpha", "lam")), 64, state_out=st, scale_out=sc)
    outs = []
    for seg in range(2):
        a = t0 + seg * T
        st2, sc2 = torch.empty_like(st), torch.empty_like(sc)
        outs.append(B.ll_attn_fwd_cont(a, st, sc, *(cut(g[n], a, a + T) for n in ("q", "k", "v", "log_alpha", "lam")),
                                       64, state_out=st2, scale_out=sc2).float().cpu().numpy())
        st, sc = st2, sc2
    assert B.ll_last_device_error() == 0
    f = {n: synth.to_f64(inp[n]) for n in ("q", "k", "v", "log_alpha", "lam")}
    full = mamba2.forward_dense_bh(f["q"], f["k"], f["v"], f["log_alpha"], f["lam"])
    assert rel_err(np.concatenate(outs, 2), full[:, :, t0:]) <= TOL_BF16
    want = _prefix_states(f, t0 + 2 * T, Ls)
    ne = [((t0 + 2 * T) >> i) & 1 == 1 for i in range(Ls)]
    true = (st * sc[..., None, None]).cpu().numpy()
    assert rel_err(true[:, :, ne], want[:, :, ne]) <= TOL_BF16
