"""GPU parity of the forward and decode step with one decay per level
(ll_attn_fwd_level_decay, ll_attn_decode_step_level_decay) against the
float64 oracle of oracle/level_decay.py."""

import numpy as np
import pytest
import torch

from oracle import level_decay as ld
from oracle.partition import levels_needed
from log_linear_attention_chunked_gb300 import synth
from tests._parity import TOL_BF16, TOL_F32, Guarded, rel_err

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS["level_decay_bf16_t16k"]


@pytest.fixture(scope="module")
def B():
    from log_linear_attention_chunked_gb300 import binding
    binding.lib()
    return binding


def _cfg(**kw):
    c = dict(W)
    c.update(kw)
    return c


def _run(B, inp, chunk, Ls=0):
    dev = torch.device("cuda")
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    la, lam = inp["log_alpha"].to(dev), inp["lam"].to(dev)
    Bn, H, T, dk = q.shape
    dv = v.shape[-1]
    shape = B.make_shape(Bn, H, T, dk, dv, lam.shape[-1], chunk, Ls, B._io(q.dtype))
    ws_n = B.ll_attn_fwd_level_decay_workspace_size(shape)
    assert ws_n > 0
    o = Guarded((Bn, H, T, dv), q.dtype)
    ws = Guarded((ws_n,), torch.uint8)
    st = sc = None
    if Ls:
        st = Guarded((Bn, H, Ls, dv, dk), torch.float32)
        sc = Guarded((Bn, H, Ls), torch.float32)
    B.ll_attn_fwd_level_decay(q, k, v, la, lam, chunk, o=o.view, workspace=ws.view,
                              state_out=st.view if st else None, scale_out=sc.view if sc else None)
    assert B.ll_last_device_error() == 0
    for g in (o, ws, st, sc):
        if g is not None:
            assert g.intact(), "write outside the buffer"
    out = o.view.float().cpu().numpy()
    if Ls:
        return out, st.view.cpu().numpy(), sc.view.cpu().numpy()
    return out


def _f64(inp):
    return {n: synth.to_f64(inp[n]) for n in ("q", "k", "v", "log_alpha", "lam")}


CASES = [
    # io, T, d, chunk, la_mode
    ("f32", 64, 16, 16, "softplus"),
    ("f32", 1, 16, 16, "softplus"),
    ("f32", 16, 32, 16, "slow"),
    ("f32", 300, 32, 32, "slow"),     # ragged
    ("f32", 512, 64, 64, "zero"),
    ("bf16", 1024, 64, 64, "softplus"),
    ("bf16", 1000, 64, 128, "slow"),  # chunk 128, ragged
    ("bf16", 2048, 128, 64, "slow"),
]


@pytest.mark.parametrize("io,T,d,chunk,la", CASES)
def test_matches_dense(B, io, T, d, chunk, la):
    cfg = _cfg(io=io, T=T, dk=d, dv=d, chunk=chunk, L=levels_needed(T))
    inp = synth.make_inputs(cfg, B=1, H=2, la_mode=la, tag=f"ld{io}{T}{d}{la}")
    out = _run(B, inp, chunk)
    f = _f64(inp)
    ref = ld.forward_dense_bh(f["q"], f["k"], f["v"], f["log_alpha"], f["lam"])
    assert rel_err(out, ref) <= (TOL_F32 if io == "f32" else TOL_BF16)


@pytest.mark.parametrize("lvl", [1, 5, 7, 9, 11])
def test_onehot_levels_slow_decay(B, lvl):
    """lam one-hot at one level: that level's bucket alone, with decays that
    keep the keys alive over the whole sequence."""
    T = 2048
    cfg = _cfg(io="f32", T=T, dk=32, dv=32, chunk=64, L=levels_needed(T))
    inp = synth.make_inputs(cfg, B=1, H=2, la_mode="slow", lam_mode="onehot", lam_level=lvl, tag=f"ldoh{lvl}")
    out = _run(B, inp, 64)
    f = _f64(inp)
    ref = ld.forward_dense_bh(f["q"], f["k"], f["v"], f["log_alpha"], f["lam"])
    assert rel_err(out, ref) <= TOL_F32


@pytest.mark.parametrize("lvl", [0, 1, 3, 5, 6, 7, 8, 10, 12])
def test_tensor_core_path_onehot_levels(B, lvl):
    """bf16, d = 128, T a multiple of 128: the tensor-core path.  lam one-hot
    at one level isolates that level's factors: levels 0..5 (the diagonal
    32-row groups), 6 and 7 (the groups below them), 8 and up (the Fenwick
    nodes across tiles), under decays that keep every key alive."""
    T = 4096
    cfg = _cfg(io="bf16", T=T, dk=128, dv=128, chunk=64, L=levels_needed(T))
    inp = synth.make_inputs(cfg, B=1, H=2, la_mode="slow", lam_mode="onehot", lam_level=lvl, tag=f"ldtc{lvl}")
    out = _run(B, inp, 64)
    f = _f64(inp)
    ref = ld.forward_dense_bh(f["q"], f["k"], f["v"], f["log_alpha"], f["lam"])
    assert rel_err(out, ref) <= TOL_BF16


@pytest.mark.parametrize("T,la", [(128, "softplus"), (256, "slow"), (1024, "softplus"), (4096, "zero"),
                                  (8192, "slow")])
def test_tensor_core_path_matches_dense(B, T, la):
    cfg = _cfg(io="bf16", T=T, dk=128, dv=128, chunk=64, L=levels_needed(T))
    inp = synth.make_inputs(cfg, B=1, H=2, la_mode=la, tag=f"ldtcd{T}{la}")
    out = _run(B, inp, 64)
    f = _f64(inp)
    if T <= 4096:
        ref = ld.forward_dense_bh(f["q"], f["k"], f["v"], f["log_alpha"], f["lam"])
        assert rel_err(out, ref) <= TOL_BF16
    else:
        rows = np.r_[0, 127, 128, 1000, 4095, 4096, 6000, T - 1]
        for h in range(2):
            ref = ld.forward_rows(f["q"][0, h], f["k"][0, h], f["v"][0, h], f["log_alpha"][0, h], f["lam"][0, h],
                                  rows)
            assert rel_err(out[0, h][rows][None, None], ref[None, None]) <= TOL_BF16, h


def test_tensor_core_and_cuda_core_paths_agree(B):
    """The same bf16 d = 128 call on both paths: T % 128 == 0 takes the
    tensor cores, one token more the CUDA cores (its first T tokens are the
    same inputs, so their outputs must agree)."""
    T = 2048
    cfg = _cfg(io="bf16", T=T + 1, dk=128, dv=128, chunk=64, L=levels_needed(T + 1))
    inp = synth.make_inputs(cfg, B=1, H=2, tag="ldpaths")
    long_out = _run(B, inp, 64)
    short = {n: x[:, :, :T].contiguous() for n, x in inp.items()}
    short_out = _run(B, short, 64)
    assert rel_err(short_out, long_out[:, :, :T]) <= 2 * TOL_BF16


def test_equal_columns_match_the_base_forward(B):
    """Every level with the same decay: the per-level path and ll_attn_fwd
    compute the same function (both checked against the oracle too)."""
    T = 777
    cfg = _cfg(io="f32", T=T, dk=32, dv=32, chunk=32, L=levels_needed(T))
    inp = synth.make_inputs(cfg, B=1, H=2, tag="ldeq")
    la1 = inp["log_alpha"][..., 3].contiguous()
    inp["log_alpha"] = la1[..., None].expand(-1, -1, -1, cfg["L"]).contiguous()
    dev = torch.device("cuda")
    q, k, v, lam = (inp[n].to(dev) for n in ("q", "k", "v", "lam"))
    o_ld = B.ll_attn_fwd_level_decay(q, k, v, inp["log_alpha"].to(dev), lam, 32)
    o_b = B.ll_attn_fwd(q, k, v, la1.to(dev), lam, 32)
    assert rel_err(o_ld.cpu().numpy(), o_b.cpu().numpy()) <= 2 * TOL_F32


@pytest.mark.parametrize("io,T,d,chunk", [("f32", 256, 16, 16), ("f32", 300, 32, 32), ("bf16", 1000, 64, 64),
                                          ("bf16", 1024, 128, 64)])
def test_state_export(B, io, T, d, chunk):
    L = levels_needed(T + 1)
    Ls = T.bit_length()
    cfg = _cfg(io=io, T=T, dk=d, dv=d, chunk=chunk, L=L)
    inp = synth.make_inputs(cfg, B=1, H=2, la_mode="slow", tag=f"ldst{io}{T}")
    out, st, sc = _run(B, inp, chunk, Ls=Ls)
    f = _f64(inp)
    tol = TOL_F32 if io == "f32" else TOL_BF16
    for h in range(2):
        S, ne = ld.states_at(f["k"][0, h], f["v"][0, h], f["log_alpha"][0, h], T, Ls)
        np.testing.assert_array_equal(sc[0, h], ne.astype(np.float32))
        true = st[0, h] * sc[0, h][:, None, None]
        assert rel_err(true[ne][None, None], S[ne][None, None]) <= tol
        assert np.all(st[0, h][~ne] == 0)


@pytest.mark.parametrize("io,d,P,n,chunk", [("f32", 32, 192, 70, 16), ("bf16", 64, 256, 40, 64),
                                            ("f32", 16, 100, 30, 32)])
def test_decode_continues_the_forward(B, io, d, P, n, chunk):
    """A prefix through the forward with state export, then single-token
    steps; every step against the oracle's dense rows of the whole sequence."""
    T = P + n
    Ls = (T + 1).bit_length()
    L = Ls + 1
    cfg = _cfg(io=io, T=T, dk=d, dv=d, chunk=chunk, L=L)
    inp = synth.make_inputs(cfg, B=2, H=2, la_mode="slow", tag=f"lddec{io}{d}{P}")
    dev = torch.device("cuda")
    q, k, v = (inp[x].to(dev) for x in ("q", "k", "v"))
    la, lam = inp["log_alpha"].to(dev), inp["lam"].to(dev)
    st = torch.empty(2, 2, Ls, d, d, device=dev)
    sc = torch.empty(2, 2, Ls, device=dev)
    cut = lambda x: x[:, :, :P].contiguous()  # noqa: E731
    B.ll_attn_fwd_level_decay(cut(q), cut(k), cut(v), cut(la), cut(lam), chunk, state_out=st, scale_out=sc)
    outs = []
    for i in range(n):
        t = torch.full((2,), P + i, dtype=torch.int64, device=dev)
        o = B.ll_attn_decode_step_level_decay(t, q[:, :, P + i].contiguous(), k[:, :, P + i].contiguous(),
                                              v[:, :, P + i].contiguous(), la[:, :, P + i, :Ls + 1].contiguous(),
                                              lam[:, :, P + i, :Ls + 1].contiguous(), st, sc)
        outs.append(o.float())
    assert B.ll_last_device_error() == 0
    out = torch.stack(outs, 2).cpu().numpy()
    f = _f64(inp)
    tol = TOL_F32 if io == "f32" else TOL_BF16
    for b in range(2):
        for h in range(2):
            ref = ld.forward_rows(f["q"][b, h], f["k"][b, h], f["v"][b, h], f["log_alpha"][b, h], f["lam"][b, h],
                                  range(P, T))
            assert rel_err(out[b, h][None, None], ref[None, None]) <= tol, (b, h)
    stn, scn = st.cpu().numpy(), sc.cpu().numpy()
    for b in range(2):
        for h in range(2):
            S, ne = ld.states_at(f["k"][b, h], f["v"][b, h], f["log_alpha"][b, h], T, Ls)
            true = stn[b, h] * scn[b, h][:, None, None]
            assert rel_err(true[ne][None, None], S[ne][None, None]) <= tol


def test_full_size_workload_sampled_rows(B):
    """The benchmark's launch (B=1, H=16, T=16384, d=128, bf16): sampled rows
    of two heads against the oracle's row form."""
    inp = synth.make_inputs(W)
    out = _run(B, inp, W["chunk"])
    f = _f64(inp)
    rng = np.random.default_rng(0)
    rows = np.unique(np.r_[0, 1, 63, 64, 4095, 8191, 16383, rng.integers(0, W["T"], 24)])
    for h in (0, 11):
        ref = ld.forward_rows(f["q"][0, h], f["k"][0, h], f["v"][0, h], f["log_alpha"][0, h], f["lam"][0, h], rows)
        assert rel_err(out[0, h][rows][None, None], ref[None, None]) <= TOL_BF16, h


def test_full_size_slow_decay_sampled_rows(B):
    inp = synth.make_inputs(W, H=2, la_mode="slow", tag="ldslow")
    out = _run(B, inp, W["chunk"])
    f = _f64(inp)
    rows = np.array([5, 700, 4096, 9000, 12345, 16383])
    for h in range(2):
        ref = ld.forward_rows(f["q"][0, h], f["k"][0, h], f["v"][0, h], f["log_alpha"][0, h], f["lam"][0, h], rows)
        assert rel_err(out[0, h][rows][None, None], ref[None, None]) <= TOL_BF16, h


def test_rejects_bad_arguments(B):
    lib = B.lib()
    shape = B.make_shape(1, 1, 64, 16, 16, 7, 16, 0, B.LL_F32)
    assert lib.ll_attn_fwd_level_decay(B.ctypes.byref(shape), *[None] * 9, 0, None) == 1
    bad = B.make_shape(1, 1, 64, 16, 16, 6, 16, 0, B.LL_F32)  # L below the levels T touches
    assert B.ll_attn_fwd_level_decay_workspace_size(bad) == 0
    big = B.make_shape(1, 1, 4097 * 64, 16, 16, 20, 64, 0, B.LL_F32)  # more than 4096 chunks
    assert B.ll_attn_fwd_level_decay_workspace_size(big) == 0


def test_tc_more_heads_than_ctas(B):
    """The tensor-core mode with B=2, H=96 (192 heads) x 2 tiles: the first
    tiles of heads 152..191 run as a CTA's second step, and the per-level
    decay table is indexed by head beyond the grid."""
    cfg = _cfg(io="bf16", T=256, dk=128, dv=128, chunk=64, L=levels_needed(256))
    inp = synth.make_inputs(cfg, B=2, H=96, la_mode="slow", tag="ldheads")
    shape = B.make_shape(2, 96, 256, 128, 128, cfg["L"], 64, 0, B.LL_BF16)
    assert B.ll_attn_fwd_level_decay_launches(shape) == 3, "tensor-core path not selected"
    out = _run(B, inp, 64)
    f = _f64(inp)
    ref = ld.forward_dense_bh(f["q"], f["k"], f["v"], f["log_alpha"], f["lam"])
    assert rel_err(out, ref) <= TOL_BF16
