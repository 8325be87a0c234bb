"""GPU parity of the tensor-core forward (bf16, d = 128, T a multiple of 128).

These shapes take the tcgen05 path of ll_attn_fwd (one persistent kernel);
each case is compared element by element with the float64 oracle.
"""

import numpy as np
import pytest
import torch

from oracle import mamba2
from oracle.partition import levels_needed
from log_linear_attention_chunked_gb300 import synth
from tests._parity import TOL_BF16, Guarded, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from log_linear_attention_chunked_gb300 import binding
    binding.lib()
    return binding


def _cfg(T, Bn=1, H=2, L=None, seed=21):
    return dict(kind="mamba2", B=Bn, H=H, T=T, dk=128, dv=128, chunk=64, L=L or levels_needed(T), io="bf16",
                seed=seed, shift=0.0)


def _run(B, inp, Ls=0):
    dev = torch.device("cuda")
    g = {n: inp[n].to(dev) for n in ("q", "k", "v", "log_alpha", "lam")}
    Bn, H, T, d = g["q"].shape
    shape = B.make_shape(Bn, H, T, d, d, g["lam"].shape[-1], 64, Ls, B.LL_BF16)
    assert B.ll_attn_fwd_launches(shape) == (2 if Ls else 1), "tensor-core path not selected"
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


def _oracle(inp):
    f = {n: synth.to_f64(inp[n]) for n in ("q", "k", "v", "log_alpha", "lam")}
    return mamba2.forward_dense_bh(f["q"], f["k"], f["v"], f["log_alpha"], f["lam"])


@pytest.mark.parametrize("la_mode,lam_mode,lvl", [
    ("softplus", "onehot", 0),   # diagonal only: q_t.k_t v_t
    ("zero", "const", 0),        # causal linear attention inside one tile
    ("softplus", "softplus", 0),
])
def test_single_tile(B, la_mode, lam_mode, lvl):
    inp = synth.make_inputs(_cfg(128), la_mode=la_mode, lam_mode=lam_mode, lam_level=lvl, tag="tc1")
    assert rel_err(_run(B, inp), _oracle(inp)) <= TOL_BF16


@pytest.mark.parametrize("T", [256, 384, 512, 1024, 2048])
@pytest.mark.parametrize("la_mode", ["softplus", "zero", "slow"])
def test_tiles_and_levels(B, T, la_mode):
    inp = synth.make_inputs(_cfg(T, Bn=2, H=2), la_mode=la_mode, tag=f"tc{T}")
    assert rel_err(_run(B, inp), _oracle(inp)) <= TOL_BF16


@pytest.mark.parametrize("lvl", [0, 3, 7, 8, 9, 10])
def test_onehot_levels(B, lvl):
    # one level at a time: intra levels 0..7, inter levels 8.. (tile bits)
    inp = synth.make_inputs(_cfg(1024), la_mode="slow", lam_mode="onehot", lam_level=lvl, tag="tcoh")
    ref = _oracle(inp)
    assert np.abs(ref).max() > 0
    assert rel_err(_run(B, inp), ref) <= TOL_BF16, lvl


def test_many_heads_odd_tile_count(B):
    # more tiles than CTAs, a partial last wave, three heads of 13 tiles
    inp = synth.make_inputs(_cfg(13 * 128, Bn=1, H=3), la_mode="slow", tag="tc13")
    assert rel_err(_run(B, inp), _oracle(inp)) <= TOL_BF16


def test_state_export(B):
    T = 1536  # 12 tiles: levels 11 (bit 3) and 12 (bit 2 of the tile count... bits of T)
    Ls = T.bit_length() + 1
    inp = synth.make_inputs(_cfg(T, H=2, L=levels_needed(T)), la_mode="slow", tag="tcexp")
    out, st, sc = _run(B, inp, Ls=Ls)
    f = {n: synth.to_f64(inp[n]) for n in ("k", "v", "log_alpha")}
    for h in range(2):
        S, ne = mamba2.states_at(f["k"][0, h], f["v"][0, h], f["log_alpha"][0, h], T, Ls)
        assert list(sc[0, h] > 0) == list(ne)
        assert rel_err(st[0, h][None, None] * sc[0, h][None, None, :, None, None], S[None, None]) <= TOL_BF16
    assert rel_err(out, _oracle(inp)) <= TOL_BF16


def test_repeated_calls_same_workspace(B):
    # per-call publication tokens: a second call on the same workspace must not
    # see the first call's nodes as already published
    dev = torch.device("cuda")
    cfg = _cfg(1024, H=2)
    a = synth.make_inputs(cfg, tag="tcrep_a")
    b = synth.make_inputs(cfg, tag="tcrep_b")
    shape = B.make_shape(1, 2, 1024, 128, 128, cfg["L"], 64, 0, B.LL_BF16)
    ws = B.alloc_workspace(B.ll_attn_fwd_workspace_size(shape), dev)
    outs = []
    for inp in (a, b, a):
        g = {n: inp[n].to(dev) for n in ("q", "k", "v", "log_alpha", "lam")}
        outs.append(B.ll_attn_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["lam"], 64, workspace=ws).float().cpu())
    assert B.ll_last_device_error() == 0
    assert rel_err(outs[0].numpy(), _oracle(a)) <= TOL_BF16
    assert rel_err(outs[1].numpy(), _oracle(b)) <= TOL_BF16
    assert torch.equal(outs[0], outs[2])  # deterministic


def _sampled_rows(T, per_tile=(0, 45, 77, 127)):
    return np.array([j * 128 + r for j in range(T // 128) for r in per_tile])


def _check_sampled(out, inp, rows):
    f = {n: synth.to_f64(inp[n]) for n in ("q", "k", "v", "log_alpha", "lam")}
    Bn, H = out.shape[:2]
    ref = np.stack([np.stack([mamba2.forward_rows(f["q"][b, h], f["k"][b, h], f["v"][b, h], f["log_alpha"][b, h],
                                                  f["lam"][b, h], rows) for h in range(H)]) for b in range(Bn)])
    return rel_err(out[:, :, rows], ref)


@pytest.mark.parametrize("la_mode", ["softplus", "slow"])
def test_more_tiles_than_ctas(B, la_mode):
    # 16 heads x 32 tiles = 512 tiles: most CTAs run 3-4 pipelined steps
    T = 4096
    inp = synth.make_inputs(_cfg(T, Bn=1, H=16), la_mode=la_mode, tag=f"tcsteps_{la_mode}")
    assert _check_sampled(_run(B, inp), inp, _sampled_rows(T)) <= TOL_BF16


def test_full_size_workload_sampled_rows(B):
    # the 16K-token, 16-head workload the benchmark times, sampled rows of every tile
    cfg = dict(synth.WORKLOADS["mamba2_bf16_t16k"])
    inp = synth.make_inputs(cfg)
    out = _run(B, inp)
    assert np.isfinite(out).all()
    assert _check_sampled(out, inp, _sampled_rows(cfg["T"], per_tile=(0, 127))) <= TOL_BF16


def test_full_size_workload_slow_decay_sampled_rows(B):
    """The benchmark's launch (B=1, H=16, T=16384: 2048 tiles, tile bits 0..6 =
    levels 8..14) with slow decay, so that keys 8K tokens back still count and
    every tile level is checked against non-vanishing values."""
    cfg = dict(synth.WORKLOADS["mamba2_bf16_t16k"])
    inp = synth.make_inputs(cfg, la_mode="slow", tag="tcslow16k")
    out = _run(B, inp)
    assert np.isfinite(out).all()
    assert _check_sampled(out, inp, _sampled_rows(cfg["T"], per_tile=(0, 127))) <= TOL_BF16


@pytest.mark.parametrize("lvl", [11, 12, 13, 14])
def test_onehot_high_tile_levels(B, lvl):
    """One-hot lambda at the tile levels of tile bits 3..6 (levels 11..14) at
    T = 16384 with slow decay: only the bucket of that level reaches the
    output, which is non-zero exactly for queries whose bit lvl-1 is set."""
    T = 16384
    inp = synth.make_inputs(_cfg(T, H=2), la_mode="slow", lam_mode="onehot", lam_level=lvl, tag=f"tcoh{lvl}")
    out = _run(B, inp)
    rows = _sampled_rows(T, per_tile=(0, 127))
    err = _check_sampled(out, inp, rows)
    assert err <= TOL_BF16, (lvl, err)
    # the level is empty for rows with bit lvl-1 clear: their outputs are exactly zero
    empty = [t for t in rows if not (t >> (lvl - 1)) & 1]
    full = [t for t in rows if (t >> (lvl - 1)) & 1]
    assert np.abs(out[:, :, empty]).max() == 0.0
    assert np.abs(out[:, :, full]).max() > 1e-2


def _run_ragged(B, inp, Ls=0):
    """ll_attn_fwd for a bf16 d=128 shape with T % 128 != 0: the whole tiles on
    the tensor cores, the remainder continued from their decode states."""
    dev = torch.device("cuda")
    g = {n: inp[n].to(dev) for n in ("q", "k", "v", "log_alpha", "lam")}
    Bn, H, T, d = g["q"].shape
    shape = B.make_shape(Bn, H, T, d, d, g["lam"].shape[-1], 64, Ls, B.LL_BF16)
    full = B.make_shape(Bn, H, T - T % 128, d, d, g["lam"].shape[-1], 64, 0, B.LL_BF16)
    # more launches than the whole-tile forward alone: the tail runs as a continuation
    assert B.ll_attn_fwd_launches(shape) > B.ll_attn_fwd_launches(full)
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


@pytest.mark.parametrize("T,la_mode", [(1000, "softplus"), (1000, "slow"), (129, "slow"), (2047, "slow")])
def test_ragged_length(B, T, la_mode):
    inp = synth.make_inputs(_cfg(T, Bn=2, H=2), la_mode=la_mode, tag=f"tcrag{T}")
    assert rel_err(_run_ragged(B, inp), _oracle(inp)) <= TOL_BF16


def test_ragged_length_state_export(B):
    T = 1000
    Ls = T.bit_length() + 1
    inp = synth.make_inputs(_cfg(T, H=2), la_mode="slow", tag="tcragexp")
    out, st, sc = _run_ragged(B, inp, Ls=Ls)
    assert rel_err(out, _oracle(inp)) <= TOL_BF16
    f = {n: synth.to_f64(inp[n]) for n in ("k", "v", "log_alpha")}
    for h in range(2):
        S, ne = mamba2.states_at(f["k"][0, h], f["v"][0, h], f["log_alpha"][0, h], T, Ls)
        assert list(sc[0, h] > 0) == list(ne)
        assert rel_err(st[0, h][None, None] * sc[0, h][None, None, :, None, None], S[None, None]) <= TOL_BF16


def test_full_size_ragged_sampled_rows(B):
    """The 16-head long-context shape with 37 tokens fewer: 127 whole tiles per
    head on the tensor cores, then a 91-token tail."""
    cfg = dict(synth.WORKLOADS["mamba2_bf16_t16k"], T=16384 - 37)
    inp = synth.make_inputs(cfg, la_mode="slow", tag="tcrag16k")
    out = _run_ragged(B, inp)
    rows = np.array(sorted(set(list(_sampled_rows(16384 - 128, per_tile=(0, 127))) + list(range(16384 - 128, 16384 - 37)))))
    assert _check_sampled(out, inp, rows) <= TOL_BF16


@pytest.mark.parametrize("lvl", [8, 11])
def test_repeated_calls_two_tiles_per_cta(B, lvl):
    """Back-to-back calls at H = 2, T = 16384 (256 tiles on 152 CTAs: most
    CTAs take two tiles, so the second tile's level decays are the first
    use of one slot of the producer's hand-over in a launch).  Shared memory
    keeps the previous launch's values there; every call must still match
    the oracle, a one-hot lambda at the first tile level (8) or a higher one
    (11) making any wrong level decay visible."""
    T = 16384
    inp = synth.make_inputs(_cfg(T, H=2), la_mode="slow", lam_mode="onehot", lam_level=lvl, tag=f"tcrep{lvl}")
    rows = _sampled_rows(T, per_tile=(0, 77))
    for _ in range(4):
        out = _run(B, inp)
        assert _check_sampled(out, inp, rows) <= TOL_BF16, lvl


def test_more_heads_than_ctas(B):
    """B=2, H=96 (192 heads) x 2 tiles: tiles are dealt as u = j * (B*H) + bh,
    so the first tiles of heads 152..191 (no inter-tile level) run as the
    second step of a CTA, after a tile with levels; slow decay keeps the
    second tiles' level-8 bucket visible."""
    inp = synth.make_inputs(_cfg(256, Bn=2, H=96), la_mode="slow", tag="tcheads")
    assert rel_err(_run(B, inp), _oracle(inp)) <= TOL_BF16
