"""GPU parity of ll_attn_bwd (log-linear Mamba-2 backward) against the float64 oracle."""

import numpy as np
import pytest
import torch

from oracle import backward
from oracle.partition import levels_needed
from log_linear_attention_chunked_gb300 import synth
from tests._parity import TOL_BF16, TOL_F32, Guarded, rel_err

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
NAMES = ("dq", "dk", "dv", "dlog_alpha", "dlam")


@pytest.fixture(scope="module")
def B():
    from log_linear_attention_chunked_gb300 import binding
    binding.lib()
    return binding


def _cfg(base, **kw):
    c = dict(W[base])
    c.update(kw)
    return c


def _run(B, inp, chunk):
    dev = torch.device("cuda")
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "dout"))
    la, lam = inp["log_alpha"].to(dev), inp["lam"].to(dev)
    Bn, H, T, dk = q.shape
    dv = v.shape[-1]
    shape = B.make_shape(Bn, H, T, dk, dv, lam.shape[-1], chunk, 0, B._io(q.dtype))
    ws = Guarded((B.ll_attn_bwd_workspace_size(shape),), torch.uint8)
    g = [Guarded(tuple(x.shape), x.dtype) for x in (q, k, v, la, lam)]
    B.ll_attn_bwd(q, k, v, la, lam, do, chunk, grads=tuple(x.view for x in g), workspace=ws.view)
    assert B.ll_last_device_error() == 0
    for x in g + [ws]:
        assert x.intact(), "write outside the buffer"
    return [x.view.float().cpu().numpy() for x in g]


def _lam(inp):
    return synth.to_f64(inp["lam"])


def _oracle(inp):
    f = {n: synth.to_f64(inp[n]) for n in ("q", "k", "v", "log_alpha", "lam", "dout")}
    return backward.backward_dense_bh(f["q"], f["k"], f["v"], f["log_alpha"], f["lam"], f["dout"])


def _assert_close(out, ref, tol, what="", lam=None):
    for name, o, r in zip(NAMES, out, ref):
        if name == "dlog_alpha":
            # dlog_alpha sums the differences dc_t = do_t.o_t - v_t.dv_t; its
            # error is measured against the larger of its own norm and the norm
            # of do_t.o_t = sum_l lam_t[l] dlam_t[l] (for T = 1 the exact value is 0)
            terms = np.abs(np.sum(np.asarray(lam, np.float64) * ref[4], axis=-1))
            den = np.maximum(np.abs(r).max(axis=-1), terms.max(axis=-1))
            e = float((np.abs(o - r).max(axis=-1) / np.maximum(den, 1e-30)).max())
        else:
            e = rel_err(o, r)
        assert e <= tol, (what, name, e)


def test_workload_fp32_t64(B):
    cfg = W["mamba2_fp32_t64"]
    inp = synth.make_inputs(cfg, dout=True)
    _assert_close(_run(B, inp, cfg["chunk"]), _oracle(inp), TOL_F32, lam=_lam(inp))


def test_workload_bf16_t2k(B):
    cfg = W["mamba2_bf16_t2k"]
    inp = synth.make_inputs(cfg, dout=True)
    _assert_close(_run(B, inp, cfg["chunk"]), _oracle(inp), TOL_BF16, lam=_lam(inp))


@pytest.mark.parametrize("T,chunk,dk,dv,io", [
    (16, 16, 16, 16, "f32"),     # single chunk (T == C)
    (32, 16, 16, 16, "f32"),     # two chunks
    (48, 16, 32, 16, "f32"),     # dk != dv, N = 3
    (96, 32, 16, 64, "bf16"),    # dk < dv
    (1, 16, 16, 16, "f32"),      # T = 1
    (37, 16, 16, 16, "f32"),     # ragged: two full chunks and 5 rows
    (100, 64, 32, 32, "bf16"),   # ragged: one full chunk and 36 rows
    (208, 16, 128, 128, "f32"),  # N = 13 chunks of a wide head
    (384, 128, 64, 64, "bf16"),  # chunk 128
    (300, 64, 128, 128, "bf16"),  # d = 128, ragged
    (1000, 32, 64, 32, "f32"),   # many chunks, ragged, every level of the tree
    # d = 128 with 64-token chunks: the register-tiled kernels
    (640, 64, 128, 128, "f32"),   # N = 10
    (200, 64, 128, 128, "f32"),   # ragged: 3 full chunks and 8 rows
    (64, 64, 128, 128, "bf16"),   # one chunk
    (1024, 128, 128, 128, "bf16"),  # chunk 128 runs as 64-token chunks
    (1, 64, 128, 128, "f32"),     # T = 1
    # bf16 with d = 128: the tensor-core kernels (128-token tiles)
    (1, 64, 128, 128, "bf16"),    # T = 1
    (129, 64, 128, 128, "bf16"),  # a second tile of one row
    (2048, 64, 128, 128, "bf16"),  # 16 tiles: levels 8..10 on the query and key sides
])
def test_shapes_and_edges(B, T, chunk, dk, dv, io):
    cfg = _cfg("mamba2_fp32_t64", io=io, T=T, dk=dk, dv=dv, L=levels_needed(T), B=2, H=3)
    inp = synth.make_inputs(cfg, tag=f"bwd{T}{dk}{dv}", dout=True)
    _assert_close(_run(B, inp, chunk), _oracle(inp), TOL_F32 if io == "f32" else TOL_BF16, (T, chunk), _lam(inp))


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("la_mode,lam_mode", [("zero", "softplus"), ("slow", "softplus"), ("softplus", "const"),
                                              ("slow", "onehot")])
def test_decay_and_lambda_variants(B, io, la_mode, lam_mode):
    cfg = _cfg("mamba2_fp32_t64", io=io, T=512, dk=32, dv=32, L=levels_needed(512), H=2, chunk=32)
    for lvl in ([0, 3, 6, 9] if lam_mode == "onehot" else [0]):
        inp = synth.make_inputs(cfg, la_mode=la_mode, lam_mode=lam_mode, lam_level=lvl,
                                tag=f"bwd{la_mode}{lam_mode}", dout=True)
        _assert_close(_run(B, inp, cfg["chunk"]), _oracle(inp), TOL_F32 if io == "f32" else TOL_BF16,
                      (la_mode, lam_mode, lvl), _lam(inp))


@pytest.mark.parametrize("la_mode,lam_mode,levels", [("zero", "softplus", [0]), ("slow", "softplus", [0]),
                                                     ("slow", "onehot", [0, 5, 7, 8, 10])])
def test_tensor_core_variants(B, la_mode, lam_mode, levels):
    """bf16 d = 128 (the tensor-core kernels): alpha = 1, slow decay, and lam
    on one level at a time, inside the diagonal 32-block (0, 5), in the
    off-diagonal blocks of a tile (7) and between tiles (8, 10)."""
    cfg = _cfg("mamba2_fp32_t64", io="bf16", T=1024, dk=128, dv=128, L=levels_needed(1024), B=1, H=2, chunk=64)
    for lvl in levels:
        inp = synth.make_inputs(cfg, la_mode=la_mode, lam_mode=lam_mode, lam_level=lvl,
                                tag=f"bwdtc{la_mode}{lam_mode}", dout=True)
        _assert_close(_run(B, inp, cfg["chunk"]), _oracle(inp), TOL_BF16, (la_mode, lam_mode, lvl), _lam(inp))


@pytest.mark.parametrize("T", [2650, 2816])
def test_tensor_core_many_items(B, T):
    """bf16 d = 128 with more (tile, head) items than two per SM: the query
    kernel then claims items from its counter and the intra kernel starts the
    CTAs with one item fewer later.  2650 tokens: 21 tiles, the last ragged
    (an odd count: the key-side nodes are cleared whole); 2816: 22 tiles (the
    odd nodes cleared by the pitched memset, the even ones stored); 16 heads."""
    cfg = _cfg("mamba2_fp32_t64", io="bf16", T=T, dk=128, dv=128, L=levels_needed(T), B=1, H=16, chunk=64)
    inp = synth.make_inputs(cfg, tag=f"bwdtcmany{T}", dout=True)
    _assert_close(_run(B, inp, cfg["chunk"]), _oracle(inp), TOL_BF16, ("many items", T), _lam(inp))


def test_tensor_core_more_heads_than_sms(B):
    """bf16 d = 128 with 160 heads of 300 tokens (three tiles, the last
    ragged): more heads than SMs, so a persistent CTA meets the ragged tile
    (staged by its threads) as a later item too, after and before TMA-loaded
    ones, and the query kernel claims items from its counter."""
    cfg = _cfg("mamba2_fp32_t64", io="bf16", T=300, dk=128, dv=128, L=levels_needed(300), B=1, H=160, chunk=64)
    inp = synth.make_inputs(cfg, tag="bwdtc160", dout=True)
    _assert_close(_run(B, inp, cfg["chunk"]), _oracle(inp), TOL_BF16, ("160 heads",), _lam(inp))


def test_extra_levels_are_zero(B):
    # lam with more levels than T reaches: their gradient is exactly 0
    cfg = _cfg("mamba2_fp32_t64", T=200, L=levels_needed(200) + 3, B=1, H=2)
    inp = synth.make_inputs(cfg, tag="bwdextra", dout=True)
    out = _run(B, inp, 16)
    assert np.all(out[4][..., levels_needed(200):] == 0.0)
    _assert_close(out, _oracle(inp), TOL_F32, lam=_lam(inp))


def test_tensor_core_many_levels_are_zero(B):
    """bf16 d = 128 with L = 40 levels: lam rows too long for the query
    kernel's shared-memory copy (read from global instead) and a second
    block of levels in the key kernel's lam . dlam; the levels past those T
    reaches have gradient exactly 0."""
    T = 1024
    cfg = _cfg("mamba2_fp32_t64", io="bf16", T=T, dk=128, dv=128, L=40, B=1, H=2, chunk=64)
    inp = synth.make_inputs(cfg, tag="bwdtcL40", dout=True)
    out = _run(B, inp, cfg["chunk"])
    assert np.all(out[4][..., levels_needed(T):] == 0.0)
    _assert_close(out, _oracle(inp), TOL_BF16, ("L = 40",), _lam(inp))


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_independent_of_chunk(B, io):
    cfg = _cfg("mamba2_fp32_t64", io=io, T=1024, dk=64, dv=64, L=levels_needed(1024), B=1, H=2)
    inp = synth.make_inputs(cfg, la_mode="slow", tag="bwdchunks", dout=True)
    ref = _oracle(inp)
    for c in (16, 32, 64, 128):
        _assert_close(_run(B, inp, c), ref, TOL_F32 if io == "f32" else TOL_BF16, c, _lam(inp))


def test_workload_bf16_t16k_sampled_rows(B):
    """The T=16384, H=16, d=128 backward at full size (the launch the
    benchmark times), checked on sampled rows: dq and dlam of query rows,
    dk and dv of key rows, and dlog_alpha through its differences
    dlog_alpha[t] - dlog_alpha[t+1] = dc_t."""
    cfg = W["mamba2_bwd_bf16_t16k"]
    inp = synth.make_inputs(cfg)
    dq, dk, dv, dla, dlam = _run(B, inp, cfg["chunk"])
    T = cfg["T"]
    rng = np.random.default_rng(1)
    rows = sorted(set([0, 1, 63, 64, 127, 128, 4095, 4096, 8191, 8192, T - 2, T - 1] +
                      list(rng.integers(0, T, 12))))
    f = {n: synth.to_f64(inp[n]) for n in ("q", "k", "v", "log_alpha", "lam", "dout")}
    for h in range(0, cfg["H"], 3):
        args = (f["q"][0, h], f["k"][0, h], f["v"][0, h], f["log_alpha"][0, h], f["lam"][0, h], f["dout"][0, h])
        rq, rl, row_term = backward.backward_query_rows(*args, rows)
        ck, cv, col_term = backward.backward_key_rows(*args, rows)
        for name, got, ref in (("dq", dq[0, h][rows], rq), ("dlam", dlam[0, h][rows], rl),
                               ("dk", dk[0, h][rows], ck), ("dv", dv[0, h][rows], cv)):
            assert rel_err(got[None, None], ref[None, None]) <= TOL_BF16, (h, name)
        nxt = np.append(dla[0, h], 0.0)
        diff = np.array([nxt[t] - nxt[t + 1] for t in rows], np.float64)
        dc = row_term - col_term
        assert np.abs(diff - dc).max() <= TOL_BF16 * np.abs(dla[0, h]).max(), h


def test_dlog_alpha_first_is_zero(B):
    # no decay acts before the first token: dlog_alpha[0] = 0 up to rounding
    cfg = _cfg("mamba2_bf16_t2k", B=1, H=4)
    inp = synth.make_inputs(cfg, tag="bwdfirst", dout=True)
    dla = _run(B, inp, 64)[3]
    for h in range(4):
        assert abs(dla[0, h, 0]) <= 1e-4 * np.abs(dla[0, h]).max()
