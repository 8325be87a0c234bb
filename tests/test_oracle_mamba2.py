"""Pins for the log-linear Mamba-2 oracle (oracle/mamba2.py).

Each pin ties the oracle to something other than itself: hand-derived
values, a textbook recurrence it must collapse to, brute-force enumeration,
or a second independent algorithm.
"""

import json
import os

import numpy as np
import pytest

from oracle import mamba2
from oracle.partition import levels_needed

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(T, dk, dv, L, seed, la="softplus"):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, dk)) / np.sqrt(dk)
    k = rng.standard_normal((T, dk)) / np.sqrt(dk)
    v = rng.standard_normal((T, dv))
    if la == "zero":
        log_alpha = np.zeros(T)
    elif la == "slow":
        log_alpha = -0.01 * rng.random(T)
    else:
        log_alpha = -np.log1p(np.exp(rng.standard_normal(T)))
    lam = np.log1p(np.exp(rng.standard_normal((T, L))))
    return q, k, v, log_alpha, lam


def test_golden_worked_forward():
    with open(os.path.join(GOLDEN, "worked_forward.json")) as f:
        g = json.load(f)
    lam = np.tile(10.0 ** np.arange(4), (8, 1))
    one = np.ones((8, 1))
    o = mamba2.forward_dense(one, one, one, np.zeros(8), lam)[:, 0]
    np.testing.assert_allclose(o, g["alpha_one"]["o"], rtol=0, atol=1e-9)
    o = mamba2.forward_dense(one[:4], one[:4], one[:4], np.full(4, -np.log(2.0)), lam[:4])[:, 0]
    np.testing.assert_allclose(o, g["alpha_half"]["o"], rtol=1e-13)
    # the brute-force and recurrent routes give the same hand values
    o = mamba2.forward_buckets(one[:4], one[:4], one[:4], np.full(4, -np.log(2.0)), lam[:4])[:, 0]
    np.testing.assert_allclose(o, g["alpha_half"]["o"], rtol=1e-13)
    o, _ = mamba2.forward_recurrent(one, one, one, np.zeros(8), lam)
    np.testing.assert_allclose(o[:, 0], g["alpha_one"]["o"], rtol=0, atol=1e-9)


def test_bucket_size_closed_form():
    # q=k=v=1, alpha=1, lam^(l) = 10^l: o_t = 1 + sum over set bits b of t of 10^(b+1) 2^b
    T = 40
    lam = np.tile(10.0 ** np.arange(levels_needed(T)), (T, 1))
    one = np.ones((T, 1))
    o = mamba2.forward_dense(one, one, one, np.zeros(T), lam)[:, 0]
    want = [1 + sum(10.0 ** (b + 1) * 2 ** b for b in range(t.bit_length()) if (t >> b) & 1) for t in range(T)]
    np.testing.assert_allclose(o, want, rtol=1e-14)


@pytest.mark.parametrize("la", ["softplus", "zero", "slow"])
@pytest.mark.parametrize("T", [1, 5, 33, 96])
def test_dense_equals_recurrent(T, la):
    L = levels_needed(T)
    q, k, v, log_alpha, lam = _rand(T, 6, 5, L, seed=T, la=la)
    d = mamba2.forward_dense(q, k, v, log_alpha, lam)
    r, _ = mamba2.forward_recurrent(q, k, v, log_alpha, lam)
    np.testing.assert_allclose(r, d, rtol=1e-11, atol=1e-11 * np.abs(d).max())


def test_dense_equals_bucket_bruteforce():
    T = 21
    q, k, v, log_alpha, lam = _rand(T, 3, 4, levels_needed(T), seed=7)
    d = mamba2.forward_dense(q, k, v, log_alpha, lam)
    b = mamba2.forward_buckets(q, k, v, log_alpha, lam)
    np.testing.assert_allclose(b, d, rtol=1e-12, atol=1e-13)


def test_rows_equal_dense():
    T = 130
    q, k, v, log_alpha, lam = _rand(T, 8, 4, levels_needed(T), seed=3)
    d = mamba2.forward_dense(q, k, v, log_alpha, lam)
    rows = [0, 1, 63, 64, 100, 129]
    np.testing.assert_allclose(mamba2.forward_rows(q, k, v, log_alpha, lam, rows), d[rows], rtol=1e-12, atol=1e-14)


def test_constant_lambda_is_mamba2_ssd():
    # all lam equal to c collapses to c * Mamba-2 (study note §3-3, §3-5)
    T = 70
    q, k, v, log_alpha, _ = _rand(T, 5, 3, 1, seed=11)
    lam = np.full((T, levels_needed(T)), 2.5)
    np.testing.assert_allclose(mamba2.forward_dense(q, k, v, log_alpha, lam),
                               2.5 * mamba2.ssd_recurrent(q, k, v, log_alpha), rtol=1e-11, atol=1e-13)


def test_alpha_one_constant_lambda_is_linear_attention():
    # alpha = 1 and lam equal: causal linear attention (study note §1-2)
    T = 50
    q, k, v, _, _ = _rand(T, 4, 4, 1, seed=12)
    lam = np.full((T, levels_needed(T)), 0.75)
    np.testing.assert_allclose(mamba2.forward_dense(q, k, v, np.zeros(T), lam),
                               0.75 * mamba2.linear_attention_recurrent(q, k, v), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("level", [0, 1, 2, 3, 4])
def test_onehot_lambda_selects_one_bucket(level):
    T = 24
    q, k, v, log_alpha, _ = _rand(T, 3, 2, 1, seed=level)
    lam = np.zeros((T, levels_needed(T)))
    lam[:, level] = 1.0
    d = mamba2.forward_dense(q, k, v, log_alpha, lam)
    from oracle.partition import buckets
    cum = np.cumsum(log_alpha)
    for t in range(T):
        want = np.zeros(2)
        for lv, lo, hi in buckets(t):
            if lv == level:
                for s in range(lo, hi):
                    want += np.exp(cum[t] - cum[s]) * (q[t] @ k[s]) * v[s]
        np.testing.assert_allclose(d[t], want, rtol=1e-12, atol=1e-14)


def test_level0_only_is_diagonal():
    T = 16
    q, k, v, log_alpha, _ = _rand(T, 4, 3, 1, seed=5)
    lam = np.zeros((T, levels_needed(T)))
    lam[:, 0] = np.linspace(0.5, 2.0, T)
    d = mamba2.forward_dense(q, k, v, log_alpha, lam)
    want = lam[:, :1] * np.sum(q * k, axis=1, keepdims=True) * v
    np.testing.assert_allclose(d, want, rtol=1e-13)


def test_linear_in_v_and_lambda():
    T = 30
    q, k, v, log_alpha, lam = _rand(T, 4, 3, levels_needed(T), seed=9)
    _, _, v2, _, lam2 = _rand(T, 4, 3, levels_needed(T), seed=10)
    f = lambda vv, ll: mamba2.forward_dense(q, k, vv, log_alpha, ll)
    np.testing.assert_allclose(f(2 * v - 3 * v2, lam), 2 * f(v, lam) - 3 * f(v2, lam), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(f(v, lam + 0.5 * lam2), f(v, lam) + 0.5 * f(v, lam2), rtol=1e-11, atol=1e-12)


def test_causality():
    T = 40
    q, k, v, log_alpha, lam = _rand(T, 4, 3, levels_needed(T), seed=13)
    d = mamba2.forward_dense(q, k, v, log_alpha, lam)
    v2 = v.copy()
    v2[25:] += 1.0
    d2 = mamba2.forward_dense(q, k, v2, log_alpha, lam)
    np.testing.assert_array_equal(d[:25], d2[:25])


def test_states_at_reproduce_outputs():
    # outputs after position P from the exported states equal the dense rows
    T, P = 45, 32
    q, k, v, log_alpha, lam = _rand(T, 4, 3, levels_needed(T), seed=14)
    S, ne = mamba2.states_at(k, v, log_alpha, P, Ls=6)
    assert list(ne) == [False] * 5 + [True]  # P = 32: one bucket of 32 keys at level 6
    states = {i + 1: S[i] for i in range(6) if ne[i]}
    outs = []
    for t in range(P, T):
        outs.append(mamba2.fenwick_step(states, t, q[t], k[t], v[t], log_alpha[t], lam[t]))
    d = mamba2.forward_dense(q, k, v, log_alpha, lam)
    np.testing.assert_allclose(np.array(outs), d[P:], rtol=1e-11, atol=1e-13)
    _, st = mamba2.forward_recurrent(q[:P], k[:P], v[:P], log_alpha[:P], lam[:P])
    np.testing.assert_allclose(st[6], S[5], rtol=1e-12)
