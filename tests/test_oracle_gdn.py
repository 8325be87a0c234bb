"""Pins for the log-linear Gated DeltaNet oracle (oracle/gdn.py)."""

import json
import os

import numpy as np
import pytest

from oracle import gdn, mamba2
from oracle.partition import levels_needed

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(T, d, L, seed, la="softplus"):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, d)) / np.sqrt(d)
    k = rng.standard_normal((T, d))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, d))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(T)))
    if la == "zero":
        log_alpha = np.zeros(T)
    else:
        log_alpha = -np.log1p(np.exp(rng.standard_normal(T) + 2.0))
    lam = np.log1p(np.exp(rng.standard_normal((T, L))))
    return q, k, v, beta, log_alpha, lam


def test_golden_two_tokens():
    with open(os.path.join(GOLDEN, "worked_gdn.json")) as f:
        g = json.load(f)
    one = np.ones((2, 1))
    v = np.array([[1.0], [2.0]])
    beta = np.array([0.5, 0.5])
    la = np.zeros(2)
    lam = np.array([[1.0, 10.0], [1.0, 10.0]])
    np.testing.assert_allclose(gdn.gdn_recurrent(one, one, v, beta, la)[:, 0], g["single_state"]["o"], rtol=1e-14)
    np.testing.assert_allclose(gdn.gdn_forward_A(one, one, v, beta, la, lam)[:, 0], g["reading_A"]["o"], rtol=1e-14)
    np.testing.assert_allclose(gdn.gdn_forward_B(one, one, v, beta, la, lam)[:, 0], g["reading_B"]["o"], rtol=1e-14)
    o, _ = gdn.gdn_recurrent_levels_A(one, one, v, beta, la, lam)
    np.testing.assert_allclose(o[:, 0], g["reading_A"]["o"], rtol=1e-14)


@pytest.mark.parametrize("la", ["softplus", "zero"])
def test_constant_lambda_is_plain_gdn(la):
    T, d = 40, 6
    q, k, v, beta, log_alpha, _ = _rand(T, d, 1, seed=1, la=la)
    lam = np.full((T, levels_needed(T)), 1.7)
    ref = 1.7 * gdn.gdn_recurrent(q, k, v, beta, log_alpha)
    for f in (gdn.gdn_forward_A, gdn.gdn_forward_B):
        np.testing.assert_allclose(f(q, k, v, beta, log_alpha, lam), ref, rtol=1e-10, atol=1e-12)


def test_orthonormal_keys_reduce_to_mamba2():
    # k_s = e_s: K K^T = I, the delta correction vanishes and GDN is
    # log-linear Mamba-2 on beta-scaled values (both readings)
    T = d = 12
    q, _, v, beta, log_alpha, lam = _rand(T, d, levels_needed(T), seed=2)
    k = np.eye(T)
    want = mamba2.forward_dense(q, k, beta[:, None] * v, log_alpha, lam)
    np.testing.assert_allclose(gdn.gdn_forward_A(q, k, v, beta, log_alpha, lam), want, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(gdn.gdn_forward_B(q, k, v, beta, log_alpha, lam), want, rtol=1e-12, atol=1e-14)


def test_beta_zero_gives_zero():
    T, d = 20, 4
    q, k, v, _, log_alpha, lam = _rand(T, d, levels_needed(T), seed=3)
    assert np.abs(gdn.gdn_forward_A(q, k, v, np.zeros(T), log_alpha, lam)).max() == 0.0


@pytest.mark.parametrize("la", ["softplus", "zero"])
@pytest.mark.parametrize("T", [7, 64, 100])
def test_dense_A_equals_level_recurrence(T, la):
    q, k, v, beta, log_alpha, lam = _rand(T, 8, levels_needed(T), seed=T, la=la)
    d = gdn.gdn_forward_A(q, k, v, beta, log_alpha, lam)
    r, _ = gdn.gdn_recurrent_levels_A(q, k, v, beta, log_alpha, lam)
    np.testing.assert_allclose(r, d, rtol=1e-10, atol=1e-10 * np.abs(d).max())


def test_rows_equal_dense_A():
    T = 90
    q, k, v, beta, log_alpha, lam = _rand(T, 5, levels_needed(T), seed=4)
    d = gdn.gdn_forward_A(q, k, v, beta, log_alpha, lam)
    rows = [0, 1, 31, 32, 63, 89]
    np.testing.assert_allclose(gdn.gdn_rows_A(q, k, v, beta, log_alpha, lam, rows), d[rows], rtol=1e-11, atol=1e-13)


def test_readings_differ_in_general():
    T = 16
    q, k, v, beta, log_alpha, lam = _rand(T, 4, levels_needed(T), seed=5, la="zero")
    a = gdn.gdn_forward_A(q, k, v, beta, log_alpha, lam)
    b = gdn.gdn_forward_B(q, k, v, beta, log_alpha, lam)
    assert np.abs(a - b).max() > 1e-3


# ---- decode (Gated DeltaNet, reading A): gdn_decode_steps


def test_decode_from_zero_equals_dense_A():
    """Decoding every token from position 0 reproduces the dense matrix form."""
    T, d = 45, 6
    q, k, v, beta, log_alpha, lam = _rand(T, d, levels_needed(T) + 1, seed=11)
    Ls = levels_needed(T)
    o, _, _ = gdn.gdn_decode_steps(np.zeros((Ls, d, d)), np.zeros(Ls, bool), 0, q, k, v, beta, log_alpha, lam)
    want = gdn.gdn_forward_A(q, k, v, beta, log_alpha, lam[:, :levels_needed(T)])
    np.testing.assert_allclose(o, want, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("t0", [1, 8, 13, 31])
def test_decode_handoff_at_any_position(t0):
    """Stopping at t0 and continuing from the returned states changes nothing."""
    T, d = 40, 5
    Ls = levels_needed(T)
    q, k, v, beta, log_alpha, lam = _rand(T, d, Ls + 1, seed=12 + t0)
    z = (np.zeros((Ls, d, d)), np.zeros(Ls, bool), 0)
    o_all, S_all, ne_all = gdn.gdn_decode_steps(*z, q, k, v, beta, log_alpha, lam)
    o1, S1, ne1 = gdn.gdn_decode_steps(*z, q[:t0], k[:t0], v[:t0], beta[:t0], log_alpha[:t0], lam[:t0])
    assert list(ne1) == [bool((t0 >> i) & 1) for i in range(Ls)]
    o2, S2, ne2 = gdn.gdn_decode_steps(S1, ne1, t0, q[t0:], k[t0:], v[t0:], beta[t0:], log_alpha[t0:], lam[t0:])
    np.testing.assert_allclose(np.concatenate([o1, o2]), o_all, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S2, S_all, rtol=1e-12, atol=1e-14)
    assert list(ne2) == list(ne_all)


def test_decode_equal_lambda_is_single_state_rule():
    """With every lambda equal the level states sum to the one gated-delta state."""
    T, d = 33, 7
    Ls = levels_needed(T)
    q, k, v, beta, log_alpha, _ = _rand(T, d, 1, seed=13)
    lam = np.full((T, Ls + 1), 0.6)
    o, S, ne = gdn.gdn_decode_steps(np.zeros((Ls, d, d)), np.zeros(Ls, bool), 0, q, k, v, beta, log_alpha, lam)
    np.testing.assert_allclose(o, 0.6 * gdn.gdn_recurrent(q, k, v, beta, log_alpha), rtol=1e-10, atol=1e-12)
    # and the stored levels of position T sum to the textbook state at T - 1
    Sref = np.zeros((d, d))
    I = np.eye(d)
    for t in range(T):
        Sref = np.exp(log_alpha[t]) * Sref @ (I - beta[t] * np.outer(k[t], k[t])) + beta[t] * np.outer(v[t], k[t])
    np.testing.assert_allclose(S[ne].sum(axis=0), Sref, rtol=1e-10, atol=1e-12)


def test_decode_rejects_levels_that_are_not_the_bits_of_t0():
    d, Ls = 4, 5
    q, k, v, beta, log_alpha, lam = _rand(2, d, Ls + 1, seed=14)
    ne = np.array([True, False, False, False, False])  # t0 = 6 has bits 1 and 2
    with pytest.raises(ValueError):
        gdn.gdn_decode_steps(np.zeros((Ls, d, d)), ne, 6, q, k, v, beta, log_alpha, lam)
