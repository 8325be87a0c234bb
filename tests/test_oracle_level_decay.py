"""Pins for the per-level-decay oracle (oracle/level_decay.py).

The variant has no worked example on the pages (the study note's §7 names it
as a follow-up idea), so the pins are the form it must reduce to (one decay
for all levels is the log-linear Mamba-2, itself pinned), hand-derived
products, closed forms obtained by counting the steps a key spends on each
level, and the brute-force and recurrent routes.
"""

import numpy as np
import pytest

from oracle import level_decay as ld
from oracle import mamba2
from oracle.partition import levels_needed


def _rand(T, dk, dv, L, seed, scale=0.3):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, dk)) / np.sqrt(dk)
    k = rng.standard_normal((T, dk)) / np.sqrt(dk)
    v = rng.standard_normal((T, dv))
    la = -scale * rng.random((T, L))
    lam = np.log1p(np.exp(rng.standard_normal((T, L))))
    return q, k, v, la, lam


@pytest.mark.parametrize("T,seed", [(1, 0), (7, 1), (16, 2), (37, 3), (64, 4)])
def test_one_decay_for_all_levels_is_the_base_form(T, seed):
    L = levels_needed(T)
    q, k, v, la, lam = _rand(T, 8, 5, L, seed)
    la_lv = np.repeat(la[:, :1], L, axis=1)
    np.testing.assert_allclose(ld.forward_dense(q, k, v, la_lv, lam),
                               mamba2.forward_dense(q, k, v, la[:, 0], lam), rtol=1e-12, atol=1e-13)


def test_hand_derived_products_t4():
    # levels of key s at steps r (from the buckets of r): key 0 is at level 1
    # at r = 1 and level 2 at r = 2, 3; key 1 at level 2 at r = 2, 3; key 2
    # at level 1 at r = 3.  With log alpha_r^(l) = -(r + 10 l) / 100:
    a = lambda r, l: np.exp(-(r + 10 * l) / 100.0)  # noqa: E731
    G = np.zeros((4, 4))
    for t in range(4):
        G[t, t] = 1.0
    G[1, 0] = a(1, 1)
    G[2, 0] = a(1, 1) * a(2, 2)
    G[3, 0] = a(1, 1) * a(2, 2) * a(3, 2)
    G[2, 1] = a(2, 2)
    G[3, 1] = a(2, 2) * a(3, 2)
    G[3, 2] = a(3, 1)
    la = np.array([[-(r + 10 * l) / 100.0 for l in range(3)] for r in range(4)])
    np.testing.assert_allclose(ld.decay_matrix(la), G, rtol=1e-14)
    # with q = k = v = 1 and lam^(l) = 10^l: o_t = sum_s 10^level(t,s) G[t, s]
    lam = np.tile(10.0 ** np.arange(3), (4, 1))
    lv = [[0], [1, 0], [2, 2, 0], [2, 2, 1, 0]]
    want = [sum(10.0 ** lv[t][s] * G[t, s] for s in range(t + 1)) for t in range(4)]
    one = np.ones((4, 1))
    np.testing.assert_allclose(ld.forward_dense(one, one, one, la, lam)[:, 0], want, rtol=1e-14)
    np.testing.assert_allclose(ld.forward_buckets(one, one, one, la, lam)[:, 0], want, rtol=1e-14)
    np.testing.assert_allclose(ld.forward_recurrent(one, one, one, la, lam)[0][:, 0], want, rtol=1e-14)


def test_constant_rate_per_level_closed_form():
    # log alpha^(m) = c_m at every step: key s spends 2^(m-1) steps on every
    # level m < level(t, s) whose bit m-1 is clear in s, none on the others,
    # and (t mod 2^(l-1)) + 1 steps on l = level(t, s).
    T = 96
    L = levels_needed(T)
    c = -0.013 * np.arange(L) - 0.002 * np.arange(L) ** 2
    la = np.tile(c, (T, 1))
    want = np.zeros((T, T))
    for t in range(T):
        for s in range(t + 1):
            if s == t:
                want[t, s] = 1.0
                continue
            l = (t ^ s).bit_length()
            e = sum(c[m] * 2 ** (m - 1) for m in range(1, l) if not (s >> (m - 1)) & 1)
            e += c[l] * ((t % 2 ** (l - 1)) + 1)
            want[t, s] = np.exp(e)
    np.testing.assert_allclose(ld.decay_matrix(la), want, rtol=1e-12)


def test_only_level_one_survives():
    # alpha^(l) = 0 above level 1: a key survives only while it has not left
    # level 1, i.e. o_t = lam_t0 (q.k_t) v_t + [t odd] lam_t1 alpha_t^(1) (q.k_{t-1}) v_{t-1}
    T = 24
    L = levels_needed(T)
    q, k, v, la, lam = _rand(T, 6, 3, L, 11)
    la[:, 2:] = -1e4
    o = ld.forward_dense(q, k, v, la, lam)
    want = np.zeros_like(o)
    for t in range(T):
        want[t] = lam[t, 0] * (q[t] @ k[t]) * v[t]
        if t % 2 == 1:
            want[t] += lam[t, 1] * np.exp(la[t, 1]) * (q[t] @ k[t - 1]) * v[t - 1]
    np.testing.assert_allclose(o, want, rtol=1e-12, atol=1e-14)


def test_column_zero_is_never_used():
    T = 40
    L = levels_needed(T)
    q, k, v, la, lam = _rand(T, 4, 4, L, 5)
    la2 = la.copy()
    la2[:, 0] = -7.0
    np.testing.assert_array_equal(ld.forward_dense(q, k, v, la, lam), ld.forward_dense(q, k, v, la2, lam))


@pytest.mark.parametrize("T,seed", [(5, 0), (13, 1), (16, 2)])
def test_brute_force_recurrent_and_dense_agree(T, seed):
    L = levels_needed(T)
    q, k, v, la, lam = _rand(T, 4, 3, L, seed, scale=1.0)
    d = ld.forward_dense(q, k, v, la, lam)
    np.testing.assert_allclose(ld.forward_buckets(q, k, v, la, lam), d, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(ld.forward_recurrent(q, k, v, la, lam)[0], d, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("T,seed", [(1, 0), (33, 1), (200, 2), (513, 3)])
def test_rows_match_dense(T, seed):
    L = levels_needed(T)
    q, k, v, la, lam = _rand(T, 8, 6, L, seed)
    d = ld.forward_dense(q, k, v, la, lam)
    rows = np.unique(np.r_[0, T - 1, np.arange(0, T, 7)])
    np.testing.assert_allclose(ld.forward_rows(q, k, v, la, lam, rows), d[rows], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(ld.forward_recurrent(q, k, v, la, lam)[0], d, rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("t0,n", [(0, 9), (5, 12), (64, 30), (77, 20)])
def test_decode_continues_the_sequence(t0, n):
    T = t0 + n
    L = levels_needed(T)
    Ls = L - 1
    q, k, v, la, lam = _rand(T, 5, 4, L, t0 + n)
    S0, ne0 = ld.states_at(k, v, la, t0, Ls)
    o, S1, ne1 = ld.decode_steps(S0, ne0, t0, q[t0:], k[t0:], v[t0:], la[t0:], lam[t0:])
    np.testing.assert_allclose(o, ld.forward_dense(q, k, v, la, lam)[t0:], rtol=1e-11, atol=1e-13)
    S_ref, ne_ref = ld.states_at(k, v, la, T, Ls)
    np.testing.assert_array_equal(ne1, ne_ref)
    np.testing.assert_allclose(S1, S_ref, rtol=1e-11, atol=1e-13)


def test_states_are_the_buckets_decayed_by_the_definition():
    # the state of level l at position P holds the keys of that bucket, each
    # with the decay Gamma(P - 1, s) of the definition
    T = 45
    L = levels_needed(T + 1)
    q, k, v, la, lam = _rand(T + 1, 3, 2, L, 9)
    G = ld.decay_matrix(la)
    S, ne = ld.states_at(k, v, la, T, L - 1)
    from oracle.partition import buckets
    for lv, lo, hi in buckets(T)[1:]:
        want = sum(G[T - 1, s] * np.outer(v[s], k[s]) for s in range(lo, hi))
        np.testing.assert_allclose(S[lv - 1], want, rtol=1e-12)
        assert ne[lv - 1]
