"""Pins for the log-linear Mamba-2 backward oracle (oracle/backward.py).

The backward is pinned to the forward oracle (itself pinned in
test_oracle_mamba2.py) by central finite differences, and to identities that
follow from the forward's linearity in lam_t, q_t and V alone.  Mutants
planted in the oracle's steps show that the pins catch plausible mistakes.
"""

import numpy as np
import pytest

from oracle import backward, mamba2
from oracle.partition import levels_needed


def _case(T, dk, dv, L, seed, la="softplus"):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, dk))
    k = rng.standard_normal((T, dk))
    v = rng.standard_normal((T, dv))
    if la == "zero":
        log_alpha = np.zeros(T)
    else:
        log_alpha = -np.log1p(np.exp(rng.standard_normal(T)))
    lam = np.log1p(np.exp(rng.standard_normal((T, L))))
    do = rng.standard_normal((T, dv))
    return q, k, v, log_alpha, lam, do


def _numeric_grads(q, k, v, log_alpha, lam, do, eps=1e-6):
    """Central differences of f = sum(forward_dense(...) * do) for every input entry."""
    args = [np.array(x, np.float64) for x in (q, k, v, log_alpha, lam)]

    def f():
        return float(np.sum(mamba2.forward_dense(*args) * do))

    grads = []
    for x in args:
        g = np.zeros_like(x)
        flat, gf = x.reshape(-1), g.reshape(-1)
        for i in range(flat.size):
            keep = flat[i]
            flat[i] = keep + eps
            fp = f()
            flat[i] = keep - eps
            fm = f()
            flat[i] = keep
            gf[i] = (fp - fm) / (2 * eps)
        grads.append(g)
    return grads


def _fd_ok(case, rtol=1e-6):
    an = backward.backward_dense(*case)
    nu = _numeric_grads(*case)
    for a, n in zip(an, nu):
        scale = max(np.abs(n).max(), 1e-300)
        if np.abs(a - n).max() > rtol * scale:
            return False
    return True


@pytest.mark.parametrize("T,dk,dv,la", [(13, 3, 2, "softplus"), (9, 2, 3, "zero"), (16, 2, 2, "softplus")])
def test_finite_differences(T, dk, dv, la):
    L = levels_needed(T) + 1  # one level no key reaches: its gradient is 0
    case = _case(T, dk, dv, L, seed=T, la=la)
    an = backward.backward_dense(*case)
    nu = _numeric_grads(*case)
    for name, a, n in zip(("dq", "dk", "dv", "dlog_alpha", "dlam"), an, nu):
        assert a.shape == n.shape, name
        np.testing.assert_allclose(a, n, rtol=0, atol=1e-6 * np.abs(n).max(), err_msg=name)
    assert np.all(an[4][:, L - 1] == 0.0)


def test_homogeneity_identities():
    # o_t is linear in lam_t (row t), in q_t, and O is linear in V and in K:
    # sum_l lam_t[l] dlam_t[l] = q_t . dq_t = do_t . o_t;  sum_s v_s . dv_s = sum_s k_s . dk_s = sum_t do_t . o_t
    T = 37
    q, k, v, la, lam, do = _case(T, 4, 3, levels_needed(T), seed=5)
    dq, dk, dv, dla, dlam = backward.backward_dense(q, k, v, la, lam, do)
    o = mamba2.forward_dense(q, k, v, la, lam)
    row = np.sum(do * o, axis=1)
    np.testing.assert_allclose(np.sum(lam * dlam, axis=1), row, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(np.sum(q * dq, axis=1), row, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(np.sum(v * dv), row.sum(), rtol=1e-11)
    np.testing.assert_allclose(np.sum(k * dk), row.sum(), rtol=1e-11)
    # Gamma never depends on alpha_0
    assert abs(dla[0]) < 1e-10 * np.abs(dla).max()


def test_linear_attention_special_case():
    # lam = 1, alpha = 1: O = tril(Q K^T) V, whose gradients are textbook:
    # dQ = tril(dO V^T) K, dK = tril(dO V^T)^T Q, dV = tril(Q K^T)^T dO
    T = 12
    q, k, v, _, _, do = _case(T, 3, 2, levels_needed(T), seed=3)
    lam = np.ones((T, levels_needed(T)))
    dq, dk, dv, dla, dlam = backward.backward_dense(q, k, v, np.zeros(T), lam, do)
    lo = np.tril(np.ones((T, T)))
    G = lo * (do @ v.T)
    np.testing.assert_allclose(dq, G @ k, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dk, G.T @ q, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dv, (lo * (q @ k.T)).T @ do, rtol=1e-12, atol=1e-12)


def test_rows_match_dense():
    T = 41
    q, k, v, la, lam, do = _case(T, 4, 5, levels_needed(T), seed=9)
    dq, dk, dv, dla, dlam = backward.backward_dense(q, k, v, la, lam, do)
    rows = np.array([0, 1, 7, 16, 31, 40])
    rq, rl, row_term = backward.backward_query_rows(q, k, v, la, lam, do, rows)
    ck, cv, col_term = backward.backward_key_rows(q, k, v, la, lam, do, rows)
    np.testing.assert_allclose(rq, dq[rows], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(rl, dlam[rows], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ck, dk[rows], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(cv, dv[rows], rtol=1e-12, atol=1e-12)
    # dc_t = dla_t - dla_{t+1}
    dc = dla - np.append(dla[1:], 0.0)
    np.testing.assert_allclose(row_term - col_term, dc[rows], rtol=1e-10, atol=1e-11)


# ---- mutants planted in the oracle's steps: the finite-difference pin must fail
_FD_CASE = _case(11, 2, 2, levels_needed(11), seed=1)


def test_unmutated_backward_passes():
    assert _fd_ok(_FD_CASE)


def test_prefix_instead_of_suffix_is_caught(monkeypatch):
    monkeypatch.setattr(backward, "suffix_sums", lambda dc: np.cumsum(dc))
    assert not _fd_ok(_FD_CASE)


def test_cumsum_sign_is_caught(monkeypatch):
    orig = backward.cumsum_grad
    monkeypatch.setattr(backward, "cumsum_grad", lambda dG, G: -orig(dG, G))
    assert not _fd_ok(_FD_CASE)


def test_column_term_dropped_is_caught(monkeypatch):
    monkeypatch.setattr(backward, "cumsum_grad", lambda dG, G: (dG * G).sum(axis=1))
    assert not _fd_ok(_FD_CASE)


def test_level_sums_by_key_row_is_caught(monkeypatch):
    # the level gradient booked to the key's row instead of the query's
    def bad(dH, L):
        T = dH.shape[0]
        out = np.zeros((T, L))
        for t in range(T):
            for s_ in range(t + 1):
                out[s_, mamba2.level_array(t, s_)] += dH[t, s_]
        return out

    monkeypatch.setattr(backward, "level_sums", bad)
    assert not _fd_ok(_FD_CASE)


def test_level_off_by_one_is_caught(monkeypatch):
    orig = backward.level_sums
    monkeypatch.setattr(backward, "level_sums", lambda dH, L: np.roll(orig(dH, L), 1, axis=1))
    assert not _fd_ok(_FD_CASE)
