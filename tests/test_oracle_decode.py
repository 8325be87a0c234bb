"""Pins for the Fenwick decode oracle (oracle/decode.py)."""

import numpy as np
import pytest

from oracle import decode, mamba2
from oracle.partition import levels_needed


def _rand(T, d, L, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, d)) / np.sqrt(d)
    k = rng.standard_normal((T, d)) / np.sqrt(d)
    v = rng.standard_normal((T, d))
    log_alpha = -np.log1p(np.exp(rng.standard_normal(T)))
    lam = np.log1p(np.exp(rng.standard_normal((T, L))))
    return q, k, v, log_alpha, lam


@pytest.mark.parametrize("P,n", [(64, 40), (37, 30), (1, 20)])
def test_decode_rows_equal_dense_rows(P, n):
    # decode outputs for positions P..P+n-1 equal the dense definition's rows
    T = P + n
    Ls = levels_needed(T + 1)
    q, k, v, log_alpha, lam = _rand(T, 5, Ls + 1, seed=P)
    S0, ne0 = mamba2.states_at(k, v, log_alpha, P, Ls)
    o, S, ne = decode.decode_steps(S0, ne0, P, q[P:], k[P:], v[P:], log_alpha[P:], lam[P:])
    d = mamba2.forward_rows(q, k, v, log_alpha, lam, range(P, T))
    np.testing.assert_allclose(o, d, rtol=1e-11, atol=1e-13)
    # final states equal the bucket sums at the end
    S1, ne1 = mamba2.states_at(k, v, log_alpha, T, Ls)
    assert list(ne) == list(ne1)
    np.testing.assert_allclose(S, S1, rtol=1e-11, atol=1e-13)


def test_aligned_block_collapses_to_one_level():
    # after 2^k steps from an aligned start only one level is non-empty
    P, n = 64, 64
    q, k, v, log_alpha, lam = _rand(P + n, 3, 9, seed=1)
    S0, ne0 = mamba2.states_at(k, v, log_alpha, P, 8)
    _, S, ne = decode.decode_steps(S0, ne0, P, q[P:], k[P:], v[P:], log_alpha[P:], lam[P:])
    assert list(np.nonzero(ne)[0] + 1) == [8]


def test_rejects_inconsistent_levels():
    S0 = np.zeros((4, 2, 2))
    ne0 = np.array([True, False, False, False])
    with pytest.raises(ValueError):
        decode.decode_steps(S0, ne0, 2, np.zeros((1, 2)), np.zeros((1, 2)), np.zeros((1, 2)), np.zeros(1), np.zeros((1, 5)))
