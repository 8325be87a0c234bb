"""Plant plausible mistakes in the oracle (on the CPU) and check a pin catches each.

Each mutant replaces one oracle function for the duration of one check; the
check is an existing pin's comparison and must now fail.
"""

import json
import os

import numpy as np
import pytest

from oracle import gdn, mamba2
from oracle.partition import levels_needed

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _case(T=24, seed=0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, 3))
    k = rng.standard_normal((T, 3))
    v = rng.standard_normal((T, 2))
    la = -np.log1p(np.exp(rng.standard_normal(T)))
    lam = np.log1p(np.exp(rng.standard_normal((T, levels_needed(T)))))
    return q, k, v, la, lam


def _golden_alpha_half_ok():
    with open(os.path.join(GOLDEN, "worked_forward.json")) as f:
        g = json.load(f)
    lam = np.tile(10.0 ** np.arange(4), (4, 1))
    one = np.ones((4, 1))
    o = mamba2.forward_dense(one, one, one, np.full(4, -np.log(2.0)), lam)[:, 0]
    return np.allclose(o, g["alpha_half"]["o"], rtol=1e-12)


def _dense_vs_recurrent_ok():
    q, k, v, la, lam = _case()
    return np.allclose(mamba2.forward_dense(q, k, v, la, lam), mamba2.forward_recurrent(q, k, v, la, lam)[0],
                       rtol=1e-10, atol=1e-12)


def test_unmutated_pins_pass():
    assert _golden_alpha_half_ok()
    assert _dense_vs_recurrent_ok()


def test_level_off_by_one_is_caught(monkeypatch):
    orig = mamba2.level_array
    monkeypatch.setattr(mamba2, "level_array", lambda t, s: np.maximum(orig(t, s) - 1, 0))
    assert not _golden_alpha_half_ok()
    assert not _dense_vs_recurrent_ok()


def test_level_exclusive_token_is_caught(monkeypatch):
    # reading the state as excluding token t (level 0 dropped)
    orig = mamba2.hier_mask
    monkeypatch.setattr(mamba2, "hier_mask", lambda lam: orig(lam) - np.diag(np.asarray(lam)[:, 0]))
    assert not _golden_alpha_half_ok()
    assert not _dense_vs_recurrent_ok()


def test_decay_closed_interval_is_caught(monkeypatch):
    # product of alpha over [s, t] instead of (s, t]
    orig = mamba2.decay_matrix
    monkeypatch.setattr(mamba2, "decay_matrix", lambda la: orig(la) * np.exp(np.asarray(la, np.float64))[None, :])
    assert not _golden_alpha_half_ok()
    assert not _dense_vs_recurrent_ok()


def test_transposed_mask_is_caught(monkeypatch):
    # lambda indexed by the key's position instead of the query's
    def bad(lam):
        lam = np.asarray(lam, np.float64)
        T = lam.shape[0]
        t = np.arange(T)[:, None]
        s = np.arange(T)[None, :]
        lv = mamba2.level_array(t, s)
        out = np.where(s <= t, lam[np.broadcast_to(s, (T, T)), lv], 0.0)
        return out
    monkeypatch.setattr(mamba2, "hier_mask", bad)
    assert not _dense_vs_recurrent_ok()


def test_gdn_missing_beta_is_caught(monkeypatch):
    with open(os.path.join(GOLDEN, "worked_gdn.json")) as f:
        g = json.load(f)
    orig = gdn.gdn_coeff
    monkeypatch.setattr(gdn, "gdn_coeff", lambda q, k, beta, la: orig(q, k, beta, la) / np.asarray(beta)[None, :])
    one = np.ones((2, 1))
    o = gdn.gdn_forward_A(one, one, np.array([[1.0], [2.0]]), np.array([0.5, 0.5]), np.zeros(2),
                          np.array([[1.0, 10.0], [1.0, 10.0]]))[:, 0]
    assert not np.allclose(o, g["reading_A"]["o"])


# ---- Gated DeltaNet decode step (gdn.gdn_level_step)

def _gdn_decode_vs_dense_ok():
    T, d = 30, 4
    rng = np.random.default_rng(21)
    q = rng.standard_normal((T, d))
    k = rng.standard_normal((T, d))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, d))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(T)))
    la = -np.log1p(np.exp(rng.standard_normal(T)))
    Ls = levels_needed(T)
    lam = np.log1p(np.exp(rng.standard_normal((T, Ls + 1))))
    o, _, _ = gdn.gdn_decode_steps(np.zeros((Ls, d, d)), np.zeros(Ls, bool), 0, q, k, v, beta, la, lam)
    return np.allclose(o, gdn.gdn_forward_A(q, k, v, beta, la, lam[:, :Ls]), rtol=1e-10, atol=1e-12)


def _step_variant(write_first=False, carry_shift=0):
    def step(states, t, q, k, v, beta, log_alpha, lam):
        P = np.exp(log_alpha) * (np.eye(k.shape[0]) - beta * np.outer(k, k))
        if write_first:  # the token's own write also goes through this step's transition
            states[0] = beta * np.outer(v, k)
        for lv in list(states):
            states[lv] = states[lv] @ P
        if not write_first:
            states[0] = beta * np.outer(v, k)
        o = sum(lam[lv] * (S @ q) for lv, S in states.items())
        j = 0
        while (t >> j) & 1:
            j += 1
        merged = states.pop(0)
        for lv in range(1, j + 1):
            merged = merged + states.pop(lv, 0)
        states[j + 1 + carry_shift] = merged + states.pop(j + 1 + carry_shift, 0)
        return o
    return step


def test_gdn_decode_unmutated_variant_passes(monkeypatch):
    monkeypatch.setattr(gdn, "gdn_level_step", _step_variant())
    assert _gdn_decode_vs_dense_ok()


def test_gdn_decode_write_transitioned_is_caught(monkeypatch):
    monkeypatch.setattr(gdn, "gdn_level_step", _step_variant(write_first=True))
    assert not _gdn_decode_vs_dense_ok()


def test_gdn_decode_carry_to_wrong_level_is_caught(monkeypatch):
    monkeypatch.setattr(gdn, "gdn_level_step", _step_variant(carry_shift=1))
    assert not _gdn_decode_vs_dense_ok()


# ----------------------------------------------------------------------------
# the per-level-decay variant
# ----------------------------------------------------------------------------
def _ld_case(T=20, seed=3):
    rng = np.random.default_rng(seed)
    L = levels_needed(T)
    q = rng.standard_normal((T, 3))
    k = rng.standard_normal((T, 3))
    v = rng.standard_normal((T, 2))
    la = -rng.random((T, L))
    lam = np.log1p(np.exp(rng.standard_normal((T, L))))
    return q, k, v, la, lam


def _ld_pins_ok():
    from oracle import level_decay as ld
    T = 24
    L = levels_needed(T)
    c = -0.05 * np.arange(L) - 0.01
    la = np.tile(c, (T, 1))
    want = np.zeros((T, T))
    for t in range(T):
        for s in range(t + 1):
            if s == t:
                want[t, s] = 1.0
                continue
            l = (t ^ s).bit_length()
            e = sum(c[m] * 2 ** (m - 1) for m in range(1, l) if not (s >> (m - 1)) & 1)
            want[t, s] = np.exp(e + c[l] * ((t % 2 ** (l - 1)) + 1))
    closed = np.allclose(ld.decay_matrix(la), want, rtol=1e-12)
    q, k, v, la, lam = _ld_case()
    routes = np.allclose(ld.forward_dense(q, k, v, la, lam), ld.forward_recurrent(q, k, v, la, lam)[0],
                         rtol=1e-10, atol=1e-12)
    return closed and routes


def test_level_decay_unmutated_pins_pass():
    assert _ld_pins_ok()


def test_level_decay_at_the_query_level_is_caught(monkeypatch):
    # every step of (s, t] decayed at the rate of level(t, s), the level the
    # key has for the query, instead of the level it occupies at each step
    from oracle import level_decay as ld

    def bad(la):
        la = np.asarray(la, np.float64)
        T = la.shape[0]
        out = np.eye(T)
        for t in range(T):
            for s in range(t):
                lv = (t ^ s).bit_length()
                out[t, s] = np.exp(la[s + 1:t + 1, lv].sum())
        return out
    monkeypatch.setattr(ld, "decay_matrix", bad)
    assert not _ld_pins_ok()


def test_level_decay_one_step_late_is_caught(monkeypatch):
    # the level of key s at step r taken as its level at step r - 1
    from oracle import level_decay as ld

    def bad(la):
        la = np.asarray(la, np.float64)
        T = la.shape[0]
        out = np.eye(T)
        for s in range(T):
            acc = 0.0
            for r in range(s + 1, T):
                acc += la[r, mamba2.level_array(r - 1, s) if r - 1 > s else 1]
                out[r, s] = np.exp(acc)
        return out
    monkeypatch.setattr(ld, "decay_matrix", bad)
    assert not _ld_pins_ok()


def test_level_decay_rate_index_off_by_one_is_caught(monkeypatch):
    # recurrent form: the state of level l decayed at the rate of level l + 1
    from oracle import level_decay as ld

    def bad(states, t, q_t, k_t, v_t, la_t, lam_t):
        for lv in list(states):
            states[lv] = states[lv] * float(np.exp(la_t[min(lv + 1, len(la_t) - 1)]))
        states[0] = np.outer(v_t, k_t)
        o = np.zeros(v_t.shape[0])
        for lv, S in states.items():
            o += lam_t[lv] * (S @ q_t)
        j = 0
        while (t >> j) & 1:
            j += 1
        merged = states.pop(0)
        for lv in range(1, j + 1):
            merged = merged + states.pop(lv)
        states[j + 1] = merged
        return o
    monkeypatch.setattr(ld, "fenwick_step", bad)
    assert not _ld_pins_ok()
