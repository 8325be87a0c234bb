"""Log-linear Mamba-2 with a decay per level, oracle (NumPy float64; test
infrastructure only).

Source: "Log-Linear Attention" study note (dimensionstp.github.io) §7
"Follow-up design", which lists a learned memory decay per level as a
follow-up idea without defining it.  Reading R21 (the plainest one that the
recurrent form of §3-3 / §3-6 supports): the memory of level l decays at its
own rate alpha_t^(l), so a key decays, at every step r, at the rate of the
level it occupies at that step:

    M(t, s) = lam_t[level(t, s)] * prod_{r = s+1..t} alpha_r^(level(r, s))

and o = (Q K^T . M) V.  In the recurrent form every level state is multiplied
by its own alpha_t^(l) where the base form multiplies all of them by alpha_t;
the carry-merge is unchanged (a key's level only grows with r, and the merged
contents decay at the rate of the level they land in).  log_alpha is [T, L]
like lam; its column 0 is never used, since a key is at level 0 only at its
own step, which applies no decay.  With every column equal to one scalar
log-decay the form is the log-linear Mamba-2 of oracle.mamba2.

Routes, cross-checked by the tests:
  ``forward_dense``      the T x T masked form (the definition);
  ``forward_rows``       the same sum for selected rows t, with the steps of
                         each key grouped by the level it occupies;
  ``forward_recurrent``  a token loop over level states with carry-merge;
  ``forward_buckets``    brute force: each bucket enumerated, each key's
                         level at each step looked up in that step's buckets.
"""

from __future__ import annotations

import numpy as np

from .mamba2 import hier_mask, level_array
from .partition import buckets


def decay_matrix(log_alpha_lv) -> np.ndarray:
    """Gamma(t, s) = exp(sum_{r=s+1..t} log_alpha_lv[r, level(r, s)]) for s <= t, else 0."""
    la = np.asarray(log_alpha_lv, np.float64)
    T = la.shape[0]
    out = np.zeros((T, T))
    for s in range(T):
        out[s, s] = 1.0
        if s + 1 < T:
            r = np.arange(s + 1, T)
            lv = level_array(r, s)
            out[s + 1:, s] = np.exp(np.cumsum(la[r, lv]))
    return out


def forward_dense(q, k, v, log_alpha_lv, lam) -> np.ndarray:
    """O = (Q K^T . Gamma . M^H) V for one (batch, head) slice."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    M = decay_matrix(log_alpha_lv) * hier_mask(lam)
    return ((q @ k.T) * M) @ v


def forward_dense_bh(q, k, v, log_alpha_lv, lam) -> np.ndarray:
    """forward_dense over leading [B, H] axes."""
    B, H = q.shape[:2]
    out = np.zeros(q.shape[:3] + (v.shape[-1],))
    for b in range(B):
        for h in range(H):
            out[b, h] = forward_dense(q[b, h], k[b, h], v[b, h], log_alpha_lv[b, h], lam[b, h])
    return out


def log_decay_rows(log_alpha_lv, t: int) -> np.ndarray:
    """log Gamma(t, s) for s = 0..t.

    The steps r in (s, t] at which key s sits at level m are the block of
    2^(m-1) positions just above s's own aligned block of that size (present
    when bit m-1 of s is clear), cut at t; the sum over r is taken block by
    block from per-level running sums.
    """
    la = np.asarray(log_alpha_lv, np.float64)
    L = la.shape[1]
    cum = np.vstack([np.zeros((1, L)), np.cumsum(la, axis=0)])  # cum[i] = sum of rows < i
    s = np.arange(t + 1)
    g = np.zeros(t + 1)
    for m in range(1, L):
        lo = ((s >> m) << m) + (1 << (m - 1))
        hi = np.minimum(lo + (1 << (m - 1)), t + 1)
        use = (((s >> (m - 1)) & 1) == 0) & (lo <= t)
        lo_c = np.minimum(lo, t + 1)
        g += np.where(use, cum[np.where(use, hi, 0), m] - cum[np.where(use, lo_c, 0), m], 0.0)
    if t > 0 and level_array(t, 0) >= L:
        raise ValueError("log_alpha_lv has too few levels for this t")
    return g


def forward_rows(q, k, v, log_alpha_lv, lam, rows) -> np.ndarray:
    """The definition evaluated for query rows ``rows`` only (one slice)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    lam = np.asarray(lam, np.float64)
    out = np.zeros((len(rows), v.shape[1]))
    for i, t in enumerate(rows):
        t = int(t)
        s = np.arange(t + 1)
        coef = (k[: t + 1] @ q[t]) * np.exp(log_decay_rows(log_alpha_lv, t)) * lam[t, level_array(t, s)]
        out[i] = coef @ v[: t + 1]
    return out


def fenwick_step(states: dict, t: int, q_t, k_t, v_t, log_alpha_t, lam_t):
    """One token of the recurrent form; ``states`` maps level -> [dv, dk].

    On entry the states hold the buckets of query t (levels >= 1), decayed to
    t - 1.  Steps:
      1. the state of level l is decayed by alpha_t^(l);
      2. the token enters level 0 as v_t k_t^T;
      3. o_t = sum_l lam_t[l] S^(l) q_t;
      4. carry: with j trailing ones in t, levels 0..j merge into level j + 1.
    On exit the states hold the buckets of query t + 1, decayed to t.
    """
    for lv in list(states):
        states[lv] = states[lv] * float(np.exp(log_alpha_t[lv]))
    states[0] = np.outer(v_t, k_t)
    o = np.zeros(v_t.shape[0])
    for lv, S in states.items():
        o += lam_t[lv] * (S @ q_t)
    j = 0
    while (t >> j) & 1:
        j += 1
    if (j + 1) in states:
        raise AssertionError("carry target level is not empty")
    merged = states.pop(0)
    for lv in range(1, j + 1):
        merged = merged + states.pop(lv)
    states[j + 1] = merged
    return o


def forward_recurrent(q, k, v, log_alpha_lv, lam):
    """Token loop over level states; returns (O, final states dict)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    lam = np.asarray(lam, np.float64)
    la = np.asarray(log_alpha_lv, np.float64)
    states: dict = {}
    out = np.zeros((q.shape[0], v.shape[1]))
    for t in range(q.shape[0]):
        out[t] = fenwick_step(states, t, q[t], k[t], v[t], la[t], lam[t])
    return out, states


def forward_buckets(q, k, v, log_alpha_lv, lam) -> np.ndarray:
    """Brute force over buckets; a key's level at step r is found by searching
    the buckets of r.  Tiny T only."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    lam = np.asarray(lam, np.float64)
    alpha = np.exp(np.asarray(log_alpha_lv, np.float64))

    def level_at(r, s):
        for lv, lo, hi in buckets(r):
            if lo <= s < hi:
                return lv
        raise AssertionError("key outside the buckets of its query")

    T = q.shape[0]
    out = np.zeros((T, v.shape[1]))
    for t in range(T):
        for lv, lo, hi in buckets(t):
            for s in range(lo, hi):
                gamma = 1.0
                for r in range(s + 1, t + 1):
                    gamma *= alpha[r, level_at(r, s)]
                out[t] += lam[t, lv] * gamma * float(q[t] @ k[s]) * v[s]
    return out


def states_at(k, v, log_alpha_lv, T_pos: int, Ls: int):
    """Level states of query position T_pos from keys 0..T_pos-1, decayed to
    T_pos - 1 (slot i is level i + 1): the recurrent form run to T_pos.

    Returns (S [Ls, dv, dk], nonempty [Ls] bool).
    """
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    la = np.asarray(log_alpha_lv, np.float64)
    dv, dk = v.shape[1], k.shape[1]
    states: dict = {}
    zero_q = np.zeros(dk)
    lam0 = np.zeros(la.shape[1])
    for t in range(T_pos):
        fenwick_step(states, t, zero_q, k[t], v[t], la[t], lam0)
    S = np.zeros((Ls, dv, dk))
    ne = np.zeros(Ls, dtype=bool)
    for lv, M in states.items():
        if lv > Ls:
            raise ValueError("Ls too small for this position")
        S[lv - 1] = M
        ne[lv - 1] = True
    return S, ne


def decode_steps(S0, nonempty0, t0: int, q, k, v, log_alpha_lv, lam):
    """len(q) decode steps from position t0 with per-level decays.

    S0 [Ls, dv, dk], nonempty0 [Ls]: the states of query t0 (decayed to t0-1);
    q, k [n, dk]; v [n, dv]; log_alpha_lv, lam [n, Ls + 1].
    Returns (o [n, dv], S [Ls, dv, dk], nonempty [Ls]) after the last step.
    """
    Ls = S0.shape[0]
    expect = [(t0 >> (lv - 1)) & 1 == 1 for lv in range(1, Ls + 1)]
    if list(map(bool, nonempty0)) != expect:
        raise ValueError("non-empty levels must be the set bits of t0")
    states = {i + 1: np.asarray(S0[i], np.float64).copy() for i in range(Ls) if nonempty0[i]}
    n = q.shape[0]
    out = np.zeros((n, v.shape[1]))
    for i in range(n):
        out[i] = fenwick_step(states, t0 + i, np.asarray(q[i], np.float64), np.asarray(k[i], np.float64),
                              np.asarray(v[i], np.float64), np.asarray(log_alpha_lv[i], np.float64),
                              np.asarray(lam[i], np.float64))
    S = np.zeros((Ls, v.shape[1], k.shape[1]))
    ne = np.zeros(Ls, dtype=bool)
    for lv, M in states.items():
        if lv == 0 or lv > Ls:
            raise ValueError(f"level {lv} cannot be stored in {Ls} slots")
        S[lv - 1] = M
        ne[lv - 1] = True
    return out, S, ne
