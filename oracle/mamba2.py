"""Log-linear Mamba-2 forward, oracle (NumPy float64; test infrastructure only).

What is computed (per batch row and head; q, k: [T, dk], v: [T, dv],
log_alpha: [T], lam: [T, L]):

    o_t = sum_{s <= t} (q_t . k_s) * Gamma(t, s) * lam_t[level(t, s)] * v_s

i.e. O = (Q K^T . M^S . M^H) V with
  * M^S(t, s) = Gamma(t, s) = prod_{r = s+1..t} alpha_r for s <= t (1 on the
    diagonal), the Mamba-2 scalar-decay semiseparable mask (reading R4), and
  * M^H(t, s) = lam_t[level(t, s)], the Fenwick hierarchical mask.

Sources: "Log-Linear Attention" study note (dimensionstp.github.io) §3-4
"Parallel form" (O = (Q K^T . M^H) V with a lower-triangular hierarchical
M^H), §3-5 (M = M^S . M^H; Log-Linear Mamba-2 keeps the Mamba-2 transition
and multiplies in M^H), §2-2 / §3-3 (o_t = sum_l lam_t^(l) q_t^T S_t^(l), one
recurrent state per bucket).  No 1/sqrt(d) scale, no normalisation, no skip
term: the pages' formulas have none.

Four independent routes are provided and cross-checked by the tests:
  ``forward_dense``      the T x T masked form (the definition);
  ``forward_rows``       the same definition evaluated for selected rows t;
  ``forward_recurrent``  a token loop over Fenwick level states with
                         carry-merge (the recurrent form);
  ``forward_buckets``    brute-force enumeration of each bucket, with the
                         decay taken as an explicit product of alphas.
"""

from __future__ import annotations

import numpy as np

from .partition import buckets


# ----------------------------------------------------------------------------
# masks
# ----------------------------------------------------------------------------
def level_array(t_idx: np.ndarray, s_idx: np.ndarray) -> np.ndarray:
    """Vectorised closed-form level (reading R1): 0 if s == t else bitlen(t ^ s).

    Valid for s <= t; entries with s > t are returned but meaningless.
    np.frexp gives x = m * 2**e with 0.5 <= m < 1, so e is the bit length of
    a positive integer x (exact for x < 2**53).
    """
    x = np.bitwise_xor(np.asarray(t_idx, dtype=np.int64), np.asarray(s_idx, dtype=np.int64))
    _, e = np.frexp(x.astype(np.float64))
    return np.where(x > 0, e, 0).astype(np.int64)


def decay_matrix(log_alpha: np.ndarray) -> np.ndarray:
    """M^S: Gamma(t, s) = exp(sum_{r=s+1..t} log_alpha_r) for s <= t, else 0."""
    la = np.asarray(log_alpha, dtype=np.float64)
    cum = np.cumsum(la)
    g = cum[:, None] - cum[None, :]
    T = la.shape[0]
    causal = np.tril(np.ones((T, T), dtype=bool))
    out = np.zeros((T, T), dtype=np.float64)
    out[causal] = np.exp(g[causal])
    return out


def hier_mask(lam: np.ndarray) -> np.ndarray:
    """M^H: lam_t[level(t, s)] for s <= t, else 0.  lam: [T, L]."""
    lam = np.asarray(lam, dtype=np.float64)
    T = lam.shape[0]
    t_idx = np.arange(T)[:, None]
    s_idx = np.arange(T)[None, :]
    lv = level_array(t_idx, s_idx)
    causal = s_idx <= t_idx
    if lv[causal].max(initial=0) >= lam.shape[1]:
        raise ValueError("lam has too few levels for this T")
    out = np.zeros((T, T), dtype=np.float64)
    rows = np.broadcast_to(t_idx, (T, T))
    out[causal] = lam[rows[causal], lv[causal]]
    return out


# ----------------------------------------------------------------------------
# the definition
# ----------------------------------------------------------------------------
def forward_dense(q, k, v, log_alpha, lam) -> np.ndarray:
    """O = (Q K^T . M^S . M^H) V for one (batch, head) slice."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    A = q @ k.T
    M = decay_matrix(log_alpha) * hier_mask(lam)
    return (A * M) @ v


def forward_dense_bh(q, k, v, log_alpha, lam) -> np.ndarray:
    """forward_dense over leading [B, H] axes: q [B,H,T,dk] ... lam [B,H,T,L]."""
    B, H = q.shape[:2]
    out = np.zeros(q.shape[:3] + (v.shape[-1],), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            out[b, h] = forward_dense(q[b, h], k[b, h], v[b, h], log_alpha[b, h], lam[b, h])
    return out


def forward_rows(q, k, v, log_alpha, lam, rows) -> np.ndarray:
    """The same definition evaluated only for query rows ``rows`` (one slice).

    Row t needs keys 0..t only, so cost is O(t * d) per row: this is how the
    long sequences are checked on sampled rows.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    lam = np.asarray(lam, np.float64)
    cum = np.cumsum(np.asarray(log_alpha, np.float64))
    out = np.zeros((len(rows), v.shape[1]), dtype=np.float64)
    for i, t in enumerate(rows):
        t = int(t)
        s = np.arange(t + 1)
        coef = (k[: t + 1] @ q[t]) * np.exp(cum[t] - cum[: t + 1]) * lam[t, level_array(t, s)]
        out[i] = coef @ v[: t + 1]
    return out


# ----------------------------------------------------------------------------
# recurrent form: Fenwick level states with carry-merge
# ----------------------------------------------------------------------------
def fenwick_step(states: dict, t: int, q_t, k_t, v_t, log_alpha_t, lam_t):
    """One token of the recurrent form.  ``states`` maps level -> [dv, dk].

    On entry the states hold the buckets of query t (levels >= 1), decayed to
    t - 1.  Steps (study note §3-3 / §3-6; drawer analogy in the zh summary):
      1. every state is decayed by alpha_t (M^S over (s, t]);
      2. the token enters level 0 as v_t k_t^T;
      3. o_t = sum_l lam_t[l] * S^(l) q_t;
      4. carry: j = number of trailing ones of t; levels 0..j are full and are
         merged (added) into level j + 1, which is empty before the merge.
    On exit the states hold the buckets of query t + 1, decayed to t.
    """
    alpha = float(np.exp(log_alpha_t))
    for lv in list(states):
        states[lv] = states[lv] * alpha
    states[0] = np.outer(v_t, k_t)
    o = np.zeros(v_t.shape[0], dtype=np.float64)
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


def forward_recurrent(q, k, v, log_alpha, lam):
    """Token loop over level states; returns (O, final states dict)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    lam = np.asarray(lam, np.float64)
    la = np.asarray(log_alpha, np.float64)
    T = q.shape[0]
    states: dict = {}
    out = np.zeros((T, v.shape[1]), dtype=np.float64)
    for t in range(T):
        out[t] = fenwick_step(states, t, q[t], k[t], v[t], la[t], lam[t])
    return out, states


def forward_buckets(q, k, v, log_alpha, lam) -> np.ndarray:
    """Brute force: o_t = sum over buckets of t of lam_t[l] * sum_{s in bucket} ...

    The decay is taken as an explicit product of alphas over (s, t], the
    buckets from the peeling procedure.  Tiny T only.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    lam = np.asarray(lam, np.float64)
    alpha = np.exp(np.asarray(log_alpha, np.float64))
    T = q.shape[0]
    out = np.zeros((T, v.shape[1]), dtype=np.float64)
    for t in range(T):
        for lv, lo, hi in buckets(t):
            for s in range(lo, hi):
                gamma = 1.0
                for r in range(s + 1, t + 1):
                    gamma *= alpha[r]
                out[t] += lam[t, lv] * gamma * float(q[t] @ k[s]) * v[s]
    return out


# ----------------------------------------------------------------------------
# textbook special cases used as pins
# ----------------------------------------------------------------------------
def ssd_recurrent(q, k, v, log_alpha) -> np.ndarray:
    """Plain Mamba-2 / SSD scalar-decay recurrence: S_t = a_t S_{t-1} + v_t k_t^T, o_t = S_t q_t."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    alpha = np.exp(np.asarray(log_alpha, np.float64))
    S = np.zeros((v.shape[1], k.shape[1]))
    out = np.zeros((q.shape[0], v.shape[1]))
    for t in range(q.shape[0]):
        S = alpha[t] * S + np.outer(v[t], k[t])
        out[t] = S @ q[t]
    return out


def linear_attention_recurrent(q, k, v) -> np.ndarray:
    """Causal linear attention (study note §1-2): S_t = S_{t-1} + v_t k_t^T, o_t = S_t q_t."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    S = np.zeros((v.shape[1], k.shape[1]))
    out = np.zeros((q.shape[0], v.shape[1]))
    for t in range(q.shape[0]):
        S = S + np.outer(v[t], k[t])
        out[t] = S @ q[t]
    return out


# ----------------------------------------------------------------------------
# level states at a position (the state a forward hands to decoding)
# ----------------------------------------------------------------------------
def states_at(k, v, log_alpha, T_pos: int, Ls: int):
    """Level states of query position T_pos built from keys 0..T_pos-1.

    Returns (S [Ls, dv, dk], nonempty [Ls] bool); slot i is level i + 1.
    S^(l) = sum_{s in bucket l of T_pos} Gamma(T_pos - 1, s) v_s k_s^T, i.e.
    the buckets of T_pos decayed to the last token seen (T_pos - 1); the new
    token T_pos (level 0) is not included.
    """
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    cum = np.cumsum(np.asarray(log_alpha, np.float64))
    dv, dk = v.shape[1], k.shape[1]
    S = np.zeros((Ls, dv, dk))
    ne = np.zeros(Ls, dtype=bool)
    for lv, lo, hi in buckets(T_pos)[1:]:
        if lv > Ls:
            raise ValueError("Ls too small for this position")
        w = np.exp(cum[T_pos - 1] - cum[lo:hi])
        S[lv - 1] = (v[lo:hi] * w[:, None]).T @ k[lo:hi]
        ne[lv - 1] = True
    return S, ne
