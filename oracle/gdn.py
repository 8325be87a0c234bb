"""Log-linear Gated DeltaNet forward, oracle (NumPy float64; test infrastructure only).

The pages name the variant but print no delta-rule equations: the study note
(dimensionstp.github.io) §3-5 says Log-Linear Gated DeltaNet lifts Gated
DeltaNet by composing its temporal mask with M^H (M = M^S . M^H), and the
gist.science (de) Technische Zusammenfassung §2 says the delta rule is
combined with the hierarchical structure.  Reading R7 fills the gap with the
standard gated delta rule

    S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t.

Unrolled, o_t = sum_{s <= t} c(t, s) v_s with

    C = (Q K^T . Gamma . causal) (I + diag(beta) SL(K K^T . Gamma))^{-1} diag(beta),

SL = strictly lower part, Gamma = M^S.  (Derivation: with the pseudo-values
u_t = beta_t (v_t - alpha_t S_{t-1} k_t) the state is S_t = sum_s Gamma(t,s)
u_s k_s^T, and u solves (I + diag(beta) SL(K K^T . Gamma)) U = diag(beta) V.)

  reading A (the one the GPU path implements): O = (C . M^H) V.  Every
      Fenwick level state follows the full gated-delta transition; the new
      write goes to level 0; merging is addition.
  reading B: O = (Q K^T . Gamma . M^H) (I + ...)^{-1} diag(beta) V, i.e.
      log-linear Mamba-2 applied to the delta-rule pseudo-values.
The pages do not decide between A and B: that parity is unpinned by the pages.
"""

from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular

from .mamba2 import decay_matrix, hier_mask, level_array


def _system(k, beta, log_alpha):
    """L = I + diag(beta) SL(K K^T . Gamma) (unit lower triangular) and Gamma."""
    k = np.asarray(k, np.float64)
    beta = np.asarray(beta, np.float64)
    G = decay_matrix(log_alpha)
    KK = (k @ k.T) * G
    L = np.eye(k.shape[0]) + beta[:, None] * np.tril(KK, -1)
    return L, G


def gdn_coeff(q, k, beta, log_alpha) -> np.ndarray:
    """C = (Q K^T . Gamma . causal) L^{-1} diag(beta)  ([T, T], lower triangular)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    L, G = _system(k, beta, log_alpha)
    A = (q @ k.T) * G  # G is zero above the diagonal
    # X = A L^{-1}  <=>  L^T X^T = A^T
    X = solve_triangular(L.T, A.T, lower=False, unit_diagonal=True).T
    return X * np.asarray(beta, np.float64)[None, :]


def gdn_forward_A(q, k, v, beta, log_alpha, lam) -> np.ndarray:
    """Reading A: O = (C . M^H) V for one (batch, head) slice."""
    C = gdn_coeff(q, k, beta, log_alpha)
    return (C * hier_mask(lam)) @ np.asarray(v, np.float64)


def gdn_forward_B(q, k, v, beta, log_alpha, lam) -> np.ndarray:
    """Reading B: O = (Q K^T . Gamma . M^H) L^{-1} diag(beta) V."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    L, G = _system(k, beta, log_alpha)
    U = solve_triangular(L, np.asarray(beta, np.float64)[:, None] * v, lower=True, unit_diagonal=True)
    return ((q @ k.T) * G * hier_mask(lam)) @ U


def gdn_rows_A(q, k, v, beta, log_alpha, lam, rows) -> np.ndarray:
    """Reading A evaluated for selected query rows only (long sequences).

    Row t of C is a_t L^{-1} diag(beta) with a_t = row t of (Q K^T . Gamma);
    it needs keys 0..t only, so row t is solved on the leading (t+1) block.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    lam = np.asarray(lam, np.float64)
    beta = np.asarray(beta, np.float64)
    cum = np.cumsum(np.asarray(log_alpha, np.float64))
    tmax = int(max(rows)) + 1
    L, _ = _system(k[:tmax], beta[:tmax], log_alpha[:tmax])
    out = np.zeros((len(rows), v.shape[1]))
    for i, t in enumerate(rows):
        t = int(t)
        a = (k[: t + 1] @ q[t]) * np.exp(cum[t] - cum[: t + 1])
        c = solve_triangular(L[: t + 1, : t + 1].T, a, lower=False, unit_diagonal=True) * beta[: t + 1]
        c = c * lam[t, level_array(t, np.arange(t + 1))]
        out[i] = c @ v[: t + 1]
    return out


def gdn_recurrent(q, k, v, beta, log_alpha) -> np.ndarray:
    """Textbook single-state gated delta rule, token by token."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    alpha = np.exp(np.asarray(log_alpha, np.float64))
    dv, dk = v.shape[1], k.shape[1]
    S = np.zeros((dv, dk))
    out = np.zeros((q.shape[0], dv))
    I = np.eye(dk)
    for t in range(q.shape[0]):
        S = alpha[t] * S @ (I - beta[t] * np.outer(k[t], k[t])) + beta[t] * np.outer(v[t], k[t])
        out[t] = S @ q[t]
    return out


def gdn_level_step(states: dict, t: int, q, k, v, beta: float, log_alpha: float, lam) -> np.ndarray:
    """One token of reading A over the Fenwick level states of query t.

    `states` maps level -> true state (d_v x d_k) for the non-empty levels of
    position t (levels >= 1), each after the transition of token t - 1, and
    is updated in place to the states of position t + 1.  Every level is
    right-multiplied by alpha_t (I - beta_t k_t k_t^T); level 0 receives
    beta_t v_t k_t^T; o_t = sum_l lam[l] S^(l) q_t; then the carry merges
    levels 0..j (j = trailing ones of t) into level j + 1 by addition.
    Returns o_t.
    """
    dk = k.shape[0]
    P = np.exp(log_alpha) * (np.eye(dk) - beta * np.outer(k, k))
    for lv in list(states):
        states[lv] = states[lv] @ P
    states[0] = beta * np.outer(v, k)
    o = np.zeros(v.shape[0])
    for lv, S in states.items():
        o += lam[lv] * (S @ q)
    j = 0
    while (t >> j) & 1:
        j += 1
    merged = states.pop(0)
    for lv in range(1, j + 1):
        merged = merged + states.pop(lv)
    assert (j + 1) not in states
    states[j + 1] = merged
    return o


def gdn_recurrent_levels_A(q, k, v, beta, log_alpha, lam):
    """Reading A as a recurrence over Fenwick level states, from position 0
    (gdn_level_step for every token).  Returns (O, final states dict)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    lam = np.asarray(lam, np.float64)
    log_alpha = np.asarray(log_alpha, np.float64)
    beta = np.asarray(beta, np.float64)
    states: dict = {}
    out = np.zeros((q.shape[0], v.shape[1]))
    for t in range(q.shape[0]):
        out[t] = gdn_level_step(states, t, q[t], k[t], v[t], float(beta[t]), float(log_alpha[t]), lam[t])
    return out, states


def gdn_decode_steps(S0, nonempty0, t0: int, q, k, v, beta, log_alpha, lam):
    """Run len(q) Gated DeltaNet (reading A) decode steps from position t0.

    S0 [Ls, dv, dk] true states, slot i = level i + 1, nonempty0 [Ls] (must be
    the set bits of t0); q, k [n, dk]; v [n, dv]; beta, log_alpha [n];
    lam [n, Ls + 1] (lam[:, 0] weights the token itself).
    Returns (o [n, dv], S [Ls, dv, dk], nonempty [Ls]) after the last step.
    """
    from .decode import states_from_array, states_to_array

    Ls = S0.shape[0]
    expect = [(t0 >> (lv - 1)) & 1 == 1 for lv in range(1, Ls + 1)]
    if list(map(bool, nonempty0)) != expect:
        raise ValueError("non-empty levels must be the set bits of t0")
    states = states_from_array(S0, nonempty0)
    n = q.shape[0]
    out = np.zeros((n, np.asarray(v).shape[1]))
    for i in range(n):
        out[i] = gdn_level_step(states, t0 + i, np.asarray(q[i], np.float64), np.asarray(k[i], np.float64),
                                np.asarray(v[i], np.float64), float(beta[i]), float(log_alpha[i]),
                                np.asarray(lam[i], np.float64))
    S, ne = states_to_array(states, Ls, np.asarray(v).shape[1], np.asarray(k).shape[1])
    return out, S, ne
