"""Log-linear Mamba-2 backward, oracle (NumPy float64; test infrastructure only).

The pages print no backward formulas.  They name the backward pass, and in
it the gradient of the lambda terms, as the hard part of an implementation
("Log-Linear Attention" study note §4-5 "Implementation notes" and §6
"Limitations"; gist.science (zh) summary §5, limitations).  What it computes
is therefore fixed by the forward alone: the exact gradient of

    O = (A . M) V,   A = Q K^T,   M = Gamma . H,
    Gamma(t, s) = exp(c_t - c_s),  c = cumsum(log_alpha),   H(t, s) = lam_t[level(t, s)]

(study note §3-4 "Parallel form", §3-5 mask composition; both masks are 0
above the diagonal), for an upstream gradient dO, written out by the chain
rule in dense T x T form:

    P  = A . M                    dV = P^T dO
    dP = (dO V^T) . causal        dA = dP . M       dQ = dA K      dK = dA^T Q
    dM = dP . A                   dH = dM . Gamma   dGamma = dM . H
    dlam_t[l] = sum over s <= t with level(t, s) = l of dH(t, s)
    dc_t      = sum_s dGamma(t, s) Gamma(t, s) - sum_t' dGamma(t', t) Gamma(t', t)
    dlog_alpha_r = sum over t >= r of dc_t         (c_t = sum_{r <= t} log_alpha_r)

``backward_dense`` is that definition; ``backward_query_rows`` and
``backward_key_rows`` evaluate the same entries for selected rows (long
sequences).  Pinned in tests by central finite differences of the forward
oracle and by homogeneity identities, not by retyping these formulas.
"""

from __future__ import annotations

import numpy as np

from .mamba2 import decay_matrix, hier_mask, level_array


def level_sums(dH: np.ndarray, L: int) -> np.ndarray:
    """dlam[t, l] = sum of dH[t, s] over the keys s <= t at level l of query t."""
    T = dH.shape[0]
    t_idx = np.arange(T)[:, None]
    s_idx = np.arange(T)[None, :]
    lv = np.broadcast_to(level_array(t_idx, s_idx), (T, T))
    rows = np.broadcast_to(t_idx, (T, T))
    causal = s_idx <= t_idx
    causal = np.broadcast_to(causal, (T, T))
    out = np.zeros((T, L), dtype=np.float64)
    np.add.at(out, (rows[causal], lv[causal]), dH[causal])
    return out


def cumsum_grad(dGamma: np.ndarray, Gamma: np.ndarray) -> np.ndarray:
    """dc_t for Gamma(t, s) = exp(c_t - c_s): c_t enters row t with + and column t with -."""
    X = dGamma * Gamma
    return X.sum(axis=1) - X.sum(axis=0)


def suffix_sums(dc: np.ndarray) -> np.ndarray:
    """dlog_alpha_r = sum_{t >= r} dc_t, the adjoint of c = cumsum(log_alpha)."""
    return np.cumsum(dc[::-1])[::-1].copy()


def backward_dense(q, k, v, log_alpha, lam, do):
    """Gradients (dq, dk, dv, dlog_alpha, dlam) of sum(O * do) for one (batch, head) slice."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    lam = np.asarray(lam, np.float64)
    T = q.shape[0]
    causal = np.tril(np.ones((T, T), dtype=bool))
    A = q @ k.T
    Gamma = decay_matrix(log_alpha)
    H = hier_mask(lam)
    M = Gamma * H
    P = A * M
    dv = P.T @ do
    dP = np.where(causal, do @ v.T, 0.0)
    dA = dP * M
    dq = dA @ k
    dk = dA.T @ q
    dM = dP * A
    dlam = level_sums(dM * Gamma, lam.shape[1])
    dla = suffix_sums(cumsum_grad(dM * H, Gamma))
    return dq, dk, dv, dla, dlam


def backward_dense_bh(q, k, v, log_alpha, lam, do):
    """backward_dense over leading [B, H] axes."""
    B, H = q.shape[:2]
    outs = [np.zeros(x.shape, np.float64) for x in (q, k, v, log_alpha, lam)]
    for b in range(B):
        for h in range(H):
            r = backward_dense(q[b, h], k[b, h], v[b, h], log_alpha[b, h], lam[b, h], do[b, h])
            for o, x in zip(outs, r):
                o[b, h] = x
    return tuple(outs)


def backward_query_rows(q, k, v, log_alpha, lam, do, rows):
    """dq_t, dlam_t and the row term of dc_t for query rows ``rows`` (one slice).

    Row t needs keys 0..t only: O(t d) per row.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    lam = np.asarray(lam, np.float64)
    cum = np.cumsum(np.asarray(log_alpha, np.float64))
    L = lam.shape[1]
    dq = np.zeros((len(rows), q.shape[1]))
    dlam = np.zeros((len(rows), L))
    row_term = np.zeros(len(rows))
    for i, t in enumerate(rows):
        t = int(t)
        s = np.arange(t + 1)
        a = k[: t + 1] @ q[t]
        g = v[: t + 1] @ do[t]
        gam = np.exp(cum[t] - cum[: t + 1])
        lv = level_array(t, s)
        h = lam[t, lv]
        dq[i] = (g * gam * h) @ k[: t + 1]
        dlam[i] = np.bincount(lv, weights=g * a * gam, minlength=L)
        row_term[i] = np.sum(g * a * gam * h)
    return dq, dlam, row_term


def backward_key_rows(q, k, v, log_alpha, lam, do, cols):
    """dk_s, dv_s and the column term of dc_s for key rows ``cols`` (one slice).

    Key s is seen by queries s..T-1: O((T - s) d) per row.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    lam = np.asarray(lam, np.float64)
    cum = np.cumsum(np.asarray(log_alpha, np.float64))
    T = q.shape[0]
    dk = np.zeros((len(cols), k.shape[1]))
    dv = np.zeros((len(cols), v.shape[1]))
    col_term = np.zeros(len(cols))
    for i, s in enumerate(cols):
        s = int(s)
        t = np.arange(s, T)
        a = q[s:] @ k[s]
        g = do[s:] @ v[s]
        gam = np.exp(cum[s:] - cum[s])
        h = lam[t, level_array(t, s)]
        dk[i] = (g * gam * h) @ q[s:]
        dv[i] = (a * gam * h) @ do[s:]
        col_term[i] = np.sum(g * a * gam * h)
    return dk, dv, col_term
