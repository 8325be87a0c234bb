"""The chunk-wise backward that the CUDA kernels implement, restated in float64
NumPy and compared with the dense gradients of the oracle (CPU only).

The decomposition: per chunk the dense in-chunk gradients and its state;
Fenwick nodes F_e of the chunk states; the query side of every set bit h of a
chunk (node e, level log2(C)+1+h), which also fills the key-side node R_e
with that chunk's queries; the key side of every chunk from the R nodes of
the blocks that hold its keys; dc_t = sum_l lam_t[l] dlam_t[l] - v_t . dv_t
and its suffix sums.  This test checks that decomposition against the
definition; it shares nothing with the kernels but the reading."""

import numpy as np
import pytest

from oracle import backward
from oracle.mamba2 import level_array
from oracle.partition import levels_needed


def chunked_backward(q, k, v, la, lam, do, C):
    T, d = q.shape
    dv_ = v.shape[1]
    L = lam.shape[1]
    lc = int(np.log2(C))
    N = (T + C - 1) // C
    pad = N * C - T

    def padz(x):
        return np.concatenate([x, np.zeros((pad,) + x.shape[1:])]) if pad else x

    q, k, v, do, la = padz(q), padz(k), padz(v), padz(do), padz(la)
    lam = padz(lam)
    nv = [min(C, T - c * C) for c in range(N)]
    gq = np.zeros_like(q)
    gk = np.zeros_like(k)
    gv = np.zeros_like(v)
    glam = np.zeros((N * C, L))
    cs = [np.cumsum(la[c * C:(c + 1) * C]) for c in range(N)]     # per chunk, inclusive
    tot = np.array([cs[c][-1] for c in range(N)])
    cum = np.cumsum(tot)                                          # running chunk totals
    S = []
    # (1) intra
    for c in range(N):
        r = slice(c * C, (c + 1) * C)
        i_ = np.arange(C)[:, None]
        j_ = np.arange(C)[None, :]
        causal = (j_ <= i_) & (i_ < nv[c])
        lv = level_array(i_, j_)
        gam = np.where(causal, np.exp(cs[c][:, None] - cs[c][None, :]), 0.0)
        Hm = np.where(causal, lam[r][np.broadcast_to(i_, (C, C)), np.minimum(lv, L - 1)], 0.0)
        A = q[r] @ k[r].T
        G = do[r] @ v[r].T
        P = A * gam * Hm
        dA = G * gam * Hm
        gq[r] += dA @ k[r]
        gk[r] += dA.T @ q[r]
        gv[r] += P.T @ do[r]
        X = np.where(causal, G * A * gam, 0.0)
        for i in range(nv[c]):  # present rows only: their levels are below L
            for j in range(i + 1):
                glam[c * C + i, lv[i, j]] += X[i, j]
        w = np.exp(cs[c][-1] - cs[c])
        S.append((w[:, None] * v[r]).T @ k[r])
    # (2) Fenwick nodes: F_i = S_i + sum over children i - 2^m of exp(decay after the child) F_child
    F = [None] * N
    for i in range(N):
        acc = S[i].copy()
        m = 0
        while (i >> m) & 1:
            j = i - (1 << m)
            acc += np.exp(cum[i] - cum[j]) * F[j]
            m += 1
        F[i] = acc
    # (3) query side, filling the key-side nodes
    R = [np.zeros((dv_, d)) for _ in range(N)]
    for c in range(N):
        r = slice(c * C, (c + 1) * C)
        for h in range(32):
            if (c >> h) == 0:
                break
            if not (c >> h) & 1:
                continue
            e = ((c >> (h + 1)) << (h + 1)) + (1 << h) - 1
            wq = np.exp(cs[c] + (cum[c - 1] - cum[e]))             # decay from the end of e to row i
            wq[nv[c]:] = 0.0
            lw = wq * lam[r][:, lc + 1 + h]
            g = (do[r] @ F[e]) * wq[:, None]                      # exp(.) F_e^T do_i
            gq[r] += lam[r][:, lc + 1 + h][:, None] * g
            glam[r, lc + 1 + h] += np.sum(g * q[r], axis=1)
            R[e] += (lw[:, None] * do[r]).T @ q[r]
    # (4) key side
    for c in range(N):
        r = slice(c * C, (c + 1) * C)
        E = np.zeros((dv_, d))
        for h in range(31):
            if (c >> h) & 1:
                continue
            e = ((c >> (h + 1)) << (h + 1)) + (1 << h) - 1
            if e + 1 >= N:
                break
            E += np.exp(cum[e] - cum[c]) * R[e]
        wdec = np.exp(cs[c][-1] - cs[c])
        gv[r] += wdec[:, None] * (k[r] @ E.T)
        gk[r] += wdec[:, None] * (v[r] @ E)
    # (5) dc and its suffix sums
    dc = np.sum(lam * glam, axis=1) - np.sum(v * gv, axis=1)
    dla = np.cumsum(dc[::-1])[::-1]
    return gq[:T], gk[:T], gv[:T], dla[:T], glam[:T]


def _case(T, d, L, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, d)) / np.sqrt(d)
    k = rng.standard_normal((T, d)) / np.sqrt(d)
    v = rng.standard_normal((T, d))
    la = -np.log1p(np.exp(rng.standard_normal(T) + 1.0))
    lam = np.log1p(np.exp(rng.standard_normal((T, L))))
    do = rng.standard_normal((T, d))
    return q, k, v, la, lam, do


@pytest.mark.parametrize("T,C", [(64, 8), (100, 8), (257, 16), (33, 32), (1, 4)])
def test_chunked_backward_equals_the_definition(T, C):
    L = levels_needed(T)
    case = _case(T, 4, L, seed=T)
    got = chunked_backward(*case, C=C)
    want = backward.backward_dense(*case)
    for name, a, b in zip(("dq", "dk", "dv", "dlog_alpha", "dlam"), got, want):
        np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-9 * max(np.abs(b).max(), 1.0), err_msg=name)
