"""Fenwick decoding, oracle (NumPy float64; test infrastructure only).

Sources: "Log-Linear Attention" study note (dimensionstp.github.io) §3-6
"Memory-efficient decoding" (O(log T) states, tied to the significant bits
of the binary representation of t) and the drawer analogy of the gist.science
(zh) summary (a new token goes into drawer 0; a full drawer is merged into the
next one), with the output rule of §3-3.

The oracle keeps true (eagerly decayed) states.  A GPU implementation may
keep a lazily applied per-level scale g (reading R9); the comparison is then
against g * S_stored.
"""

from __future__ import annotations

import numpy as np

from .mamba2 import fenwick_step


def states_from_array(S: np.ndarray, nonempty: np.ndarray) -> dict:
    """[Ls, dv, dk] + [Ls] bool -> {level: state}; slot i is level i + 1."""
    return {i + 1: np.asarray(S[i], np.float64).copy() for i in range(S.shape[0]) if nonempty[i]}


def states_to_array(states: dict, Ls: int, dv: int, dk: int):
    S = np.zeros((Ls, dv, dk))
    ne = np.zeros(Ls, dtype=bool)
    for lv, M in states.items():
        if lv == 0 or lv > Ls:
            raise ValueError(f"level {lv} cannot be stored in {Ls} slots")
        S[lv - 1] = M
        ne[lv - 1] = True
    return S, ne


def decode_steps(S0, nonempty0, t0: int, q, k, v, log_alpha, lam):
    """Run len(q) decode steps from position t0.

    S0 [Ls, dv, dk], nonempty0 [Ls]: the states of query t0 (decayed to t0-1);
    q, k [n, dk]; v [n, dv]; log_alpha [n]; lam [n, Ls + 1].
    Returns (o [n, dv], S [Ls, dv, dk], nonempty [Ls]) after the last step.
    """
    Ls = S0.shape[0]
    expect = [(t0 >> (lv - 1)) & 1 == 1 for lv in range(1, Ls + 1)]
    if list(map(bool, nonempty0)) != expect:
        raise ValueError("non-empty levels must be the set bits of t0")
    states = states_from_array(S0, nonempty0)
    n = q.shape[0]
    out = np.zeros((n, v.shape[1]))
    for i in range(n):
        out[i] = fenwick_step(states, t0 + i, np.asarray(q[i], np.float64), np.asarray(k[i], np.float64),
                              np.asarray(v[i], np.float64), float(log_alpha[i]), np.asarray(lam[i], np.float64))
    S, ne = states_to_array(states, Ls, v.shape[1], k.shape[1])
    return out, S, ne
