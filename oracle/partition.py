"""Fenwick-tree prefix partition (oracle; test infrastructure only).

Source: "Log-Linear Attention" study note (dimensionstp.github.io), §2-2
"Design intuition" and §3-2 "Fenwick tree partitioning": the prefix of t is
split into power-of-two buckets, small (fine) buckets for recent tokens and
large (coarse) ones for distant tokens, at most O(log T) of them; §3-6 ties
the number of states to the significant bits of t.

Reading R1/R3: token t is its own bucket at level 0; the remaining prefix
[0, t) is peeled Fenwick-style from t downward, one lowest set bit at a time,
and a bucket of size 2**k gets level k + 1.  Two independent codings are
given: ``buckets`` (the peeling procedure) and ``level`` (a closed form).  The
tests check that they agree, which is the pin for both.
"""

from __future__ import annotations


def level(t: int, s: int) -> int:
    """Closed form of the level of key s as seen from query t (0 <= s <= t).

    0 when s == t; otherwise floor(log2(t xor s)) + 1: the highest bit where
    s and t differ is set in t and clear in s, and every key that shares the
    bits of t above it (and has that bit clear) sits in one bucket.
    """
    if s < 0 or s > t:
        raise ValueError("level(t, s) needs 0 <= s <= t")
    if s == t:
        return 0
    return (t ^ s).bit_length()  # == floor(log2(t ^ s)) + 1


def buckets(t: int) -> list[tuple[int, int, int]]:
    """Fenwick peeling of [0, t]: list of (level, lo, hi) with keys lo <= s < hi.

    The token itself first (level 0), then the prefix [0, t) from the nearest
    bucket to the farthest: x = t; repeatedly take the lowest set bit b of x,
    emit [x - b, x) at level log2(b) + 1 and clear that bit.
    """
    if t < 0:
        raise ValueError("t must be >= 0")
    out = [(0, t, t + 1)]
    x = t
    while x > 0:
        b = x & (-x)
        out.append((b.bit_length(), x - b, x))
        x -= b
    return out


def levels_needed(T: int) -> int:
    """Number of lambda levels a sequence of length T can touch (levels 0..max)."""
    if T <= 1:
        return 1
    return (T - 1).bit_length() + 1


def nonempty_levels(t: int) -> list[int]:
    """Levels >= 1 that hold keys for query t (bit l-1 of t is set)."""
    return [lv for (lv, lo, hi) in buckets(t)[1:]]
