"""Pins for the Fenwick partition (oracle/partition.py)."""

import json
import os

import numpy as np
import pytest

from oracle import partition
from oracle.mamba2 import level_array

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_golden_buckets():
    with open(os.path.join(GOLDEN, "fenwick_buckets.json")) as f:
        g = json.load(f)
    for t, want in g["cases"].items():
        assert partition.buckets(int(t)) == [tuple(x) for x in want], t


def test_peeling_equals_closed_form_exhaustive():
    # two independent codings of the partition agree for every pair s <= t < 512
    for t in range(512):
        lv = np.full(t + 1, -1)
        for level, lo, hi in partition.buckets(t):
            assert (lv[lo:hi] == -1).all(), "buckets overlap"
            lv[lo:hi] = level
        assert (lv >= 0).all(), "buckets do not cover [0, t]"
        closed = [partition.level(t, s) for s in range(t + 1)]
        assert list(lv) == closed, t
        assert list(level_array(t, np.arange(t + 1))) == closed, t


def test_bucket_sizes_sum_and_powers_of_two():
    for t in range(2048):
        bs = partition.buckets(t)
        assert sum(hi - lo for _, lo, hi in bs) == t + 1
        assert len(bs) == 1 + bin(t).count("1")
        for level, lo, hi in bs[1:]:
            assert hi - lo == 2 ** (level - 1)
        # fine (recent) buckets first, coarse (distant) last
        sizes = [hi - lo for _, lo, hi in bs[1:]]
        assert sizes == sorted(sizes)
        his = [hi for _, lo, hi in bs]
        assert his == sorted(his, reverse=True)


@pytest.mark.parametrize("T,L", [(64, 7), (2048, 12), (16384, 15), (4096, 13), (65536, 17)])
def test_levels_needed_matches_workload_L(T, L):
    # the L of each workload equals the number of levels a length-T sequence touches
    assert partition.levels_needed(T) == L
    assert max(partition.level(T - 1, s) for s in (0, T // 2, T - 2)) == L - 1


def test_nonempty_levels_are_bits():
    for t in range(1, 300):
        want = [b + 1 for b in range(t.bit_length()) if (t >> b) & 1]
        assert sorted(partition.nonempty_levels(t)) == want


def test_level_rejects_bad_args():
    with pytest.raises(ValueError):
        partition.level(3, 4)
    with pytest.raises(ValueError):
        partition.buckets(-1)
