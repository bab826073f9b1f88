"""Stored oracle fixtures under tests/golden/ stay what the oracle and the
closed form say."""
import os

from oracle import rkv_oracle as O

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    with open(os.path.join(HERE, name)) as f:
        return [tuple(int(x) for x in line.split()) for line in f if not line.startswith("#")]


def test_tiny_fixture_closed_form():
    for t, o, n, e, slot in _rows("tiny_bookkeeping.txt"):
        assert (o, n, e, slot) == (max(0, t - 32), min(t, 32), int(t >= 33), (t - 1) % 32)


def test_chunk_fixture_matches_oracle():
    o, n = 999_990, 20
    for t, o2, n2, e, slot in _rows("chunk_bookkeeping.txt"):
        bk = O.bookkeep(o, n, 6, 32)
        assert bk.log() == (o2, n2, e, slot)
        # closed form: positions are contiguous, so origin' + fill' = origin + fill + 6
        assert o2 + n2 == o + n + 6 and n2 == min(32, n + 6) and slot == (o + n) % 32
        o, n = o2, n2
