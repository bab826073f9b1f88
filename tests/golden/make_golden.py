"""Writes the stored expected values under tests/golden/ by calling only the
oracle (oracle/).  The pages print no worked example of eviction or
re-basing values, so these fixtures are oracle outputs, pinned to the closed
form in tests/test_oracle.py::test_bookkeeping_closed_form_tiny and re-checked
against the live oracle by tests/test_golden.py.

Run from the repository root:  python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import rkv_oracle as O  # noqa: E402


def tiny_log(steps=200, capacity=32):
    rows, o, n = [], 0, 0
    for t in range(1, steps + 1):
        bk = O.bookkeep(o, n, 1, capacity)
        rows.append((t,) + bk.log())
        o, n = bk.origin, bk.fill
    return rows


def chunk_log(cs=(6,) * 12, capacity=32, origin=999_990, fill=20):
    rows, o, n = [], origin, fill
    for t, c in enumerate(cs, 1):
        bk = O.bookkeep(o, n, c, capacity)
        rows.append((t,) + bk.log())
        o, n = bk.origin, bk.fill
    return rows


def write(name, header, rows):
    with open(os.path.join(HERE, name), "w") as f:
        f.write(header)
        f.write("# step origin fill evicted first_slot\n")
        for r in rows:
            f.write(" ".join(str(x) for x in r) + "\n")


if __name__ == "__main__":
    write("tiny_bookkeeping.txt",
          "# Tiny workload: capacity 32, one token per step, 200 steps from an empty window.\n"
          "# Eviction and origin shift per the flowchart of 'Audio8 ASR Infinite: What It Actually\n"
          "# Takes to Listen Forever' (evict oldest pair, shift sliding origin forward).\n",
          tiny_log())
    write("chunk_bookkeeping.txt",
          "# Capacity 32, six tokens per step, starting at origin 999990 with 20 retained pairs.\n"
          "# Same passage; several pairs evicted per step once full.\n",
          chunk_log())
