"""Writes the stored expected values under tests/golden/ by calling only the oracle.

    python tests/golden/make_golden.py
"""
import hashlib
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def main():
    g = oracle.iq2_grid()
    with open(os.path.join(HERE, "iq2_grid.txt"), "w") as f:
        f.write("# the library's IQ2-style grid: 256 entries x 8 magnitudes, written by make_golden.py\n")
        f.write("# sha256 of the 2048 bytes: %s\n" % hashlib.sha256(g.tobytes()).hexdigest())
        for e in range(256):
            f.write(" ".join(str(int(v)) for v in g[e]) + "\n")


if __name__ == "__main__":
    main()
