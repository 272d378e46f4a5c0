"""Writes the stored expected values under tests/golden/ from the CPU oracle only.

Run from the repository root:  python tests/golden/make_golden.py
Outputs:
  nf4_table.txt  -- the 16 NF4 levels the oracle derives (hex float and decimal)
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import oracle  # noqa: E402


def main():
    L = oracle.nf4_table()
    with open(os.path.join(HERE, "nf4_table.txt"), "w") as f:
        f.write("# NF4 levels from the CPU oracle (N(0,1) quantiles with equal-share bins,\n")
        f.write("# 7 negative + exact 0 + 8 positive, each half normalised to +-1).\n")
        f.write(f"# outermost probability delta = {oracle.nf4_delta()!r}\n")
        f.write("# code  hex-float  decimal\n")
        for i, v in enumerate(L):
            f.write(f"{i:2d} {float(v).hex()} {float(v)!r}\n")


if __name__ == "__main__":
    main()
