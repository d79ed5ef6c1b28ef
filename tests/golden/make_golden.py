"""Writes the regression fixtures in this folder that are not printed on the pages.

Calls only ``oracle/``.  Run from the repository root:

    python tests/golden/make_golden.py

``nf4_levels_f32.txt``: the float32 NF4 table (hex bit patterns) the oracle
builds; tests compare the oracle against it so that an accidental change of
the table shows up.  It is a regression fixture, not an independent pin (the
pins are the invariants and the glossary page's worked example).
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import nf4  # noqa: E402


def main():
    lv = nf4.nf4_levels_f32()
    with open(os.path.join(HERE, "nf4_levels_f32.txt"), "w") as f:
        f.write("# float32 NF4 levels, index 0..15, hex bit patterns (written by make_golden.py from oracle/nf4.py)\n")
        f.write(" ".join("%08x" % int(v) for v in lv.view("uint32")) + "\n")


if __name__ == "__main__":
    main()
