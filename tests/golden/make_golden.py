"""Writes the plan golden vectors in this folder.  Calls only the oracle.

The anchor-key hash is this library's own definition (the DFlash pages fix determinism in
(mask, sample ids, step, seed) but give no hash); these files freeze that definition so a
later change to it shows up as a test failure.

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import dflash_oracle as orc  # noqa: E402


def write(name, mask, sids, step, seed, N, S, note):
    p = orc.build_plan(mask, sids, step, seed, N, S)
    B, L = mask.shape
    with open(os.path.join(HERE, name), "w") as f:
        f.write(f"# {note}\n# written by make_golden.py from the oracle's build_plan\n")
        f.write(f"B={B} L={L} N={N} S={S} step={step} seed={seed}\n")
        for b in range(B):
            f.write(f"mask{b}: " + "".join(str(int(v)) for v in mask[b]) + "\n")
        for b in range(B):
            f.write(f"sid{b}: {int(sids[b])}\n")
        for b in range(B):
            f.write(f"anchors{b}: " + " ".join(str(int(a)) for a in p["anchors"][b]) + "\n")


def main():
    mask = np.ones((4, 40), np.uint8)
    mask[1, 25:] = 0
    mask[2, 1] = 0
    mask[2, 7:9] = 0
    mask[3, 1:] = 0
    write("plan_small.txt", mask, np.array([3, -5, 123456789012, 8], np.int64), 17, 0xD1F1A5,
          6, 4, "distinct sample ids; right padding, holes and a row with no window")
    mask = np.ones((5, 33), np.uint8)
    mask[3, 20:] = 0
    write("plan_shared_sid.txt", mask, np.array([42, 42, 7, 42, 7], np.int64), 0, 2 ** 64 - 1,
          5, 16, "rows 0,1,3 share a sample id, rows 2,4 share another; row 3 is shorter")


if __name__ == "__main__":
    main()
