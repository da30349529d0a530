"""Writes tests/golden/oracle_d4_T6.txt by calling the oracle only.

The pages print no worked example, so this fixture is a regression guard for
the oracle itself: a change to the oracle's arithmetic shows up as a failing
fixture comparison.  Inputs are small hand-picked decimals (exactly
representable up to fp64 rounding of the decimal literals).

Run from the repository root: ``python tests/golden/make_golden.py``.
"""

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402

d, T, lam = 4, 6, 0.5
q = np.array([[0.5, -1.0, 0.25, 2.0], [-0.75, 0.5, 1.5, -0.25], [1.0, 1.0, -1.0, 0.0],
              [0.0, -2.0, 0.5, 0.75], [-1.25, 0.25, 0.0, 1.0], [0.5, 0.5, 0.5, -0.5]])
k = np.array([[1.0, 0.0, 2.0, -1.0], [0.5, -1.5, 0.0, 1.0], [-2.0, 1.0, 1.0, 0.5],
              [0.25, 0.25, -1.0, 2.0], [1.5, -0.5, 0.75, 0.0], [-1.0, -1.0, 1.0, 1.0]])
v = np.array([[2.0, -1.0, 0.5, 0.0], [0.0, 1.0, -1.0, 1.5], [1.0, 0.25, 0.75, -2.0],
              [-0.5, 0.5, 2.0, 1.0], [1.25, -1.25, 0.0, 0.5], [0.5, 2.0, -0.5, -1.0]])
u = np.array([[0.5, 1.0, 0.0, -0.5], [1.0, -0.5, 0.5, 0.0], [0.0, 0.25, -1.0, 1.0],
              [-0.75, 0.0, 0.5, 0.5], [0.25, 0.5, 0.25, -1.0], [1.0, 1.0, -0.5, 0.25]])
r = oracle.forward(q, k, v, u, lam, nthreads=1)


def row(name, a):
    return "%s: %s\n" % (name, " ".join(repr(float(x)) for x in np.ravel(a)))


out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_d4_T6.txt")
with open(out, "w") as f:
    f.write("# VLA forward recurrence, d=4, T=6, lambda0=0.5, A0 = I/lambda0, S0 = 0, n0 = 0.\n")
    f.write("# Written by tests/golden/make_golden.py from the fp64 oracle (regression\n")
    f.write("# fixture; the pages print no worked example).  Arrays are row-major.\n")
    f.write(row("lambda0", [lam]))
    for nm, a in (("q", q), ("k", k), ("v", v), ("u", u)):
        f.write(row(nm, a))
    for nm in ("o", "S_T", "A_T", "n_T"):
        f.write(row(nm, r[nm]))
print("wrote", out)
