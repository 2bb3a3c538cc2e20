"""Writes the regression fixture `oracle_tiny.txt` from the fp64 oracle (oracle/ only; inputs
from the seeded generator module). The pages print no worked numeric example of the layer
(their numbers are model-level accuracies and speedups), so the oracle's pins are closed forms,
invariants and hand values (tests/test_oracle.py); this fixture only freezes the oracle's
output on one tiny case so that any later change to its arithmetic shows up as a diff that
the commit making it has to justify.

    python tests/golden/make_golden.py     # rewrites tests/golden/oracle_tiny.txt
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle as O  # noqa: E402


def tiny_case():
    """d = 8 inputs, m = 6 outputs, static rank k = 2, residual rank r = 2, two samples of
    five tokens; W, b and X from one PCG64 stream."""
    rng = np.random.Generator(np.random.PCG64(20261203))
    W = rng.standard_normal((8, 6))
    b = rng.standard_normal(6)
    X = rng.standard_normal((2, 5, 8))
    return W, b, X


def compute():
    W, b, X = tiny_case()
    prep = O.prepare(W, b, "lowrank", 2, 2)
    out = {"Y_cholesky": O.forward(X, prep, solver="cholesky"),
           "Y_newton_schulz_8": O.forward(X, prep, solver="newton_schulz", ns_iters=8),
           "Y_als_t2": O.forward_als(X, prep, 2.0),
           "W_hat": prep["W_hat"]}
    return out


def main():
    out = compute()
    lines = ["# oracle output on tests/golden/make_golden.py's tiny case (fp64, 17 significant digits)"]
    for name, arr in out.items():
        flat = np.asarray(arr, dtype=np.float64).ravel()
        lines.append(f"{name} {' '.join(str(s) for s in arr.shape)}")
        lines.append(" ".join(f"{v:.17g}" for v in flat))
    with open(os.path.join(HERE, "oracle_tiny.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
