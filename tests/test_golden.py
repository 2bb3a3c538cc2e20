"""Regression check of the oracle against the frozen fixture tests/golden/oracle_tiny.txt
(written by tests/golden/make_golden.py from the oracle itself; the oracle's real pins are in
test_oracle.py). A change to the oracle's arithmetic shows up here and must be justified by the
commit that regenerates the fixture."""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden  # noqa: E402


def _load():
    with open(os.path.join(HERE, "golden", "oracle_tiny.txt")) as f:
        lines = [l.strip() for l in f if l.strip() and not l.startswith("#")]
    out = {}
    for head, body in zip(lines[0::2], lines[1::2]):
        name, *shape = head.split()
        out[name] = np.array([float(v) for v in body.split()]).reshape([int(s) for s in shape])
    return out


def test_oracle_matches_frozen_fixture():
    frozen = _load()
    now = make_golden.compute()
    assert set(frozen) == set(now)
    for name, arr in now.items():
        ref = frozen[name]
        assert arr.shape == ref.shape, name
        err = np.linalg.norm(arr - ref) / np.linalg.norm(ref)
        assert err < 1e-10, f"{name}: relative difference {err:.3e}"
