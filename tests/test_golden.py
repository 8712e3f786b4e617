"""The oracle against its stored outputs on one tiny GQA + RoPE case
(tests/golden/tiny_gqa_rope.txt, written by tests/golden/make_golden.py,
which calls only the oracle).  A regression pin: the independent pins are in
oracle_pins.py; this one fails when the oracle's arithmetic changes at all.
The tolerance (1e-12 relative) allows last-place differences between C math
libraries.  CPU only."""
import os
import sys

import numpy as np

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
sys.path.insert(0, HERE)

import make_golden  # noqa: E402


def load():
    out = {}
    with open(os.path.join(HERE, "tiny_gqa_rope.txt")) as f:
        lines = [ln for ln in f.read().splitlines() if ln and not ln.startswith("#")]
    for head, vals in zip(lines[::2], lines[1::2]):
        name, *shape = head.split()
        out[name] = np.array([float(x) for x in vals.split()]).reshape([int(s) for s in shape])
    return out


def test_oracle_matches_stored_outputs():
    stored = load()
    got = make_golden.compute()
    assert sorted(stored) == sorted(got)
    for name, ref in stored.items():
        g = got[name]
        assert g.shape == ref.shape, name
        den = np.abs(ref).max()
        assert np.abs(g - ref).max() <= 1e-12 * den, name
