"""The CPU oracle against its pins (closed forms, invariants, finite differences,
torch's attention routine).  CPU only."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_group_slice_matches_full(orc):
    """The oracle on one (batch, kv head) group equals that slice of the full run."""
    import ne_inputs
    x = ne_inputs.make_custom(B=2, T=21, Hq=6, Hkv=3, d=8, seed=81)
    q, k, v, do = (ne_inputs.as_f64(x[n]) for n in ("q", "k", "v", "do"))
    full = orc.attn_bwd(q, k, v, do, ne_inputs.ROPE_THETA)
    G = 2
    b, j = 1, 2
    part = orc.attn_bwd(oracle.group_slice(q, b, j, G), oracle.group_slice(k, b, j, 1),
                        oracle.group_slice(v, b, j, 1), oracle.group_slice(do, b, j, G),
                        ne_inputs.ROPE_THETA)
    for n, hp in (("dq", G), ("dk", 1), ("dv", 1), ("o", G)):
        assert (part[n] == oracle.group_slice(full[n], b, j, hp)).all()


def test_rejects_bad_shapes(orc):
    import numpy as np
    with pytest.raises(ValueError):
        orc.attn_fwd(np.zeros((1, 4, 3, 8)), np.zeros((1, 4, 2, 8)), np.zeros((1, 4, 2, 8)),
                     10000.0)
