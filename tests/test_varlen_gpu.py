"""Padded variable-length batches (ne_attn_fwd_varlen / ne_attn_bwd_varlen):
sequence b is its first L_b rows.  Valid rows are checked against the float64
oracle with the causal path's tolerances; padding rows must be exactly
O = 0, lse = -inf and zero gradients (outputs start as NaN, so a row the
library never writes fails).  Also: all lengths T is bitwise the causal entry
points, the padding contents do not change a valid bit, repeated calls are
bitwise equal, and the 116M SFT step's shape is sampled.  Needs an sm_103 GPU."""
import numpy as np
import pytest
import torch

import ne_inputs
import oracle
from parity_util import compare, custom_inputs, to_dev

pytestmark = pytest.mark.gpu
THETA = ne_inputs.ROPE_THETA


@pytest.fixture(scope="module")
def ne():
    import causal_gqa_attention_ne_gb300 as mod
    mod.load_library()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return mod


def _run(ne, xd, lens):
    q, k, v, do = xd["q"], xd["k"], xd["v"], xd["do"]
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    nan = float("nan")
    ws = torch.empty(ne.ne_attn_varlen_workspace_size(B, T, Hq, Hkv, d), dtype=torch.uint8,
                     device="cuda")
    o = torch.full_like(q, nan)
    lse = torch.full((B, Hq, T), nan, dtype=torch.float32, device="cuda")
    ne.ne_attn_fwd_varlen(q, k, v, o, lse, lens, ws, THETA)
    dq, dk, dv = (torch.full_like(x, nan) for x in (q, k, v))
    ne.ne_attn_bwd_varlen(q, k, v, o, lse, do, dq, dk, dv, lens, ws, THETA)
    torch.cuda.synchronize()
    status = ne.ne_attn_get_error()
    assert status == 0, f"device status {ne.NE_STATUS.get(status, status)}"
    return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}


def _check_padding(got, lens):
    for b, L in enumerate(lens):
        for n in ("o", "dq", "dk", "dv"):
            assert (got[n][b, L:] == 0).all(), (n, b, "padding rows not zero")
        assert torch.isneginf(got["lse"][b, :, L:]).all(), (b, "padding lse not -inf")


def _check_sequences(got, x, lens, which):
    """Oracle on the prefix of each sequence in `which` (a B = 1 causal problem)."""
    q, k, v, do = (ne_inputs.as_f64(x[n]) for n in ("q", "k", "v", "do"))
    for b in which:
        L = lens[b]
        if L == 0:
            continue
        sl = (slice(b, b + 1), slice(0, L))
        ref = oracle.attn_bwd(q[sl], k[sl], v[sl], do[sl], THETA)
        g = {n: got[n][sl] for n in ("o", "dq", "dk", "dv")}
        g["lse"] = got["lse"][b:b + 1, :, :L]
        compare(g, ref, q[sl], k[sl])


@pytest.mark.parametrize("B,T,Hq,Hkv,d,lens", [
    (5, 300, 12, 4, 64, [300, 0, 1, 129, 128]),
    (4, 256, 8, 2, 32, [5, 256, 200, 64]),
    (3, 200, 4, 2, 128, [200, 77, 130]),
    (3, 384, 6, 2, 64, [383, 256, 257]),
    (2, 130, 3, 1, 64, [2, 129]),
    (3, 520, 16, 4, 128, [520, 391, 9]),
])
def test_varlen_matches_oracle(ne, B, T, Hq, Hkv, d, lens):
    x = custom_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=2100 + T + Hq)
    got = _run(ne, to_dev(x), lens)
    _check_padding(got, lens)
    _check_sequences(got, x, lens, range(B))


def test_varlen_all_full_is_the_causal_path(ne):
    """Every length T: the unit tables are the full enumerations in launch
    order, so the results are the causal entry points' bit for bit."""
    x = to_dev(custom_inputs(B=3, T=300, Hq=12, Hkv=4, d=64, seed=2200))
    got = _run(ne, x, [300, 300, 300])
    o, lse = ne.attention_forward(x["q"], x["k"], x["v"], THETA)
    dq, dk, dv = ne.attention_backward(x["q"], x["k"], x["v"], o, lse, x["do"], THETA)
    torch.cuda.synchronize()
    for n, ref in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert torch.equal(got[n], ref), n


def test_varlen_padding_contents_do_not_matter(ne):
    """Other (finite) values in the padding rows of q, k, v and dO leave every
    output bit unchanged: masked probabilities are exact zeros."""
    lens = [150, 300, 1, 257]
    x = custom_inputs(B=4, T=300, Hq=6, Hkv=2, d=64, seed=2300)
    y = custom_inputs(B=4, T=300, Hq=6, Hkv=2, d=64, seed=2301)
    for b, L in enumerate(lens):
        for n in ("q", "k", "v", "do"):
            y[n][b, :L] = x[n][b, :L]
    a = _run(ne, to_dev(x), lens)
    c = _run(ne, to_dev(y), lens)
    for n in ("o", "lse", "dq", "dk", "dv"):
        assert torch.equal(a[n], c[n]), n


def test_varlen_sft_step_shape_sampled(ne):
    """The 116M SFT step's layer shape (B = 64 padded to 512, 12/4 heads,
    d = 64) with its seeded lengths, in the launch configuration the benchmark
    times: padding exact everywhere, four sequences against the oracle, and
    a second call bitwise equal (no atomics)."""
    w = ne_inputs.SFT_116M
    lens = w.seqlens()
    x = ne_inputs.make_inputs(w)
    xd = to_dev(x)
    got = _run(ne, xd, lens)
    _check_padding(got, lens)
    order = np.argsort(lens)
    _check_sequences(got, x, lens, [int(order[0]), int(order[len(lens) // 2]),
                                    int(order[-1]), 5])
    again = _run(ne, xd, lens)
    for n in ("o", "lse", "dq", "dk", "dv"):
        assert torch.equal(got[n], again[n]), n
