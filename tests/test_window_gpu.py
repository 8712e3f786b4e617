"""Sliding-window attention (ne_attn_fwd_window / ne_attn_bwd_window): query t
sees keys t-W+1 .. t.  Checked against the float64 oracle with the same
tolerances as the causal path, at windows that cut tiles in the middle, at
W = 1, at W >= T (the causal result) and through W = 0 (bitwise the causal
entry points).  Needs an sm_103 GPU."""
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


def _run(ne, xd, W):
    q, k, v, do = xd["q"], xd["k"], xd["v"], xd["do"]
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, T, dtype=torch.float32, device="cuda")
    ne.ne_attn_fwd_window(q, k, v, o, lse, W, THETA)
    ws = torch.empty(ne.ne_attn_bwd_workspace_size(B, T, Hq, Hkv, d), dtype=torch.uint8,
                     device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ne.ne_attn_bwd_window(q, k, v, o, lse, do, dq, dk, dv, ws, W, THETA)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0
    return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}


@pytest.mark.parametrize("B,T,Hq,Hkv,d,W", [(1, 300, 6, 2, 64, 100), (2, 256, 4, 4, 32, 1),
                                             (1, 384, 12, 4, 64, 129), (1, 200, 4, 2, 128, 64),
                                             (2, 130, 8, 2, 32, 300), (1, 512, 12, 4, 64, 256),
                                             (1, 640, 3, 1, 64, 191)])
def test_window_matches_oracle(ne, B, T, Hq, Hkv, d, W):
    x = custom_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=1600 + T + W)
    got = _run(ne, to_dev(x), W)
    q, k, v, do = (ne_inputs.as_f64(x[n]) for n in ("q", "k", "v", "do"))
    ref = oracle.attn_bwd(q, k, v, do, THETA, window=W)
    compare(got, ref, q, k)


@pytest.mark.parametrize("B,T,Hq,Hkv,d,W", [(1, 384, 12, 4, 64, 129), (2, 300, 4, 2, 32, 64)])
def test_window_training_pair_matches_oracle(ne, B, T, Hq, Hkv, d, W):
    x = custom_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=1650 + T + W)
    xd = to_dev(x)
    q, k, v, do = xd["q"], xd["k"], xd["v"], xd["do"]
    ws = torch.zeros(ne.ne_attn_bwd_workspace_size(B, T, Hq, Hkv, d), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, T, dtype=torch.float32, device="cuda")
    ne.ne_attn_fwd_save(q, k, v, o, lse, ws, THETA, window=W)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ne.ne_attn_bwd_saved(q, k, v, o, lse, do, dq, dk, dv, ws, THETA, window=W)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0
    q64, k64, v64, do64 = (ne_inputs.as_f64(x[n]) for n in ("q", "k", "v", "do"))
    ref = oracle.attn_bwd(q64, k64, v64, do64, THETA, window=W)
    compare({"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}, ref, q64, k64)


def test_window_zero_is_the_causal_path(ne):
    x = to_dev(custom_inputs(B=2, T=300, Hq=6, Hkv=2, d=64, seed=1700))
    got = _run(ne, x, 0)
    o, lse = ne.attention_forward(x["q"], x["k"], x["v"], THETA)
    dq, dk, dv = ne.attention_backward(x["q"], x["k"], x["v"], o, lse, x["do"], THETA)
    torch.cuda.synchronize()
    for n, ref in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert torch.equal(got[n], ref), n


def test_window_long_context_sampled(ne):
    """T = 2048 with W = 300: most key tiles of a query tile lie outside the
    window and are skipped; the oracle checks two (batch, kv head) groups."""
    from parity_util import slice_gpu
    B, T, Hq, Hkv, d, W = 2, 2048, 8, 2, 128, 300
    x = custom_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=1800)
    got = _run(ne, to_dev(x), W)
    q, k, v, do = (ne_inputs.as_f64(x[n]) for n in ("q", "k", "v", "do"))
    G = Hq // Hkv
    for (b, j) in ((0, 0), (1, 1)):
        ref = oracle.attn_bwd(oracle.group_slice(q, b, j, G), oracle.group_slice(k, b, j, 1),
                              oracle.group_slice(v, b, j, 1), oracle.group_slice(do, b, j, G),
                              THETA, window=W)
        compare(slice_gpu(got, b, j, G), ref, oracle.group_slice(q, b, j, G),
                oracle.group_slice(k, b, j, 1))
