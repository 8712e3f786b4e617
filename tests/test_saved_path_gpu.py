"""The training pair ne_attn_fwd_save / ne_attn_bwd_saved: the forward leaves
the rotated Q' and K' in the backward's workspace, the backward reuses them.
Checked against the oracle with the usual tolerances, and the stored Q' / K'
against the ones ne_attn_bwd_preprocess writes for the same inputs.  Needs an
sm_103 GPU."""
import numpy as np
import pytest
import torch

import ne_inputs
from parity_util import compare, custom_inputs, oracle_all, to_dev

pytestmark = pytest.mark.gpu
THETA = ne_inputs.ROPE_THETA


@pytest.fixture(scope="module")
def ne():
    import causal_gqa_attention_ne_gb300 as mod
    mod.load_library()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return mod


def _saved_pair(ne, xd):
    q, k, v, do = xd["q"], xd["k"], xd["v"], xd["do"]
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    ws = torch.zeros(ne.ne_attn_bwd_workspace_size(B, T, Hq, Hkv, d), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, T, dtype=torch.float32, device="cuda")
    ne.ne_attn_fwd_save(q, k, v, o, lse, ws, THETA)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ne.ne_attn_bwd_saved(q, k, v, o, lse, do, dq, dk, dv, ws, THETA)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0
    return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}, ws


def _rotated_views(ws, B, T, Hq, Hkv, d):
    def r256(x):
        return (x + 255) // 256 * 256
    off_q = r256(B * Hq * T * 4)
    off_k = off_q + r256(B * T * Hq * d * 2)
    qr = ws[off_q:off_q + B * T * Hq * d * 2].view(torch.float16).view(B, T, Hq, d)
    kr = ws[off_k:off_k + B * T * Hkv * d * 2].view(torch.float16).view(B, T, Hkv, d)
    return qr, kr


@pytest.mark.parametrize("B,T,Hq,Hkv,d", [(1, 300, 6, 2, 64), (2, 256, 4, 4, 32),
                                          (1, 384, 12, 4, 64), (1, 200, 4, 2, 128),
                                          (2, 128, 8, 2, 32)])
def test_saved_pair_matches_oracle(ne, B, T, Hq, Hkv, d):
    x = custom_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=1100 + T + d)
    got, _ = _saved_pair(ne, to_dev(x))
    ref, q64, k64 = oracle_all(x, THETA)
    compare(got, ref, q64, k64)


def test_saved_rotations_equal_the_preprocess(ne):
    B, T, Hq, Hkv, d = 2, 400, 6, 2, 64
    xd = to_dev(custom_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=1201))
    _, ws_saved = _saved_pair(ne, xd)
    o, _ = ne.attention_forward(xd["q"], xd["k"], xd["v"], THETA)
    ws_pre = torch.zeros_like(ws_saved)
    ne.ne_attn_bwd_preprocess(xd["q"], xd["k"], o, xd["do"], ws_pre, THETA)
    torch.cuda.synchronize()
    for a, b, n in zip(_rotated_views(ws_saved, B, T, Hq, Hkv, d),
                       _rotated_views(ws_pre, B, T, Hq, Hkv, d), ("Q'", "K'")):
        # one rotation routine with explicitly rounded operations: the same bits
        assert torch.equal(a, b), f"{n}: max diff {(a.float() - b.float()).abs().max().item():.3e}"


def test_saved_pair_rejects_short_workspace(ne):
    xd = to_dev(custom_inputs(B=1, T=64, Hq=2, Hkv=1, d=64, seed=1202))
    q, k, v = xd["q"], xd["k"], xd["v"]
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 64, dtype=torch.float32, device="cuda")
    ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ne.NeAttnError) as e:
        ne.ne_attn_fwd_save(q, k, v, o, lse, ws, THETA)
    assert e.value.status == 5   # NE_ERR_WORKSPACE, nothing launched


def test_saved_pair_matches_the_standalone_pair_with_many_units_per_cta(ne):
    # B64 T512 12/4 d64 (the bench layer): about seven work units per CTA, so
    # the next unit's Q' tiles are rotated and stored while a unit runs
    B, T, Hq, Hkv, d = 64, 512, 12, 4, 64
    xd = to_dev(custom_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=1203))
    got, _ = _saved_pair(ne, xd)
    o, lse = ne.attention_forward(xd["q"], xd["k"], xd["v"], THETA)
    dq, dk, dv = ne.attention_backward(xd["q"], xd["k"], xd["v"], o, lse, xd["do"], THETA)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0
    assert torch.equal(got["o"], o) and torch.equal(got["lse"], lse)
    # the forward's rotation and the preprocess's give the same Q', K' bits,
    # and both preprocess kernels sum D in the same order
    for n, a, b in (("dq", got["dq"], dq), ("dk", got["dk"], dk), ("dv", got["dv"], dv)):
        assert torch.equal(a, b), n
