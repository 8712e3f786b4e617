"""Decode against a key/value cache (ne_attn_decode) against the float64
oracle: one new token per sequence at position Tk - 1 over Tk cached keys,
i.e. the last row of causal attention.  Tolerances as for the forward (O
norm-wise relative error <= 1e-2, lse absolute error <= 1e-3).  Needs an
sm_103 GPU."""
import numpy as np
import pytest
import torch

import ne_inputs
import oracle
from parity_util import TOL_LSE, TOL_O, custom_inputs, rel_err

pytestmark = pytest.mark.gpu
THETA = ne_inputs.ROPE_THETA


@pytest.fixture(scope="module")
def ne():
    import causal_gqa_attention_ne_gb300 as mod
    mod.load_library()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return mod


def _case(B, Tk, Hq, Hkv, d, seed):
    x = custom_inputs(B=B, T=Tk, Hq=Hq, Hkv=Hkv, d=d, seed=seed)
    q1 = x["q"][:, -1].contiguous()          # [B, Hq, d]: the new token's query
    return q1, x["k"], x["v"]


@pytest.mark.parametrize("B,Tk,Hq,Hkv,d", [(2, 300, 6, 2, 64), (1, 1, 4, 2, 32),
                                           (3, 129, 8, 2, 128), (2, 1000, 12, 4, 64),
                                           (1, 513, 16, 1, 128), (4, 64, 4, 4, 32)])
def test_decode_matches_oracle(ne, B, Tk, Hq, Hkv, d):
    q1, k, v = _case(B, Tk, Hq, Hkv, d, 1400 + Tk + d)
    o, lse = ne.attention_decode(q1.cuda(), k.cuda(), v.cuda(), THETA)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0
    ro, rl = oracle.attn_decode(*(ne_inputs.as_f64(t) for t in (q1, k, v)), THETA)
    err = rel_err(o.float().cpu().numpy(), ro)
    lerr = float(np.abs(lse.cpu().double().numpy() - rl).max())
    assert err <= TOL_O, f"o: {err:.3e}"
    assert lerr <= TOL_LSE, f"lse: {lerr:.3e}"


def test_decode_is_deterministic_and_reuses_its_workspace(ne):
    q1, k, v = (t.cuda() for t in _case(2, 777, 12, 4, 64, 1500))
    ws = torch.full((ne.ne_attn_decode_workspace_size(2, 777, 12, 4, 64),), 0x7f,
                    dtype=torch.uint8, device="cuda")
    o1, l1 = ne.attention_decode(q1, k, v, THETA, workspace=ws)
    o2, l2 = ne.attention_decode(q1, k, v, THETA, workspace=ws)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_at_the_116m_chat_shape_sampled(ne):
    # the decode workload of the bench (B64, Tk 512, 12/4 heads, d64), checked
    # against the oracle on a sample of sequences
    q1, k, v = _case(64, 512, 12, 4, 64, 1501)
    o, lse = ne.attention_decode(q1.cuda(), k.cuda(), v.cuda(), THETA)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0
    rows = [0, 17, 42, 63]
    ro, rl = oracle.attn_decode(*(ne_inputs.as_f64(t[rows]) for t in (q1, k, v)), THETA)
    assert rel_err(o[rows].float().cpu().numpy(), ro) <= TOL_O
    assert float(np.abs(lse[rows].cpu().double().numpy() - rl).max()) <= TOL_LSE


def test_decode_long_cache(ne):
    # 4096 cached positions: 32 chunks merged per (b, h)
    q1, k, v = _case(2, 4096, 16, 4, 128, 1502)
    o, lse = ne.attention_decode(q1.cuda(), k.cuda(), v.cuda(), THETA)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0
    ro, rl = oracle.attn_decode(*(ne_inputs.as_f64(t) for t in (q1, k, v)), THETA)
    assert rel_err(o.float().cpu().numpy(), ro) <= TOL_O
    assert float(np.abs(lse.cpu().double().numpy() - rl).max()) <= TOL_LSE
