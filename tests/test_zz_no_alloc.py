"""ne_attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (all of it already claimed by another allocator, or a fixed budget)
and so cannot provide a workspace.  It runs the same kernels as ne_attn_bwd
on the same inputs, only with its scratch in a fixed array inside the
library, so its gradients must equal ne_attn_bwd's bit for bit, call after
call; and it must refuse shapes whose scratch does not fit that array.
Needs an sm_103 GPU.

This file is named so that pytest collects it last.
"""
import pytest
import torch

import ne_inputs
from parity_util import custom_inputs, to_dev

pytestmark = pytest.mark.gpu
THETA = ne_inputs.ROPE_THETA


@pytest.fixture(scope="module")
def ne():
    import causal_gqa_attention_ne_gb300 as mod
    mod.load_library()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return mod


def _compare_once(ne, seed, B, T, Hq, Hkv, d):
    x = to_dev(custom_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=seed))
    o, lse = ne.attention_forward(x["q"], x["k"], x["v"], THETA)
    ref = ne.attention_backward(x["q"], x["k"], x["v"], o, lse, x["do"], THETA)
    got = tuple(torch.empty_like(t) for t in ref)
    ne.ne_attn_bwd_noalloc(x["q"], x["k"], x["v"], o, lse, x["do"], *got, THETA)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        assert torch.equal(a, b), f"{name} differs from the workspace backward"


def test_noalloc_matches_workspace_backward_on_two_calls(ne):
    # two calls in a row on different inputs, the larger shape first: a
    # stale read of scratch left by the first call would change the second
    # call's gradients
    _compare_once(ne, 902, B=3, T=517, Hq=12, Hkv=4, d=64)
    _compare_once(ne, 901, B=2, T=300, Hq=6, Hkv=2, d=64)


def test_noalloc_other_head_dims(ne):
    _compare_once(ne, 903, B=1, T=260, Hq=4, Hkv=2, d=32)
    _compare_once(ne, 904, B=1, T=260, Hq=4, Hkv=4, d=128)


def test_noalloc_rejects_shapes_beyond_its_scratch(ne):
    lib = ne.load_library()
    B, T, Hq, Hkv, d = 8, 4096, 8, 8, 128
    assert ne.ne_attn_bwd_workspace_size(B, T, Hq, Hkv, d) > ne.ne_attn_bwd_noalloc_max_scratch()
    y = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    p = y.data_ptr()
    rc = lib.ne_attn_bwd_noalloc(p, p, p, p, p, p, p, p, p, B, T, Hq, Hkv, d, THETA, None)
    assert rc == 10, ne.NE_STATUS.get(rc, rc)      # NE_ERR_TOO_LARGE, nothing launched
    assert ne.ne_attn_get_error() == 0
