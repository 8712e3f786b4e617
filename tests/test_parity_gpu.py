"""CUDA path (through the C ABI) against the float64 oracle on the same seeded
inputs: every workload shape, ragged and tiny T, every supported head dim and
several GQA ratios.  Needs an sm_103 GPU."""
import numpy as np
import pytest
import torch

import ne_inputs
from parity_util import compare, custom_inputs, gpu_fwd_bwd, oracle_all, slice_gpu, to_dev

pytestmark = pytest.mark.gpu
THETA = ne_inputs.ROPE_THETA


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import causal_gqa_attention_ne_gb300 as ne
    ne.load_library()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield


def _full_case(x):
    gpu = gpu_fwd_bwd(to_dev(x), THETA)
    ref, q64, k64 = oracle_all(x, THETA)
    return compare(gpu, ref, q64, k64)


@pytest.mark.parametrize("name", ["tiny_b1_t128_h4x2_d32", "small_b16_t128_h4x2_d32",
                                  "gpt116m_b16_t512_h12x4_d64"])
def test_workload_full(name):
    w = ne_inputs.WORKLOADS[name]
    errs = _full_case(ne_inputs.make_inputs(w))
    print(name, errs)


def _sampled_case(w, layer, groups):
    x = ne_inputs.make_inputs(w, layer)
    gpu = gpu_fwd_bwd(to_dev(x), THETA)
    errs = []
    for (b, j, ref, q64, k64) in oracle_all(x, THETA, groups, w.G):
        errs.append(compare(slice_gpu(gpu, b, j, w.G), ref, q64, k64))
    return errs


def test_step_workload_one_layer_sampled():
    """One layer of the 16-layer B=64 step workload at full size, in the bench's
    launch configuration; the oracle checks 6 (batch, kv head) groups."""
    w = ne_inputs.STEP_116M
    groups = [(0, 0), (17, 1), (33, 2), (50, 3), (63, 0), (63, 3)]
    print(_sampled_case(w, 5, groups))


def test_stress_workload_every_group():
    """B4 T4096 16/4 d128 with one 8x row per (tensor, batch, head): the oracle
    checks all 16 (batch, kv head) groups (every one holds 8x rows of q, k
    and v), with the flat lse bound on every row."""
    w = ne_inputs.STRESS
    groups = [(b, j) for b in range(w.B) for j in range(w.Hkv)]
    x = ne_inputs.make_inputs(w, 0)
    for (b, j) in groups:
        for name, heads in (("q", range(j * w.G, (j + 1) * w.G)), ("k", [j]), ("v", [j])):
            ms = x[name][b, :, list(heads)].float().pow(2).mean(-1)
            assert (ms > 16).any(), (name, b, j, "no 8x row in the checked group")
    print(_sampled_case(w, 0, groups))


@pytest.mark.parametrize("T", [1, 2, 3, 17, 127, 128, 129, 200, 255, 256, 300, 383])
def test_ragged_lengths_d64(T):
    _full_case(custom_inputs(B=2, T=T, Hq=6, Hkv=2, d=64, seed=100 + T))


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 2), (6, 2), (8, 2), (5, 1), (12, 4)])
def test_head_dims_and_groups(d, Hq, Hkv):
    _full_case(custom_inputs(B=1, T=260, Hq=Hq, Hkv=Hkv, d=d, seed=7 * d + Hq + Hkv))


@pytest.mark.parametrize("d", [32, 128])
def test_ragged_other_dims(d):
    for T in (1, 5, 131):
        _full_case(custom_inputs(B=2, T=T, Hq=4, Hkv=2, d=d, seed=300 + T + d))


def test_deterministic():
    """Two backward calls on the same inputs are bitwise equal (no float atomics)."""
    import causal_gqa_attention_ne_gb300 as ne
    xd = to_dev(custom_inputs(B=3, T=400, Hq=12, Hkv=4, d=64, seed=5))
    o, lse = ne.attention_forward(xd["q"], xd["k"], xd["v"], THETA)
    o2, lse2 = ne.attention_forward(xd["q"], xd["k"], xd["v"], THETA)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    a = ne.attention_backward(xd["q"], xd["k"], xd["v"], o, lse, xd["do"], THETA)
    b = ne.attention_backward(xd["q"], xd["k"], xd["v"], o, lse, xd["do"], THETA)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_outputs_stay_in_bounds():
    """Guard regions around every output keep their fill pattern (odd T)."""
    import causal_gqa_attention_ne_gb300 as ne
    B, T, Hq, Hkv, d = 2, 133, 6, 2, 64
    xd = to_dev(custom_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=9))
    G = 4096

    def guarded(shape, dtype):
        n = int(np.prod(shape))
        buf = torch.full((n + 2 * G,), 7.0, dtype=dtype, device="cuda")
        return buf, buf[G:G + n].view(shape)

    ob, o = guarded((B, T, Hq, d), torch.bfloat16)
    lb, lse = guarded((B, Hq, T), torch.float32)
    ne.ne_attn_fwd(xd["q"], xd["k"], xd["v"], o, lse, THETA)
    qb, dq = guarded((B, T, Hq, d), torch.bfloat16)
    kb, dk = guarded((B, T, Hkv, d), torch.bfloat16)
    vb, dv = guarded((B, T, Hkv, d), torch.bfloat16)
    ws = torch.empty(ne.ne_attn_bwd_workspace_size(B, T, Hq, Hkv, d), dtype=torch.uint8,
                     device="cuda")
    ne.ne_attn_bwd(xd["q"], xd["k"], xd["v"], o, lse, xd["do"], dq, dk, dv, ws, THETA)
    torch.cuda.synchronize()
    for buf in (ob, lb, qb, kb, vb):
        assert (buf[:G] == 7.0).all() and (buf[-G:] == 7.0).all()
    assert ne.ne_attn_get_error() == 0


def test_timeout_path_reports_and_recovers():
    """A wait that can never complete ends by its limit, is reported as
    NE_ERR_TIMEOUT, and the context stays usable."""
    import causal_gqa_attention_ne_gb300 as ne
    assert ne.ne_attn_get_error() == 0
    ne.ne_attn_selftest_timeout(2_000_000)   # 2 ms
    assert ne.ne_attn_get_error() == 7
    assert ne.ne_attn_get_error() == 0       # cleared
    _full_case(custom_inputs(B=1, T=64, Hq=2, Hkv=1, d=64, seed=3))


def test_rejects_bad_arguments_on_device():
    import causal_gqa_attention_ne_gb300 as ne
    lib = ne.load_library()
    x = torch.zeros(1, 8, 2, 48, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 2, 8, dtype=torch.float32, device="cuda")
    # d = 48 unsupported
    assert lib.ne_attn_fwd(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(),
                           lse.data_ptr(), 1, 8, 2, 2, 48, 10000.0, None) == 3
    y = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    # misaligned pointer
    assert lib.ne_attn_fwd(y.data_ptr() + 2, y.data_ptr(), y.data_ptr(), y.data_ptr(),
                           lse.data_ptr(), 1, 1, 1, 1, 32, 10000.0, None) == 4
    # short workspace
    assert lib.ne_attn_bwd(*(y.data_ptr(),) * 9, y.data_ptr(), 0, 1, 1, 1, 1, 32, 10000.0,
                           None) == 5
    assert ne.ne_attn_get_error() == 0


@pytest.mark.parametrize("d", [32, 64, 128])
def test_substeps_match_full_backward(d):
    """preprocess -> dq -> dkdv through their own entry points equals ne_attn_bwd
    bitwise, also when kernels of other head dims ran in between."""
    import causal_gqa_attention_ne_gb300 as ne
    B, T, Hq, Hkv = 2, 300, 6, 2
    xd = to_dev(custom_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=40 + d))
    o, lse = ne.attention_forward(xd["q"], xd["k"], xd["v"], THETA)
    dq, dk, dv = ne.attention_backward(xd["q"], xd["k"], xd["v"], o, lse, xd["do"], THETA)
    ws = torch.empty(ne.ne_attn_bwd_workspace_size(B, T, Hq, Hkv, d), dtype=torch.uint8,
                     device="cuda")
    dq2, dk2, dv2 = torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)
    ne.ne_attn_bwd_preprocess(xd["q"], xd["k"], o, xd["do"], ws, THETA)
    ne.ne_attn_bwd_dkdv(xd["q"], xd["k"], xd["v"], lse, xd["do"], dk2, dv2, ws, THETA)
    ne.ne_attn_bwd_dq(xd["q"], xd["k"], xd["v"], lse, xd["do"], dq2, ws, THETA)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)
