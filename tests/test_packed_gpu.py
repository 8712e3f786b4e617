"""Packed variable-length batches (ne_attn_fwd_packed / ne_attn_bwd_packed):
the sequences concatenated along the rows with no padding, sequence b at
rows cu_seqlens[b] .. cu_seqlens[b+1]-1, positions restarting at 0.
Checked against the float64 oracle's packed functions with the causal
path's tolerances (empty, one-row, tile-sized and ragged sequences; every
head dim; several group sizes), against the padded entry points on the same
sequences bit for bit, and for writing no row outside the pack.  Needs an
sm_103 GPU."""
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


def _pack(lens, Hq, Hkv, d, seed):
    """Seeded [total, H, d] tensors (the usual recipe on a [1, total] batch)."""
    total = int(sum(lens))
    x = custom_inputs(B=1, T=total, Hq=Hq, Hkv=Hkv, d=d, seed=seed)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return {n: t[0].contiguous() for n, t in x.items()}, cu


def _run_packed(ne, xd, cu, guard=0):
    q, k, v, do = xd["q"], xd["k"], xd["v"], xd["do"]
    total, Hq, d = q.shape
    Hkv = k.shape[1]
    nan = float("nan")
    ws = torch.empty(ne.ne_attn_packed_workspace_size(len(cu) - 1, total, Hq, Hkv, d),
                     dtype=torch.uint8, device="cuda")
    o = torch.full_like(q, nan)
    lse = torch.full((Hq, total), nan, dtype=torch.float32, device="cuda")
    ne.ne_attn_fwd_packed(q, k, v, o, lse, cu, ws, THETA)
    dq, dk, dv = (torch.full_like(x, nan) for x in (q, k, v))
    ne.ne_attn_bwd_packed(q, k, v, o, lse, do, dq, dk, dv, cu, ws, THETA)
    torch.cuda.synchronize()
    status = ne.ne_attn_get_error()
    assert status == 0, f"device status {ne.NE_STATUS.get(status, status)}"
    return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}


CASES = [
    # (lengths, Hq, Hkv, d)
    ([300, 0, 1, 128, 129, 57], 6, 2, 64),
    ([127, 256, 5], 4, 4, 32),
    ([200, 1, 333], 8, 2, 128),
    ([512, 384, 17, 260], 12, 4, 64),
    ([1, 1, 1, 130], 5, 1, 64),
]


@pytest.mark.parametrize("lens,Hq,Hkv,d", CASES)
def test_packed_matches_oracle(ne, lens, Hq, Hkv, d):
    x, cu = _pack(lens, Hq, Hkv, d, seed=600 + sum(lens))
    got = _run_packed(ne, to_dev(x), cu)
    q, k, v, do = (ne_inputs.as_f64(x[n]) for n in ("q", "k", "v", "do"))
    ro, rl = oracle.attn_fwd_packed(q, k, v, cu, THETA)
    rg = oracle.attn_bwd_packed(q, k, v, do, cu, THETA)
    ref = {"o": ro, "lse": rl, **rg}
    print(lens, compare(got, ref))


def test_packed_equals_padded_bitwise(ne):
    """The same sequences padded to the longest: every valid row of every
    output is the same bits (the tiles, positions and masks are the same)."""
    lens = [300, 0, 129, 77, 256]
    Hq, Hkv, d = 6, 2, 64
    x, cu = _pack(lens, Hq, Hkv, d, seed=700)
    got = _run_packed(ne, to_dev(x), cu)
    B, T = len(lens), max(lens)
    pad = {n: torch.zeros(B, T, *t.shape[1:], dtype=t.dtype) for n, t in x.items()}
    for b, L in enumerate(lens):
        for n in pad:
            pad[n][b, :L] = x[n][cu[b]:cu[b] + L]
    pd = to_dev(pad)
    ws = torch.empty(ne.ne_attn_varlen_workspace_size(B, T, Hq, Hkv, d), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty_like(pd["q"])
    lse = torch.empty(B, Hq, T, dtype=torch.float32, device="cuda")
    sl = np.asarray(lens, np.int32)
    ne.ne_attn_fwd_varlen(pd["q"], pd["k"], pd["v"], o, lse, sl, ws, THETA)
    dq, dk, dv = torch.empty_like(pd["q"]), torch.empty_like(pd["k"]), torch.empty_like(pd["v"])
    ne.ne_attn_bwd_varlen(pd["q"], pd["k"], pd["v"], o, lse, pd["do"], dq, dk, dv, sl, ws, THETA)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0
    for b, L in enumerate(lens):
        r = slice(cu[b], cu[b] + L)
        for n, padded in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
            assert torch.equal(got[n][r], padded[b, :L]), (n, b)
        assert torch.equal(got["lse"][:, r], lse[b, :, :L]), ("lse", b)


def test_packed_writes_nothing_outside_the_pack(ne):
    """Outputs inside guard regions: the fill pattern around them survives
    (the last tile of each sequence is stored row by row)."""
    lens = [130, 3, 255]
    Hq, Hkv, d = 4, 2, 64
    x, cu = _pack(lens, Hq, Hkv, d, seed=701)
    xd = to_dev(x)
    total = int(cu[-1])
    G = 4096

    def guarded(shape, dtype):
        n = int(np.prod(shape))
        buf = torch.full((n + 2 * G,), 7.0, dtype=dtype, device="cuda")
        return buf, buf[G:G + n].view(shape)

    ob, o = guarded((total, Hq, d), torch.bfloat16)
    lb, lse = guarded((Hq, total), torch.float32)
    qb, dq = guarded((total, Hq, d), torch.bfloat16)
    kb, dk = guarded((total, Hkv, d), torch.bfloat16)
    vb, dv = guarded((total, Hkv, d), torch.bfloat16)
    ws = torch.empty(ne.ne_attn_packed_workspace_size(len(lens), total, Hq, Hkv, d),
                     dtype=torch.uint8, device="cuda")
    ne.ne_attn_fwd_packed(xd["q"], xd["k"], xd["v"], o, lse, cu, ws, THETA)
    ne.ne_attn_bwd_packed(xd["q"], xd["k"], xd["v"], o, lse, xd["do"], dq, dk, dv, cu, ws, THETA)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0
    for buf in (ob, lb, qb, kb, vb):
        assert (buf[:G] == 7.0).all() and (buf[-G:] == 7.0).all()
    assert torch.isfinite(o.float()).all() and torch.isfinite(dq.float()).all()


def _run_packed_dev(ne, xd, cu_dev, ws):
    q, k, v, do = xd["q"], xd["k"], xd["v"], xd["do"]
    total, Hq, d = q.shape
    nan = float("nan")
    o = torch.full_like(q, nan)
    lse = torch.full((Hq, total), nan, dtype=torch.float32, device="cuda")
    dq, dk, dv = (torch.full_like(x, nan) for x in (q, k, v))
    ne.ne_attn_fwd_packed_dev(q, k, v, o, lse, cu_dev, ws, THETA)
    ne.ne_attn_bwd_packed_dev(q, k, v, o, lse, do, dq, dk, dv, cu_dev, ws, THETA)
    return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}


@pytest.mark.parametrize("lens,Hq,Hkv,d", CASES)
def test_packed_device_offsets_equal_host(ne, lens, Hq, Hkv, d):
    """cu_seqlens in device memory (tables planned on the GPU): every output
    bitwise equal to the host-offset entry points."""
    x, cu = _pack(lens, Hq, Hkv, d, seed=800 + sum(lens))
    xd = to_dev(x)
    ref = _run_packed(ne, xd, cu)
    total = int(cu[-1])
    ws = torch.full((ne.ne_attn_packed_workspace_size(len(cu) - 1, total, Hq, Hkv, d),), 0x33,
                    dtype=torch.uint8, device="cuda")
    got = _run_packed_dev(ne, xd, torch.from_numpy(cu).cuda(), ws)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0
    for n in ref:
        assert torch.equal(got[n], ref[n]), n


def test_packed_graph_replays_with_new_offsets(ne):
    """One capture; replays after writing other offsets (same sequence count
    and total) into the same device tensor equal eager host-offset calls."""
    Hq, Hkv, d = 6, 2, 64
    x, cu0 = _pack([300, 100, 12], Hq, Hkv, d, seed=810)
    xd = to_dev(x)
    total = int(cu0[-1])
    ws = torch.zeros(ne.ne_attn_packed_workspace_size(3, total, Hq, Hkv, d), dtype=torch.uint8,
                     device="cuda")
    cu_dev = torch.from_numpy(cu0).cuda()
    out = _run_packed_dev(ne, xd, cu_dev, ws)            # warm-up outside the capture
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out = _run_packed_dev(ne, xd, cu_dev, ws)
    for lens in ([300, 100, 12], [1, 410, 1], [0, 0, 412], [129, 128, 155]):
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        cu_dev.copy_(torch.from_numpy(cu))
        for t in out.values():
            t.fill_(float("nan"))
        graph.replay()
        ref = _run_packed(ne, xd, cu)
        for n in ref:
            assert torch.equal(out[n], ref[n]), (lens, n)


def test_packed_device_bad_offsets_report_and_sanitise(ne):
    """A decreasing prefix array in device memory: NE_ERR_ARG, and the call
    runs on the monotone array (running maximum), no fault."""
    Hq, Hkv, d = 4, 2, 64
    x, _ = _pack([6, 0, 4], Hq, Hkv, d, seed=811)
    xd = to_dev(x)
    ws = torch.zeros(ne.ne_attn_packed_workspace_size(3, 10, Hq, Hkv, d), dtype=torch.uint8,
                     device="cuda")
    got = _run_packed_dev(ne, xd, torch.tensor([0, 6, 4, 10], dtype=torch.int32,
                                               device="cuda"), ws)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 9              # NE_ERR_ARG
    ref = _run_packed(ne, xd, np.asarray([0, 6, 6, 10], np.int32))
    for n in ref:
        assert torch.equal(got[n], ref[n]), n
