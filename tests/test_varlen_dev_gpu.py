"""Padded variable-length batches with the lengths in device memory
(ne_attn_fwd_varlen_dev / ne_attn_bwd_varlen_dev): the work-unit tables are
planned on the GPU.  Checked against the host-length entry points bit for
bit (tables, counts and every output), through a CUDA graph captured once
and replayed with other lengths written into the same buffer, and for a
length out of range (clamped, NE_ERR_ARG).  Needs an sm_103 GPU."""
import numpy as np
import pytest
import torch

import ne_inputs
from parity_util import custom_inputs, to_dev
from test_varlen_plan import chunks

pytestmark = pytest.mark.gpu
THETA = ne_inputs.ROPE_THETA


@pytest.fixture(scope="module")
def ne():
    import causal_gqa_attention_ne_gb300 as mod
    mod.load_library()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return mod


def _outputs(xd):
    nan = float("nan")
    q, k, v = xd["q"], xd["k"], xd["v"]
    B, T, Hq, _ = q.shape
    return {"o": torch.full_like(q, nan),
            "lse": torch.full((B, Hq, T), nan, dtype=torch.float32, device="cuda"),
            "dq": torch.full_like(q, nan), "dk": torch.full_like(k, nan),
            "dv": torch.full_like(v, nan)}


def _call(ne, xd, out, lens, ws, dev):
    q, k, v, do = xd["q"], xd["k"], xd["v"], xd["do"]
    if dev:
        ne.ne_attn_fwd_varlen_dev(q, k, v, out["o"], out["lse"], lens, ws, THETA)
        ne.ne_attn_bwd_varlen_dev(q, k, v, out["o"], out["lse"], do, out["dq"], out["dk"],
                                  out["dv"], lens, ws, THETA)
    else:
        ne.ne_attn_fwd_varlen(q, k, v, out["o"], out["lse"], lens, ws, THETA)
        ne.ne_attn_bwd_varlen(q, k, v, out["o"], out["lse"], do, out["dq"], out["dk"],
                              out["dv"], lens, ws, THETA)


def _tables(ws, B, T, Hq, Hkv, d):
    """The workspace's table regions (layout of ne_attn_varlen_workspace_size)."""
    def r256(x):
        return (x + 255) // 256 * 256
    G, tiles = Hq // Hkv, (T + 127) // 128 * B * Hkv
    nf, nq = chunks(d, G)
    off = [0, r256(4 * B)]
    off.append(off[-1] + r256(4 * tiles * nf))
    off.append(off[-1] + r256(4 * tiles * nq))
    off.append(off[-1] + r256(4 * tiles))
    w = ws.view(torch.int32).cpu().numpy()
    return {"seqlen": w[:B], "fwd": w[off[1] // 4:], "dq": w[off[2] // 4:],
            "dkv": w[off[3] // 4:], "counts": w[off[4] // 4: off[4] // 4 + 3]}


@pytest.mark.parametrize("B,T,Hq,Hkv,d,seed", [(5, 300, 6, 2, 64, 1), (3, 517, 12, 4, 64, 2),
                                               (4, 260, 4, 2, 32, 3), (3, 200, 4, 1, 128, 4)])
def test_device_plan_equals_host(ne, B, T, Hq, Hkv, d, seed):
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, T + 1, size=B).astype(np.int32)
    lens[0] = T
    xd = to_dev(custom_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=1600 + seed))
    nbytes = ne.ne_attn_varlen_workspace_size(B, T, Hq, Hkv, d)
    ws_h = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    ws_d = torch.full((nbytes,), 0x55, dtype=torch.uint8, device="cuda")
    ref, got = _outputs(xd), _outputs(xd)
    _call(ne, xd, ref, lens, ws_h, dev=False)
    _call(ne, xd, got, torch.from_numpy(lens).cuda(), ws_d, dev=True)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0
    for n in ref:
        assert torch.equal(got[n], ref[n]), n
    counts, (tf, tq, tk) = ne.ne_attn_varlen_plan(lens, T, Hq, Hkv, d)
    tab = _tables(ws_d, B, T, Hq, Hkv, d)
    assert (tab["seqlen"] == lens).all()
    assert list(tab["counts"]) == list(counts)
    assert (tab["fwd"][:counts[0]] == tf).all()
    assert (tab["dq"][:counts[1]] == tq).all()
    assert (tab["dkv"][:counts[2]] == tk).all()


def test_graph_replays_with_new_lengths(ne):
    """One capture of the forward + backward; replays after writing other
    lengths into the same device buffer equal eager host-length calls."""
    B, T, Hq, Hkv, d = 4, 384, 6, 2, 64
    xd = to_dev(custom_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=1700))
    nbytes = ne.ne_attn_varlen_workspace_size(B, T, Hq, Hkv, d)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    lens_dev = torch.tensor([384, 100, 0, 257], dtype=torch.int32, device="cuda")
    out = _outputs(xd)
    _call(ne, xd, out, lens_dev, ws, dev=True)          # warm-up outside the capture
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _call(ne, xd, out, lens_dev, ws, dev=True)
    for lens in ([384, 100, 0, 257], [1, 383, 128, 129], [384, 384, 384, 384], [0, 0, 5, 0]):
        lens_dev.copy_(torch.tensor(lens, dtype=torch.int32))
        for t in out.values():
            t.fill_(float("nan"))
        graph.replay()
        ref = _outputs(xd)
        ws_h = torch.zeros_like(ws)
        _call(ne, xd, ref, np.asarray(lens, np.int32), ws_h, dev=False)
        torch.cuda.synchronize()
        assert ne.ne_attn_get_error() == 0
        for n in ref:
            assert torch.equal(out[n], ref[n]), (lens, n)


def test_device_length_out_of_range_reports_and_clamps(ne):
    B, T, Hq, Hkv, d = 2, 200, 4, 2, 64
    xd = to_dev(custom_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=1701))
    ws = torch.zeros(ne.ne_attn_varlen_workspace_size(B, T, Hq, Hkv, d), dtype=torch.uint8,
                     device="cuda")
    out = _outputs(xd)
    _call(ne, xd, out, torch.tensor([250, -3], dtype=torch.int32, device="cuda"), ws, dev=True)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 9              # NE_ERR_ARG
    ref = _outputs(xd)
    _call(ne, xd, ref, np.asarray([200, 0], np.int32), torch.zeros_like(ws), dev=False)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0              # cleared; the clamped lengths ran
    for n in ref:
        assert torch.equal(out[n], ref[n]), n
