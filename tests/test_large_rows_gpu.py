"""Rows of q and k drawn at 8x the scale of the others (the stress shape's
outliers, and the large-norm rows real activations have): the forward makes
their scores exact (a large query row recomputed in fp32, the rows that see
a large key corrected by that pair's exact weight), so lse stays within the
flat 1e-3 bound against the float64 oracle on every row, for every head
dim, ragged T, a sliding window, padded variable-length batches and the
training pair.  More large rows than a CTA of the forward repairs (48)
report NE_WARN_PRECISION; q values beyond the fp16 range report NE_ERR_RANGE; both
leave the context usable.  Needs an sm_103 GPU."""
import numpy as np
import pytest
import torch

import ne_inputs
import oracle
from parity_util import compare, custom_inputs, gpu_fwd_bwd, oracle_all, to_dev

pytestmark = pytest.mark.gpu
THETA = ne_inputs.ROPE_THETA


@pytest.fixture(scope="module")
def ne():
    import causal_gqa_attention_ne_gb300 as mod
    mod.load_library()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return mod


def with_large_rows(x, q_rows=(), k_rows=(), v_rows=(), scale=8.0):
    """Scales rows (b, t, head) of q, k, v by `scale` (a power of two, exact in bf16)."""
    x = {n: t.clone() for n, t in x.items()}
    for name, rows in (("q", q_rows), ("k", k_rows), ("v", v_rows)):
        for (b, t, h) in rows:
            x[name][b, t, h] *= scale
    return x


# per (batch, position, head)
Q_ROWS = [(0, 0, 0), (0, 130, 0), (0, 299, 3), (1, 127, 1), (1, 200, 2), (1, 255, 3)]
K_ROWS = [(0, 5, 0), (0, 127, 0), (0, 128, 1), (1, 200, 1), (1, 299, 0)]


@pytest.mark.parametrize("d", [32, 64, 128])
def test_large_rows_flat_lse(ne, d):
    x = with_large_rows(custom_inputs(B=2, T=300, Hq=4, Hkv=2, d=d, seed=500 + d),
                        Q_ROWS, K_ROWS, v_rows=[(0, 7, 1), (1, 128, 0)])
    gpu = gpu_fwd_bwd(to_dev(x), THETA)
    ref, _, _ = oracle_all(x, THETA)
    print(d, compare(gpu, ref))


def test_large_query_and_key_in_the_same_pair(ne):
    """The large query row sees the large key (both 8x): that row is
    recomputed exactly and not corrected a second time for the key."""
    x = with_large_rows(custom_inputs(B=1, T=256, Hq=2, Hkv=1, d=64, seed=77),
                        q_rows=[(0, 200, 0), (0, 200, 1)], k_rows=[(0, 150, 0)])
    gpu = gpu_fwd_bwd(to_dev(x), THETA)
    ref, _, _ = oracle_all(x, THETA)
    print(compare(gpu, ref))


def test_large_rows_sliding_window(ne):
    B, T, Hq, Hkv, d, W = 2, 300, 4, 2, 64, 100
    x = with_large_rows(custom_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=31),
                        Q_ROWS, K_ROWS)
    xd = to_dev(x)
    o = torch.empty_like(xd["q"])
    lse = torch.empty(B, Hq, T, dtype=torch.float32, device="cuda")
    ne.ne_attn_fwd_window(xd["q"], xd["k"], xd["v"], o, lse, W, THETA)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0
    q, k, v = (ne_inputs.as_f64(x[n]) for n in ("q", "k", "v"))
    ro, rl = oracle.attn_fwd(q, k, v, THETA, window=W)
    print(compare({"o": o, "lse": lse}, {"o": ro, "lse": rl}, what=("o", "lse")))


def test_large_rows_padded_varlen(ne):
    B, T, Hq, Hkv, d = 2, 300, 4, 2, 64
    lens = [250, 300]
    x = with_large_rows(custom_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=32),
                        Q_ROWS, K_ROWS)
    xd = to_dev(x)
    ws = torch.empty(ne.ne_attn_varlen_workspace_size(B, T, Hq, Hkv, d), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty_like(xd["q"])
    lse = torch.empty(B, Hq, T, dtype=torch.float32, device="cuda")
    ne.ne_attn_fwd_varlen(xd["q"], xd["k"], xd["v"], o, lse, np.asarray(lens, np.int32), ws,
                          THETA)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0
    q, k, v = (ne_inputs.as_f64(x[n]) for n in ("q", "k", "v"))
    for b, L in enumerate(lens):
        sl = (slice(b, b + 1), slice(0, L))
        ro, rl = oracle.attn_fwd(q[sl], k[sl], v[sl], THETA)
        print(b, compare({"o": o[sl], "lse": lse[b:b + 1, :, :L]}, {"o": ro, "lse": rl},
                         what=("o", "lse")))


def test_large_rows_training_pair_equals_standalone(ne):
    """ne_attn_fwd_save corrects the same scores as ne_attn_fwd: bitwise equal
    outputs, and the backward of the pair equals the standalone backward."""
    B, T, Hq, Hkv, d = 2, 300, 6, 2, 64
    x = with_large_rows(custom_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=33),
                        [(0, 10, 4), (1, 290, 5)], [(0, 3, 1), (1, 256, 0)])
    xd = to_dev(x)
    o, lse = ne.attention_forward(xd["q"], xd["k"], xd["v"], THETA)
    dq, dk, dv = ne.attention_backward(xd["q"], xd["k"], xd["v"], o, lse, xd["do"], THETA)
    ws = torch.empty(ne.ne_attn_bwd_workspace_size(B, T, Hq, Hkv, d), dtype=torch.uint8,
                     device="cuda")
    o2, lse2 = torch.empty_like(o), torch.empty_like(lse)
    ne.ne_attn_fwd_save(xd["q"], xd["k"], xd["v"], o2, lse2, ws, THETA)
    dq2, dk2, dv2 = torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)
    ne.ne_attn_bwd_saved(xd["q"], xd["k"], xd["v"], o2, lse2, xd["do"], dq2, dk2, dv2, ws, THETA)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0
    for a, b in ((o, o2), (lse, lse2), (dq, dq2), (dk, dk2), (dv, dv2)):
        assert torch.equal(a, b)
    ref, _, _ = oracle_all(x, THETA)
    print(compare({"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}, ref))


def test_too_many_large_rows_warns(ne):
    """Sixty large key rows in one sequence (a CTA repairs up to 48 large
    rows): the forward reports NE_WARN_PRECISION, its outputs are finite,
    and the next call on ordinary inputs reports NE_OK."""
    x = with_large_rows(custom_inputs(B=1, T=200, Hq=2, Hkv=1, d=64, seed=34),
                        k_rows=[(0, s, 0) for s in range(0, 120, 2)])
    xd = to_dev(x)
    o, lse = ne.attention_forward(xd["q"], xd["k"], xd["v"], THETA)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 11          # NE_WARN_PRECISION
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    assert ne.ne_attn_get_error() == 0           # cleared
    gpu = gpu_fwd_bwd(to_dev(custom_inputs(B=1, T=200, Hq=2, Hkv=1, d=64, seed=35)),
                      THETA)
    assert gpu["o"].shape == (1, 200, 2, 64)


def test_many_large_rows_within_capacity(ne):
    """Forty large key rows and large query rows of every head in one
    sequence, within what a CTA repairs: flat lse and NE_OK (forward only:
    with this many large keys the backward's fp16 scores dominate its
    error, which the single-outlier cases bound)."""
    x = with_large_rows(custom_inputs(B=1, T=300, Hq=4, Hkv=1, d=64, seed=38),
                        q_rows=[(0, t, h) for t in (3, 150, 299) for h in range(4)],
                        k_rows=[(0, s, 0) for s in range(1, 280, 7)])
    gpu = gpu_fwd_bwd(to_dev(x), THETA, with_bwd=False)
    ref, _, _ = oracle_all(x, THETA)
    print(compare(gpu, ref, what=("o", "lse")))


def test_fp16_range_overflow_reports_and_recovers(ne):
    """A q value beyond the fp16 range (bf16 holds it) sets NE_ERR_RANGE; the
    kernels finish (no wait depends on the values) and the context stays
    usable."""
    x = custom_inputs(B=1, T=64, Hq=2, Hkv=1, d=64, seed=36)
    x["q"][0, 0, 0, :] = 1.0e5
    xd = to_dev(x)
    ne.attention_forward(xd["q"], xd["k"], xd["v"], THETA)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 8           # NE_ERR_RANGE
    assert ne.ne_attn_get_error() == 0
    gpu = gpu_fwd_bwd(to_dev(custom_inputs(B=1, T=64, Hq=2, Hkv=1, d=64, seed=37)),
                      THETA)
    ref, _, _ = oracle_all(custom_inputs(B=1, T=64, Hq=2, Hkv=1, d=64, seed=37), THETA)
    compare(gpu, ref)


def test_large_rows_packed(ne):
    """A packed batch with 8x rows of q and k in several sequences: the repair
    addresses rows through the pack's offsets; flat lse against the oracle's
    packed forward."""
    lens = [300, 1, 129, 200]
    Hq, Hkv, d = 4, 2, 64
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    total = int(cu[-1])
    x = custom_inputs(B=1, T=total, Hq=Hq, Hkv=Hkv, d=d, seed=39)
    # 8x rows at (sequence, position, head)
    for (sq, t, h) in ((0, 5, 0), (0, 299, 3), (2, 128, 1), (3, 0, 2), (3, 150, 0)):
        x["q"][0, cu[sq] + t, h] *= 8.0
    for (sq, t, j) in ((0, 40, 0), (2, 3, 1), (3, 130, 0), (1, 0, 1)):
        x["k"][0, cu[sq] + t, j] *= 8.0
    xp = {n: t[0].contiguous() for n, t in x.items()}
    xd = to_dev(xp)
    ws = torch.empty(ne.ne_attn_packed_workspace_size(len(lens), total, Hq, Hkv, d),
                     dtype=torch.uint8, device="cuda")
    o = torch.empty_like(xd["q"])
    lse = torch.empty(Hq, total, dtype=torch.float32, device="cuda")
    ne.ne_attn_fwd_packed(xd["q"], xd["k"], xd["v"], o, lse, cu, ws, THETA)
    torch.cuda.synchronize()
    assert ne.ne_attn_get_error() == 0
    q, k, v = (ne_inputs.as_f64(xp[n]) for n in ("q", "k", "v"))
    ro, rl = oracle.attn_fwd_packed(q, k, v, cu, THETA)
    print(compare({"o": o, "lse": lse}, {"o": ro, "lse": rl}, what=("o", "lse")))
