"""Checks that pin the CPU oracle to something other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with a closed form, an invariant the definition
implies, central finite differences (the pages' own validation method), or
torch's CPU attention routine.  ``tests/test_oracle.py`` runs them on the real
oracle; ``tests/test_oracle_mutations.py`` runs them on copies of the oracle
with planted mistakes and requires each mistake to be caught.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import ne_inputs

THETA = ne_inputs.ROPE_THETA


def _rel(a, b) -> float:
    """Norm-wise relative error max|a - b| / max|b|."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.abs(b).max()
    return float(np.abs(a - b).max() / (den if den > 0 else 1.0))


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ---------------------------------------------------------------- RoPE ----

def pin_rope_closed_form(orc):
    """Rotate-half RoPE on unit vectors, written out by hand.

    d = 4, theta = 10000: frequencies theta^(-2i/d) are 1 and 0.01.  Position t
    rotates the pair (x0, x2) by angle t and the pair (x1, x3) by 0.01 t.
    d = 8, theta = 100: frequencies 100^(-i/4).
    """
    T = 7
    eye = np.eye(4)
    x = np.zeros((1, T, 4, 4))
    for t in range(T):
        x[0, t] = eye
    y = orc.rope(x, 10000.0)
    for t in range(T):
        c0, s0, c1, s1 = math.cos(t), math.sin(t), math.cos(0.01 * t), math.sin(0.01 * t)
        want = np.array([
            [c0, 0.0, s0, 0.0],     # e0 -> (cos t, 0, sin t, 0)
            [0.0, c1, 0.0, s1],     # e1 -> (0, cos .01t, 0, sin .01t)
            [-s0, 0.0, c0, 0.0],    # e2 -> (-sin t, 0, cos t, 0)
            [0.0, -s1, 0.0, c1],    # e3 -> (0, -sin .01t, 0, cos .01t)
        ])
        assert np.abs(y[0, t] - want).max() < 1e-14, (t, y[0, t], want)
    # inverse rotation is the transpose
    yi = orc.rope(x, 10000.0, inverse=True)
    for t in range(T):
        c0, s0 = math.cos(t), math.sin(t)
        assert abs(yi[0, t, 0, 0] - c0) < 1e-14 and abs(yi[0, t, 0, 2] + s0) < 1e-14
    # d = 8, theta = 100, e3 at position 5: frequency 100^(-6/8)
    x8 = np.zeros((1, 6, 1, 8))
    x8[0, 5, 0, 3] = 1.0
    y8 = orc.rope(x8, 100.0)
    f3 = 100.0 ** (-0.75)
    want8 = np.zeros(8)
    want8[3] = math.cos(5 * f3)
    want8[7] = math.sin(5 * f3)
    assert np.abs(y8[0, 5, 0] - want8).max() < 1e-14, y8[0, 5, 0]


def pin_rope_identity_and_orthogonal(orc):
    """R(0) is the identity; R(t) preserves norms; R(t)^T R(t) = I."""
    x = _rand((2, 9, 3, 16), 1)
    y = orc.rope(x, THETA)
    assert np.array_equal(y[:, 0], x[:, 0])
    assert np.abs(np.linalg.norm(y, axis=-1) - np.linalg.norm(x, axis=-1)).max() < 1e-12
    back = orc.rope(y, THETA, inverse=True)
    assert np.abs(back - x).max() < 1e-12


# ------------------------------------------------------------- forward ----

def pin_relative_position(orc):
    """Shifting every position by a constant leaves the scores, hence O and lse, unchanged."""
    x = ne_inputs.make_custom(B=1, T=33, Hq=4, Hkv=2, d=16, seed=11)
    q, k, v = (ne_inputs.as_f64(x[n]) for n in ("q", "k", "v"))
    o0, l0 = orc.attn_fwd(q, k, v, THETA)
    o1, l1 = orc.attn_fwd(q, k, v, THETA, pos_offset=1000)
    assert _rel(o1, o0) < 1e-10 and np.abs(l1 - l0).max() < 1e-10


def pin_rows_sum_to_one(orc):
    """Softmax rows sum to one: with v = 1 everywhere, O = 1; O lies in the hull of v."""
    x = ne_inputs.make_custom(B=2, T=40, Hq=6, Hkv=2, d=8, seed=12)
    q, k = ne_inputs.as_f64(x["q"]), ne_inputs.as_f64(x["k"])
    ones = np.ones_like(ne_inputs.as_f64(x["v"]))
    o, _ = orc.attn_fwd(q, k, ones, THETA)
    assert np.abs(o - 1.0).max() < 1e-12
    v = ne_inputs.as_f64(x["v"])
    o, _ = orc.attn_fwd(q, k, v, THETA)
    assert o.max() <= v.max() + 1e-12 and o.min() >= v.min() - 1e-12


def pin_causality(orc):
    """O[t] and lse[t] do not depend on tokens after t (bitwise in double)."""
    x = ne_inputs.make_custom(B=1, T=24, Hq=4, Hkv=1, d=8, seed=13)
    q, k, v = (ne_inputs.as_f64(x[n]) for n in ("q", "k", "v"))
    t0 = 10
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    rng = np.random.default_rng(5)
    for a in (q2, k2, v2):
        a[:, t0 + 1:] += rng.standard_normal(a[:, t0 + 1:].shape)
    o, lse = orc.attn_fwd(q, k, v, THETA)
    o2, lse2 = orc.attn_fwd(q2, k2, v2, THETA)
    assert np.array_equal(o[:, :t0 + 1], o2[:, :t0 + 1])
    assert np.array_equal(lse[:, :, :t0 + 1], lse2[:, :, :t0 + 1])
    assert not np.array_equal(o[:, t0 + 1:], o2[:, t0 + 1:])


def pin_single_token(orc):
    """T = 1: O = v, lse = <q, k>/sqrt(d), dq = dk = 0, dv = sum of dO over the group."""
    B, Hq, Hkv, d = 2, 6, 3, 8
    q, k, v = _rand((B, 1, Hq, d), 21), _rand((B, 1, Hkv, d), 22), _rand((B, 1, Hkv, d), 23)
    do = _rand((B, 1, Hq, d), 24)
    G = Hq // Hkv
    o, lse = orc.attn_fwd(q, k, v, THETA)
    r = orc.attn_bwd(q, k, v, do, THETA)
    for b in range(B):
        for h in range(Hq):
            j = h // G
            assert np.abs(o[b, 0, h] - v[b, 0, j]).max() < 1e-14
            want = float(q[b, 0, h] @ k[b, 0, j]) / math.sqrt(d)
            assert abs(lse[b, h, 0] - want) < 1e-13
        for j in range(Hkv):
            want_dv = do[b, 0, j * G:(j + 1) * G].sum(axis=0)
            assert np.abs(r["dv"][b, 0, j] - want_dv).max() < 1e-13
    assert np.abs(r["dq"]).max() < 1e-14 and np.abs(r["dk"]).max() < 1e-14


def pin_zero_query(orc):
    """q = 0: uniform attention, O[t] = mean(v[0..t]), lse[t] = ln(t + 1)."""
    B, T, Hq, Hkv, d = 1, 50, 4, 2, 8
    k, v = _rand((B, T, Hkv, d), 31), _rand((B, T, Hkv, d), 32)
    q = np.zeros((B, T, Hq, d))
    o, lse = orc.attn_fwd(q, k, v, THETA)
    G = Hq // Hkv
    csum = np.cumsum(v, axis=1) / np.arange(1, T + 1)[None, :, None, None]
    for h in range(Hq):
        assert np.abs(o[:, :, h] - csum[:, :, h // G]).max() < 1e-12
        assert np.abs(lse[0, h] - np.log(np.arange(1, T + 1))).max() < 1e-12


def pin_fwd_bwd_agree(orc):
    """The backward's recomputed O and lse equal the forward's."""
    x = ne_inputs.make_custom(B=2, T=17, Hq=4, Hkv=2, d=8, seed=41)
    q, k, v, do = (ne_inputs.as_f64(x[n]) for n in ("q", "k", "v", "do"))
    o, lse = orc.attn_fwd(q, k, v, THETA)
    r = orc.attn_bwd(q, k, v, do, THETA)
    assert np.abs(r["o"] - o).max() < 1e-13 and np.abs(r["lse"] - lse).max() < 1e-13


# ------------------------------------------------------------ backward ----

def _loss(orc, q, k, v, do, theta):
    o, _ = orc.attn_fwd(q, k, v, theta, threads=1)
    return float((o * do).sum())


def fd_check(orc, q, k, v, do, theta, idx_per_tensor=None, h=1e-6, seed=0):
    """Central finite differences of L = sum(O * dO), compared with the analytic backward.

    Returns the worst norm-wise relative error over dq, dk, dv.  With
    ``idx_per_tensor`` set, only that many random elements per tensor are
    differenced.
    """
    r = orc.attn_bwd(q, k, v, do, theta)
    rng = np.random.default_rng(seed)
    worst = 0.0
    for name, x, g in (("q", q, r["dq"]), ("k", k, r["dk"]), ("v", v, r["dv"])):
        flat = x.reshape(-1)
        n = flat.size
        idx = np.arange(n) if idx_per_tensor is None else rng.choice(n, idx_per_tensor,
                                                                      replace=False)
        fd = np.empty(idx.size)
        for m, i in enumerate(idx):
            old = flat[i]
            flat[i] = old + h
            lp = _loss(orc, q, k, v, do, theta)
            flat[i] = old - h
            lm = _loss(orc, q, k, v, do, theta)
            flat[i] = old
            fd[m] = (lp - lm) / (2 * h)
        an = g.reshape(-1)[idx]
        worst = max(worst, _rel(an, fd))
    return worst


def pin_finite_differences(orc):
    """Every gradient element of a tiny GQA case against central differences in double."""
    x = ne_inputs.make_custom(B=1, T=5, Hq=4, Hkv=2, d=8, seed=51)
    q, k, v, do = (ne_inputs.as_f64(x[n]).copy() for n in ("q", "k", "v", "do"))
    err = fd_check(orc, q, k, v, do, THETA)
    assert err < 1e-6, err


def pin_finite_differences_tiny_workload(orc):
    """Sampled central differences on the tiny workload (B1 T128 4/2 heads d32)."""
    x = ne_inputs.make_inputs(ne_inputs.TINY)
    q, k, v, do = (ne_inputs.as_f64(x[n]).copy() for n in ("q", "k", "v", "do"))
    err = fd_check(orc, q, k, v, do, THETA, idx_per_tensor=40, seed=3)
    assert err < 1e-6, err


# --------------------------------------------------- library cross-check ----

def _torch_rope(x, theta):
    """RoPE through complex multiplication: (x_i + i x_{i+d/2}) * exp(i t theta_i)."""
    B, T, H, d = x.shape
    half = d // 2
    freq = theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / d)
    ang = torch.arange(T, dtype=torch.float64)[:, None] * freq[None, :]
    rot = torch.polar(torch.ones_like(ang), ang)[None, :, None, :]
    z = torch.complex(x[..., :half], x[..., half:]) * rot
    return torch.cat([z.real, z.imag], dim=-1)


def torch_reference(q, k, v, do, theta):
    """torch CPU float64: complex-rotation RoPE, then scaled_dot_product_attention
    (causal, GQA) and autograd for the gradients of sum(O * dO)."""
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    G = q.shape[2] // k.shape[2]
    qr = _torch_rope(tq, theta).transpose(1, 2)
    kr = _torch_rope(tk, theta).transpose(1, 2)
    vv = tv.transpose(1, 2)
    d = q.shape[-1]
    o = torch.nn.functional.scaled_dot_product_attention(
        qr, kr, vv, is_causal=True, scale=1.0 / math.sqrt(d), enable_gqa=True)
    (o * torch.tensor(do).transpose(1, 2)).sum().backward()
    with torch.no_grad():
        krep = kr.repeat_interleave(G, dim=1)
        s = qr @ krep.transpose(-1, -2) / math.sqrt(d)
        T = q.shape[1]
        mask = torch.ones(T, T, dtype=torch.bool).triu(1)
        lse = torch.logsumexp(s.masked_fill(mask, float("-inf")), dim=-1)
    return {"o": o.detach().transpose(1, 2).numpy(), "lse": lse.numpy(),
            "dq": tq.grad.numpy(), "dk": tk.grad.numpy(), "dv": tv.grad.numpy()}


def pin_torch_sdpa(orc):
    """Forward and backward against torch's CPU attention in float64 (to 1e-10)."""
    for (B, T, Hq, Hkv, d, seed) in ((2, 37, 6, 2, 16, 61), (1, 64, 4, 4, 32, 62),
                                     (1, 20, 8, 1, 8, 63)):
        x = ne_inputs.make_custom(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=seed)
        q, k, v, do = (ne_inputs.as_f64(x[n]) for n in ("q", "k", "v", "do"))
        ref = torch_reference(q, k, v, do, THETA)
        o, lse = orc.attn_fwd(q, k, v, THETA)
        r = orc.attn_bwd(q, k, v, do, THETA)
        assert _rel(o, ref["o"]) < 1e-10, ("o", _rel(o, ref["o"]))
        assert np.abs(lse - ref["lse"]).max() < 1e-10, "lse"
        for n in ("dq", "dk", "dv"):
            assert _rel(r[n], ref[n]) < 1e-10, (n, _rel(r[n], ref[n]))


def pin_gqa_is_repeated_mha(orc):
    """GQA equals MHA on K/V repeated G times per head (h reads h // G); dk and dv
    of the GQA call equal the MHA gradients summed over the G copies."""
    x = ne_inputs.make_custom(B=1, T=19, Hq=6, Hkv=2, d=8, seed=71)
    q, k, v, do = (ne_inputs.as_f64(x[n]) for n in ("q", "k", "v", "do"))
    G = 3
    kr, vr = np.repeat(k, G, axis=2), np.repeat(v, G, axis=2)
    o, lse = orc.attn_fwd(q, k, v, THETA)
    o2, lse2 = orc.attn_fwd(q, kr, vr, THETA)
    assert _rel(o, o2) < 1e-13 and np.abs(lse - lse2).max() < 1e-13
    r = orc.attn_bwd(q, k, v, do, THETA)
    r2 = orc.attn_bwd(q, kr, vr, do, THETA)
    dk2 = r2["dk"].reshape(1, 19, 2, G, 8).sum(axis=3)
    dv2 = r2["dv"].reshape(1, 19, 2, G, 8).sum(axis=3)
    assert _rel(r["dk"], dk2) < 1e-12 and _rel(r["dv"], dv2) < 1e-12
    assert _rel(r["dq"], r2["dq"]) < 1e-12


# ------------------------------------------------------- sliding window ----

def pin_window_torch_band_mask(orc):
    """Sliding window W against torch in float64: complex-rotation RoPE, then
    scaled_dot_product_attention with the band mask t - W < s <= t and
    autograd for the gradients of sum(O * dO); to 1e-10."""
    for (B, T, Hq, Hkv, d, W, seed) in ((1, 37, 6, 2, 16, 5, 111), (2, 30, 4, 4, 8, 1, 112),
                                        (1, 50, 4, 1, 8, 17, 113)):
        x = ne_inputs.make_custom(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=seed)
        q, k, v, do = (ne_inputs.as_f64(x[n]) for n in ("q", "k", "v", "do"))
        tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
        t = torch.arange(T)
        allowed = (t[None, :] <= t[:, None]) & (t[:, None] - t[None, :] < W)
        qr = _torch_rope(tq, THETA).transpose(1, 2)
        kr = _torch_rope(tk, THETA).transpose(1, 2)
        o = torch.nn.functional.scaled_dot_product_attention(
            qr, kr, tv.transpose(1, 2), attn_mask=allowed, scale=1.0 / math.sqrt(d),
            enable_gqa=True)
        (o * torch.tensor(do).transpose(1, 2)).sum().backward()
        with torch.no_grad():
            s = qr @ kr.repeat_interleave(Hq // Hkv, dim=1).transpose(-1, -2) / math.sqrt(d)
            lse = torch.logsumexp(s.masked_fill(~allowed, float("-inf")), dim=-1)
        o1, lse1 = orc.attn_fwd(q, k, v, THETA, window=W)
        r = orc.attn_bwd(q, k, v, do, THETA, window=W)
        assert _rel(o1, o.detach().transpose(1, 2).numpy()) < 1e-10, "o"
        assert np.abs(lse1 - lse.numpy()).max() < 1e-10, "lse"
        for n, g in (("dq", tq.grad), ("dk", tk.grad), ("dv", tv.grad)):
            assert _rel(r[n], g.numpy()) < 1e-10, (n, _rel(r[n], g.numpy()))


def pin_window_limits(orc):
    """W >= T is the causal mask (bitwise); W = 1 lets query t see key t only:
    O[t] = v[t], lse[t] = <q'_t, k'_t> / sqrt(d) (position t rotates both by
    the same angle, which leaves their dot product unchanged)."""
    x = ne_inputs.make_custom(B=2, T=23, Hq=4, Hkv=2, d=8, seed=115)
    q, k, v, do = (ne_inputs.as_f64(x[n]) for n in ("q", "k", "v", "do"))
    o0, l0 = orc.attn_fwd(q, k, v, THETA)
    o1, l1 = orc.attn_fwd(q, k, v, THETA, window=23)
    assert (o0 == o1).all() and (l0 == l1).all()
    r0 = orc.attn_bwd(q, k, v, do, THETA)
    r1 = orc.attn_bwd(q, k, v, do, THETA, window=40)
    for n in ("dq", "dk", "dv"):
        assert (r0[n] == r1[n]).all()
    o, lse = orc.attn_fwd(q, k, v, THETA, window=1)
    kk = np.repeat(k, 2, axis=2)
    assert _rel(o, np.repeat(v, 2, axis=2)) < 1e-13
    want = (q * kk).sum(-1).transpose(0, 2, 1) / math.sqrt(8)
    assert np.abs(lse - want).max() < 1e-12


# -------------------------------------------------------------- decode ----

def pin_decode_torch_sdpa(orc):
    """Decode against torch in float64: the query rotated at position Tk - 1 and
    keys at 0 .. Tk-1 (complex-rotation RoPE), then scaled_dot_product_attention
    of one query row over all keys (no mask), with GQA; to 1e-10."""
    for (B, Tk, Hq, Hkv, d, seed) in ((2, 23, 6, 2, 16, 91), (1, 40, 4, 4, 8, 92),
                                      (3, 1, 2, 1, 8, 93)):
        q1 = _rand((B, Hq, d), seed)
        k = _rand((B, Tk, Hkv, d), seed + 1)
        v = _rand((B, Tk, Hkv, d), seed + 2)
        qpad = np.zeros((B, Tk, Hq, d))
        qpad[:, -1] = q1
        qr = _torch_rope(torch.tensor(qpad), THETA)[:, -1:].transpose(1, 2)   # [B, Hq, 1, d]
        kr = _torch_rope(torch.tensor(k), THETA).transpose(1, 2)             # [B, Hkv, Tk, d]
        vv = torch.tensor(v).transpose(1, 2)
        o = torch.nn.functional.scaled_dot_product_attention(
            qr, kr, vv, scale=1.0 / math.sqrt(d), enable_gqa=True)[:, :, 0]
        s = qr @ kr.repeat_interleave(Hq // Hkv, dim=1).transpose(-1, -2) / math.sqrt(d)
        lse = torch.logsumexp(s[:, :, 0], dim=-1)
        o1, lse1 = orc.attn_decode(q1, k, v, THETA)
        assert _rel(o1, o.numpy()) < 1e-10, ("o", _rel(o1, o.numpy()))
        assert np.abs(lse1 - lse.numpy()).max() < 1e-10, "lse"


def pin_decode_is_last_causal_row(orc):
    """Decode equals the last row of the (separately pinned) causal forward over
    the same Tk positions, whatever the earlier query rows are."""
    B, Tk, Hq, Hkv, d = 2, 29, 6, 3, 8
    q = _rand((B, Tk, Hq, d), 95)
    k = _rand((B, Tk, Hkv, d), 96)
    v = _rand((B, Tk, Hkv, d), 97)
    o, lse = orc.attn_fwd(q, k, v, THETA)
    o1, lse1 = orc.attn_decode(q[:, -1], k, v, THETA)
    assert _rel(o1, o[:, -1]) < 1e-13 and np.abs(lse1 - lse[:, :, -1]).max() < 1e-12


def pin_decode_closed_forms(orc):
    """q = 0: uniform weights, O = mean of v over the cache, lse = ln Tk.
    Tk = 1: O = v[0] and lse = <q, k[0]> / sqrt(d) (position 0 rotates nothing)."""
    B, Tk, Hq, Hkv, d = 1, 17, 4, 2, 8
    v = _rand((B, Tk, Hkv, d), 98)
    o1, lse1 = orc.attn_decode(np.zeros((B, Hq, d)), _rand((B, Tk, Hkv, d), 99), v, THETA)
    mean = np.repeat(v.mean(axis=1), 2, axis=1)
    assert _rel(o1, mean) < 1e-13 and np.abs(lse1 - math.log(Tk)).max() < 1e-13
    q1 = _rand((2, 4, d), 100)
    k = _rand((2, 1, 2, d), 101)
    v = _rand((2, 1, 2, d), 102)
    o1, lse1 = orc.attn_decode(q1, k, v, THETA)
    kk = np.repeat(k[:, 0], 2, axis=1)
    assert _rel(o1, np.repeat(v[:, 0], 2, axis=1)) < 1e-14
    assert np.abs(lse1 - (q1 * kk).sum(-1) / math.sqrt(d)).max() < 1e-13


def pin_varlen_torch_sdpa(orc):
    """Padded variable-length batches against torch in float64: complex-rotation
    RoPE, scaled_dot_product_attention with a per-sequence mask (valid row t of
    sequence b sees keys s <= t; a padding row sees only itself, so torch stays
    finite there) and autograd of the sum of O * dO over valid rows only.  Valid
    rows of O and lse, and every gradient element, to 1e-10; padding rows of O
    exactly 0 and of lse exactly -inf; padding gradients exactly 0."""
    for (B, T, Hq, Hkv, d, lens, seed) in ((3, 37, 6, 2, 16, (37, 0, 20), 121),
                                           (4, 30, 4, 4, 8, (1, 29, 13, 30), 122),
                                           (2, 50, 4, 1, 8, (7, 33), 123)):
        x = ne_inputs.make_custom(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=seed)
        q, k, v, do = (ne_inputs.as_f64(x[n]) for n in ("q", "k", "v", "do"))
        L = torch.tensor(lens)
        t = torch.arange(T)
        valid = t[None, :] < L[:, None]                                   # [B, T]
        allowed = (t[None, None, :] <= t[None, :, None]) & valid[:, :, None]
        allowed = allowed | torch.eye(T, dtype=torch.bool)[None]         # padding: itself
        tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
        qr = _torch_rope(tq, THETA).transpose(1, 2)
        kr = _torch_rope(tk, THETA).transpose(1, 2)
        o = torch.nn.functional.scaled_dot_product_attention(
            qr, kr, tv.transpose(1, 2), attn_mask=allowed[:, None], scale=1.0 / math.sqrt(d),
            enable_gqa=True)
        dmask = valid[:, None, :, None].to(torch.float64)
        (o * torch.tensor(do).transpose(1, 2) * dmask).sum().backward()
        with torch.no_grad():
            sc = qr @ kr.repeat_interleave(Hq // Hkv, dim=1).transpose(-1, -2) / math.sqrt(d)
            lse = torch.logsumexp(sc.masked_fill(~allowed[:, None], float("-inf")), dim=-1)
        o1, lse1 = orc.attn_fwd_varlen(q, k, v, lens, THETA)
        r = orc.attn_bwd_varlen(q, k, v, do, lens, THETA)
        vm = valid.numpy()
        ot = o.detach().transpose(1, 2).numpy()
        assert _rel(o1[vm], ot[vm]) < 1e-10, "o"
        assert (o1[~vm] == 0).all(), "padding rows of O"
        lm = np.broadcast_to(vm[:, None, :], lse1.shape)
        assert np.abs(lse1[lm] - lse.numpy()[lm]).max() < 1e-10, "lse"
        assert np.isneginf(lse1[~lm]).all(), "padding rows of lse"
        for n, g in (("dq", tq.grad), ("dk", tk.grad), ("dv", tv.grad)):
            assert _rel(r[n], g.numpy()) < 1e-10, (n, _rel(r[n], g.numpy()))
            assert (r[n][~vm] == 0).all(), (n, "padding positions")


def pin_varlen_prefix_and_closed_forms(orc):
    """A causal row never sees a later key, so the valid rows of a padded batch
    equal the same rows of the plain causal forward over all T rows; a length
    of T is the causal forward, bit for bit.  L = 0: everything is padding
    (O = 0, lse = -inf, gradients 0).  L = 1: O[0] = v[0] of the head's group,
    lse[0] = <q_0, k_0> / sqrt(d) (position 0 rotates nothing), dq = dk = 0
    (the one probability is 1 whatever the score) and dv[0] = the sum of dO[0]
    over the group's query heads."""
    B, T, Hq, Hkv, d = 4, 21, 6, 2, 8
    x = ne_inputs.make_custom(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=125)
    q, k, v, do = (ne_inputs.as_f64(x[n]) for n in ("q", "k", "v", "do"))
    lens = (21, 0, 1, 9)
    o, lse = orc.attn_fwd_varlen(q, k, v, lens, THETA)
    oc, lc = orc.attn_fwd(q, k, v, THETA)
    assert (o[0] == oc[0]).all() and (lse[0] == lc[0]).all()
    assert _rel(o[3, :9], oc[3, :9]) < 1e-13 and np.abs(lse[3, :, :9] - lc[3, :, :9]).max() < 1e-12
    assert (o[1] == 0).all() and np.isneginf(lse[1]).all()
    G = Hq // Hkv
    assert _rel(o[2, 0], np.repeat(v[2, 0], G, axis=0)) < 1e-14
    want = (q[2, 0] * np.repeat(k[2, 0], G, axis=0)).sum(-1) / math.sqrt(d)
    assert np.abs(lse[2, :, 0] - want).max() < 1e-13
    r = orc.attn_bwd_varlen(q, k, v, do, lens, THETA)
    rc = orc.attn_bwd(q[:1], k[:1], v[:1], do[:1], THETA)
    for n in ("dq", "dk", "dv"):
        assert (r[n][0] == rc[n][0]).all(), n
        assert (r[n][1] == 0).all(), n
    assert np.abs(r["dq"][2, 0]).max() < 1e-14 and np.abs(r["dk"][2, 0]).max() < 1e-14
    assert _rel(r["dv"][2, 0], do[2, 0].reshape(Hkv, G, d).sum(axis=1)) < 1e-14


def _packed_case(lens, Hq, Hkv, d, seed):
    total = sum(lens)
    q = _rand((total, Hq, d), seed)
    k = _rand((total, Hkv, d), seed + 1)
    v = _rand((total, Hkv, d), seed + 2)
    do = _rand((total, Hq, d), seed + 3)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(int)
    return q, k, v, do, cu


def pin_packed_torch_sdpa(orc):
    """Packed batches against torch in float64: each sequence rotated at its
    own positions 0 .. len-1 (complex-rotation RoPE per segment), then one
    scaled_dot_product_attention over the whole pack with a block-diagonal
    causal mask, and autograd of sum(O * dO); to 1e-10."""
    for (lens, Hq, Hkv, d, seed) in (((5, 17, 1, 9), 6, 2, 16, 131), ((30,), 4, 4, 8, 135),
                                     ((12, 0, 21), 4, 1, 8, 139)):
        q, k, v, do, cu = _packed_case(lens, Hq, Hkv, d, seed)
        total = int(cu[-1])
        tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
        seg = torch.repeat_interleave(torch.arange(len(lens)), torch.tensor(lens))
        t = torch.arange(total)
        allowed = (seg[:, None] == seg[None, :]) & (t[None, :] <= t[:, None])
        qr = torch.cat([_torch_rope(tq[None, a:b], THETA) for a, b in zip(cu[:-1], cu[1:])
                        if b > a], dim=1).transpose(1, 2)
        kr = torch.cat([_torch_rope(tk[None, a:b], THETA) for a, b in zip(cu[:-1], cu[1:])
                        if b > a], dim=1).transpose(1, 2)
        o = torch.nn.functional.scaled_dot_product_attention(
            qr, kr, tv[None].transpose(1, 2), attn_mask=allowed, scale=1.0 / math.sqrt(d),
            enable_gqa=True)
        (o * torch.tensor(do)[None].transpose(1, 2)).sum().backward()
        with torch.no_grad():
            sc = qr @ kr.repeat_interleave(Hq // Hkv, dim=1).transpose(-1, -2) / math.sqrt(d)
            lse = torch.logsumexp(sc.masked_fill(~allowed, float("-inf")), dim=-1)[0]
        o1, lse1 = orc.attn_fwd_packed(q, k, v, cu, THETA)
        r = orc.attn_bwd_packed(q, k, v, do, cu, THETA)
        assert _rel(o1, o.detach()[0].transpose(0, 1).numpy()) < 1e-10, "o"
        assert np.abs(lse1 - lse.numpy()).max() < 1e-10, "lse"
        for n, g in (("dq", tq.grad), ("dk", tk.grad), ("dv", tv.grad)):
            assert _rel(r[n], g.numpy()) < 1e-10, (n, _rel(r[n], g.numpy()))


def pin_packed_single_tokens(orc):
    """A pack of one-token sequences: each token sees only itself, so
    O = v of its own token, lse = <q, k> / sqrt(d) (position 0 rotates
    nothing), dq = dk = 0 and dv = the sum of dO over the group's heads."""
    n, Hq, Hkv, d = 7, 6, 3, 8
    q, k, v, do, cu = _packed_case([1] * n, Hq, Hkv, d, 141)
    G = Hq // Hkv
    o, lse = orc.attn_fwd_packed(q, k, v, cu, THETA)
    assert _rel(o, np.repeat(v, G, axis=1)) < 1e-14
    want = (q * np.repeat(k, G, axis=1)).sum(-1).T / math.sqrt(d)
    assert np.abs(lse - want).max() < 1e-13
    r = orc.attn_bwd_packed(q, k, v, do, cu, THETA)
    assert np.abs(r["dq"]).max() < 1e-14 and np.abs(r["dk"]).max() < 1e-14
    assert _rel(r["dv"], do.reshape(n, Hkv, G, d).sum(axis=2)) < 1e-14


ALL_PINS = [
    pin_rope_closed_form,
    pin_rope_identity_and_orthogonal,
    pin_relative_position,
    pin_rows_sum_to_one,
    pin_causality,
    pin_single_token,
    pin_zero_query,
    pin_fwd_bwd_agree,
    pin_finite_differences,
    pin_finite_differences_tiny_workload,
    pin_torch_sdpa,
    pin_gqa_is_repeated_mha,
    pin_window_torch_band_mask,
    pin_window_limits,
    pin_decode_torch_sdpa,
    pin_decode_is_last_causal_row,
    pin_decode_closed_forms,
    pin_varlen_torch_sdpa,
    pin_varlen_prefix_and_closed_forms,
    pin_packed_torch_sdpa,
    pin_packed_single_tokens,
]
