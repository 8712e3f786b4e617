"""Host side of padded variable-length batches (no GPU): the work-unit tables
the library builds (ne_attn_varlen_plan returns them from the same host image
the varlen entry points copy into the workspace), the workspace size and the
argument errors of the varlen entry points.

Each table entry is an index into a kernel's full unit enumeration.  The
decoding below restates that enumeration: forward and dq take
u -> query tile m = M-1 - u // (B Hkv nchunks), then (chunk, kv head j, b);
dk/dv takes u -> key tile n = u // (B Hkv), then (j, b).  A unit is live when
its tile holds a valid row of sequence b (128 * tile < L_b).  CPU only."""
import ctypes

import numpy as np
import pytest

import causal_gqa_attention_ne_gb300 as ne


def heads_per_cta(d, G, cap):
    return max(g for g in range(1, cap + 1) if G % g == 0)


def chunks(d, G):
    fwd = G // heads_per_cta(d, G, {32: 4, 64: 3, 128: 2}[d])
    dq = G // (1 if d == 128 else heads_per_cta(d, G, {32: 4, 64: 3}[d]))
    return fwd, dq


CASES = [
    # (lengths, T, Hq, Hkv, d)
    ([300, 0, 128, 129, 512], 512, 12, 4, 64),
    ([1, 2, 3], 130, 4, 2, 32),
    ([0, 0], 64, 8, 8, 128),
    ([512] * 6, 512, 12, 4, 64),
    (list(np.random.default_rng(7).integers(0, 1001, 37)), 1000, 6, 2, 128),
    (list(np.random.default_rng(8).integers(0, 385, 64)), 384, 16, 4, 32),
    # d = 128, G = 4: the forward, dq and dk/dv tables hold 2, 4 and 1 units per
    # tile, so their regions in the workspace image differ in size
    ([520, 391, 9], 520, 16, 4, 128),
    (list(np.random.default_rng(9).integers(0, 513, 64)), 512, 16, 4, 128),
]


@pytest.mark.parametrize("lens,T,Hq,Hkv,d", CASES)
def test_unit_tables(lens, T, Hq, Hkv, d):
    B, G, M = len(lens), Hq // Hkv, (T + 127) // 128
    mt = [(L + 127) // 128 for L in lens]
    counts, (tf, tq, tk) = ne.ne_attn_varlen_plan(lens, T, Hq, Hkv, d)
    nf, nq = chunks(d, G)
    for table, nch, name in ((tf, nf, "fwd"), (tq, nq, "dq")):
        per_m = B * Hkv * nch
        assert len(table) == len(set(table.tolist())), name          # no unit twice
        assert ((table >= 0) & (table < M * per_m)).all(), name
        units = []
        for u in table.tolist():
            m = M - 1 - u // per_m
            rem = u % per_m
            c, j, b = rem % nch, (rem // nch) % Hkv, rem // nch // Hkv
            units.append((m, b, j, c))
        want = {(m, b, j, c) for b in range(B) for m in range(mt[b]) for j in range(Hkv)
                for c in range(nch)}
        assert set(units) == want, name                               # exactly the live ones
        ms = [u[0] for u in units]
        assert ms == sorted(ms, reverse=True), name                   # decreasing work
    per_n = B * Hkv
    assert len(tk) == len(set(tk.tolist()))
    assert ((tk >= 0) & (tk < M * per_n)).all()
    units = [(u // per_n, (u % per_n) // Hkv, u % Hkv) for u in tk.tolist()]
    want = {(n, b, j) for b in range(B) for n in range(mt[b]) for j in range(Hkv)}
    assert set(units) == want
    work = [mt[b] - n for (n, b, j) in units]
    assert work == sorted(work, reverse=True)
    assert counts == [len(tf), len(tq), len(tk)]
    assert ne.ne_attn_varlen_plan(lens, T, Hq, Hkv, d, with_tables=False)[0] == counts


def test_all_full_lengths_list_every_unit_in_launch_order():
    """With every length T the tables are the full enumerations, in order: the
    varlen launch then does exactly what the causal launch does."""
    B, T, Hq, Hkv, d = 3, 300, 12, 4, 64
    counts, (tf, tq, tk) = ne.ne_attn_varlen_plan([T] * B, T, Hq, Hkv, d)
    M = (T + 127) // 128
    nf, nq = chunks(d, Hq // Hkv)
    assert (tf == np.arange(M * B * Hkv * nf)).all()
    assert (tq == np.arange(M * B * Hkv * nq)).all()
    assert (tk == np.arange(M * B * Hkv)).all()


def test_workspace_size():
    def r256(x):
        return (x + 255) // 256 * 256
    for (B, T, Hq, Hkv, d) in ((64, 512, 12, 4, 64), (3, 7, 5, 1, 32), (2, 1000, 16, 4, 128)):
        G, tiles = Hq // Hkv, (T + 127) // 128 * B * Hkv
        nf, nq = chunks(d, G)
        M = (T + 127) // 128
        # + the device-side plan's counts (int32 [4]) and scratch (int32 [2B + 2(M + 2)])
        tables = r256(4 * B) + r256(4 * tiles * nf) + r256(4 * tiles * nq) + r256(4 * tiles) + \
            r256(16) + r256(4 * (2 * B + 2 * (M + 2)))
        assert ne.ne_attn_varlen_workspace_size(B, T, Hq, Hkv, d) == \
            tables + ne.ne_attn_bwd_workspace_size(B, T, Hq, Hkv, d)
    assert ne.ne_attn_varlen_workspace_size(1, 8, 3, 2, 64) == 0      # Hq % Hkv != 0


def test_argument_errors():
    lib = ne.load_library()
    buf = ctypes.create_string_buffer(1 << 16)
    a = (ctypes.addressof(buf) + 15) // 16 * 16
    ok = (ctypes.c_int32 * 2)(5, 8)
    bad = (ctypes.c_int32 * 2)(5, 9)
    neg = (ctypes.c_int32 * 2)(-1, 8)
    ws = ne.ne_attn_varlen_workspace_size(2, 8, 2, 2, 64)
    fwd, bwd = lib.ne_attn_fwd_varlen, lib.ne_attn_bwd_varlen
    args = (2, 8, 2, 2, 64, 10000.0, None)
    assert fwd(a, a, a, a, a, None, a, ws, *args) == 1                # NE_ERR_NULL: seqlens
    assert fwd(a, a, a, a, a, bad, a, ws, *args) == 9                 # a length above T
    assert fwd(a, a, a, a, a, neg, a, ws, *args) == 9                 # a negative length
    assert fwd(a, a, a, a, a, ok, a, 16, *args) == 5                  # short workspace
    assert fwd(a + 2, a, a, a, a, ok, a, ws, *args) == 4              # alignment
    assert fwd(a, a, a, a, a, ok, a, ws, 2, 8, 2, 2, 48, 10000.0, None) == 3   # d
    assert bwd(*([a] * 9), None, a, ws, *args) == 1
    assert bwd(*([a] * 9), bad, a, ws, *args) == 9
    assert bwd(*([a] * 9), ok, a, ws - 1, *args) == 5                 # needs the whole size
    assert bwd(*([a] * 6), a + 8, a, a, ok, a, ws, *args) == 4        # dq alignment
    counts = (ctypes.c_int32 * 3)()
    assert lib.ne_attn_varlen_plan(bad, 2, 8, 2, 2, 64, None, None, None, 0, counts) == 9
    assert lib.ne_attn_varlen_plan(ok, 2, 8, 3, 2, 64, None, None, None, 0, counts) == 2
    assert lib.ne_attn_varlen_plan(ok, 2, 8, 2, 2, 64, None, None, None, 0, None) == 1
    assert lib.ne_attn_varlen_plan(None, 2, 8, 2, 2, 64, None, None, None, 0, counts) == 1
    assert lib.ne_attn_varlen_plan(ok, 2, 8, 2, 2, 48, None, None, None, 0, counts) == 3
    assert lib.ne_attn_varlen_plan(ok, 2, 8, 2, 2, 64, None, None, None, 0, counts) == 0
    assert list(counts) == [4, 4, 4]      # 2 sequences x 1 tile x 2 kv heads (G = 1)
