"""The C-ABI library on the host: it loads, exports every entry point
include/ne_attn.h declares, and rejects bad arguments before any device work
(so these run without a GPU).  CPU only."""
import ctypes
import os
import re
import subprocess

import pytest

import causal_gqa_attention_ne_gb300 as ne

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ne_attn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ne_attn_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return ne.load_library()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ne_attn_fwd", "ne_attn_bwd", "ne_attn_bwd_workspace_size",
                     "ne_attn_get_error", "ne_attn_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    exported = subprocess.run(["nm", "-D", "--defined-only", ne.lib_path()],
                              capture_output=True, text=True, check=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}$", exported, re.M), f"{n} not exported"
        assert hasattr(lib, n)
    assert set(ne._binding.EXPORTED) == set(names)


def test_status_strings(lib):
    for code in range(12):
        s = ne.ne_attn_status_string(code)
        assert s and s != "unknown status"
    assert ne.ne_attn_status_string(99) == "unknown status"


def test_workspace_size(lib):
    # D (fp32 B*Hq*T) + Q' (fp16 B*T*Hq*d) + K' (fp16 B*T*Hkv*d), 256-aligned each
    def r256(x):
        return (x + 255) // 256 * 256
    for (B, T, Hq, Hkv, d) in ((1, 128, 4, 2, 32), (16, 512, 12, 4, 64), (4, 4096, 16, 4, 128),
                               (3, 7, 5, 1, 64)):
        want = r256(B * Hq * T * 4) + r256(B * T * Hq * d * 2) + r256(B * T * Hkv * d * 2)
        assert ne.ne_attn_bwd_workspace_size(B, T, Hq, Hkv, d) == want
    assert ne.ne_attn_bwd_workspace_size(1, 8, 3, 2, 64) == 0      # Hq % Hkv != 0
    assert ne.ne_attn_bwd_workspace_size(1, 8, 2, 2, 48) == 0      # unsupported d


def _fwd(lib, ptrs, B=1, T=8, Hq=2, Hkv=2, d=64, theta=10000.0):
    return lib.ne_attn_fwd(*ptrs, B, T, Hq, Hkv, d, theta, None)


def test_forward_argument_errors(lib):
    buf = ctypes.create_string_buffer(4096 + 64)
    a = (ctypes.addressof(buf) + 15) // 16 * 16
    ok = [a, a, a, a, a]
    assert _fwd(lib, [None, a, a, a, a]) == 1                       # NE_ERR_NULL
    assert _fwd(lib, ok, B=0) == 2                                  # NE_ERR_SHAPE
    assert _fwd(lib, ok, Hq=3, Hkv=2) == 2                          # Hq % Hkv
    assert _fwd(lib, ok, d=48) == 3                                 # NE_ERR_UNSUPPORTED
    assert _fwd(lib, ok, theta=0.0) == 9                            # NE_ERR_ARG
    assert _fwd(lib, ok, theta=float("nan")) == 9
    assert _fwd(lib, [a + 2, a, a, a, a]) == 4                      # NE_ERR_ALIGN


def test_backward_argument_errors(lib):
    buf = ctypes.create_string_buffer(4096)
    a = (ctypes.addressof(buf) + 15) // 16 * 16
    args = [a] * 9
    # short workspace
    assert lib.ne_attn_bwd(*args, a, 0, 1, 8, 2, 2, 64, 10000.0, None) == 5
    # null gradient
    assert lib.ne_attn_bwd(*args[:6], None, a, a, a, 1 << 20, 1, 8, 2, 2, 64, 10000.0,
                           None) == 1
    # no-allocation variant: shape whose scratch exceeds its fixed buffer
    assert lib.ne_attn_bwd_noalloc(*args, 8, 4096, 8, 8, 128, 10000.0, None) == 10
    assert lib.ne_attn_bwd_noalloc(*args, 1, 8, 3, 2, 64, 10000.0, None) == 2
    # pointer checks come first, as in ne_attn_bwd: an oversized shape with a
    # NULL or misaligned pointer reports the pointer
    for i in range(9):
        bad = list(args)
        bad[i] = None
        assert lib.ne_attn_bwd_noalloc(*bad, 8, 4096, 8, 8, 128, 10000.0, None) == 1
    for i in (0, 1, 2, 3, 5, 6, 7, 8):          # 16-byte tensors (lse at 4 needs 4 bytes)
        bad = list(args)
        bad[i] = a + 2
        assert lib.ne_attn_bwd_noalloc(*bad, 1, 8, 2, 2, 64, 10000.0, None) == 4
        assert lib.ne_attn_bwd(*bad, a, 1 << 20, 1, 8, 2, 2, 64, 10000.0, None) == 4


def test_varlen_device_lengths_argument_errors(lib):
    buf = ctypes.create_string_buffer(1 << 16)
    a = (ctypes.addressof(buf) + 15) // 16 * 16
    ws = ne.ne_attn_varlen_workspace_size(2, 8, 2, 2, 64)
    args = (2, 8, 2, 2, 64, 10000.0, None)
    fwd, bwd = lib.ne_attn_fwd_varlen_dev, lib.ne_attn_bwd_varlen_dev
    assert fwd(a, a, a, a, a, None, a, ws, *args) == 1                # NE_ERR_NULL: seqlens
    assert fwd(a, a, a, a, a, a + 2, a, ws, *args) == 4               # lengths 4-byte aligned
    assert fwd(a, a, a, a, a, a, a, 16, *args) == 5                   # short workspace
    assert fwd(a, a, a, a, a, a, a, ws, 2, 8, 3, 2, 64, 10000.0, None) == 2
    assert bwd(*([a] * 9), None, a, ws, *args) == 1
    assert bwd(*([a] * 9), a, a, ws - 1, *args) == 5


def test_decode_workspace_size_and_argument_errors(lib):
    def r256(x):
        return (x + 255) // 256 * 256
    for (B, Tk, Hq, Hkv, d) in ((1, 1, 4, 2, 32), (64, 512, 12, 4, 64), (3, 1000, 16, 4, 128)):
        rows = B * Hq * ((Tk + 127) // 128)
        assert ne.ne_attn_decode_workspace_size(B, Tk, Hq, Hkv, d) == r256(rows * d * 4) + \
            r256(rows * 2 * 4)
    assert ne.ne_attn_decode_workspace_size(1, 8, 3, 2, 64) == 0      # Hq % Hkv != 0
    buf = ctypes.create_string_buffer(1 << 16)
    a = (ctypes.addressof(buf) + 15) // 16 * 16
    ws = 1 << 15
    dec = lib.ne_attn_decode
    assert dec(None, a, a, a, a, a, ws, 1, 8, 2, 2, 64, 10000.0, None) == 1    # NE_ERR_NULL
    assert dec(a, a, a, a, a, a, ws, 1, 0, 2, 2, 64, 10000.0, None) == 2       # Tk = 0
    assert dec(a, a, a, a, a, a, ws, 1, 8, 2, 2, 48, 10000.0, None) == 3       # d
    assert dec(a, a, a, a, a, a, ws, 1, 8, 34, 2, 64, 10000.0, None) == 3      # group of 17
    assert dec(a, a, a, a, a, a, 0, 1, 8, 2, 2, 64, 10000.0, None) == 5        # workspace
    assert dec(a + 2, a, a, a, a, a, ws, 1, 8, 2, 2, 64, 10000.0, None) == 4   # alignment


def test_window_argument_errors(lib):
    buf = ctypes.create_string_buffer(4096 + 64)
    a = (ctypes.addressof(buf) + 15) // 16 * 16
    assert lib.ne_attn_fwd_window(a, a, a, a, a, 1, 8, 2, 2, 64, 10000.0, -1, None) == 9
    assert lib.ne_attn_bwd_window(*([a] * 10), 1 << 20, 1, 8, 2, 2, 64, 10000.0, -3, None) == 9


def test_packed_workspace_size_and_argument_errors(lib):
    def r256(x):
        return (x + 255) // 256 * 256
    # [lengths][cu][fwd units][dq units][dk/dv units][plan counts][plan scratch]
    # + the backward workspace of
    # a [1][total] batch; live tiles per kv head <= total // 128 + nseq
    nseq, total, Hq, Hkv, d = 3, 300, 12, 4, 64
    tiles = (total // 128 + nseq) * Hkv
    M = (total + 127) // 128     # + the device-side plan's counts and scratch
    want = (r256(4 * nseq) + r256(4 * (nseq + 1)) + r256(4 * tiles) + r256(4 * tiles) +
            r256(4 * tiles) + r256(16) + r256(4 * (2 * nseq + 2 * (M + 2))) +
            ne.ne_attn_bwd_workspace_size(1, total, Hq, Hkv, d))
    assert ne.ne_attn_packed_workspace_size(nseq, total, Hq, Hkv, d) == want
    assert ne.ne_attn_packed_workspace_size(0, total, Hq, Hkv, d) == 0
    assert ne.ne_attn_packed_workspace_size(1, 0, Hq, Hkv, d) == 0
    buf = ctypes.create_string_buffer(1 << 16)
    a = (ctypes.addressof(buf) + 15) // 16 * 16
    ws = 1 << 15

    def fwd(cu, nseq, total, wsb=ws, d=64):
        arr = (ctypes.c_int32 * len(cu))(*cu) if cu is not None else None
        return lib.ne_attn_fwd_packed(a, a, a, a, a, arr, a, wsb, nseq, total, 2, 2, d,
                                      10000.0, None)

    assert fwd(None, 2, 10) == 1                 # NE_ERR_NULL
    assert fwd([0, 10], 0, 10) == 2              # no sequences
    assert fwd([0, 0], 1, 0) == 2                # empty pack
    assert fwd([1, 10], 1, 10) == 9              # cu[0] != 0
    assert fwd([0, 6, 4, 10], 3, 10) == 9        # decreasing
    assert fwd([0, 4, 9], 2, 10) == 9            # cu[nseq] != total
    assert fwd([0, 4, 10], 2, 10, d=48) == 3     # head dim
    assert fwd([0, 4, 10], 2, 10, wsb=0) == 5    # workspace
    cu = (ctypes.c_int32 * 3)(0, 4, 10)
    assert lib.ne_attn_bwd_packed(a, a, a, a, a, a, a, a, a, cu, a, 0, 2, 10, 2, 2, 64,
                                  10000.0, None) == 5
    dev = lib.ne_attn_fwd_packed_dev
    assert dev(a, a, a, a, a, None, a, ws, 2, 10, 2, 2, 64, 10000.0, None) == 1
    assert dev(a, a, a, a, a, a + 2, a, ws, 2, 10, 2, 2, 64, 10000.0, None) == 4
    assert dev(a, a, a, a, a, a, a, ws, 0, 10, 2, 2, 64, 10000.0, None) == 2
    assert dev(a, a, a, a, a, a, a, 0, 2, 10, 2, 2, 64, 10000.0, None) == 5
    assert lib.ne_attn_bwd_packed_dev(a, a, a, a, a, a, a, a, a, None, a, 1 << 15, 2, 10, 2, 2,
                                      64, 10000.0, None) == 1
