"""CPU oracle for causal GQA attention with RoPE (forward and backward), float64.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only users.  The CUDA library never calls
into this package and this package never imports the CUDA library.

The arithmetic lives in ``ne_oracle.c`` (plain C, double precision, the full
T x T score matrix).  This module compiles it on first use with the host C
compiler and wraps it with ctypes.  What it computes, and where on the pages
each step comes from, is stated in the header of ``ne_oracle.c``:

* "NanoEuler: a GPT-2-scale LLM built from scratch in C and CUDA",
  technical specification (RoPE on queries and keys; GQA; decoder-only) and
  validation section (analytic gradients checked by central finite
  differences in double precision);
* "Rebuilding GPT-2 in one 100KB C/CUDA file (NanoEuler 116M walkthrough)",
  section 3.4 (tiled FlashAttention with an online softmax, which is an exact
  reorganisation of softmax attention, so the oracle is softmax attention).

Every function is pinned by tests in ``tests/test_oracle.py`` against closed
forms, invariants, finite differences and torch's CPU attention routine.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ne_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libne_oracle.so")
_lock = threading.Lock()
_lib = None

_DP = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile ne_oracle.c into libne_oracle.so next to it (gcc, OpenMP, -O2)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


def _bind(path: str):
    lib = ctypes.CDLL(path)
    lib.ne_oracle_rope.restype = ctypes.c_int
    lib.ne_oracle_rope.argtypes = [_DP, _DP] + [ctypes.c_int] * 4 + [
        ctypes.c_double, ctypes.c_long, ctypes.c_int]
    lib.ne_oracle_fwd.restype = ctypes.c_int
    lib.ne_oracle_fwd.argtypes = [_DP] * 5 + [ctypes.c_int] * 5 + [
        ctypes.c_double, ctypes.c_long, ctypes.c_int, ctypes.c_int]
    lib.ne_oracle_bwd.restype = ctypes.c_int
    lib.ne_oracle_bwd.argtypes = [_DP] * 10 + [ctypes.c_int] * 5 + [
        ctypes.c_double, ctypes.c_long, ctypes.c_int, ctypes.c_int]
    lib.ne_oracle_decode.restype = ctypes.c_int
    lib.ne_oracle_decode.argtypes = [_DP] * 5 + [ctypes.c_int] * 5 + [
        ctypes.c_double, ctypes.c_long]
    _IP = ctypes.POINTER(ctypes.c_int)
    lib.ne_oracle_fwd_varlen.restype = ctypes.c_int
    lib.ne_oracle_fwd_varlen.argtypes = [_DP] * 5 + [_IP] + [ctypes.c_int] * 5 + [
        ctypes.c_double, ctypes.c_long, ctypes.c_int]
    lib.ne_oracle_bwd_varlen.restype = ctypes.c_int
    lib.ne_oracle_bwd_varlen.argtypes = [_DP] * 7 + [_IP] + [ctypes.c_int] * 5 + [
        ctypes.c_double, ctypes.c_long, ctypes.c_int]
    lib.ne_oracle_fwd_packed.restype = ctypes.c_int
    lib.ne_oracle_fwd_packed.argtypes = [_DP] * 5 + [_IP] + [ctypes.c_int] * 4 + [
        ctypes.c_double, ctypes.c_long, ctypes.c_int]
    lib.ne_oracle_bwd_packed.restype = ctypes.c_int
    lib.ne_oracle_bwd_packed.argtypes = [_DP] * 7 + [_IP] + [ctypes.c_int] * 4 + [
        ctypes.c_double, ctypes.c_long, ctypes.c_int]
    lib.ne_oracle_max_threads.restype = ctypes.c_int
    return lib


def _c(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float64)


def _p(x):
    return None if x is None else x.ctypes.data_as(_DP)


class Oracle:
    """The oracle's entry points bound to one compiled copy of ne_oracle.c."""

    def __init__(self, lib):
        self._lib = lib

    def max_threads(self) -> int:
        return self._lib.ne_oracle_max_threads()

    def rope(self, x, theta: float, pos_offset: int = 0, inverse: bool = False):
        """Rotate-half RoPE of a [B, T, H, d] array: R(t + pos_offset) x, or R^T x if inverse."""
        x = _c(x)
        B, T, H, d = x.shape
        y = np.empty_like(x)
        rc = self._lib.ne_oracle_rope(_p(x), _p(y), B, T, H, d, float(theta), int(pos_offset),
                                      int(inverse))
        if rc:
            raise ValueError(f"ne_oracle_rope rejected shape {x.shape}")
        return y

    def attn_fwd(self, q, k, v, theta: float, pos_offset: int = 0, threads: int = 0,
                 window: int = 0):
        """Causal GQA attention with RoPE (window W > 0: query t sees keys t-W+1 .. t).
        Returns (o [B,T,Hq,d], lse [B,Hq,T])."""
        q, k, v = _c(q), _c(k), _c(v)
        B, T, Hq, d = q.shape
        Hkv = k.shape[2]
        if k.shape != (B, T, Hkv, d) or v.shape != k.shape:
            raise ValueError("k and v must be [B, T, Hkv, d] matching q")
        o = np.empty_like(q)
        lse = np.empty((B, Hq, T), dtype=np.float64)
        rc = self._lib.ne_oracle_fwd(_p(q), _p(k), _p(v), _p(o), _p(lse), B, T, Hq, Hkv, d,
                                     float(theta), int(pos_offset), int(threads), int(window))
        if rc:
            raise ValueError(f"ne_oracle_fwd failed with code {rc}")
        return o, lse

    def attn_bwd(self, q, k, v, do, theta: float, pos_offset: int = 0, threads: int = 0,
                 window: int = 0):
        """Gradients of sum(O * dO): dict with dq, dk, dv and the oracle's o, lse, D."""
        q, k, v, do = _c(q), _c(k), _c(v), _c(do)
        B, T, Hq, d = q.shape
        Hkv = k.shape[2]
        if do.shape != q.shape or k.shape != (B, T, Hkv, d) or v.shape != k.shape:
            raise ValueError("shape mismatch")
        dq = np.empty_like(q)
        dk = np.empty_like(k)
        dv = np.empty_like(v)
        o = np.empty_like(q)
        lse = np.empty((B, Hq, T), dtype=np.float64)
        D = np.empty((B, Hq, T), dtype=np.float64)
        rc = self._lib.ne_oracle_bwd(_p(q), _p(k), _p(v), _p(do), _p(dq), _p(dk), _p(dv),
                                     _p(o), _p(lse), _p(D), B, T, Hq, Hkv, d, float(theta),
                                     int(pos_offset), int(threads), int(window))
        if rc:
            raise ValueError(f"ne_oracle_bwd failed with code {rc}")
        return {"dq": dq, "dk": dk, "dv": dv, "o": o, "lse": lse, "D": D}


    def attn_decode(self, q1, k, v, theta: float, pos_offset: int = 0):
        """One new token per sequence against a [B, Tk, Hkv, d] key/value cache whose
        last row is the token's own: the last row of causal attention over Tk
        positions.  q1 is [B, Hq, d].  Returns (o1 [B, Hq, d], lse1 [B, Hq])."""
        q1, k, v = _c(q1), _c(k), _c(v)
        B, Hq, d = q1.shape
        Tk, Hkv = k.shape[1], k.shape[2]
        if k.shape != (B, Tk, Hkv, d) or v.shape != k.shape:
            raise ValueError("k and v must be [B, Tk, Hkv, d] matching q1")
        o1 = np.empty_like(q1)
        lse1 = np.empty((B, Hq), dtype=np.float64)
        rc = self._lib.ne_oracle_decode(_p(q1), _p(k), _p(v), _p(o1), _p(lse1), B, Tk, Hq, Hkv,
                                        d, float(theta), int(pos_offset))
        if rc:
            raise ValueError(f"ne_oracle_decode failed with code {rc}")
        return o1, lse1


    def _seqlens(self, seqlens, B: int):
        sl = np.ascontiguousarray(np.asarray(seqlens).reshape(-1), dtype=np.intc)
        if sl.shape != (B,):
            raise ValueError(f"seqlens must hold {B} lengths")
        return sl

    def attn_fwd_varlen(self, q, k, v, seqlens, theta: float, pos_offset: int = 0,
                        threads: int = 0):
        """Padded variable-length batch: sequence b is its first seqlens[b] rows, a
        causal problem of its own; padding rows get O = 0 and lse = -inf.
        Returns (o [B,T,Hq,d], lse [B,Hq,T])."""
        q, k, v = _c(q), _c(k), _c(v)
        B, T, Hq, d = q.shape
        Hkv = k.shape[2]
        if k.shape != (B, T, Hkv, d) or v.shape != k.shape:
            raise ValueError("k and v must be [B, T, Hkv, d] matching q")
        sl = self._seqlens(seqlens, B)
        o = np.empty_like(q)
        lse = np.empty((B, Hq, T), dtype=np.float64)
        rc = self._lib.ne_oracle_fwd_varlen(
            _p(q), _p(k), _p(v), _p(o), _p(lse), sl.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
            B, T, Hq, Hkv, d, float(theta), int(pos_offset), int(threads))
        if rc:
            raise ValueError(f"ne_oracle_fwd_varlen failed with code {rc}")
        return o, lse

    def attn_bwd_varlen(self, q, k, v, do, seqlens, theta: float, pos_offset: int = 0,
                        threads: int = 0):
        """Gradients of the sum of O * dO over the valid rows of a padded
        variable-length batch; 0 on padding positions.  Dict with dq, dk, dv."""
        q, k, v, do = _c(q), _c(k), _c(v), _c(do)
        B, T, Hq, d = q.shape
        Hkv = k.shape[2]
        if do.shape != q.shape or k.shape != (B, T, Hkv, d) or v.shape != k.shape:
            raise ValueError("shape mismatch")
        sl = self._seqlens(seqlens, B)
        dq = np.empty_like(q)
        dk = np.empty_like(k)
        dv = np.empty_like(v)
        rc = self._lib.ne_oracle_bwd_varlen(
            _p(q), _p(k), _p(v), _p(do), _p(dq), _p(dk), _p(dv),
            sl.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), B, T, Hq, Hkv, d, float(theta),
            int(pos_offset), int(threads))
        if rc:
            raise ValueError(f"ne_oracle_bwd_varlen failed with code {rc}")
        return {"dq": dq, "dk": dk, "dv": dv}


    def _cu(self, cu_seqlens, total: int):
        cu = np.ascontiguousarray(np.asarray(cu_seqlens).reshape(-1), dtype=np.intc)
        if cu.shape[0] < 2 or cu[0] != 0 or cu[-1] != total or (np.diff(cu) < 0).any():
            raise ValueError("cu_seqlens must start at 0, not decrease and end at the pack length")
        return cu

    def attn_fwd_packed(self, q, k, v, cu_seqlens, theta: float, pos_offset: int = 0,
                        threads: int = 0):
        """Packed variable-length batch: q [total, Hq, d], k and v [total, Hkv, d];
        sequence b is tokens cu_seqlens[b] .. cu_seqlens[b+1]-1, a causal problem
        of its own (positions restart at 0).  Returns (o [total,Hq,d], lse [Hq,total])."""
        q, k, v = _c(q), _c(k), _c(v)
        total, Hq, d = q.shape
        Hkv = k.shape[1]
        if k.shape != (total, Hkv, d) or v.shape != k.shape:
            raise ValueError("k and v must be [total, Hkv, d] matching q")
        cu = self._cu(cu_seqlens, total)
        o = np.zeros_like(q)
        lse = np.full((Hq, total), -np.inf)
        rc = self._lib.ne_oracle_fwd_packed(
            _p(q), _p(k), _p(v), _p(o), _p(lse), cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
            cu.shape[0] - 1, Hq, Hkv, d, float(theta), int(pos_offset), int(threads))
        if rc:
            raise ValueError(f"ne_oracle_fwd_packed failed with code {rc}")
        return o, lse

    def attn_bwd_packed(self, q, k, v, do, cu_seqlens, theta: float, pos_offset: int = 0,
                        threads: int = 0):
        """Gradients of sum(O * dO) for a packed batch.  Dict with dq, dk, dv."""
        q, k, v, do = _c(q), _c(k), _c(v), _c(do)
        total, Hq, d = q.shape
        Hkv = k.shape[1]
        if do.shape != q.shape or k.shape != (total, Hkv, d) or v.shape != k.shape:
            raise ValueError("shape mismatch")
        cu = self._cu(cu_seqlens, total)
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        rc = self._lib.ne_oracle_bwd_packed(
            _p(q), _p(k), _p(v), _p(do), _p(dq), _p(dk), _p(dv),
            cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), cu.shape[0] - 1, Hq, Hkv, d,
            float(theta), int(pos_offset), int(threads))
        if rc:
            raise ValueError(f"ne_oracle_bwd_packed failed with code {rc}")
        return {"dq": dq, "dk": dk, "dv": dv}


def compile_source(src_path: str, lib_path: str) -> str:
    """Compile one copy of the oracle's C source into a shared library."""
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src_path, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib_path)
    return lib_path


def load_from(lib_path: str) -> Oracle:
    """Bind an Oracle to a specific compiled copy (tests use this for planted mistakes)."""
    return Oracle(_bind(lib_path))


def default() -> Oracle:
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(_bind(build()))
    return _lib


def max_threads() -> int:
    return default().max_threads()


def rope(x, theta: float, pos_offset: int = 0, inverse: bool = False):
    return default().rope(x, theta, pos_offset, inverse)


def attn_fwd(q, k, v, theta: float, pos_offset: int = 0, threads: int = 0, window: int = 0):
    return default().attn_fwd(q, k, v, theta, pos_offset, threads, window)


def attn_bwd(q, k, v, do, theta: float, pos_offset: int = 0, threads: int = 0,
             window: int = 0):
    return default().attn_bwd(q, k, v, do, theta, pos_offset, threads, window)


def attn_decode(q1, k, v, theta: float, pos_offset: int = 0):
    return default().attn_decode(q1, k, v, theta, pos_offset)


def attn_fwd_varlen(q, k, v, seqlens, theta: float, pos_offset: int = 0, threads: int = 0):
    return default().attn_fwd_varlen(q, k, v, seqlens, theta, pos_offset, threads)


def attn_bwd_varlen(q, k, v, do, seqlens, theta: float, pos_offset: int = 0, threads: int = 0):
    return default().attn_bwd_varlen(q, k, v, do, seqlens, theta, pos_offset, threads)


def attn_fwd_packed(q, k, v, cu_seqlens, theta: float, pos_offset: int = 0, threads: int = 0):
    return default().attn_fwd_packed(q, k, v, cu_seqlens, theta, pos_offset, threads)


def attn_bwd_packed(q, k, v, do, cu_seqlens, theta: float, pos_offset: int = 0,
                    threads: int = 0):
    return default().attn_bwd_packed(q, k, v, do, cu_seqlens, theta, pos_offset, threads)


def group_slice(x: np.ndarray, b: int, j: int, heads_per_group: int):
    """Slice one (batch b, kv head j) group out of a [B, T, H, d] array, H = Hq or Hkv.

    Groups are independent in the definition (query head h only reads kv head
    h // G), so the oracle on a group slice equals the same slice of the
    oracle on the whole tensor.
    """
    return x[b:b + 1, :, j * heads_per_group:(j + 1) * heads_per_group, :]
