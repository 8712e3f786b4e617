"""ctypes binding of libne_attn.so with the same entry-point names as the C ABI.

Argument marshalling only: shape/dtype/device checks that keep the raw
pointers in bounds, then one call into the library.  Streams are torch's
current CUDA stream unless one is given.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

from . import _build

NE_STATUS = {
    0: "NE_OK", 1: "NE_ERR_NULL", 2: "NE_ERR_SHAPE", 3: "NE_ERR_UNSUPPORTED", 4: "NE_ERR_ALIGN",
    5: "NE_ERR_WORKSPACE", 6: "NE_ERR_CUDA", 7: "NE_ERR_TIMEOUT", 8: "NE_ERR_RANGE",
    9: "NE_ERR_ARG", 10: "NE_ERR_TOO_LARGE", 11: "NE_WARN_PRECISION",
}

EXPORTED = ("ne_attn_fwd", "ne_attn_bwd", "ne_attn_bwd_workspace_size", "ne_attn_bwd_preprocess",
            "ne_attn_bwd_dq", "ne_attn_bwd_dkdv", "ne_attn_get_error", "ne_attn_status_string",
            "ne_attn_set_wait_limit_ns", "ne_attn_selftest_timeout", "ne_attn_bwd_noalloc",
            "ne_attn_bwd_noalloc_max_scratch", "ne_attn_fwd_save", "ne_attn_bwd_saved",
            "ne_attn_bwd_preprocess_d", "ne_attn_decode", "ne_attn_decode_workspace_size",
            "ne_attn_fwd_window", "ne_attn_bwd_window", "ne_attn_varlen_workspace_size",
            "ne_attn_fwd_varlen", "ne_attn_bwd_varlen", "ne_attn_varlen_plan",
            "ne_attn_packed_workspace_size", "ne_attn_fwd_packed", "ne_attn_bwd_packed",
            "ne_attn_fwd_varlen_dev", "ne_attn_bwd_varlen_dev", "ne_attn_fwd_packed_dev",
            "ne_attn_bwd_packed_dev")

_lock = threading.Lock()
_lib = None


class NeAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {NE_STATUS.get(status, status)} "
                         f"({_status_text(status)})")


def lib_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = True):
    """Load libne_attn.so (building it first if it is absent)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB):
            if not build_if_missing:
                raise RuntimeError(f"{_build.LIB} is missing; run causal_gqa_attention_ne_gb300"
                                   "._build.build() (needs nvcc)")
            _build.build()
        lib = ctypes.CDLL(_build.LIB)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.ne_attn_fwd.argtypes = [vp] * 5 + [i] * 5 + [f, vp]
        lib.ne_attn_fwd.restype = i
        lib.ne_attn_bwd.argtypes = [vp] * 10 + [sz] + [i] * 5 + [f, vp]
        lib.ne_attn_bwd.restype = i
        lib.ne_attn_fwd_save.argtypes = [vp] * 6 + [sz] + [i] * 5 + [f, i, vp]
        lib.ne_attn_fwd_save.restype = i
        lib.ne_attn_bwd_saved.argtypes = [vp] * 10 + [sz] + [i] * 5 + [f, i, vp]
        lib.ne_attn_bwd_saved.restype = i
        lib.ne_attn_bwd_preprocess_d.argtypes = [vp] * 3 + [sz] + [i] * 5 + [vp]
        lib.ne_attn_bwd_preprocess_d.restype = i
        lib.ne_attn_bwd_preprocess.argtypes = [vp] * 5 + [sz] + [i] * 5 + [f, vp]
        lib.ne_attn_bwd_preprocess.restype = i
        lib.ne_attn_bwd_dq.argtypes = [vp] * 7 + [sz] + [i] * 5 + [f, vp]
        lib.ne_attn_bwd_dq.restype = i
        lib.ne_attn_bwd_dkdv.argtypes = [vp] * 8 + [sz] + [i] * 5 + [f, vp]
        lib.ne_attn_bwd_dkdv.restype = i
        lib.ne_attn_bwd_workspace_size.argtypes = [i] * 5
        lib.ne_attn_bwd_workspace_size.restype = sz
        lib.ne_attn_get_error.argtypes = [vp]
        lib.ne_attn_get_error.restype = i
        lib.ne_attn_status_string.argtypes = [i]
        lib.ne_attn_status_string.restype = ctypes.c_char_p
        lib.ne_attn_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        lib.ne_attn_set_wait_limit_ns.restype = None
        lib.ne_attn_selftest_timeout.argtypes = [ctypes.c_uint64, vp]
        lib.ne_attn_selftest_timeout.restype = i
        lib.ne_attn_bwd_noalloc.argtypes = [vp] * 9 + [i] * 5 + [f, vp]
        lib.ne_attn_bwd_noalloc.restype = i
        lib.ne_attn_bwd_noalloc_max_scratch.argtypes = []
        lib.ne_attn_bwd_noalloc_max_scratch.restype = sz
        lib.ne_attn_fwd_window.argtypes = [vp] * 5 + [i] * 5 + [f, i, vp]
        lib.ne_attn_fwd_window.restype = i
        lib.ne_attn_bwd_window.argtypes = [vp] * 10 + [sz] + [i] * 5 + [f, i, vp]
        lib.ne_attn_bwd_window.restype = i
        lib.ne_attn_decode.argtypes = [vp] * 6 + [sz] + [i] * 5 + [f, vp]
        lib.ne_attn_decode.restype = i
        lib.ne_attn_decode_workspace_size.argtypes = [i] * 5
        lib.ne_attn_decode_workspace_size.restype = sz
        lib.ne_attn_varlen_workspace_size.argtypes = [i] * 5
        lib.ne_attn_varlen_workspace_size.restype = sz
        lib.ne_attn_fwd_varlen.argtypes = [vp] * 7 + [sz] + [i] * 5 + [f, vp]
        lib.ne_attn_fwd_varlen.restype = i
        lib.ne_attn_bwd_varlen.argtypes = [vp] * 11 + [sz] + [i] * 5 + [f, vp]
        lib.ne_attn_bwd_varlen.restype = i
        lib.ne_attn_fwd_varlen_dev.argtypes = [vp] * 7 + [sz] + [i] * 5 + [f, vp]
        lib.ne_attn_fwd_varlen_dev.restype = i
        lib.ne_attn_bwd_varlen_dev.argtypes = [vp] * 11 + [sz] + [i] * 5 + [f, vp]
        lib.ne_attn_bwd_varlen_dev.restype = i
        lib.ne_attn_varlen_plan.argtypes = [vp] + [i] * 5 + [vp] * 3 + [sz, vp]
        lib.ne_attn_varlen_plan.restype = i
        lib.ne_attn_packed_workspace_size.argtypes = [i] * 5
        lib.ne_attn_packed_workspace_size.restype = sz
        lib.ne_attn_fwd_packed.argtypes = [vp] * 7 + [sz] + [i] * 5 + [f, vp]
        lib.ne_attn_fwd_packed.restype = i
        lib.ne_attn_bwd_packed.argtypes = [vp] * 11 + [sz] + [i] * 5 + [f, vp]
        lib.ne_attn_bwd_packed.restype = i
        lib.ne_attn_fwd_packed_dev.argtypes = [vp] * 7 + [sz] + [i] * 5 + [f, vp]
        lib.ne_attn_fwd_packed_dev.restype = i
        lib.ne_attn_bwd_packed_dev.argtypes = [vp] * 11 + [sz] + [i] * 5 + [f, vp]
        lib.ne_attn_bwd_packed_dev.restype = i
        _lib = lib
        return lib


def _status_text(status: int) -> str:
    try:
        return load_library(build_if_missing=False).ne_attn_status_string(status).decode()
    except Exception:  # the library may be the thing that failed to load
        return "see ne_attn.h"


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(x: torch.Tensor, name: str, shape, dtype) -> None:
    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if x.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if x.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {x.dtype}")
    if tuple(x.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(x.shape)}")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _dims(q: torch.Tensor, k: torch.Tensor):
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q and k must be [B, T, H, d]")
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    return B, T, Hq, Hkv, d


def ne_attn_fwd(q, k, v, o, lse, rope_theta: float = 10000.0, stream=None) -> None:
    """Forward into caller-allocated o [B,T,Hq,d] bf16 and lse [B,Hq,T] fp32."""
    B, T, Hq, Hkv, d = _dims(q, k)
    bf = torch.bfloat16
    _check(q, "q", (B, T, Hq, d), bf)
    _check(k, "k", (B, T, Hkv, d), bf)
    _check(v, "v", (B, T, Hkv, d), bf)
    _check(o, "o", (B, T, Hq, d), bf)
    _check(lse, "lse", (B, Hq, T), torch.float32)
    rc = load_library().ne_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                    lse.data_ptr(), B, T, Hq, Hkv, d, float(rope_theta),
                                    _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_fwd")


def _workspace_ptr(workspace):
    if workspace.device.type != "cuda" or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def ne_attn_fwd_save(q, k, v, o, lse, workspace, rope_theta: float = 10000.0,
                     stream=None, window: int = 0) -> None:
    """ne_attn_fwd that also leaves Q' and K' in `workspace` for ne_attn_bwd_saved."""
    B, T, Hq, Hkv, d = _dims(q, k)
    bf = torch.bfloat16
    _check(q, "q", (B, T, Hq, d), bf)
    _check(k, "k", (B, T, Hkv, d), bf)
    _check(v, "v", (B, T, Hkv, d), bf)
    _check(o, "o", (B, T, Hq, d), bf)
    _check(lse, "lse", (B, Hq, T), torch.float32)
    wp, wbytes = _workspace_ptr(workspace)
    rc = load_library().ne_attn_fwd_save(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), wp, wbytes, B, T, Hq, Hkv, d,
                                         float(rope_theta), int(window), _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_fwd_save")


def ne_attn_bwd_saved(q, k, v, o, lse, do, dq, dk, dv, workspace, rope_theta: float = 10000.0,
                      stream=None, window: int = 0) -> None:
    """ne_attn_bwd on a workspace filled by ne_attn_fwd_save (D is recomputed, Q'/K' reused)."""
    B, T, Hq, Hkv, d = _dims(q, k)
    bf = torch.bfloat16
    for x, n, h in ((q, "q", Hq), (k, "k", Hkv), (v, "v", Hkv), (o, "o", Hq), (do, "do", Hq),
                    (dq, "dq", Hq), (dk, "dk", Hkv), (dv, "dv", Hkv)):
        _check(x, n, (B, T, h, d), bf)
    _check(lse, "lse", (B, Hq, T), torch.float32)
    wp, wbytes = _workspace_ptr(workspace)
    rc = load_library().ne_attn_bwd_saved(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                          o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                                          dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), wp, wbytes,
                                          B, T, Hq, Hkv, d, float(rope_theta), int(window),
                                          _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_bwd_saved")


def ne_attn_bwd_preprocess_d(o, do, workspace, Hkv: int, stream=None) -> None:
    """D = rowsum(dO * O) into the workspace only (first step of ne_attn_bwd_saved)."""
    B, T, Hq, d = o.shape
    for x, n in ((o, "o"), (do, "do")):
        _check(x, n, (B, T, Hq, d), torch.bfloat16)
    wp, wbytes = _workspace_ptr(workspace)
    rc = load_library().ne_attn_bwd_preprocess_d(o.data_ptr(), do.data_ptr(), wp, wbytes, B, T,
                                                 Hq, Hkv, d, _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_bwd_preprocess_d")


def ne_attn_bwd_workspace_size(B: int, T: int, Hq: int, Hkv: int, d: int) -> int:
    return int(load_library().ne_attn_bwd_workspace_size(B, T, Hq, Hkv, d))


def ne_attn_bwd(q, k, v, o, lse, do, dq, dk, dv, workspace, rope_theta: float = 10000.0,
                stream=None) -> None:
    """Backward into caller-allocated dq, dk, dv; workspace is a uint8 CUDA tensor."""
    B, T, Hq, Hkv, d = _dims(q, k)
    bf = torch.bfloat16
    for x, n, h in ((q, "q", Hq), (k, "k", Hkv), (v, "v", Hkv), (o, "o", Hq), (do, "do", Hq),
                    (dq, "dq", Hq), (dk, "dk", Hkv), (dv, "dv", Hkv)):
        _check(x, n, (B, T, h, d), bf)
    _check(lse, "lse", (B, Hq, T), torch.float32)
    if workspace.device.type != "cuda" or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    wbytes = workspace.numel() * workspace.element_size()
    rc = load_library().ne_attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                    lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                    dv.data_ptr(), workspace.data_ptr(), wbytes, B, T, Hq, Hkv,
                                    d, float(rope_theta), _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_bwd")


def _bwd_common(q, k, v, lse, do, workspace):
    B, T, Hq, Hkv, d = _dims(q, k)
    bf = torch.bfloat16
    for x, n, h in ((q, "q", Hq), (k, "k", Hkv), (v, "v", Hkv), (do, "do", Hq)):
        _check(x, n, (B, T, h, d), bf)
    _check(lse, "lse", (B, Hq, T), torch.float32)
    if workspace.device.type != "cuda" or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    return B, T, Hq, Hkv, d, workspace.numel() * workspace.element_size()


def ne_attn_bwd_preprocess(q, k, o, do, workspace, rope_theta: float = 10000.0,
                           stream=None) -> None:
    """D = rowsum(dO * O) and the rotated fp16 Q', K' into the workspace (first
    backward step)."""
    B, T, Hq, Hkv, d = _dims(q, k)
    for x, n, h in ((q, "q", Hq), (k, "k", Hkv), (o, "o", Hq), (do, "do", Hq)):
        _check(x, n, (B, T, h, d), torch.bfloat16)
    if workspace.device.type != "cuda" or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    wbytes = workspace.numel() * workspace.element_size()
    rc = load_library().ne_attn_bwd_preprocess(q.data_ptr(), k.data_ptr(), o.data_ptr(),
                                               do.data_ptr(), workspace.data_ptr(), wbytes, B, T,
                                               Hq, Hkv, d, float(rope_theta), _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_bwd_preprocess")


def ne_attn_bwd_dq(q, k, v, lse, do, dq, workspace, rope_theta: float = 10000.0,
                   stream=None) -> None:
    B, T, Hq, Hkv, d, wbytes = _bwd_common(q, k, v, lse, do, workspace)
    _check(dq, "dq", (B, T, Hq, d), torch.bfloat16)
    rc = load_library().ne_attn_bwd_dq(q.data_ptr(), k.data_ptr(), v.data_ptr(), lse.data_ptr(),
                                       do.data_ptr(), dq.data_ptr(), workspace.data_ptr(), wbytes,
                                       B, T, Hq, Hkv, d, float(rope_theta), _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_bwd_dq")


def ne_attn_bwd_dkdv(q, k, v, lse, do, dk, dv, workspace, rope_theta: float = 10000.0,
                     stream=None) -> None:
    B, T, Hq, Hkv, d, wbytes = _bwd_common(q, k, v, lse, do, workspace)
    _check(dk, "dk", (B, T, Hkv, d), torch.bfloat16)
    _check(dv, "dv", (B, T, Hkv, d), torch.bfloat16)
    rc = load_library().ne_attn_bwd_dkdv(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                         lse.data_ptr(), do.data_ptr(), dk.data_ptr(),
                                         dv.data_ptr(), workspace.data_ptr(), wbytes, B, T, Hq,
                                         Hkv, d, float(rope_theta), _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_bwd_dkdv")


def ne_attn_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, rope_theta: float = 10000.0,
                        stream=None) -> None:
    """Backward into caller-allocated dq, dk, dv without any workspace: the
    library's fixed scratch array stands in for it (see ne_attn.h for its size
    limit and for why concurrent calls on one device must be serialised)."""
    B, T, Hq, Hkv, d = _dims(q, k)
    bf = torch.bfloat16
    for x, n, h in ((q, "q", Hq), (k, "k", Hkv), (v, "v", Hkv), (o, "o", Hq), (do, "do", Hq),
                    (dq, "dq", Hq), (dk, "dk", Hkv), (dv, "dv", Hkv)):
        _check(x, n, (B, T, h, d), bf)
    _check(lse, "lse", (B, Hq, T), torch.float32)
    rc = load_library().ne_attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                            o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                                            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, T, Hq,
                                            Hkv, d, float(rope_theta), _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_bwd_noalloc")


def ne_attn_bwd_noalloc_max_scratch() -> int:
    return int(load_library().ne_attn_bwd_noalloc_max_scratch())


def ne_attn_get_error(stream=None) -> int:
    """Synchronise the stream; return (and clear) the device-side status code."""
    return int(load_library().ne_attn_get_error(_stream_ptr(stream)))


def ne_attn_status_string(status: int) -> str:
    return load_library().ne_attn_status_string(int(status)).decode()


def ne_attn_set_wait_limit_ns(limit_ns: int) -> None:
    load_library().ne_attn_set_wait_limit_ns(int(limit_ns))


def ne_attn_selftest_timeout(limit_ns: int, stream=None) -> None:
    rc = load_library().ne_attn_selftest_timeout(int(limit_ns), _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_selftest_timeout")


# ---- conveniences that allocate outputs with torch (device memory only) ----

def ne_attn_fwd_window(q, k, v, o, lse, window: int, rope_theta: float = 10000.0,
                       stream=None) -> None:
    """ne_attn_fwd with a sliding window: query t sees keys t-window+1 .. t (0: causal)."""
    B, T, Hq, Hkv, d = _dims(q, k)
    bf = torch.bfloat16
    _check(q, "q", (B, T, Hq, d), bf)
    _check(k, "k", (B, T, Hkv, d), bf)
    _check(v, "v", (B, T, Hkv, d), bf)
    _check(o, "o", (B, T, Hq, d), bf)
    _check(lse, "lse", (B, Hq, T), torch.float32)
    rc = load_library().ne_attn_fwd_window(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                           lse.data_ptr(), B, T, Hq, Hkv, d, float(rope_theta),
                                           int(window), _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_fwd_window")


def ne_attn_bwd_window(q, k, v, o, lse, do, dq, dk, dv, workspace, window: int,
                       rope_theta: float = 10000.0, stream=None) -> None:
    """ne_attn_bwd with a sliding window (the forward's `window`)."""
    B, T, Hq, Hkv, d = _dims(q, k)
    bf = torch.bfloat16
    for x, n, h in ((q, "q", Hq), (k, "k", Hkv), (v, "v", Hkv), (o, "o", Hq), (do, "do", Hq),
                    (dq, "dq", Hq), (dk, "dk", Hkv), (dv, "dv", Hkv)):
        _check(x, n, (B, T, h, d), bf)
    _check(lse, "lse", (B, Hq, T), torch.float32)
    wp, wbytes = _workspace_ptr(workspace)
    rc = load_library().ne_attn_bwd_window(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                           o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                                           dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), wp, wbytes,
                                           B, T, Hq, Hkv, d, float(rope_theta), int(window),
                                           _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_bwd_window")


def ne_attn_decode_workspace_size(B: int, Tk: int, Hq: int, Hkv: int, d: int) -> int:
    return int(load_library().ne_attn_decode_workspace_size(B, Tk, Hq, Hkv, d))


def ne_attn_decode(q, k_cache, v_cache, o, lse, workspace, rope_theta: float = 10000.0,
                   stream=None) -> None:
    """Decode: q [B,Hq,d] (one new token per sequence, at position Tk-1) against
    k_cache / v_cache [B,Tk,Hkv,d]; writes o [B,Hq,d] bf16 and lse [B,Hq] fp32."""
    if q.dim() != 3 or k_cache.dim() != 4:
        raise ValueError("q must be [B, Hq, d] and k_cache [B, Tk, Hkv, d]")
    B, Hq, d = q.shape
    Tk, Hkv = k_cache.shape[1], k_cache.shape[2]
    bf = torch.bfloat16
    _check(q, "q", (B, Hq, d), bf)
    _check(k_cache, "k_cache", (B, Tk, Hkv, d), bf)
    _check(v_cache, "v_cache", (B, Tk, Hkv, d), bf)
    _check(o, "o", (B, Hq, d), bf)
    _check(lse, "lse", (B, Hq), torch.float32)
    wp, wbytes = _workspace_ptr(workspace)
    rc = load_library().ne_attn_decode(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                       o.data_ptr(), lse.data_ptr(), wp, wbytes, B, Tk, Hq, Hkv,
                                       d, float(rope_theta), _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_decode")


def attention_decode(q, k_cache, v_cache, rope_theta: float = 10000.0, stream=None,
                     workspace=None):
    """Allocate o, lse (and a workspace if none is given) and run ne_attn_decode."""
    B, Hq, d = q.shape
    Tk, Hkv = k_cache.shape[1], k_cache.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(max(ne_attn_decode_workspace_size(B, Tk, Hq, Hkv, d), 16),
                                dtype=torch.uint8, device=q.device)
    ne_attn_decode(q, k_cache, v_cache, o, lse, workspace, rope_theta, stream)
    return o, lse


def _host_seqlens(seqlens, B: int):
    """seqlens as a contiguous host int32 array of B lengths (the library reads it
    on the host during the call)."""
    if isinstance(seqlens, torch.Tensor):
        if seqlens.device.type != "cpu":
            raise ValueError("seqlens must be in host memory (a list, array or CPU tensor)")
        seqlens = seqlens.numpy()
    sl = np.ascontiguousarray(np.asarray(seqlens).reshape(-1), dtype=np.int32)
    if sl.shape != (B,):
        raise ValueError(f"seqlens must hold {B} lengths, got {sl.shape[0]}")
    return sl


def ne_attn_varlen_workspace_size(B: int, T: int, Hq: int, Hkv: int, d: int) -> int:
    return int(load_library().ne_attn_varlen_workspace_size(B, T, Hq, Hkv, d))


def ne_attn_varlen_plan(seqlens, T: int, Hq: int, Hkv: int, d: int, with_tables: bool = True):
    """Host-only: the live work units of a padded variable-length batch.  Returns
    (counts [fwd, dq, dkdv], [fwd table, dq table, dkdv table] or None)."""
    sl = np.ascontiguousarray(np.asarray(seqlens).reshape(-1), dtype=np.int32)
    B = int(sl.shape[0])
    cap = ((T + 127) // 128) * B * Hq if with_tables else 0
    tabs = [np.zeros(max(cap, 1), dtype=np.int32) for _ in range(3)]
    counts = np.zeros(3, dtype=np.int32)
    ptr = (lambda a: a.ctypes.data) if with_tables else (lambda a: None)
    rc = load_library().ne_attn_varlen_plan(sl.ctypes.data, B, T, Hq, Hkv, d, ptr(tabs[0]),
                                            ptr(tabs[1]), ptr(tabs[2]), cap, counts.ctypes.data)
    if rc:
        raise NeAttnError(rc, "ne_attn_varlen_plan")
    if not with_tables:
        return counts.tolist(), None
    return counts.tolist(), [t[:c].copy() for t, c in zip(tabs, counts.tolist())]


def ne_attn_fwd_varlen(q, k, v, o, lse, seqlens, workspace, rope_theta: float = 10000.0,
                       stream=None) -> None:
    """Padded variable-length forward: sequence b is its first seqlens[b] rows (host
    lengths); padding rows get o = 0 and lse = -inf."""
    B, T, Hq, Hkv, d = _dims(q, k)
    bf = torch.bfloat16
    _check(q, "q", (B, T, Hq, d), bf)
    _check(k, "k", (B, T, Hkv, d), bf)
    _check(v, "v", (B, T, Hkv, d), bf)
    _check(o, "o", (B, T, Hq, d), bf)
    _check(lse, "lse", (B, Hq, T), torch.float32)
    sl = _host_seqlens(seqlens, B)
    wp, wbytes = _workspace_ptr(workspace)
    rc = load_library().ne_attn_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                           lse.data_ptr(), sl.ctypes.data, wp, wbytes, B, T, Hq,
                                           Hkv, d, float(rope_theta), _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_fwd_varlen")


def ne_attn_bwd_varlen(q, k, v, o, lse, do, dq, dk, dv, seqlens, workspace,
                       rope_theta: float = 10000.0, stream=None) -> None:
    """Padded variable-length backward (o, lse from ne_attn_fwd_varlen); padding
    positions of dq, dk, dv get 0."""
    B, T, Hq, Hkv, d = _dims(q, k)
    bf = torch.bfloat16
    for x, n, h in ((q, "q", Hq), (k, "k", Hkv), (v, "v", Hkv), (o, "o", Hq), (do, "do", Hq),
                    (dq, "dq", Hq), (dk, "dk", Hkv), (dv, "dv", Hkv)):
        _check(x, n, (B, T, h, d), bf)
    _check(lse, "lse", (B, Hq, T), torch.float32)
    sl = _host_seqlens(seqlens, B)
    wp, wbytes = _workspace_ptr(workspace)
    rc = load_library().ne_attn_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                           o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                                           dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                           sl.ctypes.data, wp, wbytes, B, T, Hq, Hkv, d,
                                           float(rope_theta), _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_bwd_varlen")


def _dev_seqlens(seqlens, B: int):
    """Lengths already in device memory: an int32 CUDA tensor of B entries."""
    if not isinstance(seqlens, torch.Tensor) or seqlens.device.type != "cuda" or \
            seqlens.dtype != torch.int32 or seqlens.numel() != B or not seqlens.is_contiguous():
        raise ValueError(f"seqlens must be a contiguous int32 CUDA tensor of {B} lengths")
    return seqlens.data_ptr()


def ne_attn_fwd_varlen_dev(q, k, v, o, lse, seqlens, workspace, rope_theta: float = 10000.0,
                           stream=None) -> None:
    """ne_attn_fwd_varlen with the lengths in device memory (an int32 CUDA tensor):
    the unit tables are planned on the GPU, so the call can be captured into a
    CUDA graph and replayed with other lengths in the same tensor."""
    B, T, Hq, Hkv, d = _dims(q, k)
    bf = torch.bfloat16
    _check(q, "q", (B, T, Hq, d), bf)
    _check(k, "k", (B, T, Hkv, d), bf)
    _check(v, "v", (B, T, Hkv, d), bf)
    _check(o, "o", (B, T, Hq, d), bf)
    _check(lse, "lse", (B, Hq, T), torch.float32)
    sp = _dev_seqlens(seqlens, B)
    wp, wbytes = _workspace_ptr(workspace)
    rc = load_library().ne_attn_fwd_varlen_dev(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                               o.data_ptr(), lse.data_ptr(), sp, wp, wbytes, B,
                                               T, Hq, Hkv, d, float(rope_theta),
                                               _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_fwd_varlen_dev")


def ne_attn_bwd_varlen_dev(q, k, v, o, lse, do, dq, dk, dv, seqlens, workspace,
                           rope_theta: float = 10000.0, stream=None) -> None:
    """ne_attn_bwd_varlen with the lengths in device memory (see ne_attn_fwd_varlen_dev)."""
    B, T, Hq, Hkv, d = _dims(q, k)
    bf = torch.bfloat16
    for x, n, h in ((q, "q", Hq), (k, "k", Hkv), (v, "v", Hkv), (o, "o", Hq), (do, "do", Hq),
                    (dq, "dq", Hq), (dk, "dk", Hkv), (dv, "dv", Hkv)):
        _check(x, n, (B, T, h, d), bf)
    _check(lse, "lse", (B, Hq, T), torch.float32)
    sp = _dev_seqlens(seqlens, B)
    wp, wbytes = _workspace_ptr(workspace)
    rc = load_library().ne_attn_bwd_varlen_dev(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                               o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                                               dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), sp,
                                               wp, wbytes, B, T, Hq, Hkv, d, float(rope_theta),
                                               _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_bwd_varlen_dev")


def _host_cu(cu_seqlens, total: int):
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32).reshape(-1))
    if cu.shape[0] < 2:
        raise ValueError("cu_seqlens needs at least two entries")
    return cu


def _packed_dims(q, k):
    if q.dim() != 3 or k.dim() != 3:
        raise ValueError("packed q and k are [total, H, d]")
    total, Hq, d = q.shape
    return total, Hq, k.shape[1], d


def ne_attn_packed_workspace_size(nseq: int, total: int, Hq: int, Hkv: int, d: int) -> int:
    return int(load_library().ne_attn_packed_workspace_size(nseq, total, Hq, Hkv, d))


def ne_attn_fwd_packed(q, k, v, o, lse, cu_seqlens, workspace, rope_theta: float = 10000.0,
                       stream=None) -> None:
    """Packed variable-length forward: q [total, Hq, d], k and v [total, Hkv, d],
    sequence b is rows cu_seqlens[b] .. cu_seqlens[b+1]-1 (host offsets); lse
    is [Hq, total]."""
    total, Hq, Hkv, d = _packed_dims(q, k)
    bf = torch.bfloat16
    _check(q, "q", (total, Hq, d), bf)
    _check(k, "k", (total, Hkv, d), bf)
    _check(v, "v", (total, Hkv, d), bf)
    _check(o, "o", (total, Hq, d), bf)
    _check(lse, "lse", (Hq, total), torch.float32)
    cu = _host_cu(cu_seqlens, total)
    wp, wbytes = _workspace_ptr(workspace)
    rc = load_library().ne_attn_fwd_packed(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                           lse.data_ptr(), cu.ctypes.data, wp, wbytes,
                                           cu.shape[0] - 1, total, Hq, Hkv, d, float(rope_theta),
                                           _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_fwd_packed")


def ne_attn_bwd_packed(q, k, v, o, lse, do, dq, dk, dv, cu_seqlens, workspace,
                       rope_theta: float = 10000.0, stream=None) -> None:
    """Packed variable-length backward (o, lse from ne_attn_fwd_packed)."""
    total, Hq, Hkv, d = _packed_dims(q, k)
    bf = torch.bfloat16
    for x, n, h in ((q, "q", Hq), (k, "k", Hkv), (v, "v", Hkv), (o, "o", Hq), (do, "do", Hq),
                    (dq, "dq", Hq), (dk, "dk", Hkv), (dv, "dv", Hkv)):
        _check(x, n, (total, h, d), bf)
    _check(lse, "lse", (Hq, total), torch.float32)
    cu = _host_cu(cu_seqlens, total)
    wp, wbytes = _workspace_ptr(workspace)
    rc = load_library().ne_attn_bwd_packed(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                           o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                                           dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                           cu.ctypes.data, wp, wbytes, cu.shape[0] - 1, total,
                                           Hq, Hkv, d, float(rope_theta), _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_bwd_packed")


def _dev_cu(cu_seqlens):
    """A prefix array already in device memory: an int32 CUDA tensor of nseq + 1 entries."""
    if not isinstance(cu_seqlens, torch.Tensor) or cu_seqlens.device.type != "cuda" or \
            cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or \
            cu_seqlens.numel() < 2 or not cu_seqlens.is_contiguous():
        raise ValueError("cu_seqlens must be a contiguous 1-D int32 CUDA tensor of nseq + 1 offsets")
    return cu_seqlens.data_ptr(), cu_seqlens.numel() - 1


def ne_attn_fwd_packed_dev(q, k, v, o, lse, cu_seqlens, workspace, rope_theta: float = 10000.0,
                           stream=None) -> None:
    """ne_attn_fwd_packed with cu_seqlens in device memory (an int32 CUDA tensor):
    the unit tables are planned on the GPU, so the call can be captured into a
    CUDA graph and replayed with other offsets in the same tensor."""
    total, Hq, Hkv, d = _packed_dims(q, k)
    bf = torch.bfloat16
    _check(q, "q", (total, Hq, d), bf)
    _check(k, "k", (total, Hkv, d), bf)
    _check(v, "v", (total, Hkv, d), bf)
    _check(o, "o", (total, Hq, d), bf)
    _check(lse, "lse", (Hq, total), torch.float32)
    cp, nseq = _dev_cu(cu_seqlens)
    wp, wbytes = _workspace_ptr(workspace)
    rc = load_library().ne_attn_fwd_packed_dev(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                               o.data_ptr(), lse.data_ptr(), cp, wp, wbytes,
                                               nseq, total, Hq, Hkv, d, float(rope_theta),
                                               _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_fwd_packed_dev")


def ne_attn_bwd_packed_dev(q, k, v, o, lse, do, dq, dk, dv, cu_seqlens, workspace,
                           rope_theta: float = 10000.0, stream=None) -> None:
    """ne_attn_bwd_packed with cu_seqlens in device memory (see ne_attn_fwd_packed_dev)."""
    total, Hq, Hkv, d = _packed_dims(q, k)
    bf = torch.bfloat16
    for x, n, h in ((q, "q", Hq), (k, "k", Hkv), (v, "v", Hkv), (o, "o", Hq), (do, "do", Hq),
                    (dq, "dq", Hq), (dk, "dk", Hkv), (dv, "dv", Hkv)):
        _check(x, n, (total, h, d), bf)
    _check(lse, "lse", (Hq, total), torch.float32)
    cp, nseq = _dev_cu(cu_seqlens)
    wp, wbytes = _workspace_ptr(workspace)
    rc = load_library().ne_attn_bwd_packed_dev(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                               o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                                               dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), cp,
                                               wp, wbytes, nseq, total, Hq, Hkv, d,
                                               float(rope_theta), _stream_ptr(stream))
    if rc:
        raise NeAttnError(rc, "ne_attn_bwd_packed_dev")


def attention_forward(q, k, v, rope_theta: float = 10000.0, stream=None):
    """Allocate o and lse on q's device and run ne_attn_fwd.  Returns (o, lse)."""
    B, T, Hq, Hkv, d = _dims(q, k)
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, T, dtype=torch.float32, device=q.device)
    ne_attn_fwd(q, k, v, o, lse, rope_theta, stream)
    return o, lse


def attention_backward(q, k, v, o, lse, do, rope_theta: float = 10000.0, stream=None,
                       workspace=None):
    """Allocate dq, dk, dv (and a workspace if none is given) and run ne_attn_bwd."""
    B, T, Hq, Hkv, d = _dims(q, k)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if workspace is None:
        workspace = torch.empty(ne_attn_bwd_workspace_size(B, T, Hq, Hkv, d),
                                dtype=torch.uint8, device=q.device)
    ne_attn_bwd(q, k, v, o, lse, do, dq, dk, dv, workspace, rope_theta, stream)
    return dq, dk, dv
