"""Causal grouped-query attention with rotary embeddings for GB300 (sm_103a).

Thin Python binding over the C ABI in ``include/ne_attn.h`` (``libne_attn.so``,
built in-tree by ``_build.py``).  The functions below only marshal torch
tensors into pointers, sizes and the current CUDA stream; every step of the
computation runs in the library's CUDA kernels.  There is no CPU fallback:
if the library is missing or the device is not an sm_103 GPU, calls raise.
"""
from ._binding import (  # noqa: F401
    NE_STATUS,
    NeAttnError,
    attention_backward,
    attention_decode,
    attention_forward,
    lib_path,
    load_library,
    ne_attn_bwd,
    ne_attn_bwd_dkdv,
    ne_attn_bwd_noalloc,
    ne_attn_bwd_noalloc_max_scratch,
    ne_attn_fwd_save,
    ne_attn_bwd_saved,
    ne_attn_bwd_preprocess_d,
    ne_attn_bwd_dq,
    ne_attn_bwd_preprocess,
    ne_attn_bwd_workspace_size,
    ne_attn_decode,
    ne_attn_decode_workspace_size,
    ne_attn_fwd,
    ne_attn_fwd_window,
    ne_attn_bwd_window,
    ne_attn_fwd_varlen,
    ne_attn_bwd_varlen,
    ne_attn_fwd_varlen_dev,
    ne_attn_bwd_varlen_dev,
    ne_attn_varlen_plan,
    ne_attn_varlen_workspace_size,
    ne_attn_packed_workspace_size,
    ne_attn_fwd_packed,
    ne_attn_bwd_packed,
    ne_attn_fwd_packed_dev,
    ne_attn_bwd_packed_dev,
    ne_attn_get_error,
    ne_attn_selftest_timeout,
    ne_attn_set_wait_limit_ns,
    ne_attn_status_string,
)

__all__ = [
    "NE_STATUS", "NeAttnError", "attention_backward", "attention_decode", "attention_forward",
    "lib_path", "ne_attn_decode", "ne_attn_decode_workspace_size", "ne_attn_fwd_window",
    "ne_attn_bwd_window", "ne_attn_fwd_varlen", "ne_attn_bwd_varlen", "ne_attn_varlen_plan",
    "ne_attn_fwd_varlen_dev", "ne_attn_bwd_varlen_dev",
    "ne_attn_varlen_workspace_size", "ne_attn_packed_workspace_size", "ne_attn_fwd_packed",
    "ne_attn_bwd_packed", "ne_attn_fwd_packed_dev", "ne_attn_bwd_packed_dev",
    "load_library", "ne_attn_bwd", "ne_attn_bwd_dkdv", "ne_attn_bwd_dq",
    "ne_attn_bwd_noalloc", "ne_attn_bwd_noalloc_max_scratch", "ne_attn_fwd_save",
    "ne_attn_bwd_saved", "ne_attn_bwd_preprocess_d",
    "ne_attn_bwd_preprocess", "ne_attn_bwd_workspace_size", "ne_attn_fwd",
    "ne_attn_get_error", "ne_attn_selftest_timeout", "ne_attn_set_wait_limit_ns",
    "ne_attn_status_string",
]
