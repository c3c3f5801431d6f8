"""ctypes loader for libmtpattn.so (the C ABI declared in include/mtpattn.h and
include/fmha_fp8_varlen.h).

There is no fallback: if the library is missing the import of this module's
``lib()`` raises, so no caller can silently run anything else.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmtpattn.so")

_c_int, _c_i32, _c_i64, _c_size, _c_float = (ctypes.c_int, ctypes.c_int32, ctypes.c_int64,
                                             ctypes.c_size_t, ctypes.c_float)
_vp = ctypes.c_void_p

# name -> (restype, argtypes), in the order of include/mtpattn.h, then include/fmha_fp8_varlen.h
SIGNATURES = {
    "mtp_verify_attn_num_segments": (_c_i32, [_c_i32, _c_i32, _c_i32, _c_i32]),
    "mtp_verify_attn_workspace_size": (_c_size, [_c_i32, _c_i32, _c_i32]),
    "mtp_verify_attn_fwd": (_c_int, [
        _vp, _c_i64, _c_i64,            # q, strides
        _vp, _vp, _c_i64,               # k_cache, v_cache, num_pages
        _vp, _c_i32,                    # block_tables, max_pages_per_seq
        _vp, _vp,                       # seq_lens, cu_seqlens_q
        _c_i32, _c_i32, _c_i32, _c_i32,  # num_seqs, total_q, num_q_heads, num_kv_heads
        _vp, _vp, _c_float, _c_i32,     # k_descale, v_descale, softmax_scale, num_segments
        _vp, _c_size,                   # workspace, workspace_bytes
        _vp, _c_i64, _c_i64,            # out, strides
        _vp, _vp]),                     # status, stream
    "mtp_verify_attn_fwd_qp_fp8": (_c_int, [
        _vp, _c_i64, _c_i64, _vp, _vp, _c_i64, _vp, _c_i32, _vp, _vp,
        _c_i32, _c_i32, _c_i32, _c_i32, _vp, _vp, _c_float, _c_i32,
        _vp, _c_size, _vp, _c_i64, _c_i64, _vp, _vp]),
    "mtp_verify_attn_fwd_static_scratch": (_c_int, [
        _vp, _c_i64, _c_i64, _vp, _vp, _c_i64, _vp, _c_i32, _vp, _vp,
        _c_i32, _c_i32, _c_i32, _c_i32, _vp, _vp, _c_float, _c_i32,
        _vp, _c_i64, _c_i64, _vp, _vp]),
    "mtp_verify_attn_set_deterministic": (None, [_c_i32]),
    "mtp_verify_attn_get_deterministic": (_c_i32, []),
    "mtp_verify_attn_set_scheduling": (_c_i32, [_c_i32]),
    "mtp_verify_attn_get_scheduling": (_c_i32, []),
    "mtp_verify_attn_strerror": (ctypes.c_char_p, [_c_int]),
    "mtpattn_stream_read": (_c_int, [_vp, _c_size, _vp, _c_i32, _vp]),
    "mtpattn_stream_read_default_blocks": (_c_i32, []),
    # include/fmha_fp8_varlen.h
    "fmha_fwd_fp8_varlen": (_c_int, [
        _vp, _c_i64, _c_i64,            # q, strides (bytes)
        _vp, _c_i64, _c_i64,            # k, strides
        _vp, _c_i64, _c_i64,            # v, strides
        _vp, _vp,                       # cu_seqlens_q, cu_seqlens_k
        _c_i32, _c_i32, _c_i32,         # num_seqs, total_q, total_k
        _c_i32, _c_i32,                 # max_seqlen_q, max_seqlen_k
        _c_i32, _c_i32,                 # num_q_heads, num_kv_heads
        _vp, _vp, _vp,                  # q/k/v descales
        _c_float, _c_i32,               # softmax_scale, causal
        _vp, _c_i64, _c_i64,            # out, strides (elements)
        _vp, _vp, _vp]),                # lse, status, stream
}

_LIB = None


def load(path: str) -> ctypes.CDLL:
    """Load a build of the library at ``path`` with the C signatures attached."""
    handle = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    return handle


def lib() -> ctypes.CDLL:
    """The loaded library (raises RuntimeError if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m paged_fp8_speculative_gb300.build`")
        _LIB = load(LIB_PATH)
    return _LIB
