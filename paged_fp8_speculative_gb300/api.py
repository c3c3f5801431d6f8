"""Python binding of the C ABI (argument marshalling only).

Every function has the name of the C entry point it calls.  PyTorch supplies
device memory and the current stream; every step of the computation runs in
the library's CUDA kernels.
"""
from __future__ import annotations

import contextlib
import math
from typing import Optional

import torch

from ._lib import lib

HEAD_DIM = 256
PAGE_SIZE = 16
MAX_SEGMENTS = 64

OK, E_ARG, E_UNSUPPORTED, E_DEVICE, E_WORKSPACE, E_LAUNCH = 0, -1, -2, -3, -4, -5
E_SCRATCH_LIMIT = -6
STATIC_SCRATCH_BYTES = 32 << 20
ERR_QLEN, ERR_QLEN_GT_SEQ, ERR_PAGE, ERR_SEQ_TOO_LONG, ERR_TIMEOUT = 1, 2, 4, 8, 16
WORKSPACE_HEADER_BYTES = 4352     # MTPATTN_WORKSPACE_HEADER_BYTES: tile and call counters


class MtpAttnError(RuntimeError):
    def __init__(self, code: int):
        self.code = code
        super().__init__(f"mtpattn status {code}: {mtp_verify_attn_strerror(code)}")


def mtp_verify_attn_strerror(code: int) -> str:
    return lib().mtp_verify_attn_strerror(int(code)).decode()


def mtp_verify_attn_num_segments(num_seqs: int, num_kv_heads: int, max_pages_per_seq: int,
                                 device: int = -1) -> int:
    r = lib().mtp_verify_attn_num_segments(num_seqs, num_kv_heads, max_pages_per_seq, device)
    if r < 0:
        raise MtpAttnError(r)
    return r


def mtp_verify_attn_workspace_size(total_q: int, num_q_heads: int, num_segments: int) -> int:
    return int(lib().mtp_verify_attn_workspace_size(total_q, num_q_heads, num_segments))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


def _temporaries_on(stream, device, needed: bool):
    """Context for the temporaries a wrapper makes for a call (descale tensors from Python
    floats, a zeroed workspace, out, lse): when the call runs on a stream other than the
    current one, they are made on that stream, so that they are written in its order, before
    the library's kernels read them, and their memory is not handed out again while those
    kernels may still use it.  Nothing to do when the call makes none, or runs on the current
    stream (entering a stream context costs microseconds of host time per call)."""
    if not needed or stream is None or device.type != "cuda":
        return contextlib.nullcontext()
    ts = stream if isinstance(stream, torch.cuda.Stream) else \
        torch.cuda.ExternalStream(int(stream), device=device)
    return torch.cuda.stream(ts)


def _descale(x, device) -> torch.Tensor:
    if isinstance(x, torch.Tensor):
        return x
    return torch.full((1,), float(x), dtype=torch.float32, device=device)


def _check_args(q, k_cache, v_cache, block_tables, seq_lens, cu_seqlens_q, kd, vd, out):
    """The shape, dtype and layout checks both entry points share (the C side checks
    pointers, strides, alignment and the envelope, but cannot see shapes)."""
    if q.dtype != torch.bfloat16 or q.dim() != 3 or q.shape[2] != HEAD_DIM or q.stride(2) != 1:
        raise ValueError("q must be bf16 [total_q, H_q, 256] with unit stride on head_dim")
    if k_cache.dtype not in (torch.uint8, torch.float8_e4m3fn) or v_cache.dtype != k_cache.dtype:
        raise ValueError("k_cache / v_cache must be uint8 or float8_e4m3fn codes")
    if k_cache.dim() != 4 or k_cache.shape[1] != PAGE_SIZE or k_cache.shape[3] != HEAD_DIM:
        raise ValueError("k_cache must be [num_pages, 16, H_kv, 256]")
    if v_cache.shape != k_cache.shape or not k_cache.is_contiguous() or not v_cache.is_contiguous():
        raise ValueError("k_cache and v_cache must be contiguous and of the same shape")
    for name, t in (("block_tables", block_tables), ("seq_lens", seq_lens),
                    ("cu_seqlens_q", cu_seqlens_q)):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 tensor")
    num_seqs = seq_lens.numel()
    if seq_lens.dim() != 1 or block_tables.dim() != 2 or block_tables.shape[0] != num_seqs or \
            cu_seqlens_q.dim() != 1 or cu_seqlens_q.numel() != num_seqs + 1:
        raise ValueError("block_tables [B, max_pages], seq_lens [B], cu_seqlens_q [B+1]")
    for name, t in (("k_descale", kd), ("v_descale", vd)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.numel() != 1:
            raise ValueError(f"{name} must be a 1-element float32 tensor")
    total_q, hq, _ = q.shape
    if out is not None and (out.dtype != torch.bfloat16 or tuple(out.shape) != (total_q, hq, HEAD_DIM)
                            or out.stride(2) != 1):
        raise ValueError("out must be bf16 [total_q, H_q, 256] with unit stride on head_dim")
    return num_seqs, total_q, hq, k_cache.shape[2]


def _verify_fwd(entry, q, k_cache, v_cache, block_tables, seq_lens, cu_seqlens_q, k_descale,
                v_descale, softmax_scale, num_segments, out, workspace, status, stream):
    dev = q.device
    makes = (out is None or workspace is None or not isinstance(k_descale, torch.Tensor) or
             not isinstance(v_descale, torch.Tensor))
    with _temporaries_on(stream, dev, makes):
        kd = _descale(k_descale, dev)
        vd = _descale(v_descale, dev)
        num_seqs, total_q, hq, hkv = _check_args(q, k_cache, v_cache, block_tables, seq_lens,
                                                 cu_seqlens_q, kd, vd, out)
        # None / 0: the library chooses S (and may then share the partial slots out by
        # length); a workspace made here is sized for the S it will choose, a given one is
        # checked by the library.
        chosen = int(num_segments or 0)
        if out is None:
            out = torch.empty(total_q, hq, HEAD_DIM, dtype=torch.bfloat16, device=dev)
        if workspace is None:
            S = chosen or mtp_verify_attn_num_segments(num_seqs, hkv, block_tables.shape[1],
                                                       dev.index if dev.index is not None else -1)
            need = mtp_verify_attn_workspace_size(total_q, hq, S)
            workspace = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
    rc = entry(
        _ptr(q), q.stride(0), q.stride(1),
        _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
        _ptr(block_tables), block_tables.shape[1],
        _ptr(seq_lens), _ptr(cu_seqlens_q),
        num_seqs, total_q, hq, hkv,
        _ptr(kd), _ptr(vd), float(softmax_scale), chosen,
        _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(out), out.stride(0), out.stride(1),
        _ptr(status), _stream_handle(stream))
    if rc != OK:
        raise MtpAttnError(rc)
    return out


def mtp_verify_attn_fwd(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                        block_tables: torch.Tensor, seq_lens: torch.Tensor,
                        cu_seqlens_q: torch.Tensor, k_descale, v_descale,
                        softmax_scale: float, num_segments: Optional[int] = None,
                        out: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None,
                        status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Paged fp8 verify / draft-extend / decode attention; returns ``out`` (bf16).

    q [total_q, H_q, 256] bf16; k_cache / v_cache [num_pages, 16, H_kv, 256]
    uint8 or float8_e4m3fn codes; block_tables [B, max_pages] int32; seq_lens [B]
    int32; cu_seqlens_q [B+1] int32; descales 1-element float32 device tensors
    (a Python float is copied to the device).  ``num_segments`` None or 0 lets the library
    choose S; a long sequence may then take more than S pieces when short ones use fewer
    (the workspace's rows x S partial slots are shared out by length).  ``status`` is an optional int32
    device word that collects device-side error bits (ERR_*).  Without ``workspace`` a zeroed
    one is allocated for this call; a decode loop passes its own (zeroed once, reused by every
    call on the stream) so that no call allocates.
    """
    return _verify_fwd(lib().mtp_verify_attn_fwd, q, k_cache, v_cache, block_tables, seq_lens,
                       cu_seqlens_q, k_descale, v_descale, softmax_scale, num_segments, out,
                       workspace, status, stream)


def mtp_verify_attn_fwd_qp_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                               block_tables: torch.Tensor, seq_lens: torch.Tensor,
                               cu_seqlens_q: torch.Tensor, k_descale, v_descale,
                               softmax_scale: float, num_segments: Optional[int] = None,
                               out: Optional[torch.Tensor] = None,
                               workspace: Optional[torch.Tensor] = None,
                               status: Optional[torch.Tensor] = None,
                               stream=None) -> torch.Tensor:
    """mtp_verify_attn_fwd with Q and P rounded once to e4m3 (the pages' precision class,
    about 0.15 std of error instead of 0.01); planned scheduling only, so batches of more
    (sequence, KV head) units than SMs raise MtpAttnError(E_UNSUPPORTED)."""
    return _verify_fwd(lib().mtp_verify_attn_fwd_qp_fp8, q, k_cache, v_cache, block_tables,
                       seq_lens, cu_seqlens_q, k_descale, v_descale, softmax_scale,
                       num_segments, out, workspace, status, stream)


def mtp_verify_attn_fwd_static_scratch(q: torch.Tensor, k_cache: torch.Tensor,
                                       v_cache: torch.Tensor, block_tables: torch.Tensor,
                                       seq_lens: torch.Tensor, cu_seqlens_q: torch.Tensor,
                                       k_descale: torch.Tensor, v_descale: torch.Tensor,
                                       softmax_scale: float, num_segments: int, out: torch.Tensor,
                                       status: Optional[torch.Tensor] = None,
                                       stream=None) -> torch.Tensor:
    """The attention without a caller workspace, for callers that cannot allocate.

    The split-KV partials go to the library's own static device array
    (STATIC_SCRATCH_BYTES per GPU), so this wrapper allocates nothing either:
    ``out``, the descale tensors (1-element float32 device tensors, not Python
    floats) and every input are the caller's, and they get the same checks as in
    mtp_verify_attn_fwd.  Calls that overlap on the GPU share that array and race;
    serialise them.
    """
    if out is None:
        raise ValueError("out is required: this entry point allocates nothing")
    num_seqs, total_q, hq, hkv = _check_args(q, k_cache, v_cache, block_tables, seq_lens,
                                             cu_seqlens_q, k_descale, v_descale, out)
    rc = lib().mtp_verify_attn_fwd_static_scratch(
        _ptr(q), q.stride(0), q.stride(1),
        _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
        _ptr(block_tables), block_tables.shape[1],
        _ptr(seq_lens), _ptr(cu_seqlens_q),
        num_seqs, total_q, hq, hkv,
        _ptr(k_descale), _ptr(v_descale), float(softmax_scale), int(num_segments),
        _ptr(out), out.stride(0), out.stride(1),
        _ptr(status), _stream_handle(stream))
    if rc != OK:
        raise MtpAttnError(rc)
    return out


def mtp_verify_attn_set_deterministic(on: bool) -> None:
    """Fixed page ranges per piece (bit-identical repeats) instead of balanced tile sharing."""
    lib().mtp_verify_attn_set_deterministic(1 if on else 0)


def mtp_verify_attn_get_deterministic() -> bool:
    return bool(lib().mtp_verify_attn_get_deterministic())


SCHED_CHUNKED = 0
SCHED_PLANNED = 1


def mtp_verify_attn_set_scheduling(mode: int) -> None:
    """Chunked (0, sized for max_pages) or planned (1, sized from seq_lens on the device)."""
    rc = lib().mtp_verify_attn_set_scheduling(int(mode))
    if rc != OK:
        raise ValueError(f"unknown scheduling mode {mode}")


def mtp_verify_attn_get_scheduling() -> int:
    return int(lib().mtp_verify_attn_get_scheduling())


def mtpattn_stream_read(buf: torch.Tensor, sink: Optional[torch.Tensor] = None, blocks: int = 0,
                        stream=None) -> torch.Tensor:
    """Read every byte of ``buf`` once (streaming-read ceiling probe); returns the sink."""
    if blocks == 0:
        blocks = int(lib().mtpattn_stream_read_default_blocks())
        if blocks <= 0:
            raise MtpAttnError(blocks)
    with _temporaries_on(stream, buf.device, sink is None):
        if sink is None:
            sink = torch.empty(blocks, dtype=torch.int32, device=buf.device)
    nbytes = buf.numel() * buf.element_size()
    rc = lib().mtpattn_stream_read(_ptr(buf), nbytes, _ptr(sink), blocks, _stream_handle(stream))
    if rc != OK:
        raise MtpAttnError(rc)
    return sink


# ---- fp8 varlen prefill (include/fmha_fp8_varlen.h) ---------------------------------------------

HEAD_DIM_QK = 192
HEAD_DIM_V = 128
ERR_CU = 32


def fmha_fwd_fp8_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, q_descale, k_descale,
                        v_descale, cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor,
                        max_seqlen_q: int, max_seqlen_k: int, softmax_scale: Optional[float] = None,
                        is_causal: bool = False, return_lse: bool = False,
                        out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                        status: Optional[torch.Tensor] = None, stream=None):
    """fp8 varlen prefill attention (q/k head dim 192, v 128); returns out, or (out, lse).

    q [total_q, H_q, 192], k [total_k, H_kv, 192], v [total_k, H_kv, 128]: uint8 or
    float8_e4m3fn codes with unit stride on the head dim; cu_seqlens_q / cu_seqlens_k int32
    [B+1]; descales 1-element float32 device tensors (a Python float is copied to the
    device); softmax_scale defaults to 1/sqrt(192); out bf16 [total_q, H_q, 128]; lse float32
    [H_q, total_q] (natural log), allocated when return_lse and not given.
    """
    for name, t, d in (("q", q, HEAD_DIM_QK), ("k", k, HEAD_DIM_QK), ("v", v, HEAD_DIM_V)):
        if t.dtype not in (torch.uint8, torch.float8_e4m3fn) or t.dim() != 3 or t.shape[2] != d \
                or t.stride(2) != 1:
            raise ValueError(f"{name} must be e4m3 codes [rows, heads, {d}] with unit stride on "
                             "the head dim")
    if k.shape[:2] != v.shape[:2]:
        raise ValueError("k and v must have the same rows and heads")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if t.dtype != torch.int32 or not t.is_contiguous() or t.dim() != 1:
            raise ValueError(f"{name} must be a contiguous int32 vector")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both have num_seqs + 1 entries")
    dev = q.device
    makes = (out is None or (return_lse and lse is None) or
             not all(isinstance(x, torch.Tensor) for x in (q_descale, k_descale, v_descale)))
    with _temporaries_on(stream, dev, makes):
        qd, kd, vd = (_descale(x, dev) for x in (q_descale, k_descale, v_descale))
        for name, t in (("q_descale", qd), ("k_descale", kd), ("v_descale", vd)):
            if t.dtype != torch.float32 or t.numel() != 1:
                raise ValueError(f"{name} must be a 1-element float32 tensor")
        total_q, hq, _ = q.shape
        total_k, hkv, _ = k.shape
        if out is None:
            out = torch.empty(total_q, hq, HEAD_DIM_V, dtype=torch.bfloat16, device=dev)
        if out.dtype != torch.bfloat16 or tuple(out.shape) != (total_q, hq, HEAD_DIM_V) or \
                out.stride(2) != 1:
            raise ValueError("out must be bf16 [total_q, H_q, 128] with unit stride on the head "
                             "dim")
        if return_lse and lse is None:
            lse = torch.empty(hq, total_q, dtype=torch.float32, device=dev)
        if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (hq, total_q)
                                or not lse.is_contiguous()):
            raise ValueError("lse must be a contiguous float32 [H_q, total_q] tensor")
    scale = 1.0 / math.sqrt(HEAD_DIM_QK) if softmax_scale is None else float(softmax_scale)
    rc = lib().fmha_fwd_fp8_varlen(
        _ptr(q), q.stride(0), q.stride(1), _ptr(k), k.stride(0), k.stride(1),
        _ptr(v), v.stride(0), v.stride(1), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
        cu_seqlens_q.numel() - 1, total_q, total_k, int(max_seqlen_q), int(max_seqlen_k), hq, hkv,
        _ptr(qd), _ptr(kd), _ptr(vd), scale, 1 if is_causal else 0,
        _ptr(out), out.stride(0), out.stride(1), _ptr(lse), _ptr(status), _stream_handle(stream))
    if rc != OK:
        raise MtpAttnError(rc)
    return (out, lse) if return_lse else out
