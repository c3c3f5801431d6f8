"""Host-only tests of the C ABI (no GPU): the library loads, exports exactly what
include/mtpattn.h declares, sizes the workspace, and refuses bad arguments with
the documented status codes before it touches any device state."""
from __future__ import annotations

import ctypes
import glob
import os
import re

import pytest
import torch

from paged_fp8_speculative_gb300 import _lib, api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


def declared_functions():
    names = []
    for header in HEADERS:
        src = open(header).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\**\s+\**([A-Za-z_]\w*)\s*\(", src,
                            flags=re.M)
    return names


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert set(names) == set(_lib.SIGNATURES), names
    assert len(names) == len(set(names))
    assert "mtp_verify_attn_fwd" in names and "fmha_fwd_fp8_varlen" in names


def test_library_exports_every_declared_symbol():
    lib = _lib.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings():
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert api.mtp_verify_attn_strerror(code) not in ("", "unknown status")
    assert api.mtp_verify_attn_strerror(-99) == "unknown status"


def test_workspace_header_size_agrees():
    # the header macro, the binding's constant and the library's sizing (no rows: header only)
    src = open(os.path.join(ROOT, "include", "mtpattn.h")).read()
    m = re.search(r"#define MTPATTN_WORKSPACE_HEADER_BYTES (\d+)", src)
    assert m and int(m.group(1)) == api.WORKSPACE_HEADER_BYTES
    assert api.mtp_verify_attn_workspace_size(0, 1, 1) == api.WORKSPACE_HEADER_BYTES


def test_workspace_size():
    f = api.mtp_verify_attn_workspace_size
    rows = 64 * 16
    lse = (rows * 16 * 4 + 255) // 256 * 256
    h = api.WORKSPACE_HEADER_BYTES
    assert f(64, 16, 16) == h + lse + rows * 16 * 256 * 4
    assert f(7, 8, 3) == h + ((7 * 8 * 3 * 4 + 255) // 256 * 256) + ((7 * 8 * 3 * 1024 + 255) // 256 * 256)
    assert f(64, 16, 0) == 0 and f(64, 16, 65) == 0 and f(-1, 16, 4) == 0 and f(4, 0, 4) == 0


# A call whose every argument is valid on the host side; pointers are fake but
# aligned and are never dereferenced before the device checks.
FAKE = 0x10000


def good_args(**over):
    a = dict(q=FAKE, q_st=16 * 256, q_sh=256, k=FAKE, v=FAKE, num_pages=10, bt=FAKE, max_pages=5,
             sl=FAKE, cu=FAKE, num_seqs=2, total_q=8, hq=16, hkv=1, kd=FAKE, vd=FAKE, scale=0.0625,
             S=4, ws=FAKE, ws_bytes=1 << 30, out=FAKE, o_st=16 * 256, o_sh=256, status=None,
             stream=None)
    a.update(over)
    return a


def call(a, entry="mtp_verify_attn_fwd"):
    return getattr(_lib.lib(), entry)(
        a["q"], a["q_st"], a["q_sh"], a["k"], a["v"], a["num_pages"], a["bt"], a["max_pages"],
        a["sl"], a["cu"], a["num_seqs"], a["total_q"], a["hq"], a["hkv"], a["kd"], a["vd"],
        a["scale"], a["S"], a["ws"], a["ws_bytes"], a["out"], a["o_st"], a["o_sh"], a["status"],
        a["stream"])


REFUSALS = [
    (dict(q=None), api.E_ARG),
    (dict(k=None), api.E_ARG),
    (dict(bt=None), api.E_ARG),
    (dict(kd=None), api.E_ARG),
    (dict(out=None), api.E_ARG),
    (dict(num_seqs=-1), api.E_ARG),
    (dict(total_q=1), api.E_ARG),                     # fewer query tokens than sequences
    (dict(num_pages=0), api.E_ARG),
    (dict(max_pages=0), api.E_ARG),
    (dict(q_sh=100), api.E_ARG),                      # stride not a multiple of 8 elements
    (dict(o_st=0), api.E_ARG),
    (dict(q=FAKE + 8), api.E_ARG),                    # not 16-byte aligned
    (dict(scale=float("nan")), api.E_ARG),
    (dict(hkv=0), api.E_ARG),
    (dict(hq=12, hkv=1), api.E_UNSUPPORTED),          # ratio 12
    (dict(hq=32, hkv=1), api.E_UNSUPPORTED),          # ratio 32
    (dict(hq=16, hkv=3), api.E_UNSUPPORTED),          # not a multiple
    (dict(total_q=9), api.E_UNSUPPORTED),             # q_len > 4 somewhere
    (dict(S=65), api.E_UNSUPPORTED),
    (dict(S=-2), api.E_UNSUPPORTED),
    (dict(ws=None), api.E_WORKSPACE),
    (dict(ws=FAKE + 16), api.E_WORKSPACE),            # not 256-byte aligned
    (dict(ws_bytes=1000), api.E_WORKSPACE),
]


ENTRIES = ["mtp_verify_attn_fwd", "mtp_verify_attn_fwd_qp_fp8"]


@pytest.mark.parametrize("entry", ENTRIES)
@pytest.mark.parametrize("over,code", REFUSALS)
def test_refusals_before_any_launch(over, code, entry):
    """Both precision tiers share the checks (the fp8 tier adds its own after them)."""
    assert call(good_args(**over), entry) == code


@pytest.mark.parametrize("entry", ENTRIES)
def test_empty_batch_is_a_no_op(entry):
    assert call(good_args(num_seqs=0, total_q=0), entry) == api.OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_no_device_is_reported():
    assert call(good_args()) == api.E_DEVICE
    assert call(good_args(), "mtp_verify_attn_fwd_qp_fp8") == api.E_DEVICE
    assert _lib.lib().mtp_verify_attn_num_segments(16, 1, 100, -1) == api.E_DEVICE
    assert _lib.lib().mtpattn_stream_read(FAKE, 1024, FAKE, 4, None) == api.E_DEVICE


def test_num_segments_argument_checks():
    f = _lib.lib().mtp_verify_attn_num_segments
    assert f(0, 1, 10, -1) == api.E_ARG
    assert f(4, 0, 10, -1) == api.E_ARG
    assert f(4, 1, 0, -1) == api.E_ARG


def test_stream_read_argument_checks():
    f = _lib.lib().mtpattn_stream_read
    assert f(None, 1024, FAKE, 4, None) == api.E_ARG
    assert f(FAKE, 1000, FAKE, 4, None) == api.E_ARG       # not a multiple of 16
    assert f(FAKE, 1024, None, 4, None) == api.E_ARG


def test_deterministic_switch():
    assert not api.mtp_verify_attn_get_deterministic()
    api.mtp_verify_attn_set_deterministic(True)
    try:
        assert api.mtp_verify_attn_get_deterministic()
    finally:
        api.mtp_verify_attn_set_deterministic(False)
    assert not api.mtp_verify_attn_get_deterministic()


def test_scheduling_switch():
    assert api.mtp_verify_attn_get_scheduling() == api.SCHED_PLANNED      # the default
    api.mtp_verify_attn_set_scheduling(api.SCHED_CHUNKED)
    try:
        assert api.mtp_verify_attn_get_scheduling() == api.SCHED_CHUNKED
        assert _lib.lib().mtp_verify_attn_set_scheduling(2) == api.E_ARG
        assert api.mtp_verify_attn_get_scheduling() == api.SCHED_CHUNKED
    finally:
        api.mtp_verify_attn_set_scheduling(api.SCHED_PLANNED)
    assert api.mtp_verify_attn_get_scheduling() == api.SCHED_PLANNED


def test_static_wrapper_checks_shapes_before_the_call():
    """The allocation-free wrapper gets the same shape checks as the workspace wrapper, and
    takes descales only as tensors (so that it allocates nothing)."""
    from paged_fp8_speculative_gb300 import synth
    b = synth.make_batch([40, 20], [4, 2], 16, 1, seed=1)
    kd = torch.ones(1, dtype=torch.float32)
    out = torch.empty_like(b.q)
    f = api.mtp_verify_attn_fwd_static_scratch
    base = dict(q=b.q, k_cache=b.k_cache, v_cache=b.v_cache, block_tables=b.block_tables,
                seq_lens=b.seq_lens, cu_seqlens_q=b.cu_seqlens_q, k_descale=kd, v_descale=kd,
                softmax_scale=0.0625, num_segments=4, out=out)
    bad = [dict(block_tables=b.block_tables.t()),                 # not contiguous
           dict(k_cache=b.k_cache[0]),                             # wrong rank
           dict(v_cache=b.v_cache[:1]),                            # shape differs from K
           dict(k_descale=1.0),                                    # not a tensor
           dict(v_descale=torch.ones(2)),                          # not one element
           dict(out=out[:, :8]),                                   # wrong shape
           dict(out=None),                                         # it would need allocating
           dict(q=b.q.float()),                                    # wrong dtype
           dict(cu_seqlens_q=b.cu_seqlens_q[:-1])]                 # wrong length
    for over in bad:
        with pytest.raises(ValueError):
            f(**(base | over))


def prefill_call(**over):
    a = dict(q=FAKE, qt=2 * 192, qh=192, k=FAKE, kt=192, kh=192, v=FAKE, vt=128, vh=128,
             cq=FAKE, ck=FAKE, B=1, tq=4, tk=4, mq=4, mk=4, hq=2, hkv=1, qd=FAKE, kd=FAKE, vd=FAKE,
             scale=0.07, causal=0, out=FAKE, ot=256, oh=128, lse=None, status=None, stream=None)
    a.update(over)
    return _lib.lib().fmha_fwd_fp8_varlen(
        a["q"], a["qt"], a["qh"], a["k"], a["kt"], a["kh"], a["v"], a["vt"], a["vh"], a["cq"],
        a["ck"], a["B"], a["tq"], a["tk"], a["mq"], a["mk"], a["hq"], a["hkv"], a["qd"], a["kd"],
        a["vd"], a["scale"], a["causal"], a["out"], a["ot"], a["oh"], a["lse"], a["status"],
        a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(q=None), api.E_ARG), (dict(cq=None), api.E_ARG), (dict(vd=None), api.E_ARG),
    (dict(qt=200), api.E_ARG),                 # byte stride not a multiple of 16
    (dict(vh=8), api.E_ARG),
    (dict(ot=4), api.E_ARG),                   # element stride not a multiple of 8
    (dict(q=FAKE + 8), api.E_ARG),             # base not 16-byte aligned
    (dict(causal=2), api.E_ARG), (dict(B=-1), api.E_ARG), (dict(hq=0), api.E_ARG),
    (dict(scale=float("nan")), api.E_ARG),
    (dict(hq=3, hkv=2), api.E_UNSUPPORTED),
])
def test_prefill_refusals(over, code):
    assert prefill_call(**over) == code


def test_prefill_empty_batch_is_a_no_op():
    assert prefill_call(B=0, tq=0) == api.OK
    assert prefill_call(tq=0, mq=0) == api.OK
    assert prefill_call(mq=0) == api.E_ARG         # queries, but none allowed per sequence


def test_prefill_wrapper_checks_shapes():
    from paged_fp8_speculative_gb300 import synth
    b = synth.make_prefill_batch([5, 3], [4, 6], 4, 2, seed=1)
    f = api.fmha_fwd_fp8_varlen
    base = dict(q=b.q, k=b.k, v=b.v, q_descale=b.q_descale, k_descale=b.k_descale,
                v_descale=b.v_descale, cu_seqlens_q=b.cu_seqlens_q, cu_seqlens_k=b.cu_seqlens_k,
                max_seqlen_q=5, max_seqlen_k=6)
    for over in (dict(q=b.q[:, :, :128]), dict(v=b.k), dict(k=b.k[:, :1]),
                 dict(cu_seqlens_k=b.cu_seqlens_k[:-1]), dict(cu_seqlens_q=b.cu_seqlens_q.long()),
                 dict(out=torch.empty(8, 4, 128)), dict(q_descale=torch.ones(2))):
        with pytest.raises(ValueError):
            f(**(base | over))


def test_prefill_causal_pair_count_closed_form():
    """The flop count's closed form of the causal pairs against a direct sum."""
    from paged_fp8_speculative_gb300.synth import _causal_pairs
    for lq, lk in ((1, 1), (5, 3), (3, 5), (100, 100), (64, 300), (300, 64), (7, 0)):
        direct = sum(max(0, min(lk, i + lk - lq + 1)) for i in range(lq))
        assert _causal_pairs(lq, lk) == direct, (lq, lk)


def test_wrappers_enter_no_stream_context_unless_they_must():
    """Entering a stream context costs microseconds of host time per call, enough to make
    short eager calls host-bound: the wrappers enter one only to make temporaries for a call
    on a stream other than the current one."""
    import contextlib
    dev = torch.device("cuda", 0)
    for stream, needed in ((None, True), (None, False), (12345, False)):
        assert isinstance(api._temporaries_on(stream, dev, needed), contextlib.nullcontext)
    assert isinstance(api._temporaries_on(12345, torch.device("cpu"), True),
                      contextlib.nullcontext)
