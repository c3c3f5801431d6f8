"""Calls on several streams at once.

Two verify batches on two streams (each with its own workspace, as the header requires of
calls that overlap) and a prefill on a third run interleaved, several times each, so that
their grids overlap on the GPU and their CTAs contend for SMs and tensor memory.  In
deterministic mode every output must equal, bit for bit, the same call made alone.
"""
from __future__ import annotations

import pytest
import torch

from paged_fp8_speculative_gb300 import api, synth

pytestmark = pytest.mark.gpu


def verify_call(b, S, ws, out, stream):
    kd = torch.tensor([b.k_descale], dtype=torch.float32, device="cuda")
    vd = torch.tensor([b.v_descale], dtype=torch.float32, device="cuda")

    def call():
        api.mtp_verify_attn_fwd(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                                b.cu_seqlens_q, kd, vd, b.softmax_scale, num_segments=S, out=out,
                                workspace=ws, stream=stream)
    return call


def prefill_call(p, lq, lk, out, stream):
    def call():
        api.fmha_fwd_fp8_varlen(p.q, p.k, p.v, p.q_descale, p.k_descale, p.v_descale,
                                p.cu_seqlens_q, p.cu_seqlens_k, lq, lk, is_causal=True, out=out,
                                stream=stream)
    return call


@pytest.mark.parametrize("sched", [api.SCHED_PLANNED, api.SCHED_CHUNKED],
                         ids=["planned", "chunked"])
def test_concurrent_calls_match_calls_alone(sched):
    a = synth.make_batch([9000] * 4, 4, 16, 1, seed=91).to("cuda")
    b = synth.make_batch([6, 3000, 12000, 700, 45], [1, 4, 2, 3, 4], 16, 2, seed=92,
                         kv_recipe="unit").to("cuda")
    lq, lk = [1024, 300], [1024, 900]
    p = synth.make_prefill_batch(lq, lk, 16, 4, seed=93).to("cuda")
    S = 8
    streams = [torch.cuda.Stream() for _ in range(3)]
    wa = torch.zeros(api.mtp_verify_attn_workspace_size(a.total_q, a.num_q_heads, S),
                     dtype=torch.uint8, device="cuda")
    wb = torch.zeros(api.mtp_verify_attn_workspace_size(b.total_q, b.num_q_heads, S),
                     dtype=torch.uint8, device="cuda")
    oa, ob = torch.empty_like(a.q), torch.empty_like(b.q)
    op = torch.empty(sum(lq), 16, 128, dtype=torch.bfloat16, device="cuda")
    calls = [verify_call(a, S, wa, oa, streams[0]), verify_call(b, S, wb, ob, streams[1]),
             prefill_call(p, max(lq), max(lk), op, streams[2])]
    api.mtp_verify_attn_set_scheduling(sched)
    api.mtp_verify_attn_set_deterministic(True)
    try:
        refs = []
        for call, o in zip(calls, (oa, ob, op)):              # each alone
            torch.cuda.synchronize()
            call()
            torch.cuda.synchronize()
            refs.append(o.clone())
        for o in (oa, ob, op):
            o.zero_()
        torch.cuda.synchronize()
        for s in streams:
            s.wait_stream(torch.cuda.current_stream())
        for _ in range(6):                                     # interleaved on three streams
            for call in calls:
                call()
        torch.cuda.synchronize()
    finally:
        api.mtp_verify_attn_set_scheduling(api.SCHED_PLANNED)
        api.mtp_verify_attn_set_deterministic(False)
    for name, o, r in zip(("verify a", "verify b", "prefill"), (oa, ob, op), refs):
        assert torch.equal(o.view(torch.int16), r.view(torch.int16)), name


def test_wrapper_temporaries_follow_the_call_stream():
    """A call on a side stream while the current stream is still busy: the temporaries the
    wrappers make (descales passed as Python floats, the zeroed workspace, out, lse) must be
    made on the call's stream, in its order, not on the busy current one, or the kernels would
    read them before they are written."""
    b = synth.make_batch([3000, 700, 40], [4, 1, 3], 16, 1, seed=94, k_descale=0.5,
                         v_descale=2.0).to("cuda")
    lq, lk = [300, 128], [500, 128]
    p = synth.make_prefill_batch(lq, lk, 8, 2, seed=95).to("cuda")
    api.mtp_verify_attn_set_deterministic(True)
    try:
        def verify(stream=None):
            return api.mtp_verify_attn_fwd(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                                           b.cu_seqlens_q, b.k_descale, b.v_descale,
                                           b.softmax_scale, num_segments=4, stream=stream)

        def prefill(stream=None):
            return api.fmha_fwd_fp8_varlen(p.q, p.k, p.v, p.q_descale, p.k_descale, p.v_descale,
                                           p.cu_seqlens_q, p.cu_seqlens_k, max(lq), max(lk),
                                           is_causal=True, return_lse=True, stream=stream)

        ref_v = verify()
        ref_o, ref_l = prefill()
        torch.cuda.synchronize()
        # memory the current stream's allocator would hand out next, filled with ones bits
        junk = torch.full((64 << 20,), -1, dtype=torch.int32, device="cuda")
        del junk
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        torch.cuda._sleep(50_000_000)                   # keeps the current stream busy
        got_v = verify(side)
        got_o, got_l = prefill(side)
        side.synchronize()
        assert torch.equal(got_v.view(torch.int16), ref_v.view(torch.int16))
        assert torch.equal(got_o.view(torch.int16), ref_o.view(torch.int16))
        assert torch.equal(got_l.view(torch.int32), ref_l.view(torch.int32))
        torch.cuda.synchronize()
    finally:
        api.mtp_verify_attn_set_deterministic(False)


def test_calls_from_several_host_threads():
    """Host threads calling at once (the ctypes calls release the interpreter lock): the
    library's per-device caches (tensor maps, kernel attributes) are shared by them.  Each
    thread has its own stream, workspace and output; every output must equal the same call
    made alone, bit for bit (deterministic mode)."""
    import threading
    batches = [synth.make_batch([2000 + 700 * i, 300, 5000 - 900 * i], [4, 2, 3], 16, 1,
                                seed=96 + i).to("cuda") for i in range(4)]
    S = 6
    api.mtp_verify_attn_set_deterministic(True)
    try:
        refs = []
        for b in batches:
            refs.append(api.mtp_verify_attn_fwd(b.q, b.k_cache, b.v_cache, b.block_tables,
                                                b.seq_lens, b.cu_seqlens_q, b.k_descale,
                                                b.v_descale, b.softmax_scale, num_segments=S))
        torch.cuda.synchronize()
        errors = []

        def worker(i):
            try:
                b = batches[i]
                s = torch.cuda.Stream()
                ws = torch.zeros(api.mtp_verify_attn_workspace_size(b.total_q, b.num_q_heads, S),
                                 dtype=torch.uint8, device="cuda")
                out = torch.empty_like(b.q)
                torch.cuda.synchronize()
                for _ in range(20):
                    api.mtp_verify_attn_fwd(b.q, b.k_cache, b.v_cache, b.block_tables,
                                            b.seq_lens, b.cu_seqlens_q, b.k_descale,
                                            b.v_descale, b.softmax_scale, num_segments=S,
                                            out=out, workspace=ws, stream=s)
                s.synchronize()
                if not torch.equal(out.view(torch.int16), refs[i].view(torch.int16)):
                    errors.append(f"thread {i}: output differs")
            except Exception as e:                      # reported below, in the test's thread
                errors.append(f"thread {i}: {e!r}")

        threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(batches))]
        for t in threads:
            t.start()
        for t in threads:
            t.join(timeout=300)
        assert not any(t.is_alive() for t in threads)
        torch.cuda.synchronize()
    finally:
        api.mtp_verify_attn_set_deterministic(False)
    assert not errors, errors
