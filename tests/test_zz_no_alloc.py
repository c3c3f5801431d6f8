"""The allocation-free entry point (mtp_verify_attn_fwd_static_scratch).

Some callers cannot call cudaMalloc (a host inside another framework's memory
pool, launches issued during CUDA graph capture, loops that must never
synchronise the device), so this entry point keeps its split-KV partials in a
library-owned static device array.  The test calls it through the C ABI twice in
a row, on different batches, and checks each output against the regular entry
point (which uses a caller workspace): bit for bit, under deterministic
scheduling.  It also checks that a call too large for the array is refused;
that the first call of a fresh process, made on a non-default stream under
balanced scheduling, matches the oracle (the one-time clear of the array's
counter header is ordered on the caller's stream); and that a call which sets a
device error bit leaves the shared header zero, so the next call still matches
the workspace entry point bit for bit; and, over random batches sized around the
array, that a call is refused exactly when its partials would not fit.
This file is collected last so a stop-at-first-failure run has run every other
test before it; it passes alone in a fresh process as well.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

from paged_fp8_speculative_gb300 import _lib, api, synth

pytestmark = pytest.mark.gpu

TOL = 0.01


def _c_call(b, kd, vd, S, out, status):
    """Call the C symbol directly with raw device pointers (no Python-side allocation)."""
    return _lib.lib().mtp_verify_attn_fwd_static_scratch(
        b.q.data_ptr(), b.q.stride(0), b.q.stride(1), b.k_cache.data_ptr(), b.v_cache.data_ptr(),
        b.k_cache.shape[0], b.block_tables.data_ptr(), b.block_tables.shape[1],
        b.seq_lens.data_ptr(), b.cu_seqlens_q.data_ptr(), b.num_seqs, b.total_q,
        b.num_q_heads, b.num_kv_heads, kd.data_ptr(), vd.data_ptr(), b.softmax_scale, S,
        out.data_ptr(), out.stride(0), out.stride(1), status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def _regular(b, kd, vd, S):
    return api.mtp_verify_attn_fwd(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                                   b.cu_seqlens_q, kd, vd, b.softmax_scale, num_segments=S)


@pytest.mark.parametrize("mode", [api.SCHED_PLANNED, api.SCHED_CHUNKED], ids=["planned", "chunked"])
def test_static_scratch_matches_regular_entry_point_twice(mode):
    # Deterministic scheduling, so the two entry points must agree bit for bit.
    api.mtp_verify_attn_set_deterministic(True)
    api.mtp_verify_attn_set_scheduling(mode)
    try:
        _static_vs_regular()
    finally:
        api.mtp_verify_attn_set_deterministic(False)
        api.mtp_verify_attn_set_scheduling(api.SCHED_PLANNED)


def _static_vs_regular():
    batches = [
        synth.make_batch([3000, 1000, 77], [4, 2, 1], 16, 1, seed=901, k_descale=0.5,
                         v_descale=2.0).to("cuda"),
        synth.make_batch([500, 2500], [3, 4], 16, 2, seed=902).to("cuda"),
    ]
    for b, S in zip(batches, (16, 5)):
        kd = torch.tensor([b.k_descale], dtype=torch.float32, device="cuda")
        vd = torch.tensor([b.v_descale], dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        ref = _regular(b, kd, vd, S)
        out = torch.full_like(b.q, float("nan"))
        rc = _c_call(b, kd, vd, S, out, status)
        assert rc == api.OK, api.mtp_verify_attn_strerror(rc)
        torch.cuda.synchronize()
        assert status.item() == 0
        r = ref.float().cpu().numpy().astype(np.float64)
        o = out.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(o).all()
        assert np.abs(o - r).max() / r.std() <= TOL
        assert np.array_equal(o, r)


def test_static_scratch_refuses_calls_beyond_its_size():
    b = synth.make_batch([2000] * 16, 4, 16, 1, seed=903).to("cuda")
    kd = torch.ones(1, dtype=torch.float32, device="cuda")
    out = torch.empty_like(b.q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    need = api.mtp_verify_attn_workspace_size(b.total_q, b.num_q_heads, 64)
    assert need > api.STATIC_SCRATCH_BYTES
    assert _c_call(b, kd, kd, 64, out, status) == api.E_SCRATCH_LIMIT
    assert api.mtp_verify_attn_workspace_size(b.total_q, b.num_q_heads, 16) <= api.STATIC_SCRATCH_BYTES
    assert _c_call(b, kd, kd, 16, out, status) == api.OK
    torch.cuda.synchronize()
    assert status.item() == 0


def test_static_scratch_after_a_device_error_is_bit_identical():
    """A call whose block table names a page outside the pool sets ERR_PAGE; the shared
    array's tile counters must still be back at zero afterwards, so the next (valid) call
    equals the workspace entry point bit for bit under deterministic scheduling."""
    api.mtp_verify_attn_set_deterministic(True)
    try:
        b = synth.make_batch([2500, 700, 40], [4, 3, 1], 16, 1, seed=904, k_descale=0.5,
                             v_descale=2.0).to("cuda")
        kd = torch.tensor([b.k_descale], dtype=torch.float32, device="cuda")
        vd = torch.tensor([b.v_descale], dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        bad_bt = b.block_tables.clone()
        bad_bt[0, 5] = b.k_cache.shape[0] + 3
        bad = synth.PagedBatch(b.q, b.k_cache, b.v_cache, bad_bt, b.seq_lens, b.cu_seqlens_q,
                               b.k_descale, b.v_descale, b.softmax_scale, 1, 16)
        out = torch.empty_like(b.q)
        assert _c_call(bad, kd, vd, 8, out, status) == api.OK
        torch.cuda.synchronize()
        assert status.item() & api.ERR_PAGE
        assert out[:4].abs().max().item() == 0          # the bad sequence's rows are zeros
        status.zero_()
        ref = _regular(b, kd, vd, 8)
        out2 = torch.full_like(b.q, float("nan"))
        assert _c_call(b, kd, vd, 8, out2, status) == api.OK
        torch.cuda.synchronize()
        assert status.item() == 0
        assert torch.equal(out2, ref)
    finally:
        api.mtp_verify_attn_set_deterministic(False)


_FRESH = textwrap.dedent("""
    import sys
    import numpy as np
    import torch
    sys.path.insert(0, {root!r})
    import oracle
    from paged_fp8_speculative_gb300 import api, synth
    from tests.helpers import oracle_args
    assert not api.mtp_verify_attn_get_deterministic()      # balanced tile sharing
    batch = synth.make_batch([6000, 3000, 900], [4, 2, 3], 16, 1, seed=905, k_descale=0.5,
                             v_descale=2.0)
    side = torch.cuda.Stream()                              # a non-default stream
    with torch.cuda.stream(side):
        gb = batch.to("cuda")
        kd = torch.tensor([gb.k_descale], dtype=torch.float32, device="cuda")
        vd = torch.tensor([gb.v_descale], dtype=torch.float32, device="cuda")
        out = torch.empty_like(gb.q)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        api.mtp_verify_attn_fwd_static_scratch(gb.q, gb.k_cache, gb.v_cache, gb.block_tables,
                                               gb.seq_lens, gb.cu_seqlens_q, kd, vd,
                                               gb.softmax_scale, 16, out, status=status,
                                               stream=side)
    side.synchronize()
    ref = oracle.verify_attention(*oracle_args(batch))
    got = out.float().cpu().numpy().astype(np.float64)
    err = oracle.excess_over_half_ulp(got, ref)
    assert status.item() == 0, status.item()
    assert np.isfinite(got).all() and err <= {tol}, err
    print("fresh-process static call ok", err)
""")


def test_static_scratch_first_call_on_a_side_stream_in_a_fresh_process():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FRESH.format(root=root, tol=TOL)], cwd=root,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr


def test_static_scratch_random_batches_around_its_size():
    """Random batches whose split-KV partials need a little less or a little more than the
    static array: each call is refused with E_SCRATCH_LIMIT exactly when the workspace it
    would need exceeds STATIC_SCRATCH_BYTES, and otherwise matches the workspace entry point
    bit for bit (deterministic scheduling)."""
    rng = np.random.default_rng(904)
    api.mtp_verify_attn_set_deterministic(True)
    refused = accepted = 0
    try:
        for case in range(24):
            B = int(rng.integers(4, 33))
            ql = [int(x) for x in rng.integers(1, 5, size=B)]
            ctx = [int(x) for x in rng.integers(4, 3000, size=B)]
            hq = int(rng.choice([8, 16]))
            rows = sum(ql) * hq
            # S around the value at which rows * S partial slots fill the array
            S = int(np.clip(api.STATIC_SCRATCH_BYTES // (rows * 1028) + rng.integers(-2, 3), 1, 64))
            b = synth.make_batch(ctx, ql, hq, 1, seed=905 + case).to("cuda")
            kd = torch.full((1,), 0.5, dtype=torch.float32, device="cuda")
            vd = torch.full((1,), 2.0, dtype=torch.float32, device="cuda")
            out = torch.empty_like(b.q)
            status = torch.zeros(1, dtype=torch.int32, device="cuda")
            need = api.mtp_verify_attn_workspace_size(b.total_q, hq, S)
            rc = _c_call(b, kd, vd, S, out, status)
            if need > api.STATIC_SCRATCH_BYTES:
                assert rc == api.E_SCRATCH_LIMIT, (case, need, rc)
                refused += 1
                continue
            assert rc == api.OK, (case, need, rc)
            torch.cuda.synchronize()
            assert status.item() == 0, (case, status.item())
            ref = _regular(b, kd, vd, S)
            torch.cuda.synchronize()
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), case
            accepted += 1
    finally:
        api.mtp_verify_attn_set_deterministic(False)
    assert refused > 0 and accepted > 0, (refused, accepted)
