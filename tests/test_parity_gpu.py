"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Tolerance.  The method's stated bound is max|gpu - oracle| / std(out) <= 0.01
for a kernel that keeps Q and P in bf16/fp32 precision.  The output itself is
bf16, and rounding the exact value to bf16 alone costs up to half a bf16 ulp
(2^-8 of the leading power of two), which for the largest outputs of a
Gaussian-like output tensor is 0.008-0.016 std.  So each element is granted
half a bf16 ulp of the exact value on top of the 0.01 std budget
(oracle.excess_over_half_ulp).  Index and page handling is checked bit-exactly
through segment-count invariance on data whose result does not depend on the
summation order.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from paged_fp8_speculative_gb300 import api, synth
from tests.helpers import oracle_args

pytestmark = pytest.mark.gpu

TOL = 0.01


@pytest.fixture(params=[api.SCHED_CHUNKED, api.SCHED_PLANNED], ids=["chunked", "planned"])
def sched(request):
    """Run the test under both ways of laying out the pieces."""
    api.mtp_verify_attn_set_scheduling(request.param)
    yield request.param
    api.mtp_verify_attn_set_scheduling(api.SCHED_PLANNED)


def run_gpu(batch, num_segments=None, status=None, block_tables=None, out=None, q=None):
    d = batch
    kd = torch.tensor([d.k_descale], dtype=torch.float32, device="cuda")
    vd = torch.tensor([d.v_descale], dtype=torch.float32, device="cuda")
    o = api.mtp_verify_attn_fwd(d.q if q is None else q, d.k_cache, d.v_cache,
                                d.block_tables if block_tables is None else block_tables,
                                d.seq_lens, d.cu_seqlens_q, kd, vd, d.softmax_scale,
                                num_segments=num_segments, status=status, out=out)
    torch.cuda.synchronize()
    return o


def check(batch, num_segments=None, tol=TOL):
    gb = batch.to("cuda")
    got = run_gpu(gb, num_segments).float().cpu().numpy().astype(np.float64)
    ref = oracle.verify_attention(*oracle_args(batch))
    err = oracle.excess_over_half_ulp(got, ref)
    raw = oracle.max_err_over_std(got, ref)
    assert np.isfinite(got).all()
    assert err <= tol, f"excess error {err:.4g} std (raw {raw:.4g})"
    return err, raw


CASES = {
    # the configurations' small parity shapes
    "tiny_2x1000_gqa16": lambda: synth.workload("verify_tiny", seed=1),
    "tiny_unit_recipe": lambda: synth.workload("verify_tiny", seed=2, kv_recipe="unit"),
    "tiny_descales": lambda: synth.make_batch([1000, 1000], 4, 16, 1, seed=3, k_descale=0.5,
                                              v_descale=2.0),
    "gqa8": lambda: synth.make_batch([1000, 1000], 4, 8, 1, seed=4),
    "kv2_777": lambda: synth.workload("verify_2x777_kv2", seed=5),
    "3x8000": lambda: synth.make_batch([8000] * 3, 4, 16, 1, seed=6),
    # ragged draft extend and q_len 1 decode over a context mix with a partial last page
    "ragged_extend": lambda: synth.make_batch([6, 17, 250, 1031, 4099, 33], [1, 4, 2, 3, 4, 1],
                                              16, 1, seed=7, k_descale=0.5, v_descale=2.0),
    "decode": lambda: synth.make_batch([6, 17, 250, 1031, 4099, 33], 1, 16, 1, seed=8,
                                       k_descale=0.5, v_descale=2.0),
    "ragged_gqa8_kv2": lambda: synth.make_batch([4, 40, 300, 1500], [4, 1, 3, 2], 16, 2, seed=9),
    "tiny_contexts": lambda: synth.make_batch([1, 2, 3, 4, 5, 16, 17], [1, 1, 2, 4, 4, 3, 1],
                                              16, 1, seed=10, kv_recipe="unit"),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_parity_against_oracle(name, sched):
    check(CASES[name]())


@pytest.mark.parametrize("S", [1, 2, 3, 5, 16, 63, 64])
def test_any_segment_count_matches_oracle(S, sched):
    check(synth.make_batch([1000, 345, 80], [4, 2, 3], 16, 1, seed=20 + S, k_descale=0.5,
                           v_descale=2.0), num_segments=S)


def test_segment_count_invariance_uniform_keys(sched):
    """All keys equal => the exact output is the mean of the visible V rows.  Every
    segment count must give the same result up to float32 re-association; a
    missed or double-counted page would move it by far more."""
    batch = synth.make_batch([1000, 345, 80, 17], [4, 2, 3, 1], 16, 1, seed=30, kv_recipe="unit")
    batch.k_cache.fill_(0x38)
    ref = oracle.verify_attention(*oracle_args(batch))
    gb = batch.to("cuda")
    outs = []
    for S in (1, 2, 4, 7, 16, 33, 64):
        o = run_gpu(gb, S).float().cpu().numpy()
        assert oracle.excess_over_half_ulp(o, ref) <= 1e-3
        outs.append(o)
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= 2 ** -6 * np.abs(outs[0]).max()


def test_underflow_spike_closed_form(sched):
    """q[0] = 8, K_0[0] = 14, V_0 = +1, every other V = -1 over 16384 keys:
    exact out = (e^7 - 16383) / (e^7 + 16383) = -0.874524 in every coordinate."""
    n, D = 16384, 256
    k = torch.zeros(n // 16, 16, 1, D, dtype=torch.uint8)
    k[0, 0, 0, 0] = 0x56
    v = torch.full((n // 16, 16, 1, D), 0xB8, dtype=torch.uint8)
    v[0, 0, 0, :] = 0x38
    q = torch.zeros(1, 16, D, dtype=torch.bfloat16)
    q[0, :, 0] = 8.0
    bt = torch.randperm(n // 16, dtype=torch.int32)[None]
    kc = torch.empty_like(k); vc = torch.empty_like(v)
    kc[bt[0].long()] = k; vc[bt[0].long()] = v
    batch = synth.PagedBatch(q, kc, vc, bt, torch.tensor([n], dtype=torch.int32),
                             torch.tensor([0, 1], dtype=torch.int32), 1.0, 1.0, 1.0 / 16, 1, 16)
    expect = (math.exp(7) - (n - 1)) / (math.exp(7) + (n - 1))
    for S in (1, 16, 64):
        o = run_gpu(batch.to("cuda"), S).float().cpu().numpy()
        assert np.abs(o - expect).max() <= 2 ** -8


def test_page_permutation_is_bit_identical(sched):
    """Moving every page to another place in the pool and rewriting the block table to match
    leaves the output bit for bit unchanged (fixed page ranges, so the summation order is
    the same): the kernel reads exactly the pages the table names."""
    batch = synth.make_batch([1000, 345, 80, 4099], [4, 2, 3, 1], 16, 1, seed=40, spare_pages=37,
                             k_descale=0.5, v_descale=2.0)
    n = batch.k_cache.shape[0]
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(41))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(n)
    moved = synth.PagedBatch(batch.q, batch.k_cache[perm], batch.v_cache[perm],
                             torch.where(batch.block_tables >= 0, inv[batch.block_tables.long().clamp(min=0)].int(),
                                         batch.block_tables),
                             batch.seq_lens, batch.cu_seqlens_q, batch.k_descale, batch.v_descale,
                             batch.softmax_scale, batch.num_kv_heads, 16)
    api.mtp_verify_attn_set_deterministic(True)
    try:
        for S in (1, 7, 16):
            a = run_gpu(batch.to("cuda"), S)
            b = run_gpu(moved.to("cuda"), S)
            assert torch.equal(a, b), S
    finally:
        api.mtp_verify_attn_set_deterministic(False)


def test_strided_q_and_out_views(sched):
    batch = synth.make_batch([300, 700], [3, 4], 16, 1, seed=40)
    ref = oracle.verify_attention(*oracle_args(batch))
    gb = batch.to("cuda")
    big_q = torch.zeros(gb.total_q, 3 * 16, 256, dtype=torch.bfloat16, device="cuda")
    big_q[:, 16:32] = gb.q                               # q as a slice of a fused projection
    big_o = torch.zeros(gb.total_q, 2, 16, 256, dtype=torch.bfloat16, device="cuda")
    out = big_o[:, 1]
    run_gpu(gb, 4, q=big_q[:, 16:32], out=out)
    assert oracle.excess_over_half_ulp(out.float().cpu().numpy(), ref) <= TOL
    assert big_o[:, 0].abs().max().item() == 0


def test_repeatable_and_graph_replay_bit_identical(sched):
    """Deterministic scheduling: repeated calls and a graph replay are bit-identical."""
    api.mtp_verify_attn_set_deterministic(True)
    try:
        _repeatable_and_graph_replay()
    finally:
        api.mtp_verify_attn_set_deterministic(False)


def _repeatable_and_graph_replay():
    batch = synth.make_batch([5000, 2000], 4, 16, 1, seed=50).to("cuda")
    kd = torch.tensor([batch.k_descale], device="cuda")
    vd = torch.tensor([batch.v_descale], device="cuda")
    S = 8
    ws = torch.zeros(api.mtp_verify_attn_workspace_size(batch.total_q, 16, S), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty_like(batch.q)
    args = (batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.seq_lens,
            batch.cu_seqlens_q, kd, vd, batch.softmax_scale)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        api.mtp_verify_attn_fwd(*args, num_segments=S, out=out, workspace=ws)
    torch.cuda.synchronize()
    eager = out.clone()
    api.mtp_verify_attn_fwd(*args, num_segments=S, out=out, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    g = torch.cuda.CUDAGraph()
    out.zero_()
    with torch.cuda.graph(g, stream=s):
        api.mtp_verify_attn_fwd(*args, num_segments=S, out=out, workspace=ws, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    # descales are read on the device at replay time
    kd.fill_(batch.k_descale * 2)
    g.replay()
    torch.cuda.synchronize()
    assert not torch.equal(out, eager)


def test_balanced_scheduling_repeats_within_reassociation(sched):
    """Balanced scheduling (the default) lets the pieces of a unit share its tiles: the
    split differs from call to call, the result only by float32 re-association, the tile
    counters in the workspace header are back at zero after every call, and its two call
    counters (main-kernel CTAs counted in and out) agree after every call and advance."""
    assert not api.mtp_verify_attn_get_deterministic()
    batch = synth.make_batch([5000, 5000], 4, 16, 1, seed=51, k_descale=0.5, v_descale=2.0)
    ref = oracle.verify_attention(*oracle_args(batch))
    gb = batch.to("cuda")
    kd = torch.tensor([gb.k_descale], device="cuda")
    vd = torch.tensor([gb.v_descale], device="cuda")
    ws = torch.zeros(api.mtp_verify_attn_workspace_size(gb.total_q, 16, 16), dtype=torch.uint8,
                     device="cuda")
    outs = []
    seen = []
    for _ in range(4):
        o = api.mtp_verify_attn_fwd(gb.q, gb.k_cache, gb.v_cache, gb.block_tables, gb.seq_lens,
                                    gb.cu_seqlens_q, kd, vd, gb.softmax_scale, num_segments=16,
                                    workspace=ws)
        torch.cuda.synchronize()
        assert ws[:4096].count_nonzero().item() == 0
        started, finished = ws[4096:4104].view(torch.int32).tolist()
        assert started == finished
        seen.append(started)
        outs.append(o.float().cpu().numpy().astype(np.float64))
    steps = np.diff(seen)
    assert (steps > 0).all() and (steps == steps[0]).all()      # one grid's CTAs per call
    for o in outs:
        assert oracle.excess_over_half_ulp(o, ref) <= TOL
    scale = np.abs(outs[0]).max()
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= 2 ** -7 * scale


def test_deterministic_mode_matches_oracle(sched):
    api.mtp_verify_attn_set_deterministic(True)
    try:
        check(synth.make_batch([5000, 5000, 31], [4, 2, 1], 16, 1, seed=52), num_segments=16)
    finally:
        api.mtp_verify_attn_set_deterministic(False)


def test_device_errors_set_status_and_zero_rows(sched):
    # Rows of the valid sequences are compared bit for bit across calls: fixed page ranges.
    api.mtp_verify_attn_set_deterministic(True)
    try:
        _device_errors()
    finally:
        api.mtp_verify_attn_set_deterministic(False)


def _device_errors():
    batch = synth.make_batch([100, 200, 64], [4, 4, 2], 16, 1, seed=60).to("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = run_gpu(batch, 4, status=status)
    assert status.item() == 0
    # q_len > seq_len for sequence 2
    bad = synth.PagedBatch(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                           torch.tensor([100, 200, 1], dtype=torch.int32, device="cuda"),
                           batch.cu_seqlens_q, batch.k_descale, batch.v_descale,
                           batch.softmax_scale, 1, 16)
    o2 = run_gpu(bad, 4, status=status)
    assert status.item() & api.ERR_QLEN_GT_SEQ
    assert o2[8:].abs().max().item() == 0
    assert torch.equal(o2[:8], o[:8])
    # a block-table entry outside the pool for sequence 1
    status.zero_()
    bt = batch.block_tables.clone()
    bt[1, 3] = batch.k_cache.shape[0] + 5
    o3 = run_gpu(batch, 4, status=status, block_tables=bt)
    assert status.item() & api.ERR_PAGE
    assert o3[4:8].abs().max().item() == 0
    assert torch.equal(o3[:4], o[:4]) and torch.equal(o3[8:], o[8:])


@pytest.mark.parametrize("det", [False, True])
def test_planned_with_wide_block_table(det):
    """Planned scheduling with a block table twice as wide as the sequences need: the plan
    sizes the pieces from the lengths (not from max_pages), in both tile-sharing and
    fixed-range mode."""
    api.mtp_verify_attn_set_deterministic(det)
    try:
        for S in (4, 16):
            check(synth.make_batch([3000] * 6, 4, 16, 1, seed=80 + S, max_pages=376,
                                   k_descale=0.5, v_descale=2.0), num_segments=S)
    finally:
        api.mtp_verify_attn_set_deterministic(False)


@pytest.mark.parametrize("nseq,hkv,S", [(100, 1, 16), (70, 2, 4), (150, 1, 2), (40, 4, 64),
                                        (32, 1, 16), (33, 1, 16), (16, 2, 64), (9, 1, 3)])
def test_planned_many_units_ragged(nseq, hkv, S, sched):
    """Many (sequence, KV head) units with log-uniform lengths: the plan's general path (up to
    8 units per lane of the planning warp, the binary searches over the piece size and the
    slots), its 32-way searches for at most 32 units, and with more units than SMs
    (nseq x hkv = 160) the chunked fallback."""
    ctx = synth.log_uniform_contexts(nseq, 6, 3000, seed=nseq + hkv)
    ql = synth.uniform_q_lens(nseq, 1, 4, seed=nseq + 7)
    ctx = [max(c, q) for c, q in zip(ctx, ql)]
    check(synth.make_batch(ctx, ql, 8 * hkv, hkv, seed=100 + nseq, kv_recipe="unit",
                           k_descale=0.5, v_descale=2.0), num_segments=S)


@pytest.mark.parametrize("nseq,hkv,S", [(300, 1, 8), (200, 4, 3), (200, 4, 1)])
def test_many_units_chunked_pieces(nseq, hkv, S, sched):
    """More units than SMs: both switches run the chunked kernel, whose persistent CTAs walk
    several units each and whose chunks straddle unit boundaries."""
    ctx = synth.log_uniform_contexts(nseq, 6, 1500, seed=nseq + hkv)
    ql = synth.uniform_q_lens(nseq, 1, 4, seed=nseq + 7)
    ctx = [max(c, q) for c, q in zip(ctx, ql)]
    check(synth.make_batch(ctx, ql, 8 * hkv, hkv, seed=100 + nseq, kv_recipe="unit",
                           k_descale=0.5, v_descale=2.0), num_segments=S)


def test_scheduling_switch_refuses_unknown_modes():
    with pytest.raises(ValueError):
        api.mtp_verify_attn_set_scheduling(7)
    assert api.mtp_verify_attn_get_scheduling() == api.SCHED_PLANNED


def test_host_pointers_are_refused():
    batch = synth.make_batch([100], 4, 16, 1, seed=70)
    gb = batch.to("cuda")
    with pytest.raises(api.MtpAttnError) as ei:
        api.mtp_verify_attn_fwd(gb.q, gb.k_cache, gb.v_cache, batch.block_tables, gb.seq_lens,
                                gb.cu_seqlens_q, torch.ones(1, device="cuda"),
                                torch.ones(1, device="cuda"), 0.0625, num_segments=2)
    assert ei.value.code == api.E_DEVICE


def test_num_segments_heuristic_on_device():
    sms = torch.cuda.get_device_properties(0).multi_processor_count

    def chunked(b, hkv, v):
        share = -(-(b * hkv * v) // sms)
        return min(64, -(-v // share) + 1)

    def planned(b, hkv, v):
        u = b * hkv
        if u > min(256, sms):
            return chunked(b, hkv, v)
        return max(1, min(64, sms - u + 1, -(-v // 8)))

    cases = ((16, 1, 2188), (1, 1, 3), (1000, 8, 100), (4, 1, 2188), (8, 1, 6563), (100, 1, 400))
    assert api.mtp_verify_attn_get_scheduling() == api.SCHED_PLANNED
    for args in cases:
        s = api.mtp_verify_attn_num_segments(*args)
        assert 1 <= s <= 64 and s == planned(*args), (args, s)
    api.mtp_verify_attn_set_scheduling(api.SCHED_CHUNKED)
    try:
        for args in cases:
            s = api.mtp_verify_attn_num_segments(*args)
            assert 1 <= s <= 64 and s == chunked(*args), (args, s)
    finally:
        api.mtp_verify_attn_set_scheduling(api.SCHED_PLANNED)


@pytest.mark.parametrize("name,S", [("verify_16x35k_gqa16", 16), ("verify_16x35k_gqa8", 16),
                                    ("verify_4x35k_gqa16", 64), ("verify_16x70k_gqa16", 16),
                                    ("draft_extend_8", 0), ("decode_8", 0)])
def test_full_size_sampled_against_oracle(name, S, sched):
    """The benchmark shapes at full size, in the launch configuration the bench
    times, checked on sampled sequences the oracle computes one by one."""
    _full_size(name, S, "amax")


@pytest.mark.parametrize("name,S", [("verify_16x35k_gqa16", 16), ("verify_16x70k_gqa16", 16),
                                    ("draft_extend_8", 0)])
def test_full_size_unit_recipe_sampled_against_oracle(name, S, sched):
    """The same at full size with K/V codes e4m3(x), x ~ N(0, 1): logits of order one, so
    tens of thousands of comparable weights accumulate in every row.  This exercises the
    lazy rescaling and the scaled hi/lo encoding of P over 35k-70k keys, which the
    near-argmax softmax of the per-tensor-amax recipe leaves mostly idle."""
    _full_size(name, S, "unit")


def _full_size(name, S, recipe):
    batch = synth.workload(name, seed=1, device="cuda", kv_recipe=recipe)
    got = run_gpu(batch, S or None).float().cpu().numpy().astype(np.float64)
    args = oracle_args(batch)
    B = batch.num_seqs
    # the longest sequence too: in the ragged batches it is the one unit cut into S pieces,
    # whose rows the reduce merges with a second round of loads
    longest = int(np.argmax(batch.seq_lens.cpu().numpy()))
    seqs = sorted({0, B - 1, B // 2, longest})
    rows = oracle.verify_attention_rows(*args, seqs=seqs)
    cu = batch.cu_seqlens_q.cpu().tolist()
    ref = np.concatenate([rows[b] for b in seqs])
    res = np.concatenate([got[cu[b]:cu[b + 1]] for b in seqs])
    assert oracle.excess_over_half_ulp(res, ref) <= TOL


POOL_MARKER = 0x7fd00d1e


def _pool_rows(ws, batch, S):
    """Output rows whose first split slot carries the slot-pool redirect."""
    rows = batch.total_q * batch.num_q_heads
    h = api.WORKSPACE_HEADER_BYTES
    lse = ws[h:h + rows * S * 4].view(torch.int32).view(rows, S).cpu()
    return (lse[:, 0] == POOL_MARKER).nonzero().flatten().tolist()


@pytest.mark.parametrize("det", [False, True], ids=["balanced", "deterministic"])
@pytest.mark.parametrize("ctx,ql,hq,hkv", [
    ([20000, 30, 500, 7], [4, 1, 2, 3], 16, 1),
    ([9, 41000, 64, 300, 15, 2], [1, 4, 4, 2, 1, 1], 16, 1),
    ([12000, 100, 2], [3, 4, 1], 16, 2),
    ([30000, 17, 200], [1, 1, 1], 8, 1),          # decode, GQA 8
])
def test_slot_pool_long_unit_takes_more_than_s_pieces(ctx, ql, hq, hkv, det):
    """When the library chooses S, one long sequence among short ones may take more than S
    pieces (the workspace's rows x S partial slots are shared out by length).  The output
    matches the oracle, and the workspace shows that the pool layout was used."""
    api.mtp_verify_attn_set_deterministic(det)
    try:
        batch = synth.make_batch(ctx, ql, hq, hkv, seed=sum(ctx) % 997, kv_recipe="unit",
                                 k_descale=0.5, v_descale=2.0)
        gb = batch.to("cuda")
        S = api.mtp_verify_attn_num_segments(gb.num_seqs, hkv, gb.block_tables.shape[1])
        kd = torch.tensor([gb.k_descale], device="cuda")
        vd = torch.tensor([gb.v_descale], device="cuda")
        ws = torch.zeros(api.mtp_verify_attn_workspace_size(gb.total_q, hq, S), dtype=torch.uint8,
                         device="cuda")
        out = api.mtp_verify_attn_fwd(gb.q, gb.k_cache, gb.v_cache, gb.block_tables, gb.seq_lens,
                                      gb.cu_seqlens_q, kd, vd, gb.softmax_scale, num_segments=0,
                                      workspace=ws)
        torch.cuda.synchronize()
        ref = oracle.verify_attention(*oracle_args(batch))
        got = out.float().cpu().numpy().astype(np.float64)
        assert oracle.excess_over_half_ulp(got, ref) <= TOL
        assert len(_pool_rows(ws, gb, S)) == gb.total_q * hq        # every row redirected
        assert ws[:4096].count_nonzero().item() == 0                  # counters reset
        # with an explicit S the same batch keeps the row-major slots and the same result
        ws.zero_()
        out2 = api.mtp_verify_attn_fwd(gb.q, gb.k_cache, gb.v_cache, gb.block_tables,
                                       gb.seq_lens, gb.cu_seqlens_q, kd, vd, gb.softmax_scale,
                                       num_segments=S, workspace=ws)
        torch.cuda.synchronize()
        assert _pool_rows(ws, gb, S) == []
        got2 = out2.float().cpu().numpy().astype(np.float64)
        assert oracle.excess_over_half_ulp(got2, ref) <= TOL
    finally:
        api.mtp_verify_attn_set_deterministic(False)


def test_slot_pool_device_errors_zero_rows():
    """A bad page in the long unit under the pool layout: its rows are zeros, ERR_PAGE is set,
    the other sequences' rows are unaffected (bit for bit, fixed page ranges)."""
    api.mtp_verify_attn_set_deterministic(True)
    try:
        batch = synth.make_batch([15000, 40, 300], [4, 2, 1], 16, 1, seed=77).to("cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        good = run_gpu(batch, None, status=status)
        assert status.item() == 0
        bt = batch.block_tables.clone()
        bt[0, 700] = -5
        bad = run_gpu(batch, None, status=status, block_tables=bt)
        assert status.item() & api.ERR_PAGE
        assert bad[:4].abs().max().item() == 0
        assert torch.equal(bad[4:], good[4:])
    finally:
        api.mtp_verify_attn_set_deterministic(False)


def test_slot_pool_then_row_major_in_one_workspace():
    """Calls of both layouts alternate on one workspace without clearing it: a redirect left
    by a pool call is never followed by a call that uses the row-major slots."""
    a = synth.make_batch([20000, 30, 500, 7], [4, 1, 2, 3], 16, 1, seed=78)
    b = synth.make_batch([3000] * 4, [4, 1, 2, 3], 16, 1, seed=79)
    ga, gbb = a.to("cuda"), b.to("cuda")
    kd = torch.ones(1, device="cuda")
    S = max(api.mtp_verify_attn_num_segments(4, 1, ga.block_tables.shape[1]),
            api.mtp_verify_attn_num_segments(4, 1, gbb.block_tables.shape[1]))
    ws = torch.zeros(api.mtp_verify_attn_workspace_size(ga.total_q, 16, S), dtype=torch.uint8,
                     device="cuda")
    refs = {id(a): oracle.verify_attention(*oracle_args(a)),
            id(b): oracle.verify_attention(*oracle_args(b))}
    for host, dev, s in ((a, ga, 0), (b, gbb, 4), (a, ga, 0), (b, gbb, 0)):
        o = api.mtp_verify_attn_fwd(dev.q, dev.k_cache, dev.v_cache, dev.block_tables,
                                    dev.seq_lens, dev.cu_seqlens_q, kd, kd, dev.softmax_scale,
                                    num_segments=s, workspace=ws)
        torch.cuda.synchronize()
        got = o.float().cpu().numpy().astype(np.float64)
        assert oracle.excess_over_half_ulp(got, refs[id(host)]) <= TOL
