"""Decode rows are verify rows, every call runs its kernels exactly once, and a sequence's rows
do not depend on its place in the batch.

Row t of a verify sequence (context L, q_len n) attends to keys 0 .. L - n + t, the keys a
q_len-1 decode of the same query token over a context of L - n + t + 1 keys, through the same
block table, attends to (the verify-row / decode identity the oracle is pinned to).  With one
segment no call splits a sequence's keys, so both calls accumulate a row's keys in the same
order: the decode batch built from a verify batch's rows must give the same bf16 outputs bit
for bit, under both schedulings and in both tile modes.  The masked keys of the verify's last
tile contribute exact zeros.

The workspace header documents two call counters that the main kernel's CTAs increment when
they start and after their last write: over N calls on one workspace (eager, then replays of
a captured graph) both must grow by the same grid size per call, and the tile counters must be
back at zero after each call.  A call whose kernels ran twice, or not at all, would show.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_fp8_speculative_gb300 import api, synth
from paged_fp8_speculative_gb300.synth import PagedBatch
from tests.helpers import oracle_args

pytestmark = pytest.mark.gpu


def decode_batch_of(batch: PagedBatch) -> PagedBatch:
    """One q_len-1 sequence per query token of `batch`: the token's row of q, its sequence's
    block table and the context that ends at that token."""
    cu = batch.cu_seqlens_q.tolist()
    lens = batch.seq_lens.tolist()
    rows, ctx, seq = [], [], []
    for b, L in enumerate(lens):
        n = cu[b + 1] - cu[b]
        for t in range(n):
            rows.append(cu[b] + t)
            ctx.append(L - n + t + 1)
            seq.append(b)
    dev = batch.q.device
    return PagedBatch(batch.q[rows].contiguous(), batch.k_cache, batch.v_cache,
                      batch.block_tables[seq].contiguous(),
                      torch.tensor(ctx, dtype=torch.int32, device=dev),
                      torch.arange(len(rows) + 1, dtype=torch.int32, device=dev),
                      batch.k_descale, batch.v_descale, batch.softmax_scale, batch.num_kv_heads,
                      batch.page_size)


def run(b: PagedBatch, S: int, ws: torch.Tensor | None = None) -> torch.Tensor:
    kd = torch.tensor([b.k_descale], dtype=torch.float32, device="cuda")
    vd = torch.tensor([b.v_descale], dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = api.mtp_verify_attn_fwd(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                                  b.cu_seqlens_q, kd, vd, b.softmax_scale, num_segments=S,
                                  workspace=ws, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return out


BATCHES = {
    # q_len 1..4, contexts around page and tile boundaries and a long one
    "gqa16": lambda: synth.make_batch([4, 17, 130, 1031, 4099, 2048, 20000], [4, 1, 3, 4, 2, 4, 4],
                                      16, 1, seed=71, k_descale=0.5, v_descale=2.0),
    "gqa8_kv2": lambda: synth.make_batch([9, 300, 1500, 129], [2, 4, 3, 4], 16, 2, seed=72,
                                         kv_recipe="unit"),
}


@pytest.mark.parametrize("det", [False, True], ids=["balanced", "fixed"])
@pytest.mark.parametrize("sched", [api.SCHED_PLANNED, api.SCHED_CHUNKED],
                         ids=["planned", "chunked"])
@pytest.mark.parametrize("name", list(BATCHES))
def test_decode_rows_bit_identical_to_verify_rows(name, sched, det):
    batch = BATCHES[name]()
    api.mtp_verify_attn_set_scheduling(sched)
    api.mtp_verify_attn_set_deterministic(det)
    try:
        v = batch.to("cuda")
        verify = run(v, 1)
        decode = run(decode_batch_of(v), 1)
    finally:
        api.mtp_verify_attn_set_scheduling(api.SCHED_PLANNED)
        api.mtp_verify_attn_set_deterministic(False)
    assert decode.shape == verify.shape
    diff = (decode.view(torch.int16) != verify.view(torch.int16)).sum().item()
    assert diff == 0, f"{diff} of {verify.numel()} outputs differ"
    # and both are the oracle's attention
    got = verify.float().cpu().numpy().astype(np.float64)
    assert oracle.excess_over_half_ulp(got, oracle.verify_attention(*oracle_args(batch))) <= 0.01


def header_counters(ws: torch.Tensor):
    words = ws[:api.WORKSPACE_HEADER_BYTES].view(torch.int32).cpu()
    return words[:1024].clone(), int(words[1024]), int(words[1025])


@pytest.mark.parametrize("sched", [api.SCHED_PLANNED, api.SCHED_CHUNKED],
                         ids=["planned", "chunked"])
def test_each_call_runs_its_kernels_once(sched):
    batch = synth.make_batch([700, 33, 2500], [4, 2, 1], 16, 1, seed=73).to("cuda")
    S = 4
    ws = torch.zeros(api.mtp_verify_attn_workspace_size(batch.total_q, batch.num_q_heads, S),
                     dtype=torch.uint8, device="cuda")
    kd = torch.tensor([batch.k_descale], dtype=torch.float32, device="cuda")
    vd = torch.tensor([batch.v_descale], dtype=torch.float32, device="cuda")
    out = torch.empty_like(batch.q)
    api.mtp_verify_attn_set_scheduling(sched)
    try:
        def call():
            api.mtp_verify_attn_fwd(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                    batch.seq_lens, batch.cu_seqlens_q, kd, vd,
                                    batch.softmax_scale, num_segments=S, out=out, workspace=ws)

        call()
        torch.cuda.synchronize()
        tiles, started, finished = header_counters(ws)
        grid = started
        assert grid > 0 and finished == started and int(tiles.abs().sum()) == 0
        for n in range(2, 5):                                  # eager calls
            call()
            torch.cuda.synchronize()
            tiles, started, finished = header_counters(ws)
            assert (started, finished) == (n * grid, n * grid), (n, started, finished, grid)
            assert int(tiles.abs().sum()) == 0
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):                 # capture launches nothing
            call()
        torch.cuda.synchronize()
        assert header_counters(ws)[1] == 4 * grid
        for r in range(1, 4):                                  # graph replays
            g.replay()
            torch.cuda.synchronize()
            tiles, started, finished = header_counters(ws)
            assert (started, finished) == ((4 + r) * grid, (4 + r) * grid), (r, started, finished)
            assert int(tiles.abs().sum()) == 0
    finally:
        api.mtp_verify_attn_set_scheduling(api.SCHED_PLANNED)


def permuted(batch: PagedBatch, perm) -> PagedBatch:
    """The same sequences in the order `perm` (q rows, block tables, lengths moved together)."""
    cu = batch.cu_seqlens_q.tolist()
    rows = [r for b in perm for r in range(cu[b], cu[b + 1])]
    ql = [cu[b + 1] - cu[b] for b in perm]
    dev = batch.q.device
    return PagedBatch(batch.q[rows].contiguous(), batch.k_cache, batch.v_cache,
                      batch.block_tables[list(perm)].contiguous(),
                      batch.seq_lens[list(perm)].contiguous(),
                      torch.tensor([0] + list(np.cumsum(ql)), dtype=torch.int32, device=dev),
                      batch.k_descale, batch.v_descale, batch.softmax_scale, batch.num_kv_heads,
                      batch.page_size), rows


@pytest.mark.parametrize("S", [1, 4, 0], ids=["S1", "S4", "library_S"])
def test_sequence_order_does_not_change_any_row(S):
    """Planned scheduling cuts every (sequence, KV head) unit by its length alone, so in
    deterministic mode a unit's pieces, and the order the reduce merges them in, do not depend
    on where the sequence sits in the batch: reordering the sequences reorders the output rows
    and changes no bit."""
    batch = synth.make_batch([17, 5000, 260, 1031, 9000, 3], [2, 4, 1, 3, 4, 1], 16, 2, seed=74,
                             kv_recipe="unit").to("cuda")
    api.mtp_verify_attn_set_deterministic(True)
    try:
        base = run(batch, S)
        for seed in range(3):
            perm = np.random.default_rng(seed).permutation(batch.num_seqs).tolist()
            pb, rows = permuted(batch, perm)
            got = run(pb, S)
            assert torch.equal(got.view(torch.int16), base[rows].view(torch.int16)), (perm, S)
    finally:
        api.mtp_verify_attn_set_deterministic(False)


def test_a_sequence_alone_equals_the_same_sequence_in_a_batch():
    """With one segment every unit is computed whole by one CTA: a sequence's rows do not
    depend on which other sequences share the call."""
    batch = synth.make_batch([900, 4100, 33, 2500], [3, 4, 1, 2], 16, 1, seed=75).to("cuda")
    api.mtp_verify_attn_set_deterministic(True)
    try:
        together = run(batch, 1)
        cu = batch.cu_seqlens_q.tolist()
        for b in range(batch.num_seqs):
            alone, rows = permuted(batch, [b])
            got = run(alone, 1)
            want = together[cu[b]:cu[b + 1]]
            assert torch.equal(got.view(torch.int16), want.view(torch.int16)), b
    finally:
        api.mtp_verify_attn_set_deterministic(False)
