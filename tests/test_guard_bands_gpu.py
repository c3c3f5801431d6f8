"""Writes stay inside their buffers and inputs are left as they were.

Every output the kernels write (verify: out and the workspace; prefill: out and lse) is a view
into a larger buffer whose other bytes hold a pattern: guard bands before and after, and the
gaps that padded row and head strides leave inside `out`.  After the call the pattern must be
intact, the outputs must be right (verify: the oracle; prefill: bit for bit the same call into
plain contiguous buffers), and every input (q, the caches, block tables, lengths, descales; q,
k, v and cu_seqlens for the prefill) must be bit-identical to a copy taken before the call.
Verify runs under both schedulings, with an explicit segment count and with the library's
choice (whose slot pool lays the partials out by length).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_fp8_speculative_gb300 import api, synth
from tests.helpers import oracle_args

pytestmark = pytest.mark.gpu

PAT16 = -0x3EA1            # 0xC15F as int16: a bf16 value no kernel writes by chance
PAT8 = 0xA5
GUARD = 4096               # guard band bytes (a multiple of 256: keeps the workspace aligned)


def guarded_out(rows: int, heads: int, dim: int, pad_head: int, pad_row: int):
    """A bf16 [rows, heads, dim] view with `pad_head` spare elements after each head's dim and
    `pad_row` after each row, inside guard bands; returns (view, backing int16 buffer)."""
    hs = dim + pad_head
    rs = heads * hs + pad_row
    g = GUARD // 2
    back = torch.full((2 * g + rows * rs,), PAT16, dtype=torch.int16, device="cuda")
    view = back[g:g + rows * rs].view(torch.bfloat16).as_strided((rows, heads, dim), (rs, hs, 1))
    return view, back


def written_mask(rows: int, heads: int, dim: int, pad_head: int, pad_row: int) -> torch.Tensor:
    hs = dim + pad_head
    rs = heads * hs + pad_row
    g = GUARD // 2
    m = torch.zeros(2 * g + rows * rs, dtype=torch.bool)
    idx = (torch.arange(rows)[:, None, None] * rs + torch.arange(heads)[None, :, None] * hs +
           torch.arange(dim)[None, None, :]).reshape(-1)
    m[g + idx] = True
    return m


def snapshot(*ts):
    return [t.clone() for t in ts]


def unchanged(before, after) -> bool:
    return all(torch.equal(a.view(torch.uint8) if a.dtype != torch.uint8 else a,
                           b.view(torch.uint8) if b.dtype != torch.uint8 else b)
               for a, b in zip(before, after))


@pytest.mark.parametrize("S", [5, 0], ids=["S5", "library_S"])
@pytest.mark.parametrize("sched", [api.SCHED_PLANNED, api.SCHED_CHUNKED],
                         ids=["planned", "chunked"])
def test_verify_writes_only_out_and_workspace(sched, S):
    batch = synth.make_batch([6, 250, 4099, 1031, 33, 20000], [1, 4, 2, 3, 4, 4], 16, 1, seed=81,
                             k_descale=0.5, v_descale=2.0)
    b = batch.to("cuda")
    hq, tq = b.num_q_heads, b.total_q
    S_lib = S or api.mtp_verify_attn_num_segments(b.num_seqs, b.num_kv_heads,
                                                  b.block_tables.shape[1])
    need = api.mtp_verify_attn_workspace_size(tq, hq, S_lib)
    wback = torch.full((2 * GUARD + need,), PAT8, dtype=torch.uint8, device="cuda")
    ws = wback[GUARD:GUARD + need]
    ws.zero_()
    out, oback = guarded_out(tq, hq, 256, pad_head=8, pad_row=24)
    kd = torch.tensor([b.k_descale], dtype=torch.float32, device="cuda")
    vd = torch.tensor([b.v_descale], dtype=torch.float32, device="cuda")
    inputs = (b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, b.cu_seqlens_q, kd, vd)
    before = snapshot(*inputs)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mtp_verify_attn_set_scheduling(sched)
    try:
        for _ in range(2):                      # the second call reuses the workspace
            api.mtp_verify_attn_fwd(*inputs[:6], kd, vd, b.softmax_scale, num_segments=S, out=out,
                                    workspace=ws, status=status)
        torch.cuda.synchronize()
    finally:
        api.mtp_verify_attn_set_scheduling(api.SCHED_PLANNED)
    assert status.item() == 0
    assert bool((wback[:GUARD] == PAT8).all()) and bool((wback[GUARD + need:] == PAT8).all())
    mask = written_mask(tq, hq, 256, 8, 24).to("cuda")
    assert bool((oback[~mask] == PAT16).all()), "a write outside out's elements"
    assert unchanged(before, inputs), "an input changed"
    got = out.float().cpu().numpy().astype(np.float64)
    assert oracle.excess_over_half_ulp(got, oracle.verify_attention(*oracle_args(batch))) <= 0.01


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_prefill_writes_only_out_and_lse(causal):
    lq, lk = [130, 0, 257, 64], [200, 5, 257, 40]
    batch = synth.make_prefill_batch(lq, lk, 8, 2, seed=82)
    b = batch.to("cuda")
    tq, hq = sum(lq), 8
    out, oback = guarded_out(tq, hq, 128, pad_head=16, pad_row=8)
    g = GUARD // 4
    lback = torch.full((2 * g + hq * tq,), float("nan"), dtype=torch.float32, device="cuda")
    lback.view(torch.int32)[:] = 0x7FC0A5A5
    lse = lback[g:g + hq * tq].view(hq, tq)
    inputs = (b.q, b.k, b.v, b.cu_seqlens_q, b.cu_seqlens_k)
    before = snapshot(*inputs)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.fmha_fwd_fp8_varlen(b.q, b.k, b.v, b.q_descale, b.k_descale, b.v_descale, b.cu_seqlens_q,
                            b.cu_seqlens_k, max(lq), max(lk), is_causal=causal, return_lse=True,
                            out=out, lse=lse, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    mask = written_mask(tq, hq, 128, 16, 8).to("cuda")
    assert bool((oback[~mask] == PAT16).all()), "a write outside out's elements"
    lw = lback.view(torch.int32)
    assert bool((lw[:g] == 0x7FC0A5A5).all()) and bool((lw[g + hq * tq:] == 0x7FC0A5A5).all())
    assert unchanged(before, inputs), "an input changed"
    # the same call into plain contiguous buffers: the kernel is deterministic, so the strided
    # outputs must hold the same bits
    ref_out, ref_lse = api.fmha_fwd_fp8_varlen(b.q, b.k, b.v, b.q_descale, b.k_descale, b.v_descale,
                                               b.cu_seqlens_q, b.cu_seqlens_k, max(lq), max(lk),
                                               is_causal=causal, return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(out.contiguous().view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))
