"""Randomised differential test of the verify / extend / decode attention.

Seeded random batches (1 to 40 sequences, contexts of 1 to 9000 tokens with a log-uniform
spread, q_len 1 to 4, GQA 8 or 16, 1 to 4 KV heads, an explicit segment count or the
library's choice, both K/V recipes, descales other than 1, spare pages in the pool) go through
planned scheduling with balanced tile sharing, planned scheduling with fixed page ranges and
chunked scheduling.  Every call must leave the status word clear; the three results must agree
to within the float32 re-association of the split-KV merge; every case's longest sequence and
one more are checked against the oracle.  The plan's device-side searches, the slot pool and
the chunk layout each take different paths through the index arithmetic, so a case one of
them gets wrong shows up as a disagreement.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_fp8_speculative_gb300 import api, synth
from tests.helpers import oracle_args

pytestmark = pytest.mark.gpu

CASES = 200


def random_batch(rng: np.random.Generator):
    B = int(rng.integers(1, 41))
    ctx = np.exp(rng.uniform(0.0, np.log(9000.0), size=B)).astype(int)
    ctx = np.maximum(ctx, 1)
    ql = [int(min(rng.integers(1, 5), c)) for c in ctx]
    ratio = int(rng.choice([8, 16]))
    hkv = int(rng.choice([1, 1, 2, 4]))
    recipe = str(rng.choice(["amax", "unit"]))
    kd, vd = float(rng.choice([1.0, 0.5])), float(rng.choice([1.0, 2.0]))
    S = int(rng.choice([0, 0, 1, 2, 5, 16, 64]))
    spare = int(rng.integers(0, 8))
    batch = synth.make_batch([int(c) for c in ctx], ql, ratio * hkv, hkv,
                             seed=int(rng.integers(1 << 30)), kv_recipe=recipe, k_descale=kd,
                             v_descale=vd, spare_pages=spare)
    return batch, S


def agree(a: np.ndarray, b: np.ndarray) -> float:
    """Two bf16 results of the same arithmetic in different summation orders: each element may
    round to either neighbour of its float32 value, so one bf16 ulp is granted; the rest, over
    the standard deviation of the output."""
    excess = np.maximum(0.0, np.abs(a - b) - oracle.bf16_ulp(b))
    sd = float(b.std())
    return float(excess.max()) / sd if sd > 0 else float(excess.max())


def run(b, S, sched, det):
    api.mtp_verify_attn_set_scheduling(sched)
    api.mtp_verify_attn_set_deterministic(det)
    try:
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        kd = torch.tensor([b.k_descale], dtype=torch.float32, device="cuda")
        vd = torch.tensor([b.v_descale], dtype=torch.float32, device="cuda")
        out = api.mtp_verify_attn_fwd(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                                      b.cu_seqlens_q, kd, vd, b.softmax_scale, num_segments=S,
                                      status=status)
        torch.cuda.synchronize()
        assert status.item() == 0, status.item()
        return out.float().cpu().numpy().astype(np.float64)
    finally:
        api.mtp_verify_attn_set_scheduling(api.SCHED_PLANNED)
        api.mtp_verify_attn_set_deterministic(False)


@pytest.mark.parametrize("block", range(8))
def test_random_batches_agree_across_schedulings_and_with_the_oracle(block):
    rng = np.random.default_rng(1000 + block)
    for case in range(CASES // 8):
        batch, S = random_batch(rng)
        b = batch.to("cuda")
        planned = run(b, S, api.SCHED_PLANNED, False)
        fixed = run(b, S, api.SCHED_PLANNED, True)
        chunked = run(b, S, api.SCHED_CHUNKED, False)
        tag = (block, case, batch.seq_lens.tolist()[:6], S, b.num_q_heads, b.num_kv_heads)
        # the same arithmetic in a different summation order
        assert agree(fixed, planned) <= 0.01, tag
        assert agree(chunked, planned) <= 0.01, tag
        # and against the exact definition on two sequences (the longest, and another)
        lens = batch.seq_lens.numpy()
        seqs = sorted({int(np.argmax(lens)), int(rng.integers(len(lens)))})
        rows = oracle.verify_attention_rows(*oracle_args(batch), seqs=seqs)
        cu = batch.cu_seqlens_q.tolist()
        ref = np.concatenate([rows[s] for s in seqs])
        got = np.concatenate([planned[cu[s]:cu[s + 1]] for s in seqs])
        assert oracle.excess_over_half_ulp(got, ref) <= 0.01, tag
