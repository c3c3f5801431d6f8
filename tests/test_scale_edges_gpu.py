"""Degenerate and signed scales.

With softmax_scale = 0 every visible key has the same weight, so each output row is the mean
of the V rows its query sees (times v_descale): a closed form, checked on the oracle too.  A
negative k_descale (or a negative softmax_scale) flips the order of the logits, so the row
maximum the online softmax tracks comes from the smallest raw logit; a negative v_descale flips
the output's sign.  Both kernels must follow the definition for every sign.  And q scaled by
a power of two with the inverse softmax scale (the same logits) gives the verify kernel's
output bit for bit, from 2^-60 to 2^60.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import prefill as oprefill
from paged_fp8_speculative_gb300 import api, synth
from tests.helpers import oracle_args

pytestmark = pytest.mark.gpu

TOL = 0.01


def verify_run(batch, S):
    b = batch.to("cuda")
    kd = torch.tensor([b.k_descale], dtype=torch.float32, device="cuda")
    vd = torch.tensor([b.v_descale], dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = api.mtp_verify_attn_fwd(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                                  b.cu_seqlens_q, kd, vd, b.softmax_scale, num_segments=S,
                                  status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return out.float().cpu().numpy().astype(np.float64)


def mean_of_visible_v(batch) -> np.ndarray:
    """softmax_scale = 0: row t of sequence b is v_descale times the mean of V rows
    0 .. L - q_len + t of its KV head."""
    vc = batch.v_cache.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    cu = batch.cu_seqlens_q.tolist()
    ratio = batch.num_q_heads // batch.num_kv_heads
    out = np.zeros(tuple(batch.q.shape))
    for b, L in enumerate(batch.seq_lens.tolist()):
        n = cu[b + 1] - cu[b]
        idx = np.arange(L)
        phys = batch.block_tables[b].numpy()[idx // 16]
        V = vc[phys, idx % 16]                           # [L, H_kv, 256]
        csum = np.cumsum(V, axis=0)
        for t in range(n):
            last = L - n + t
            for h in range(batch.num_q_heads):
                out[cu[b] + t, h] = batch.v_descale * csum[last, h // ratio] / (last + 1)
    return out


@pytest.mark.parametrize("S", [1, 7])
def test_verify_zero_softmax_scale_is_the_mean_of_visible_values(S):
    batch = synth.make_batch([1, 5, 300, 2049], [1, 4, 3, 4], 16, 1, seed=101, kv_recipe="unit",
                             v_descale=2.0, softmax_scale=0.0)
    got = verify_run(batch, S)
    closed = mean_of_visible_v(batch)
    ref = oracle.verify_attention(*oracle_args(batch))
    assert np.abs(ref - closed).max() <= 1e-12 * max(1.0, np.abs(closed).max())
    assert oracle.excess_over_half_ulp(got, closed) <= TOL


@pytest.mark.parametrize("kd,vd,scale", [(-0.5, 2.0, 1 / 16), (1.0, -1.0, 1 / 16),
                                         (0.5, 1.0, -1 / 16)],
                         ids=["neg_k_descale", "neg_v_descale", "neg_scale"])
@pytest.mark.parametrize("sched", [api.SCHED_PLANNED, api.SCHED_CHUNKED],
                         ids=["planned", "chunked"])
def test_verify_signed_scales_follow_the_definition(kd, vd, scale, sched):
    batch = synth.make_batch([40, 700, 3000], [4, 2, 4], 16, 1, seed=102, kv_recipe="unit",
                             k_descale=kd, v_descale=vd, softmax_scale=scale)
    api.mtp_verify_attn_set_scheduling(sched)
    try:
        got = verify_run(batch, 5)
    finally:
        api.mtp_verify_attn_set_scheduling(api.SCHED_PLANNED)
    ref = oracle.verify_attention(*oracle_args(batch))
    assert oracle.excess_over_half_ulp(got, ref) <= TOL


@pytest.mark.parametrize("kd_sign,vd_sign,scale", [(1, 1, 0.0), (-1, 1, None), (1, -1, None),
                                                   (1, 1, -1 / 192 ** 0.5)],
                         ids=["zero_scale", "neg_k_descale", "neg_v_descale", "neg_scale"])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_prefill_signed_and_zero_scales_follow_the_definition(kd_sign, vd_sign, scale, causal):
    lq, lk = [200, 64, 130], [300, 64, 90]
    b = synth.make_prefill_batch(lq, lk, 4, 2, seed=103)
    kd, vd = kd_sign * b.k_descale, vd_sign * b.v_descale
    g = b.to("cuda")
    out, lse = api.fmha_fwd_fp8_varlen(g.q, g.k, g.v, b.q_descale, kd, vd, g.cu_seqlens_q,
                                       g.cu_seqlens_k, max(lq), max(lk), softmax_scale=scale,
                                       is_causal=causal, return_lse=True)
    torch.cuda.synchronize()
    ref, ref_lse = oprefill.varlen_prefill_attention(
        b.q.numpy(), b.k.numpy(), b.v.numpy(), b.cu_seqlens_q.numpy(), b.cu_seqlens_k.numpy(),
        b.q_descale, kd, vd, softmax_scale=scale, causal=causal, return_lse=True)
    got = out.float().cpu().numpy().astype(np.float64)
    assert oracle.excess_over_half_ulp(got, ref) <= TOL
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(lse.cpu().numpy()))
    bound = 1e-3 * max(1.0, np.abs(ref_lse[fin]).max())
    assert np.abs(lse.cpu().numpy()[fin] - ref_lse[fin]).max() <= bound


@pytest.mark.parametrize("k", [-60, -20, 20, 60])
def test_verify_q_scaled_by_a_power_of_two_with_the_inverse_scale_is_bit_identical(k):
    """q times 2^k with softmax_scale times 2^-k: the same logits.  The kernel scales each Q row
    by a power of two before its e4m3 split and folds the inverse into the logit scale, so the
    output must be bit-identical to the unscaled call, from tiny to huge query magnitudes."""
    batch = synth.make_batch([333, 1200], [4, 3], 16, 1, seed=104, kv_recipe="unit",
                             k_descale=0.5, v_descale=2.0)
    api.mtp_verify_attn_set_deterministic(True)
    try:
        base = verify_run(batch, 3)
        batch.q = (batch.q.double() * 2.0 ** k).to(torch.bfloat16)
        batch.softmax_scale = batch.softmax_scale * 2.0 ** -k
        scaled = verify_run(batch, 3)
    finally:
        api.mtp_verify_attn_set_deterministic(False)
    assert np.array_equal(base, scaled)
