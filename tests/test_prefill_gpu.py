"""GPU parity of the fp8 varlen prefill attention (include/fmha_fp8_varlen.h) against the
CPU oracle (oracle.prefill), through the C ABI.

Tolerance.  Q, K and V are the e4m3 inputs themselves, so the kernel's roundings beyond
float32 re-association are P and the bf16 output.  P enters the PV products as f16 (11
significant bits, finer than bf16's 8), so the bound is the one stated for kernels whose Q
and P stay bf16/fp32: max|gpu - oracle| / std(out) <= 0.01, after granting each element
half a bf16 ulp of the exact value (oracle.excess_over_half_ulp).  (A single e4m3 P, 4
significant bits, measured 0.26 std on the causal 1500 x 1800 case.)  The log-sum-exp is
formed from the unrounded probabilities in float32 and must agree to 1e-3.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import prefill as oprefill
from paged_fp8_speculative_gb300 import api, synth

pytestmark = pytest.mark.gpu

TOL = 0.01
LSE_TOL = 1e-3


def run(b, causal, return_lse=True, **kw):
    g = b.to("cuda")
    res = api.fmha_fwd_fp8_varlen(g.q, g.k, g.v, g.q_descale, g.k_descale, g.v_descale,
                                  g.cu_seqlens_q, g.cu_seqlens_k, g.max_seqlen_q, g.max_seqlen_k,
                                  is_causal=causal, return_lse=return_lse, **kw)
    torch.cuda.synchronize()
    return res


def reference(b, causal):
    return oprefill.varlen_prefill_attention(
        b.q.cpu().numpy(), b.k.cpu().numpy(), b.v.cpu().numpy(), b.cu_seqlens_q.cpu().numpy(),
        b.cu_seqlens_k.cpu().numpy(), b.q_descale, b.k_descale, b.v_descale, causal=causal,
        return_lse=True)


def check(b, causal):
    out, lse = run(b, causal)
    ref, ref_lse = reference(b, causal)
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    err = oracle.excess_over_half_ulp(got, ref) if np.abs(ref).max() > 0 else np.abs(got).max()
    assert err <= TOL, f"excess error {err:.4g} std (raw {oracle.max_err_over_std(got, ref):.4g})"
    gl = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(gl), fin)                # -inf exactly where no key is seen
    if fin.any():
        assert np.abs(gl[fin] - ref_lse[fin]).max() <= LSE_TOL
    return err


CASES = {
    "single_200": ([200], [200], 2, 2),
    "ragged": ([1, 130, 257, 64, 5], [1, 130, 300, 0, 700], 4, 2),
    "lq_gt_lk": ([300], [100], 2, 1),
    "gqa8": ([129], [513], 8, 1),
    "long": ([1500], [1800], 4, 4),
    "many_seqs": ([97, 13, 128, 256, 1, 77, 200, 64, 33, 150, 9, 128],
                  [97, 40, 128, 200, 3, 77, 260, 64, 1, 150, 9, 300], 4, 4),
}


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_matches_oracle(name, causal):
    lq, lk, hq, hkv = CASES[name]
    check(synth.make_prefill_batch(lq, lk, hq, hkv, seed=100 + sorted(CASES).index(name)), causal)


def test_prefill_underflow_spike_closed_form():
    """The probability-underflow example of the aiter PR #7375 page's review: q[0] = 8,
    k_0[0] = 14, every other q and k coordinate 0, v_0 = +1 and every other v = -1 over
    16384 keys, scale 1/sqrt(192): exact out = (e^a - 16383) / (e^a + 16383) = -0.6699 with
    a = 112 / sqrt(192).  An fp8 P that flushed the 16383 small probabilities to zero would
    give +1."""
    n = 16384
    q = torch.zeros(1, 1, 192, dtype=torch.uint8)
    q[0, 0, 0] = 0x50                                   # 8.0 in e4m3
    k = torch.zeros(n, 1, 192, dtype=torch.uint8)
    k[0, 0, 0] = 0x56                                   # 14.0
    v = torch.full((n, 1, 128), 0xB8, dtype=torch.uint8)  # -1.0
    v[0] = 0x38                                         # +1.0
    b = synth.PrefillBatch(q, k, v, torch.tensor([0, 1], dtype=torch.int32),
                           torch.tensor([0, n], dtype=torch.int32), 1.0, 1.0, 1.0, 1, n)
    a = 112 / math.sqrt(192)
    expect = (math.exp(a) - (n - 1)) / (math.exp(a) + (n - 1))
    for causal in (False, True):
        out, lse = run(b, causal)
        o = out.float().cpu().numpy()
        assert np.abs(o - expect).max() <= 0.02, (o.min(), o.max(), expect)
        assert abs(lse.item() - math.log(math.exp(a) + n - 1)) <= LSE_TOL


def test_prefill_chunked_merge_equals_one_causal_call():
    """Chunked prefill, as the page tests it: a non-causal call of the chunk's queries over the
    prefix keys and a causal call over the chunk's own keys, merged by their log-sum-exps,
    equal one causal call over prefix + chunk."""
    P, C, hq = 300, 200, 4
    whole = synth.make_prefill_batch([C], [P + C], hq, hq, seed=11)
    pre = synth.PrefillBatch(whole.q, whole.k[:P], whole.v[:P], whole.cu_seqlens_q,
                             torch.tensor([0, P], dtype=torch.int32), whole.q_descale,
                             whole.k_descale, whole.v_descale, C, P)
    chunk = synth.PrefillBatch(whole.q, whole.k[P:], whole.v[P:], whole.cu_seqlens_q,
                               torch.tensor([0, C], dtype=torch.int32), whole.q_descale,
                               whole.k_descale, whole.v_descale, C, C)
    o_all, l_all = run(whole, True)
    o1, l1 = run(pre, False)
    o2, l2 = run(chunk, True)
    l1, l2 = l1.double().T[..., None], l2.double().T[..., None]          # [tq, hq, 1]
    m = torch.maximum(l1, l2)
    w1, w2 = torch.exp(l1 - m), torch.exp(l2 - m)
    merged = (w1 * o1.double() + w2 * o2.double()) / (w1 + w2)
    ref, _ = reference(whole, True)
    got = merged.cpu().numpy()
    assert oracle.excess_over_half_ulp(got, ref) <= TOL
    assert oracle.excess_over_half_ulp(o_all.float().cpu().numpy().astype(np.float64), ref) <= TOL
    lse_merged = (m + torch.log(w1 + w2)).squeeze(-1).T
    assert (lse_merged - l_all.double()).abs().max().item() <= 2 * LSE_TOL


def test_prefill_strided_views_and_no_lse():
    b = synth.make_prefill_batch([100, 60], [120, 60], 2, 2, seed=12)
    ref, _ = reference(b, True)
    g = b.to("cuda")
    big_q = torch.zeros(g.q.shape[0], 6, 192, dtype=torch.uint8, device="cuda")
    big_q[:, 2:4] = g.q                                   # q as a slice of a fused projection
    big_o = torch.zeros(g.q.shape[0], 3, 2, 128, dtype=torch.bfloat16, device="cuda")
    out = big_o[:, 1]
    api.fmha_fwd_fp8_varlen(big_q[:, 2:4], g.k, g.v, g.q_descale, g.k_descale, g.v_descale,
                            g.cu_seqlens_q, g.cu_seqlens_k, g.max_seqlen_q, g.max_seqlen_k,
                            is_causal=True, out=out)
    torch.cuda.synchronize()
    assert oracle.excess_over_half_ulp(out.float().cpu().numpy().astype(np.float64), ref) <= TOL
    assert big_o[:, 0].abs().max().item() == 0 and big_o[:, 2].abs().max().item() == 0


def test_prefill_bad_cu_seqlens_set_status():
    b = synth.make_prefill_batch([64, 64], [64, 64], 2, 2, seed=13).to("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad_k = torch.tensor([0, 64, 999], dtype=torch.int32, device="cuda")     # past total_k
    out = torch.zeros(128, 2, 128, dtype=torch.bfloat16, device="cuda")
    api.fmha_fwd_fp8_varlen(b.q, b.k, b.v, b.q_descale, b.k_descale, b.v_descale, b.cu_seqlens_q,
                            bad_k, 64, 64, out=out, status=status)
    torch.cuda.synchronize()
    assert status.item() & api.ERR_CU
    assert out[64:].abs().max().item() == 0                 # the bad sequence is not written
    assert out[:64].abs().max().item() > 0


def test_prefill_sequence_longer_than_max_seqlen_q_sets_status():
    """max_seqlen_q sizes the grid: a sequence with more queries than it is flagged, not
    half-written; the others are computed."""
    b = synth.make_prefill_batch([300, 100], [300, 120], 2, 2, seed=15)
    ref, _ = reference(b, False)
    g = b.to("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros(400, 2, 128, dtype=torch.bfloat16, device="cuda")
    api.fmha_fwd_fp8_varlen(g.q, g.k, g.v, g.q_descale, g.k_descale, g.v_descale, g.cu_seqlens_q,
                            g.cu_seqlens_k, 100, 300, out=out, status=status)
    torch.cuda.synchronize()
    assert status.item() & api.ERR_CU
    assert out[:300].abs().max().item() == 0                # the long sequence is not written
    got = out[300:].float().cpu().numpy().astype(np.float64)
    assert oracle.excess_over_half_ulp(got, ref[300:]) <= TOL


def test_prefill_sequence_alone_equals_the_same_sequence_in_a_batch():
    """Each CTA computes one (query tile, head, sequence) from that sequence's keys alone: a
    sequence's rows and LSEs are the same bits whether it runs alone or packed with others."""
    lq, lk = [130, 300, 64], [200, 300, 500]
    b = synth.make_prefill_batch(lq, lk, 4, 2, seed=16)
    out, lse = run(b, True)
    q0 = k0 = 0
    for i in range(len(lq)):
        one = synth.PrefillBatch(b.q[q0:q0 + lq[i]], b.k[k0:k0 + lk[i]], b.v[k0:k0 + lk[i]],
                                 torch.tensor([0, lq[i]], dtype=torch.int32),
                                 torch.tensor([0, lk[i]], dtype=torch.int32), b.q_descale,
                                 b.k_descale, b.v_descale, lq[i], lk[i])
        o1, l1 = run(one, True)
        assert torch.equal(o1.view(torch.int16), out[q0:q0 + lq[i]].view(torch.int16)), i
        assert torch.equal(l1.view(torch.int32), lse[:, q0:q0 + lq[i]].view(torch.int32)), i
        q0 += lq[i]
        k0 += lk[i]


def test_prefill_repeatable():
    b = synth.make_prefill_batch([300, 200], [400, 200], 4, 2, seed=14)
    a1, _ = run(b, True)
    a2, _ = run(b, True)
    assert torch.equal(a1, a2)


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_prefill_full_size_sampled(causal):
    """The bench's shape at full size (1 x 12288 queries over 14336 keys, 96 query and KV
    heads, one launch as the bench times it), checked on sampled row blocks of three heads.
    A block of rows [i0, i0 + n) is the oracle's own sub-problem: those rows over the first
    i0 + n + Lk - Lq keys (causal; bottom-right alignment then gives every row the same
    visible keys as in the whole sequence) or over all keys (not causal)."""
    lq, lk, hq = 12288, 14336, 96
    b = synth.make_prefill_batch([lq], [lk], hq, hq, seed=15, device="cuda")
    out, lse = run(b, causal)
    got = out.float().cpu().numpy().astype(np.float64)
    gl = lse.cpu().numpy().astype(np.float64)
    q, k, v = b.q.cpu(), b.k.cpu(), b.v.cpu()
    for h in (0, 47, 95):
        for i0, n in ((0, 64), (6016, 128), (lq - 96, 96)):
            nk = min(lk, i0 + n + lk - lq) if causal else lk
            ref, ref_lse = oprefill.varlen_prefill_attention(
                q[i0:i0 + n, h:h + 1].numpy(), k[:nk, h:h + 1].numpy(), v[:nk, h:h + 1].numpy(),
                np.array([0, n]), np.array([0, nk]), b.q_descale, b.k_descale, b.v_descale,
                causal=causal, return_lse=True)
            res = got[i0:i0 + n, h:h + 1]
            assert oracle.excess_over_half_ulp(res, ref) <= TOL, (h, i0)
            assert np.abs(gl[h, i0:i0 + n] - ref_lse[0]).max() <= LSE_TOL, (h, i0)
