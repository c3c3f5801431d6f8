"""GPU parity of the fp8 Q/P tier (mtp_verify_attn_fwd_qp_fp8).

The tier rounds each query row (scaled by a power of two) and each probability once to
e4m3, the precision class of the pages' kernel (aiter PR #5190 page, "Kernel notes"; its
correctness table reports max|err| / std(out) of 0.075-0.090 and its notes put the fp8
quantisation floor at 0.13 std).  Two checks:

* against the exact fp64 oracle, on K/V codes e4m3(x), x ~ N(0, 1) (logits of order one):
  max|err| / std(out) <= 0.3 (measured 0.12-0.24 on these cases).  The 0.15 of the fp8
  class is not met on this data, and the model below shows the error is the roundings'
  own: the model alone is 0.14-0.26 std from the exact attention on the same batches, and
  on the 2 x 1000 batch each rounding by itself (Q rounded with P exact, or P rounded with
  Q exact) already costs 0.135-0.14.  The pages' 0.075-0.090 must come from data with a
  narrower spread of logits than N(0, 1) at head dim 256;
* against a model of the tier's own arithmetic (the same two roundings, the same 128-key
  tiles, lazy reference maximum and probability scaling; one piece per sequence so the
  tile order is fixed), which pins the implementation of the roundings themselves:
  max|err| / std(out) <= 0.03 (what remains is float32 against float64 arithmetic, which
  flips an occasional rounding decision).

With the per-tensor-amax codes and unit descales of the benchmark recipe the logits have a
standard deviation near 90, and a 3-bit rounding of Q moves them by whole units: no fp8
tier meets a bound there, and none is claimed.
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

TOL_FP8 = 0.3         # against the exact attention (see above)
TOL_MODEL = 0.03      # against the model of the tier's roundings


def e4m3_round(x: torch.Tensor) -> torch.Tensor:
    """Round to the nearest e4m3 value (ties to even), as float64."""
    return x.to(torch.float8_e4m3fn).to(torch.float64)


def tier_model(batch, tile=128, tau=3.0) -> np.ndarray:
    """The fp8 tier's arithmetic in float64 for one piece per sequence: Q row x scaled by
    2^a (max |x| 2^a in [128, 256)) and rounded to e4m3; per 128-key tile, a reference
    maximum m raised only when the tile beats it by more than tau (log2 units); p =
    2^(s - m + 8 - tau) summed unrounded into l and rounded to e4m3 for P V; rescaling of
    l and O by 2^(m_old - m_new); out = v_descale O / l."""
    q = batch.q.cpu().to(torch.float64)
    kc = batch.k_cache.cpu().view(torch.float8_e4m3fn).to(torch.float64)
    vc = batch.v_cache.cpu().view(torch.float8_e4m3fn).to(torch.float64)
    P = batch.page_size
    ratio = batch.num_q_heads // batch.num_kv_heads
    out = np.zeros(q.shape)
    cu = batch.cu_seqlens_q.cpu().tolist()
    c = batch.softmax_scale * batch.k_descale / math.log(2.0)
    for b, L in enumerate(batch.seq_lens.cpu().tolist()):
        idx = torch.arange(L)
        phys = batch.block_tables.cpu()[b, idx // P].long()
        K = kc[phys, idx % P]                   # [L, Hkv, D]
        V = vc[phys, idx % P]
        ql = cu[b + 1] - cu[b]
        for t in range(ql):
            vis = L - ql + t + 1
            for h in range(batch.num_q_heads):
                x = q[cu[b] + t, h]
                mx = float(x.abs().max())
                a = 8 - math.frexp(mx)[1] if mx > 0 else 0
                xr = e4m3_round(x * 2.0 ** a)
                s = (K[:vis, h // ratio] @ xr) * (c * 2.0 ** -a)
                m, l = -math.inf, 0.0
                o = torch.zeros(V.shape[-1], dtype=torch.float64)
                for j0 in range(0, vis, tile):
                    st = s[j0:j0 + tile]
                    mt = float(st.max())
                    alpha = 1.0
                    if m == -math.inf or mt > m + tau:
                        if m != -math.inf:
                            alpha = 2.0 ** (m - mt)
                        m = mt
                    pf = torch.exp2(st - m + (8.0 - tau))
                    l = l * alpha + float(pf.sum())
                    o = o * alpha + e4m3_round(pf) @ V[j0:j0 + len(st), h // ratio]
                out[cu[b] + t, h] = (batch.v_descale * o / l).numpy()
    return out


def run_tier(batch, qp_fp8=True, num_segments=None):
    kd = torch.tensor([batch.k_descale], dtype=torch.float32, device="cuda")
    vd = torch.tensor([batch.v_descale], dtype=torch.float32, device="cuda")
    fwd = api.mtp_verify_attn_fwd_qp_fp8 if qp_fp8 else api.mtp_verify_attn_fwd
    o = fwd(batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.seq_lens,
            batch.cu_seqlens_q, kd, vd, batch.softmax_scale, num_segments=num_segments)
    torch.cuda.synchronize()
    return o.float().cpu().numpy().astype(np.float64)


# The pages' correctness table (context, sequences, GQA, KV heads, descales) and the ragged
# draft-extend and decode mixes, with K/V codes e4m3(x), x ~ N(0, 1).
CASES = {
    "2x1000_gqa16": lambda: synth.make_batch([1000, 1000], 4, 16, 1, seed=41, kv_recipe="unit"),
    "2x1000_descales": lambda: synth.make_batch([1000, 1000], 4, 16, 1, seed=42, kv_recipe="unit",
                                                k_descale=0.5, v_descale=2.0),
    "2x1000_gqa8": lambda: synth.make_batch([1000, 1000], 4, 8, 1, seed=43, kv_recipe="unit"),
    "3x8000_gqa16": lambda: synth.make_batch([8000] * 3, 4, 16, 1, seed=44, kv_recipe="unit"),
    "2x777_kv2": lambda: synth.make_batch([777, 777], 4, 32, 2, seed=45, kv_recipe="unit"),
    "ragged_extend": lambda: synth.make_batch([6, 17, 250, 1031, 4099, 33], [1, 4, 2, 3, 4, 1],
                                              16, 1, seed=46, kv_recipe="unit", k_descale=0.5,
                                              v_descale=2.0),
    "decode": lambda: synth.make_batch([6, 17, 250, 1031, 4099, 33], 1, 16, 1, seed=47,
                                       kv_recipe="unit"),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_qp_fp8_within_the_fp8_bound(name):
    batch = CASES[name]()
    ref = oracle.verify_attention(*oracle_args(batch))
    got = run_tier(batch.to("cuda"))
    assert np.isfinite(got).all()
    err = oracle.max_err_over_std(got, ref)
    assert err <= TOL_FP8, f"fp8 tier error {err:.4g} std"


@pytest.mark.parametrize("name", ["2x1000_gqa16", "2x1000_descales", "2x777_kv2", "ragged_extend"])
def test_qp_fp8_matches_the_model_of_its_roundings(name):
    batch = CASES[name]()
    model = tier_model(batch)
    got = run_tier(batch.to("cuda"), num_segments=1)
    err = oracle.max_err_over_std(got, model)
    assert err <= TOL_MODEL, f"fp8 tier against its model: {err:.4g} std"


def test_qp_fp8_rounds_and_the_exact_tier_does_not():
    """On the same batch the fp8 tier's error is several times the exact tier's: the
    roundings really happen in one entry point and not in the other."""
    batch = synth.make_batch([3000, 2000], 4, 16, 1, seed=48, kv_recipe="unit")
    ref = oracle.verify_attention(*oracle_args(batch))
    gb = batch.to("cuda")
    e_fp8 = oracle.max_err_over_std(run_tier(gb, True), ref)
    e_exact = oracle.max_err_over_std(run_tier(gb, False), ref)
    assert e_exact <= 0.02
    assert e_fp8 >= 3 * e_exact
    assert e_fp8 <= TOL_FP8


@pytest.mark.parametrize("S", [1, 4, 16, 64])
def test_qp_fp8_any_segment_count(S):
    batch = synth.make_batch([1000, 345, 80], [4, 2, 3], 16, 1, seed=49, kv_recipe="unit",
                             k_descale=0.5, v_descale=2.0)
    ref = oracle.verify_attention(*oracle_args(batch))
    assert oracle.max_err_over_std(run_tier(batch.to("cuda"), num_segments=S), ref) <= TOL_FP8


def test_qp_fp8_underflow_spike():
    """The probability-underflow case (one key 7 nats above 16383 others, V = +1 on it and
    -1 elsewhere; exact out = (e^7 - 16383) / (e^7 + 16383) in every coordinate).  A
    probability is rounded after scaling by 2^(8 - 3) against the row's reference maximum,
    so the tail weights (2^-5.1 after scaling) stay normal e4m3 numbers instead of rounding
    to zero: the result keeps the exact sign and is within the 3-bit rounding of the tail."""
    n, D = 16384, 256
    k = torch.zeros(n // 16, 16, 1, D, dtype=torch.uint8)
    k[0, 0, 0, 0] = 0x56                       # 14
    v = torch.full((n // 16, 16, 1, D), 0xB8, dtype=torch.uint8)    # -1
    v[0, 0, 0, :] = 0x38                       # +1
    q = torch.zeros(1, 16, D, dtype=torch.bfloat16)
    q[0, :, 0] = 8.0
    bt = torch.randperm(n // 16, dtype=torch.int32)[None]
    kc = torch.empty_like(k)
    vc = torch.empty_like(v)
    kc[bt[0].long()] = k
    vc[bt[0].long()] = v
    batch = synth.PagedBatch(q, kc, vc, bt, torch.tensor([n], dtype=torch.int32),
                             torch.tensor([0, 1], dtype=torch.int32), 1.0, 1.0, 1.0 / 16, 1, 16)
    expect = (math.exp(7) - (n - 1)) / (math.exp(7) + (n - 1))
    o = run_tier(batch.to("cuda"))
    assert np.abs(o - expect).max() <= 0.03


def test_qp_fp8_full_size_sampled():
    """The headline shape at full size (16 x 35k, GQA 16, S = 16) on sampled sequences."""
    batch = synth.workload("verify_16x35k_gqa16", seed=1, device="cuda", kv_recipe="unit")
    got = run_tier(batch, num_segments=16)
    args = oracle_args(batch)
    seqs = [0, 7, 15]
    rows = oracle.verify_attention_rows(*args, seqs=seqs)
    cu = batch.cu_seqlens_q.cpu().tolist()
    ref = np.concatenate([rows[b] for b in seqs])
    res = np.concatenate([got[cu[b]:cu[b + 1]] for b in seqs])
    assert oracle.max_err_over_std(res, ref) <= TOL_FP8


def test_qp_fp8_refuses_batches_planned_scheduling_does_not_take():
    """More (sequence, KV head) units than SMs: E_UNSUPPORTED, nothing launched."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    batch = synth.make_batch([40] * (sms + 1), 1, 16, 1, seed=50, kv_recipe="unit").to("cuda")
    with pytest.raises(api.MtpAttnError) as e:
        run_tier(batch)
    assert e.value.code == api.E_UNSUPPORTED


def test_qp_fp8_graph_replay_bit_identical():
    """Deterministic scheduling: the tier's call captured in a CUDA graph replays bit for bit
    like the eager call, and the descales are read on the device at replay time."""
    api.mtp_verify_attn_set_deterministic(True)
    try:
        batch = synth.make_batch([5000, 2000], 4, 16, 1, seed=51, kv_recipe="unit").to("cuda")
        kd = torch.tensor([batch.k_descale], device="cuda")
        vd = torch.tensor([batch.v_descale], device="cuda")
        S = 8
        ws = torch.zeros(api.mtp_verify_attn_workspace_size(batch.total_q, 16, S),
                         dtype=torch.uint8, device="cuda")
        out = torch.empty_like(batch.q)
        args = (batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.seq_lens,
                batch.cu_seqlens_q, kd, vd, batch.softmax_scale)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            api.mtp_verify_attn_fwd_qp_fp8(*args, num_segments=S, out=out, workspace=ws)
        torch.cuda.synchronize()
        eager = out.clone()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            api.mtp_verify_attn_fwd_qp_fp8(*args, num_segments=S, out=out, workspace=ws, stream=s)
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
        kd.fill_(batch.k_descale * 2)
        g.replay()
        torch.cuda.synchronize()
        assert not torch.equal(out, eager)
    finally:
        api.mtp_verify_attn_set_deterministic(False)
