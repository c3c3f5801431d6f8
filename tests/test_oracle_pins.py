"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each test names what fixes the expected value: a library routine that
implements the same definition independently, a closed form, an invariant of
the mathematics, or a value printed on the pages (tests/golden/).
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_fp8_speculative_gb300 import synth
from tests.helpers import dense_sdpa_reference, oracle_args

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --- number formats -----------------------------------------------------------------------

def test_e4m3_table_matches_torch_for_all_codes():
    """All 256 codes against PyTorch's float8_e4m3fn -> float64 conversion."""
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = oracle.E4M3_TABLE
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.isnan(ours[[0x7F, 0xFF]]).all() and np.isnan(ours).sum() == 2


def test_e4m3_spec_values():
    """Values fixed by the OCP E4M3 definition."""
    assert oracle.e4m3_value(0x7E) == 448.0            # largest finite
    assert oracle.e4m3_value(0xFE) == -448.0
    assert oracle.e4m3_value(0x08) == 2.0 ** -6        # smallest normal
    assert oracle.e4m3_value(0x01) == 2.0 ** -9        # smallest subnormal
    assert oracle.e4m3_value(0x07) == 7 * 2.0 ** -9    # largest subnormal
    assert oracle.e4m3_value(0x38) == 1.0
    assert oracle.e4m3_value(0xB8) == -1.0
    assert oracle.e4m3_value(0x56) == 14.0
    assert oracle.e4m3_value(0x80) == 0.0 and math.copysign(1, oracle.e4m3_value(0x80)) < 0


def test_bf16_decode_matches_torch():
    bits = torch.arange(0, 65536, 7, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    ours = oracle.bf16_bits_to_f64(bits.numpy())
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert oracle.bf16_bits_to_f64(np.array([0x3F80, 0xC000, 0x4100], np.uint16)).tolist() == [1.0, -2.0, 8.0]


def test_bf16_ulp_against_torch_nextafter():
    x = torch.tensor([1.0, 1.5, 3.0, 300.0, -0.01, 2.0 ** -130], dtype=torch.bfloat16)
    up = torch.nextafter(x.abs(), torch.tensor(float("inf"), dtype=torch.bfloat16))
    ref = (up.double() - x.abs().double()).numpy()
    assert np.array_equal(oracle.bf16_ulp(x.double().numpy()), ref)


# --- brute force ----------------------------------------------------------------------------

@pytest.mark.parametrize("case", [
    dict(contexts=[37, 200, 16], q_lens=[4, 3, 1], hq=16, hkv=1, kd=0.5, vd=2.0, recipe="unit"),
    dict(contexts=[150, 64], q_lens=[2, 4], hq=8, hkv=1, kd=1.0, vd=1.0, recipe="amax"),
    dict(contexts=[77, 129], q_lens=[4, 4], hq=32, hkv=2, kd=0.75, vd=1.25, recipe="unit"),
    dict(contexts=[5, 4, 33], q_lens=[1, 4, 2], hq=16, hkv=2, kd=1.5, vd=0.5, recipe="amax"),
])
def test_oracle_matches_dense_sdpa(case):
    """Brute-force dense attention (torch SDPA, float64) on tiny shuffled-page inputs."""
    batch = synth.make_batch(case["contexts"], case["q_lens"], case["hq"], case["hkv"],
                             seed=11, kv_recipe=case["recipe"], k_descale=case["kd"],
                             v_descale=case["vd"], spare_pages=5, max_pages=20)
    got = oracle.verify_attention(*oracle_args(batch))
    ref = dense_sdpa_reference(batch)
    scale = np.abs(ref).max()
    assert np.abs(got - ref).max() <= 1e-12 * scale


# --- closed forms ---------------------------------------------------------------------------

def _make_codes(pool, hkv, D, fill):
    return np.full((pool, 16, hkv, D), fill, dtype=np.uint8)


def test_uniform_keys_give_mean_of_visible_values():
    """All keys equal => every visible key has weight 1/n: out = v_descale * mean(V_0..V_pos)."""
    rng = np.random.default_rng(3)
    L, ql, D, pool = 45, 4, 256, 6
    k = _make_codes(pool, 1, D, 0x38)                       # every key coordinate 1.0
    v = rng.integers(0, 0x7E, size=(pool, 16, 1, D), dtype=np.uint8)
    bt = np.array([[4, 0, 2, -1, -1]], np.int32)
    q = torch.randn(ql, 16, D).to(torch.bfloat16).view(torch.int16).numpy()
    out = oracle.verify_attention(q, k, v, bt, [L], [0, ql], 0.7, 1.5, 0.0625, 1)
    vals = oracle.E4M3_TABLE[v]
    keys = np.array([vals[bt[0, i // 16], i % 16, 0] for i in range(L)])
    for t in range(ql):
        n = L - ql + t + 1
        expect = 1.5 * keys[:n].mean(axis=0)
        assert np.allclose(out[t], expect[None, :], rtol=1e-13, atol=1e-13)


def test_single_key_and_descale_linearity():
    """L = 1: out = v_descale * V_0 exactly; out is linear in v_descale;
    halving k_descale while doubling softmax_scale leaves out unchanged."""
    rng = np.random.default_rng(5)
    D = 256
    k = rng.integers(0, 0x7E, size=(3, 16, 1, D), dtype=np.uint8)
    v = rng.integers(0, 0x7E, size=(3, 16, 1, D), dtype=np.uint8)
    q = torch.randn(1, 8, D).to(torch.bfloat16).view(torch.int16).numpy()
    bt = np.array([[2]], np.int32)
    out = oracle.verify_attention(q, k, v, bt, [1], [0, 1], 1.0, 3.0, 0.1, 1)
    assert np.array_equal(out[0], np.broadcast_to(3.0 * oracle.E4M3_TABLE[v[2, 0, 0]], (8, D)))

    batch = synth.make_batch([300], 4, 16, 1, seed=8, kv_recipe="unit", k_descale=1.0,
                             v_descale=1.0)
    a = list(oracle_args(batch))
    base = oracle.verify_attention(*a)
    a2 = list(a); a2[7] = 2.0
    assert np.array_equal(oracle.verify_attention(*a2), 2.0 * base)
    a3 = list(a); a3[6] = 0.5; a3[8] = 2.0 * a[8]
    assert np.allclose(oracle.verify_attention(*a3), base, rtol=1e-12, atol=1e-12)


def _spike_case(D, keys, q00, k00):
    """One query row over ``keys`` keys: q[0] = q00, K_0[0] = k00, V_0 = +1, V_i = -1."""
    pages = keys // 16
    k = np.zeros((pages, 16, 1, D), np.uint8)
    k[0, 0, 0, 0] = [c for c in range(256) if oracle.e4m3_value(c) == k00][0]
    v = np.full((pages, 16, 1, D), 0xB8, np.uint8)    # -1.0
    v[0, 0, 0, :] = 0x38                               # +1.0
    q = np.zeros((1, 1, D), np.uint16)
    q[0, 0, 0] = np.array([q00], np.float32).view(np.uint32)[0] >> 16
    bt = np.arange(pages, dtype=np.int32)[None, :]
    out = oracle.verify_attention(q, k, v, bt, [keys], [0, 1], 1.0, 1.0, 1.0 / math.sqrt(D), 1)
    return out[0, 0]


def test_underflow_spike_printed_value():
    """The exact answer the aiter PR #7375 review prints for its underflow case (D = 192)."""
    with open(os.path.join(GOLDEN, "underflow_spike.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for D, keys, q00, k00, printed, decimals in rows:
        D, keys, decimals = int(D), int(keys), int(decimals)
        out = _spike_case(D, keys, float(q00), float(k00))
        assert np.allclose(out, out[0])
        assert abs(out[0] - float(printed)) <= 0.5 * 10.0 ** -decimals


@pytest.mark.parametrize("D,keys", [(256, 16384), (256, 35008), (192, 16384)])
def test_underflow_spike_closed_form(D, keys):
    """out = (e^a - (n-1)) / (e^a + (n-1)), a = 8 * 14 / sqrt(D), n keys."""
    a = 8.0 * 14.0 / math.sqrt(D)
    n = keys
    expect = (math.exp(a) - (n - 1)) / (math.exp(a) + (n - 1))
    out = _spike_case(D, keys, 8.0, 14.0)
    assert np.allclose(out, expect, rtol=1e-12, atol=1e-12)
    if D == 256 and keys == 16384:
        assert round(expect, 6) == -0.874524


# --- invariants -----------------------------------------------------------------------------

def test_page_permutation_is_bit_identical():
    """Permuting the physical pages and remapping the block table changes nothing."""
    batch = synth.make_batch([200, 95], [4, 2], 16, 2, seed=21, kv_recipe="unit", spare_pages=7,
                             k_descale=0.5, v_descale=2.0)
    a = oracle_args(batch)
    base = oracle.verify_attention(*a)
    pool = a[1].shape[0]
    perm = np.random.default_rng(0).permutation(pool)       # new slot of old page i = perm[i]
    k2 = np.empty_like(a[1]); v2 = np.empty_like(a[2])
    k2[perm] = a[1]; v2[perm] = a[2]
    bt = a[3].copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    out = oracle.verify_attention(a[0], k2, v2, bt, *a[4:])
    assert np.array_equal(out, base)


def test_verify_rows_equal_plain_decode():
    """Row t of a verify batch = q_len-1 decode of the same query at context L - q_len + t + 1."""
    batch = synth.make_batch([130], 4, 16, 1, seed=31, kv_recipe="amax", k_descale=0.5,
                             v_descale=2.0)
    q, k, v, bt, sl, cu, kd, vd, sc, hkv = oracle_args(batch)
    out = oracle.verify_attention(q, k, v, bt, sl, cu, kd, vd, sc, hkv)
    for t in range(4):
        ctx = 130 - 4 + t + 1
        dec = oracle.verify_attention(q[t:t + 1], k, v, bt, [ctx], [0, 1], kd, vd, sc, hkv)
        assert np.array_equal(dec[0], out[t])


def test_causal_reach():
    """Changing key L-q_len+t+1 (just past the reach of token t) leaves row t unchanged and
    changes row t+1; unused block-table entries (-1) are never read."""
    batch = synth.make_batch([70], 4, 8, 1, seed=41, kv_recipe="unit", max_pages=9)
    q, k, v, bt, sl, cu, kd, vd, sc, hkv = oracle_args(batch)
    base = oracle.verify_attention(q, k, v, bt, sl, cu, kd, vd, sc, hkv)
    for t in range(3):
        i = 70 - 4 + t + 1
        k2 = k.copy(); v2 = v.copy()
        k2[bt[0, i // 16], i % 16] ^= 0x11
        v2[bt[0, i // 16], i % 16] ^= 0x22
        out = oracle.verify_attention(q, k2, v2, bt, sl, cu, kd, vd, sc, hkv)
        assert np.array_equal(out[:t + 1], base[:t + 1])
        assert not np.array_equal(out[t + 1], base[t + 1])
    assert (bt[0, 5:] == -1).all()


def test_gqa_groups_are_contiguous():
    """With two KV heads, query heads 0..r-1 read KV head 0 and r..2r-1 read KV head 1:
    swapping the two KV heads' data swaps the two halves of the output."""
    batch = synth.make_batch([90], 3, 16, 2, seed=51, kv_recipe="unit")
    q, k, v, bt, sl, cu, kd, vd, sc, hkv = oracle_args(batch)
    base = oracle.verify_attention(q, k, v, bt, sl, cu, kd, vd, sc, hkv)
    qs = np.concatenate([q[:, 8:], q[:, :8]], axis=1)
    out = oracle.verify_attention(qs, k[:, :, ::-1].copy(), v[:, :, ::-1].copy(), bt, sl, cu, kd,
                                  vd, sc, hkv)
    assert np.array_equal(out[:, :8], base[:, 8:])
    assert np.array_equal(out[:, 8:], base[:, :8])


def test_rejects_q_len_beyond_seq_len():
    q = np.zeros((4, 16, 256), np.uint16)
    k = np.zeros((1, 16, 1, 256), np.uint8)
    with pytest.raises(ValueError):
        oracle.verify_attention(q, k, k, np.zeros((1, 1), np.int32), [3], [0, 4], 1.0, 1.0, 1.0, 1)


# --- error measures -------------------------------------------------------------------------

def test_error_measures_on_hand_example():
    ref = np.array([1.0, -1.0, 3.0, -3.0])            # population std = sqrt(5)
    res = ref + np.array([0.0, 0.5, 0.0, -0.25])
    assert math.isclose(oracle.max_err_over_std(res, ref), 0.5 / math.sqrt(5.0))
    # half a bf16 ulp at 3.0 is 2^-7 (spacing 2^-6 in [2, 4)), at 1.0 it is 2^-8
    assert math.isclose(oracle.excess_over_half_ulp(res, ref),
                        (0.5 - 2.0 ** -8) / math.sqrt(5.0))
    assert oracle.excess_over_half_ulp(ref + np.array([2.0 ** -8, 0, 2.0 ** -7, 0]), ref) == 0.0
