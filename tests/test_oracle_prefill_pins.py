"""Pins for oracle/prefill.py, the exact fp8 varlen prefill attention (q/k 192, v 128).

Each pin fixes the oracle to something other than itself:
  * brute force: per sequence, torch scaled_dot_product_attention in float64 on tensors
    decoded with PyTorch's float8_e4m3fn, with an explicitly built bottom-right mask and GQA
    expanded by repeat_interleave; the log-sum-exp against torch.logsumexp of the masked
    logits;
  * the value the aiter PR #7375 page prints for its probability-underflow example
    (tests/golden/underflow_spike.txt), and the closed form behind it;
  * the page's chunked-prefill property: one call over prefix + chunk equals a call over
    the prefix and a causal call over the chunk merged by their log-sum-exps;
  * closed forms and invariants: uniform keys give the mean of the visible values, a single
    query row with causal masking equals the non-causal row, descale linearity, rows that
    see no key.
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest
import torch

from oracle import prefill

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "underflow_spike.txt")


def _codes(gen: torch.Generator, shape, std=1.0) -> np.ndarray:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32) * std
    return x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _batch(lq, lk, hq, hkv, seed):
    g = torch.Generator().manual_seed(seed)
    tq, tk = sum(lq), sum(lk)
    q = _codes(g, (tq, hq, 192))
    k = _codes(g, (tk, hkv, 192))
    v = _codes(g, (tk, hkv, 128))
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int64)
    ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int64)
    return q, k, v, cq, ck


def _dec(codes: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64)


def _brute(q, k, v, cq, ck, qd, kd, vd, scale, causal):
    """(out [tq, hq, 128], lse [hq, tq]) by torch SDPA and logsumexp, per sequence."""
    import torch.nn.functional as F
    hq, hkv = q.shape[1], k.shape[1]
    r = hq // hkv
    Q, K, V = _dec(q) * qd, _dec(k) * kd, _dec(v) * vd
    out = torch.zeros(q.shape[0], hq, 128, dtype=torch.float64)
    lse = torch.full((hq, q.shape[0]), -math.inf, dtype=torch.float64)
    seen = torch.zeros(q.shape[0], dtype=torch.bool)
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])
        lq, lk = q1 - q0, k1 - k0
        if lq == 0 or lk == 0:
            continue
        mask = torch.ones(lq, lk, dtype=torch.bool)
        if causal:
            ii = torch.arange(lq)[:, None]
            jj = torch.arange(lk)[None, :]
            mask = jj <= ii + (lk - lq)
        rows = mask.any(dim=1)
        qb = Q[q0:q1].transpose(0, 1)                                  # [hq, lq, 192]
        kb = K[k0:k1].transpose(0, 1).repeat_interleave(r, dim=0)     # [hq, lk, 192]
        vb = V[k0:k1].transpose(0, 1).repeat_interleave(r, dim=0)
        o = F.scaled_dot_product_attention(qb[:, rows], kb, vb, attn_mask=mask[rows], scale=scale)
        out[q0:q1][rows] = o.transpose(0, 1)
        s = torch.einsum("hid,hjd->hij", qb, kb) * scale
        s = s.masked_fill(~mask, -math.inf)
        lse[:, q0:q1][:, rows] = torch.logsumexp(s[:, rows], dim=-1)
        seen[q0:q1] = rows
    return out.numpy(), lse.numpy(), seen.numpy()


CASES = {
    "equal": ([40, 75], [40, 75], 4, 4),
    "q_shorter": ([17, 33], [90, 64], 4, 2),
    "q_longer": ([50, 9], [20, 9], 8, 2),
    "empty_kv": ([12, 30, 5], [0, 44, 5], 2, 1),
    "one_query": ([1, 1, 1], [300, 7, 1], 4, 1),
}


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_matches_brute_force(name, causal):
    lq, lk, hq, hkv = CASES[name]
    q, k, v, cq, ck = _batch(lq, lk, hq, hkv, seed=300 + len(name) * 7 + int(causal))
    qd, kd, vd, scale = 0.75, 1.5, 2.0, 0.0625
    out, lse = prefill.varlen_prefill_attention(q, k, v, cq, ck, qd, kd, vd, scale, causal,
                                                return_lse=True)
    # the brute force applies the descales to the tensors and the scale to the logits
    ref, ref_lse, seen = _brute(q, k, v, cq, ck, qd, kd, vd, scale, causal)
    assert np.allclose(out[seen], ref[seen], rtol=1e-11, atol=1e-12)
    assert np.allclose(lse[:, seen], ref_lse[:, seen], rtol=1e-12, atol=1e-12)
    # rows that see no key: output 0, log-sum-exp -inf
    assert not out[~seen].any()
    assert np.all(np.isneginf(lse[:, ~seen]))


def test_prefill_default_scale_is_one_over_sqrt_192():
    q, k, v, cq, ck = _batch([9], [23], 2, 2, seed=41)
    a = prefill.varlen_prefill_attention(q, k, v, cq, ck, 1.0, 1.0, 1.0)
    b = prefill.varlen_prefill_attention(q, k, v, cq, ck, 1.0, 1.0, 1.0, 1.0 / math.sqrt(192))
    assert np.array_equal(a, b)


def _code_of(value: float) -> int:
    code = int(torch.tensor([value]).to(torch.float8_e4m3fn).view(torch.uint8)[0])
    assert float(torch.tensor([code], dtype=torch.uint8).view(torch.float8_e4m3fn).float()) == value
    return code


def test_prefill_printed_underflow_value():
    """The page's example: non-causal, 64 queries, 16384 keys, one head, unit descales,
    default scale; Q[:,0,0] = 8, K[0,0,0] = 14, other Q/K coordinates 0; V = +1 on the first
    key and -1 elsewhere.  The page prints the exact output as -0.6699."""
    rows = [line.split() for line in open(GOLDEN) if line.strip() and not line.startswith("#")]
    dim, keys, q00, k00, printed, decimals = rows[0]
    assert int(dim) == 192
    keys, sq = int(keys), 64
    q = np.zeros((sq, 1, 192), np.uint8)
    k = np.zeros((keys, 1, 192), np.uint8)
    v = np.full((keys, 1, 128), _code_of(-1.0), np.uint8)
    q[:, 0, 0] = _code_of(float(q00))
    k[0, 0, 0] = _code_of(float(k00))
    v[0] = _code_of(1.0)
    out, lse = prefill.varlen_prefill_attention(q, k, v, [0, sq], [0, keys], 1.0, 1.0, 1.0,
                                                return_lse=True)
    assert np.all(np.round(out, int(decimals)) == float(printed))
    # the closed form behind the printed value, and its log-sum-exp
    big = math.exp(float(q00) * float(k00) / math.sqrt(192))
    exact = (big - (keys - 1)) / (big + (keys - 1))
    assert np.allclose(out, exact, rtol=0, atol=1e-12)
    assert np.allclose(lse, math.log(big + keys - 1), rtol=1e-13)


def _merge(o1, l1, o2, l2):
    """Two results over disjoint key sets combined by their log-sum-exps (test arithmetic)."""
    a, b = l1.T[..., None], l2.T[..., None]
    m = np.maximum(a, b)
    w1, w2 = np.exp(a - m), np.exp(b - m)
    return (w1 * o1 + w2 * o2) / (w1 + w2), (m[..., 0] + np.log(w1 + w2)[..., 0]).T


@pytest.mark.parametrize("prefix,chunk", [(64, 16), (1, 40), (300, 1)])
def test_chunked_prefill_merge(prefix, chunk):
    """One causal call over prefix + chunk equals a call over the prefix (every chunk query
    sees all of it) and a causal call over the chunk, merged by their log-sum-exps."""
    g = torch.Generator().manual_seed(prefix * 1000 + chunk)
    hq, hkv = 4, 2
    q = _codes(g, (chunk, hq, 192))
    k = _codes(g, (prefix + chunk, hkv, 192))
    v = _codes(g, (prefix + chunk, hkv, 128))
    args = (0.5, 1.25, 1.5, 0.07)
    full, lf = prefill.varlen_prefill_attention(q, k, v, [0, chunk], [0, prefix + chunk], *args,
                                                causal=True, return_lse=True)
    o1, l1 = prefill.varlen_prefill_attention(q, k[:prefix], v[:prefix], [0, chunk], [0, prefix],
                                              *args, causal=False, return_lse=True)
    o2, l2 = prefill.varlen_prefill_attention(q, k[prefix:], v[prefix:], [0, chunk], [0, chunk],
                                              *args, causal=True, return_lse=True)
    om, lm = _merge(o1, l1, o2, l2)
    assert np.allclose(full, om, rtol=1e-12, atol=1e-13)
    assert np.allclose(lf, lm, rtol=1e-13, atol=1e-13)


def test_uniform_keys_give_the_mean_of_visible_values():
    g = torch.Generator().manual_seed(7)
    lq, lk, hq = 10, 6, 2
    q = _codes(g, (lq, hq, 192))
    k = np.repeat(_codes(g, (1, 1, 192)), lk, axis=0)
    v = _codes(g, (lk, 1, 128))
    vd = 1.75
    out = prefill.varlen_prefill_attention(q, k, v, [0, lq], [0, lk], 0.5, 2.0, vd, causal=True)
    V = _dec(v)[:, 0, :].numpy()
    for i in range(lq):
        n = i + lk - lq + 1                      # bottom-right: the last query sees all keys
        want = vd * V[:n].mean(axis=0) if n > 0 else np.zeros(128)
        for h in range(hq):
            assert np.allclose(out[i, h], want, rtol=1e-13, atol=1e-14)


def test_single_query_causal_equals_non_causal():
    q, k, v, cq, ck = _batch([1, 1], [50, 3], 4, 4, seed=11)
    a = prefill.varlen_prefill_attention(q, k, v, cq, ck, 1.0, 1.0, 1.0, 0.1, causal=True)
    b = prefill.varlen_prefill_attention(q, k, v, cq, ck, 1.0, 1.0, 1.0, 0.1, causal=False)
    assert np.array_equal(a, b)


def test_causal_reach_is_bottom_right():
    """Changing key j moves query i exactly when j <= i + Lk - Lq."""
    q, k, v, cq, ck = _batch([6], [9], 1, 1, seed=12)
    base = prefill.varlen_prefill_attention(q, k, v, cq, ck, 1.0, 1.0, 1.0, 0.1, causal=True)
    g = torch.Generator().manual_seed(99)
    for j in range(9):
        k2, v2 = k.copy(), v.copy()
        k2[j] = _codes(g, (1, 192), std=2.0)
        v2[j] = _codes(g, (1, 128), std=2.0)
        moved = prefill.varlen_prefill_attention(q, k2, v2, cq, ck, 1.0, 1.0, 1.0, 0.1,
                                                 causal=True)
        for i in range(6):
            changed = not np.array_equal(moved[i], base[i])
            assert changed == (j <= i + 9 - 6), (i, j)


def test_descale_linearity():
    q, k, v, cq, ck = _batch([7, 5], [11, 13], 4, 2, seed=13)
    a = prefill.varlen_prefill_attention(q, k, v, cq, ck, 1.0, 1.0, 1.0, 0.05)
    b = prefill.varlen_prefill_attention(q, k, v, cq, ck, 1.0, 1.0, 2.0, 0.05)
    c = prefill.varlen_prefill_attention(q, k, v, cq, ck, 0.5, 2.0, 1.0, 0.05)
    d = prefill.varlen_prefill_attention(q, k, v, cq, ck, 1.0, 1.0, 1.0, 0.1)
    e = prefill.varlen_prefill_attention(q, k, v, cq, ck, 2.0, 1.0, 1.0, 0.05)
    assert np.array_equal(b, 2.0 * a)
    assert np.allclose(c, a, rtol=1e-14, atol=0)
    assert np.allclose(d, e, rtol=1e-14, atol=0)


def test_gqa_groups_are_contiguous():
    q, k, v, cq, ck = _batch([5], [8], 4, 2, seed=14)
    full = prefill.varlen_prefill_attention(q, k, v, cq, ck, 1.0, 1.0, 1.0, 0.1)
    for h in range(4):
        g = h // 2
        one = prefill.varlen_prefill_attention(q[:, h:h + 1], k[:, g:g + 1], v[:, g:g + 1], cq, ck,
                                               1.0, 1.0, 1.0, 0.1)
        assert np.array_equal(full[:, h], one[:, 0])


@pytest.mark.parametrize("bad", ["dim", "heads", "cu", "cu_len"])
def test_rejects_bad_arguments(bad):
    q, k, v, cq, ck = _batch([3], [4], 2, 2, seed=15)
    if bad == "dim":
        q = q[..., :128]
    elif bad == "heads":
        k, v = np.concatenate([k, k, k], axis=1)[:, :3], np.concatenate([v, v, v], axis=1)[:, :3]
        q = np.concatenate([q, q], axis=1)[:, :4]
    elif bad == "cu":
        cq = np.array([0, 4])
    else:
        cq = np.array([0, 1, 3])
    with pytest.raises(ValueError):
        prefill.varlen_prefill_attention(q, k, v, cq, ck, 1.0, 1.0, 1.0)
