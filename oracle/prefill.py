"""Exact fp8 varlen prefill attention (query/key head dim 192, value head dim 128), in float64.

Test infrastructure only (see the package docstring).  This is the definition that a
prefill kernel is to be checked against; the library has no prefill entry point yet.

The operation (aiter PR #7375 page, "Summary", "Changes" and the self-review's list of
the shapes the kernel serves):

* Packed varlen (THD) layout: ``q`` is ``[total_q, H_q, 192]``, ``k`` is
  ``[total_k, H_kv, 192]`` and ``v`` is ``[total_k, H_kv, 128]``, all e4m3 codes.  Sequence
  b owns query rows ``cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1`` and key/value rows
  ``cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1``.  Query and key counts may differ, and a
  sequence may have no keys.
* One float32 descale each for q, k and v (per tensor).  Reading taken here: the q and k
  descales multiply the logits together with ``softmax_scale``, the v descale multiplies
  the output; all three are linear, so this equals attention over the dequantised tensors.
* ``softmax_scale`` defaults to 1/sqrt(192): the page's probability-underflow example uses
  the default scale, and its printed -0.6699 comes out with this one.
* Causal masking is bottom-right aligned: query i (0-based within its sequence) of a
  sequence with Lq queries and Lk keys sees keys j <= i + Lk - Lq.  Non-causal queries see
  every key of their sequence.
* GQA: query head h reads KV head h // (H_q / H_kv) (contiguous groups).
* A query that sees no key (Lk = 0, or causal with i + Lk - Lq < 0) gets output 0 and
  log-sum-exp -inf.
* The optional log-sum-exp is the natural logarithm of sum_j exp(s_j) over the visible
  logits s_j, laid out heads by query rows, ``[H_q, total_q]``, as the page states for the
  varlen API.  The base is a reading: the page does not give it.

The softmax is the plain one: subtract the row maximum, exponentiate, normalise.
"""
from __future__ import annotations

import math

import numpy as np

from .formats import E4M3_TABLE

HEAD_DIM_QK = 192
HEAD_DIM_V = 128


def _cu(values, total: int, name: str) -> list[int]:
    cu = [int(x) for x in np.asarray(values).reshape(-1)]
    if not cu or cu[0] != 0 or cu[-1] != total or any(b < a for a, b in zip(cu, cu[1:])):
        raise ValueError(f"{name} must rise from 0 to {total}")
    return cu


def visible_keys(i: int, lq: int, lk: int, causal: bool) -> int:
    """How many keys (a prefix 0 .. n-1 of the sequence's keys) query i sees."""
    if not causal:
        return lk
    return max(0, min(lk, i + lk - lq + 1))


def varlen_prefill_attention(q_codes, k_codes, v_codes, cu_seqlens_q, cu_seqlens_k,
                             q_descale: float, k_descale: float, v_descale: float,
                             softmax_scale: float | None = None, causal: bool = False,
                             return_lse: bool = False):
    """out ``[total_q, H_q, 128]`` float64, and lse ``[H_q, total_q]`` when asked for."""
    q_codes = np.asarray(q_codes, dtype=np.uint8)
    k_codes = np.asarray(k_codes, dtype=np.uint8)
    v_codes = np.asarray(v_codes, dtype=np.uint8)
    total_q, hq, dq = q_codes.shape
    total_k, hkv, dk = k_codes.shape
    if dq != HEAD_DIM_QK or dk != HEAD_DIM_QK or v_codes.shape != (total_k, hkv, HEAD_DIM_V):
        raise ValueError("q/k head dim must be 192 and v head dim 128, k and v of equal rows")
    if hkv <= 0 or hq % hkv:
        raise ValueError("the query heads must be a multiple of the KV heads")
    cq = _cu(cu_seqlens_q, total_q, "cu_seqlens_q")
    ck = _cu(cu_seqlens_k, total_k, "cu_seqlens_k")
    if len(cq) != len(ck):
        raise ValueError("cu_seqlens_q and cu_seqlens_k must describe the same sequences")
    scale = 1.0 / math.sqrt(HEAD_DIM_QK) if softmax_scale is None else float(softmax_scale)
    logit_scale = scale * float(q_descale) * float(k_descale)
    ratio = hq // hkv

    out = np.zeros((total_q, hq, HEAD_DIM_V), dtype=np.float64)
    lse = np.full((hq, total_q), -np.inf, dtype=np.float64)
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        lq, lk = q1 - q0, k1 - k0
        for h in range(hq):
            g = h // ratio
            Q = E4M3_TABLE[q_codes[q0:q1, h, :]]
            K = E4M3_TABLE[k_codes[k0:k1, g, :]]
            V = E4M3_TABLE[v_codes[k0:k1, g, :]]
            S = logit_scale * (Q @ K.T)                      # [lq, lk]
            for i in range(lq):
                n = visible_keys(i, lq, lk, causal)
                if n == 0:
                    continue                                 # output 0, lse -inf
                s = S[i, :n]
                m = s.max()
                p = np.exp(s - m)
                den = p.sum()
                out[q0 + i, h, :] = float(v_descale) * (p @ V[:n]) / den
                lse[h, q0 + i] = m + math.log(den)
    return (out, lse) if return_lse else out

