"""Exact paged attention for verify, draft extend and decode, in float64.

Test infrastructure only (see the package docstring).

The operation (aiter PR #5190 page, "Motivation", "Modifications" and
"Kernel notes"; SGLang PR #37465 page, "Modifications"):

* Each sequence b has ``q_len`` query tokens (1..4) packed in ``q`` starting at
  ``cu_seqlens_q[b]``, and ``seq_lens[b]`` keys in a paged NHD cache.  Reading
  taken here: ``seq_lens`` counts the current query tokens too (their K/V are
  already in the cache), so the last query token sees every key.
* Causal over the last ``q_len`` positions, bottom-right aligned (the mask the
  aiter PR #7375 page calls "causal (bottom-right aligned)"): query token t of
  a sequence of length L sees keys 0 .. L - q_len + t.
* GQA: query head j reads KV head j // ratio, ratio = H_q / H_kv (contiguous
  groups; the pages give only the ratios 16 and 8).
* K/V are e4m3 codes with per-tensor float32 descales.  Reading: the K descale
  multiplies the logits together with softmax_scale, and the V descale
  multiplies the output; both are linear, so this is the same as attending
  over dequantised K = k_descale * e4m3(code) and V = v_descale * e4m3(code).
* Logical page p of sequence b lives in physical page block_tables[b][p];
  key i is slot i % page_size of logical page i // page_size.

Softmax is computed in the plain way (subtract the row max, exponentiate,
normalise) over all visible keys at once.  Split-KV segments and the LSE
merge of the CUDA path are a re-association of the same sums and have no
counterpart here.
"""
from __future__ import annotations

import numpy as np

from .formats import E4M3_TABLE, bf16_bits_to_f64


def kv_head_of(q_head: int, ratio: int) -> int:
    """KV head read by query head ``q_head`` (contiguous GQA groups)."""
    return q_head // ratio


def last_visible_key(seq_len: int, q_len: int, t: int) -> int:
    """Index of the last key query token ``t`` may attend to (bottom-right causal)."""
    return seq_len - q_len + t


def gather_keys(codes: np.ndarray, block_table_row: np.ndarray, seq_len: int, kv_head: int
                ) -> np.ndarray:
    """Decoded float64 rows 0 .. seq_len-1 of one sequence and one KV head.

    ``codes`` is the uint8 page pool ``[num_pages, page_size, H_kv, D]``.
    Only the first ceil(seq_len / page_size) block-table entries are read.
    """
    page_size = codes.shape[1]
    rows = np.empty((seq_len, codes.shape[3]), dtype=np.float64)
    for i in range(0, seq_len, page_size):
        phys = int(block_table_row[i // page_size])
        if not 0 <= phys < codes.shape[0]:
            raise IndexError(f"block table entry {phys} outside the page pool")
        n = min(page_size, seq_len - i)
        rows[i:i + n] = E4M3_TABLE[codes[phys, :n, kv_head, :]]
    return rows


def _as_bits(q) -> np.ndarray:
    q = np.asarray(q)
    if q.dtype not in (np.uint16, np.int16):
        raise TypeError("q must be given as bf16 bit patterns (uint16 or int16)")
    return q


def verify_attention_rows(q_bits, k_codes, v_codes, block_tables, seq_lens, cu_seqlens_q,
                          k_descale: float, v_descale: float, softmax_scale: float,
                          num_kv_heads: int, seqs=None) -> dict:
    """Exact outputs for the sequences in ``seqs`` (all if None).

    Returns {b: float64 array [q_len_b, H_q, D]} so large batches can be
    checked on a sample of sequences.
    """
    q = bf16_bits_to_f64(_as_bits(q_bits))
    k_codes = np.asarray(k_codes, dtype=np.uint8)
    v_codes = np.asarray(v_codes, dtype=np.uint8)
    block_tables = np.asarray(block_tables)
    seq_lens = np.asarray(seq_lens)
    cu = np.asarray(cu_seqlens_q)
    total_q, num_q_heads, head_dim = q.shape
    if num_q_heads % num_kv_heads:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    ratio = num_q_heads // num_kv_heads
    if seqs is None:
        seqs = range(len(seq_lens))
    result = {}
    for b in seqs:
        L = int(seq_lens[b])
        q0, q1 = int(cu[b]), int(cu[b + 1])
        ql = q1 - q0
        if ql < 1 or ql > L:
            raise ValueError(f"sequence {b}: need 1 <= q_len <= seq_len (q_len={ql}, seq_len={L})")
        out_b = np.zeros((ql, num_q_heads, head_dim), dtype=np.float64)
        for h in range(num_kv_heads):
            K = gather_keys(k_codes, block_tables[b], L, h)
            V = gather_keys(v_codes, block_tables[b], L, h)
            for j in range(num_q_heads):
                if kv_head_of(j, ratio) != h:
                    continue
                for t in range(ql):
                    n = last_visible_key(L, ql, t) + 1
                    s = softmax_scale * k_descale * (K[:n] @ q[q0 + t, j])
                    w = np.exp(s - s.max())
                    w /= w.sum()
                    out_b[t, j] = v_descale * (w @ V[:n])
        result[b] = out_b
    return result


def verify_attention(q_bits, k_codes, v_codes, block_tables, seq_lens, cu_seqlens_q,
                     k_descale: float, v_descale: float, softmax_scale: float,
                     num_kv_heads: int) -> np.ndarray:
    """Exact float64 output ``[total_q, H_q, D]`` for the whole batch."""
    q_bits = _as_bits(q_bits)
    cu = np.asarray(cu_seqlens_q)
    out = np.zeros(q_bits.shape, dtype=np.float64)
    rows = verify_attention_rows(q_bits, k_codes, v_codes, block_tables, seq_lens, cu,
                                 k_descale, v_descale, softmax_scale, num_kv_heads)
    for b, ob in rows.items():
        out[int(cu[b]):int(cu[b + 1])] = ob
    return out
