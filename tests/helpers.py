"""Test helpers: marshal a synthetic batch into the oracle's numpy inputs."""
from __future__ import annotations

import numpy as np
import torch


def oracle_args(batch):
    """Positional arguments for oracle.verify_attention from a PagedBatch."""
    cpu = lambda t: t.detach().cpu()
    return (cpu(batch.q).view(torch.int16).numpy(),
            cpu(batch.k_cache).numpy(), cpu(batch.v_cache).numpy(),
            cpu(batch.block_tables).numpy(), cpu(batch.seq_lens).numpy(),
            cpu(batch.cu_seqlens_q).numpy(), batch.k_descale, batch.v_descale,
            batch.softmax_scale, batch.num_kv_heads)


def dense_sdpa_reference(batch) -> np.ndarray:
    """Brute-force dense attention through torch SDPA in float64.

    Independent of the oracle: it decodes e4m3 with PyTorch's float8_e4m3fn and
    bf16 with PyTorch's bfloat16, gathers every key of a sequence with one
    fancy-index over (page, slot), builds the bottom-right causal mask with
    torch.tril and expands GQA with repeat_interleave.
    """
    import torch.nn.functional as F
    q = batch.q.cpu().to(torch.float64)
    kc = batch.k_cache.cpu().view(torch.float8_e4m3fn).to(torch.float64)
    vc = batch.v_cache.cpu().view(torch.float8_e4m3fn).to(torch.float64)
    P = batch.page_size
    Hkv = batch.num_kv_heads
    ratio = batch.num_q_heads // Hkv
    out = torch.zeros_like(q)
    cu = batch.cu_seqlens_q.cpu().tolist()
    for b, L in enumerate(batch.seq_lens.cpu().tolist()):
        idx = torch.arange(L)
        phys = batch.block_tables.cpu()[b, idx // P].long()
        K = kc[phys, idx % P]            # [L, Hkv, D]
        V = vc[phys, idx % P]
        ql = cu[b + 1] - cu[b]
        qb = q[cu[b]:cu[b + 1]].transpose(0, 1)                          # [Hq, ql, D]
        Kx = K.transpose(0, 1).repeat_interleave(ratio, dim=0) * batch.k_descale
        Vx = V.transpose(0, 1).repeat_interleave(ratio, dim=0) * batch.v_descale
        mask = torch.ones(ql, L, dtype=torch.bool).tril(diagonal=L - ql)
        o = F.scaled_dot_product_attention(qb, Kx, Vx, attn_mask=mask,
                                           scale=batch.softmax_scale)
        out[cu[b]:cu[b + 1]] = o.transpose(0, 1)
    return out.numpy()
