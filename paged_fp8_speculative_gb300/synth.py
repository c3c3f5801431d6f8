"""Seeded synthetic inputs for paged fp8 verify / draft-extend / decode attention.

This module only *makes inputs*: query activations, a paged fp8 K/V page pool,
block tables and the per-sequence length metadata.  It holds none of the
attention arithmetic, so both the CUDA path and the CPU oracle can take their
inputs from it without sharing any of the method.

Shapes follow the serving layout described on the aiter PR #5190 page
("gfx950 assembly MTP-verify attention for head_dim 256 fp8 paged KV",
Motivation and Modifications) and the SGLang PR #37465 page ("gfx950 assembly
attention for EAGLE verify, draft extend and decode", Modifications):

* ``q``            bf16  ``[total_q, H_q, D]`` packed (THD) query rows
* ``k_cache``      uint8 ``[num_pages, page_size, H_kv, D]`` e4m3 codes (NHD pages)
* ``v_cache``      uint8 same shape
* ``block_tables`` int32 ``[B, max_pages]`` logical page -> physical page, -1 where unused
* ``seq_lens``     int32 ``[B]``  context length including the current query tokens
* ``cu_seqlens_q`` int32 ``[B + 1]`` prefix sums of the per-sequence query counts

Two K/V value recipes are offered:

* ``"amax"``: x ~ N(0, 1) per element, divided by amax(|x|)/448 over the whole
  tensor and rounded to e4m3 (the per-tensor quantisation that the benchmark
  configurations describe).  The descale handed to the kernel is the
  configuration's own number, not the quantisation scale.
* ``"unit"``: x ~ N(0, 1) rounded to e4m3 directly, which keeps the logits O(1).

The e4m3 rounding uses PyTorch's own ``float8_e4m3fn`` cast after clamping to
the finite range: a library routine, independent of the oracle's decoder and of
the kernels' hardware conversions.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import torch

E4M3_MAX = 448.0


def quantize_e4m3(x: torch.Tensor, recipe: str) -> torch.Tensor:
    """Round a float tensor to e4m3 codes (uint8) with the given recipe."""
    x = x.float()
    if recipe == "amax":
        amax = x.abs().max().clamp_min(1e-30)
        x = x * (E4M3_MAX / amax)
    elif recipe != "unit":
        raise ValueError(f"unknown K/V recipe {recipe!r}")
    x = x.clamp(-E4M3_MAX, E4M3_MAX)
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


@dataclass
class PagedBatch:
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_tables: torch.Tensor
    seq_lens: torch.Tensor
    cu_seqlens_q: torch.Tensor
    k_descale: float
    v_descale: float
    softmax_scale: float
    num_kv_heads: int
    page_size: int
    # Extra block tables over the same page pool (rotating replicas for cold-L2
    # timing).  ``block_tables`` is replica 0.
    replica_tables: List[torch.Tensor] = field(default_factory=list)

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.numel())

    @property
    def total_q(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_q_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def head_dim(self) -> int:
        return int(self.q.shape[2])

    def kv_bytes(self) -> int:
        """K and V bytes one call reads: sum_b C_b * H_kv * D * 2."""
        return int(self.seq_lens.long().sum().item()) * self.num_kv_heads * self.head_dim * 2

    def to(self, device) -> "PagedBatch":
        mv = lambda t: t.to(device)
        return PagedBatch(mv(self.q), mv(self.k_cache), mv(self.v_cache), mv(self.block_tables),
                          mv(self.seq_lens), mv(self.cu_seqlens_q), self.k_descale, self.v_descale,
                          self.softmax_scale, self.num_kv_heads, self.page_size,
                          [mv(t) for t in self.replica_tables])


def log_uniform_contexts(n: int, lo: int, hi: int, seed: int) -> List[int]:
    """Contexts C_b = round(exp(U(ln lo, ln hi))), the draft / decode length mix."""
    g = torch.Generator().manual_seed(seed)
    u = torch.rand(n, generator=g, dtype=torch.float64)
    return [int(round(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo))))) for x in u]


def uniform_q_lens(n: int, lo: int, hi: int, seed: int) -> List[int]:
    g = torch.Generator().manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


def make_batch(contexts: Sequence[int], q_lens: Sequence[int] | int, num_q_heads: int,
               num_kv_heads: int, *, head_dim: int = 256, page_size: int = 16, seed: int = 0,
               kv_recipe: str = "amax", k_descale: float = 1.0, v_descale: float = 1.0,
               softmax_scale: Optional[float] = None, replicas: int = 1, spare_pages: int = 0,
               max_pages: Optional[int] = None, device: str = "cpu") -> PagedBatch:
    """Build one verify / extend / decode batch over a shuffled page pool.

    ``contexts[b]`` is seq_lens[b] (it includes the q_len[b] current tokens).
    The pool holds exactly the pages all replicas need plus ``spare_pages``;
    each replica's block table is a disjoint slice of one random permutation
    of the pool, so logical neighbours are never physical neighbours.
    Generation runs on ``device`` (CUDA for full-size benchmark pools).
    """
    B = len(contexts)
    if isinstance(q_lens, int):
        q_lens = [q_lens] * B
    assert len(q_lens) == B
    for c, ql in zip(contexts, q_lens):
        if ql < 1 or c < ql:
            raise ValueError(f"need 1 <= q_len <= seq_len, got q_len={ql} seq_len={c}")
    if num_q_heads % num_kv_heads:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(head_dim)
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(seed)

    n_pages = [(c + page_size - 1) // page_size for c in contexts]
    per_replica = sum(n_pages)
    pool = per_replica * replicas + spare_pages
    mp = max(n_pages) if max_pages is None else max_pages
    assert mp >= max(n_pages)

    total_q = sum(q_lens)
    q = torch.randn(total_q, num_q_heads, head_dim, generator=g, device=dev).to(torch.bfloat16)

    shape = (pool, page_size, num_kv_heads, head_dim)
    k_cache = quantize_e4m3(torch.randn(shape, generator=g, device=dev), kv_recipe)
    v_cache = quantize_e4m3(torch.randn(shape, generator=g, device=dev), kv_recipe)

    perm = torch.randperm(pool, generator=g, device=dev).to(torch.int32)
    tables = []
    for r in range(replicas):
        bt = torch.full((B, mp), -1, dtype=torch.int32, device=dev)
        off = r * per_replica
        for b in range(B):
            bt[b, :n_pages[b]] = perm[off:off + n_pages[b]]
            off += n_pages[b]
        tables.append(bt)

    seq_lens = torch.tensor(list(contexts), dtype=torch.int32, device=dev)
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(list(q_lens), dtype=torch.int32), 0)
    return PagedBatch(q, k_cache, v_cache, tables[0], seq_lens, cu.to(dev), float(k_descale),
                      float(v_descale), float(softmax_scale), num_kv_heads, page_size, tables[1:])


# Named workloads (sizes as the benchmark configurations state them):
# name -> (contexts, q_lens, H_q, H_kv, k_descale, v_descale)
def workload_spec(name: str):
    if name == "verify_tiny":            # 2 x 1000, q_len 4, 16/1, descales 1.0
        return [1000] * 2, [4] * 2, 16, 1, 1.0, 1.0
    if name == "verify_16x35k_gqa16":    # production verify shape
        return [35000] * 16, [4] * 16, 16, 1, 0.5, 2.0
    if name == "verify_16x70k_gqa16":
        return [70000] * 16, [4] * 16, 16, 1, 0.5, 2.0
    if name == "verify_2x777_kv2":       # 32 q heads on 2 KV heads
        return [777] * 2, [4] * 2, 32, 2, 1.0, 1.0
    if name == "verify_16x35k_gqa8":
        return [35000] * 16, [4] * 16, 8, 1, 0.5, 2.0
    if name == "verify_4x35k_gqa16":     # run with num_segments 64
        return [35000] * 4, [4] * 4, 16, 1, 0.5, 2.0
    if name in ("draft_extend_8", "decode_8"):
        ctx = log_uniform_contexts(8, 6, 105000, seed=4000)
        ql = uniform_q_lens(8, 1, 4, seed=4001) if name == "draft_extend_8" else [1] * 8
        return ctx, ql, 16, 1, 0.5, 2.0
    raise KeyError(name)


def workload(name: str, *, seed: int = 0, replicas: int = 1, device: str = "cpu",
             kv_recipe: str = "amax") -> PagedBatch:
    ctx, ql, hq, hkv, kd, vd = workload_spec(name)
    return make_batch(ctx, ql, hq, hkv, seed=seed, k_descale=kd, v_descale=vd,
                      replicas=replicas, device=device, kv_recipe=kv_recipe)


WORKLOADS = ("verify_tiny", "verify_16x35k_gqa16", "verify_16x70k_gqa16", "verify_2x777_kv2",
             "verify_16x35k_gqa8", "verify_4x35k_gqa16", "draft_extend_8", "decode_8")


# ---- fp8 varlen prefill inputs (aiter PR #7375 page) ---------------------------------------------

@dataclass
class PrefillBatch:
    q: torch.Tensor             # uint8 e4m3 codes [total_q, H_q, 192]
    k: torch.Tensor             # uint8 e4m3 codes [total_k, H_kv, 192]
    v: torch.Tensor             # uint8 e4m3 codes [total_k, H_kv, 128]
    cu_seqlens_q: torch.Tensor  # int32 [B + 1]
    cu_seqlens_k: torch.Tensor  # int32 [B + 1]
    q_descale: float
    k_descale: float
    v_descale: float
    max_seqlen_q: int
    max_seqlen_k: int

    def to(self, device) -> "PrefillBatch":
        mv = lambda t: t.to(device)
        return PrefillBatch(mv(self.q), mv(self.k), mv(self.v), mv(self.cu_seqlens_q),
                            mv(self.cu_seqlens_k), self.q_descale, self.k_descale, self.v_descale,
                            self.max_seqlen_q, self.max_seqlen_k)

    def flops(self, causal: bool) -> int:
        """Both products over the visible (query, key) pairs: 2 * (192 + 128) per pair and
        query head (the page's TFLOPS count)."""
        hq = int(self.q.shape[1])
        cq = self.cu_seqlens_q.tolist()
        ck = self.cu_seqlens_k.tolist()
        pairs = 0
        for b in range(len(cq) - 1):
            lq, lk = cq[b + 1] - cq[b], ck[b + 1] - ck[b]
            if not causal:
                pairs += lq * lk
            else:
                pairs += sum(max(0, min(lk, i + lk - lq + 1)) for i in range(lq)) if lq < 4096 \
                    else _causal_pairs(lq, lk)
        return 2 * (192 + 128) * pairs * hq


def _causal_pairs(lq: int, lk: int) -> int:
    """sum_i clamp(i + lk - lq + 1, 0, lk) over i < lq, in closed form."""
    total = 0
    # rows with the full key set: i + lk - lq + 1 >= lk  <=>  i >= lq - 1
    lo = max(0, lq - lk)                 # first row that sees at least one key: i >= lq - lk
    full = lq - 1                        # only the last row sees every key when lq <= lk
    if lo <= full:
        n = full - lo                    # rows lo .. full - 1 see i + lk - lq + 1 keys
        first = lo + lk - lq + 1
        total += n * first + n * (n - 1) // 2
    total += lk                          # the last row
    return total


def quantize_per_tensor(x: torch.Tensor):
    """e4m3 codes of x / (amax / 448) and the descale amax / 448 (the page's recipe)."""
    amax = float(x.abs().max().clamp_min(1e-30))
    s = amax / E4M3_MAX
    codes = (x / s).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, s


def make_prefill_batch(lq: Sequence[int], lk: Sequence[int], num_q_heads: int, num_kv_heads: int,
                       *, seed: int = 0, device: str = "cpu") -> PrefillBatch:
    """Packed varlen fp8 prefill inputs: q, k, v ~ N(0, 1), each quantised per tensor to e4m3
    with descale amax / 448 (the page's benchmark recipe)."""
    if len(lq) != len(lk):
        raise ValueError("lq and lk must have one entry per sequence")
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(seed)
    tq, tk = sum(lq), sum(lk)
    q, qd = quantize_per_tensor(torch.randn(tq, num_q_heads, 192, generator=g, device=dev))
    k, kd = quantize_per_tensor(torch.randn(max(tk, 1), num_kv_heads, 192, generator=g, device=dev))
    v, vd = quantize_per_tensor(torch.randn(max(tk, 1), num_kv_heads, 128, generator=g, device=dev))
    k, v = k[:tk], v[:tk]
    cq = torch.zeros(len(lq) + 1, dtype=torch.int32)
    ck = torch.zeros(len(lk) + 1, dtype=torch.int32)
    cq[1:] = torch.cumsum(torch.tensor(list(lq), dtype=torch.int32), 0)
    ck[1:] = torch.cumsum(torch.tensor(list(lk), dtype=torch.int32), 0)
    return PrefillBatch(q, k, v, cq.to(dev), ck.to(dev), qd, kd, vd, max(lq), max(lk))
