"""Randomised parity of the fp8 varlen prefill against the oracle.

Seeded random packed batches (1 to 8 sequences, 0 to 700 queries and keys each, including
empty query or key sets and more queries than keys, GQA 1, 2, 4 or 8, 1 to 3 KV heads, causal
or not) are run through the kernel and compared with the oracle at the bf16-class bound
(half a bf16 ulp granted, 0.01 std) and on the log-sum-exp (1e-3, -inf exactly where a query
sees no key).
"""
from __future__ import annotations

import numpy as np
import pytest

from paged_fp8_speculative_gb300 import synth
from tests.test_prefill_gpu import check

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("block", range(4))
def test_random_prefill_batches_match_the_oracle(block):
    rng = np.random.default_rng(2000 + block)
    for case in range(10):
        B = int(rng.integers(1, 9))
        lq = [int(x) for x in rng.integers(0, 701, size=B)]
        lk = [int(x) if rng.random() > 0.1 else 0 for x in rng.integers(1, 701, size=B)]
        if sum(lq) == 0:
            lq[0] = 1
        if sum(lk) == 0:
            lk[0] = 1
        hkv = int(rng.integers(1, 4))
        hq = hkv * int(rng.choice([1, 2, 4, 8]))
        causal = bool(rng.integers(0, 2))
        b = synth.make_prefill_batch(lq, lk, hq, hkv, seed=int(rng.integers(1 << 30)))
        check(b, causal)
