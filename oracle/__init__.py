"""CPU oracle for paged fp8 split-KV verify / draft-extend / decode attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code with the CUDA path (no kernels,
headers, tables, constants or helpers) and imports nothing from the product
package.

What it computes is the plain definition of the operation, in float64, with no
segments, no blocking and no online softmax:

    out[q0+t, j, :] = v_descale * sum_i softmax_i(s) * V_i
    s_i = softmax_scale * k_descale * <q[q0+t, j, :], K_i>,  i = 0 .. L - q_len + t

with K_i, V_i the e4m3 codes of key i of sequence b and KV head j // ratio,
gathered through the block table (aiter PR #5190 page, "Motivation" and
"Kernel notes"; SGLang PR #37465 page, "Modifications").

Pinned by tests/test_oracle_pins.py against: PyTorch's float8_e4m3fn and
bfloat16 conversions (all codes), brute-force dense attention through
torch scaled_dot_product_attention in float64, closed forms (uniform keys,
single key, the probability-underflow spike case including the value printed
on the aiter PR #7375 page), and invariants (page permutation, decode
equivalence, descale linearity, causal reach).  tests/test_oracle_mutants.py
plants plausible mistakes here and checks that the pins catch them.

``oracle.prefill`` is the same kind of definition for the second workload, fp8 varlen
prefill attention with query/key head dim 192 and value head dim 128 (aiter PR #7375
page); it is pinned by tests/test_oracle_prefill_pins.py and
tests/test_oracle_prefill_mutants.py.  The library has no prefill kernel yet.
"""
from .formats import E4M3_TABLE, e4m3_value, bf16_bits_to_f64, bf16_ulp
from .attention import (kv_head_of, last_visible_key, gather_keys, verify_attention,
                        verify_attention_rows)
from .metrics import max_err_over_std, excess_over_half_ulp
from . import prefill

__all__ = ["E4M3_TABLE", "e4m3_value", "bf16_bits_to_f64", "bf16_ulp", "kv_head_of",
           "last_visible_key", "gather_keys", "verify_attention", "verify_attention_rows",
           "max_err_over_std", "excess_over_half_ulp", "prefill"]
