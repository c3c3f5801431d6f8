"""Plant plausible mistakes in the oracle (on the CPU) and check the pins catch each one.

Each mutation is a textual edit of oracle/attention.py or oracle/formats.py:
a dropped term, a wrong index or sign, a transposed operand, an off-by-one in
the causal reach.  The mutated source is executed into a fresh namespace (the
real oracle is untouched) and run through a compact copy of the pins: brute
force against torch SDPA, the uniform-key mean, the spike closed form and the
e4m3 table against PyTorch.
"""
from __future__ import annotations

import math
import os
import types

import numpy as np
import pytest
import torch

from paged_fp8_speculative_gb300 import synth
from tests.helpers import dense_sdpa_reference, oracle_args

ORACLE_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")


def _load(formats_edit=None, attention_edit=None):
    with open(os.path.join(ORACLE_DIR, "formats.py")) as f:
        fsrc = f.read()
    with open(os.path.join(ORACLE_DIR, "attention.py")) as f:
        asrc = f.read()
    for src_name, edit in (("f", formats_edit), ("a", attention_edit)):
        if edit is None:
            continue
        old, new = edit
        src = fsrc if src_name == "f" else asrc
        assert src.count(old) >= 1, f"mutation target not found: {old!r}"
        src = src.replace(old, new)
        if src_name == "f":
            fsrc = src
        else:
            asrc = src
    fmod = types.ModuleType("oracle_mut_formats")
    exec(compile(fsrc, "formats_mut.py", "exec"), fmod.__dict__)
    amod = types.ModuleType("oracle_mut_attention")
    amod.__dict__.update(E4M3_TABLE=fmod.E4M3_TABLE, bf16_bits_to_f64=fmod.bf16_bits_to_f64)
    asrc = asrc.replace("from .formats import E4M3_TABLE, bf16_bits_to_f64", "")
    exec(compile(asrc, "attention_mut.py", "exec"), amod.__dict__)
    return fmod, amod


_BATCHES = None


def _batches():
    global _BATCHES
    if _BATCHES is None:
        _BATCHES = [
            synth.make_batch([77, 40], [4, 2], 32, 2, seed=61, kv_recipe="unit", k_descale=0.75,
                             v_descale=1.25, spare_pages=3),
            synth.make_batch([50, 21, 33], [3, 1, 4], 16, 1, seed=62, kv_recipe="amax",
                             k_descale=1.5, v_descale=0.5),
        ]
    return _BATCHES


def _pins_pass(fmod, amod) -> bool:
    # e4m3 table against PyTorch
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ok = ~np.isnan(ref)
    if not np.array_equal(fmod.E4M3_TABLE[ok], ref[ok]):
        return False
    # bf16 decode against PyTorch
    bits = torch.arange(0, 65536, 97, dtype=torch.int32).to(torch.int16)
    rb = bits.view(torch.bfloat16).to(torch.float64).numpy()
    ob = fmod.bf16_bits_to_f64(bits.numpy())
    fin = np.isfinite(rb)
    if not np.array_equal(ob[fin], rb[fin]):
        return False
    # brute force
    for batch in _batches():
        try:
            got = amod.verify_attention(*oracle_args(batch))
        except (IndexError, ValueError):
            return False
        ref = dense_sdpa_reference(batch)
        if not np.abs(got - ref).max() <= 1e-12 * np.abs(ref).max():
            return False
    # uniform keys -> mean of V
    L, ql, D = 45, 4, 256
    k = np.full((4, 16, 1, D), 0x38, np.uint8)
    v = np.random.default_rng(3).integers(0, 0x7E, size=(4, 16, 1, D), dtype=np.uint8)
    bt = np.array([[3, 1, 0]], np.int32)
    q = torch.randn(ql, 16, D).to(torch.bfloat16).view(torch.int16).numpy()
    out = amod.verify_attention(q, k, v, bt, [L], [0, ql], 0.7, 1.5, 0.0625, 1)
    vals = fmod.E4M3_TABLE[v]
    keys = np.array([vals[bt[0, i // 16], i % 16, 0] for i in range(L)])
    for t in range(ql):
        if not np.allclose(out[t], 1.5 * keys[:L - ql + t + 1].mean(axis=0)[None], rtol=1e-12,
                           atol=1e-12):
            return False
    # spike closed form, D = 256, 4096 keys
    n, D = 4096, 256
    kk = np.zeros((n // 16, 16, 1, D), np.uint8); kk[0, 0, 0, 0] = 0x56
    vv = np.full((n // 16, 16, 1, D), 0xB8, np.uint8); vv[0, 0, 0, :] = 0x38
    qq = np.zeros((1, 1, D), np.uint16); qq[0, 0, 0] = 0x4100
    o = amod.verify_attention(qq, kk, vv, np.arange(n // 16, dtype=np.int32)[None], [n], [0, 1],
                              1.0, 1.0, 1.0 / 16, 1)
    e = math.exp(7.0)
    return bool(np.allclose(o, (e - (n - 1)) / (e + (n - 1)), rtol=1e-12, atol=1e-12))


def test_unmutated_oracle_passes_the_compact_pins():
    assert _pins_pass(*_load())


MUTATIONS = {
    "gqa_modulo": (None, ("return q_head // ratio", "return q_head % ratio")),
    "reach_minus_one": (None, ("return seq_len - q_len + t", "return seq_len - q_len + t - 1")),
    "no_causal_mask": (None, ("return seq_len - q_len + t", "return seq_len - 1")),
    "same_reach_all_tokens": (None, ("return seq_len - q_len + t", "return seq_len - q_len")),
    "count_off_by_one": (None, ("n = last_visible_key(L, ql, t) + 1", "n = last_visible_key(L, ql, t)")),
    "wrong_kv_head_in_gather": (None, ("codes[phys, :n, kv_head, :]", "codes[phys, :n, 0, :]")),
    "slot_page_swapped": (None, ("int(block_table_row[i // page_size])", "int(block_table_row[i % page_size])")),
    "dropped_k_descale": (None, ("softmax_scale * k_descale * (K[:n]", "softmax_scale * (K[:n]")),
    "v_descale_on_logits": (None, ("softmax_scale * k_descale * (K[:n]", "softmax_scale * v_descale * (K[:n]")),
    "dropped_v_descale": (None, ("out_b[t, j] = v_descale * (w @ V[:n])", "out_b[t, j] = (w @ V[:n])")),
    "keys_for_values": (None, ("out_b[t, j] = v_descale * (w @ V[:n])", "out_b[t, j] = v_descale * (w @ K[:n])")),
    "no_normalisation": (None, ("w /= w.sum()", "pass")),
    "query_row_without_offset": (None, ("(K[:n] @ q[q0 + t, j])", "(K[:n] @ q[t, j])")),
    "e4m3_bias_8": (("2.0 ** (exp_field - 7)", "2.0 ** (exp_field - 8)"), None),
    "e4m3_subnormal_scale": (("(mant / 8.0) * 2.0 ** (1 - 7)", "(mant / 8.0) * 2.0 ** (0 - 7)"), None),
    "e4m3_sign_bit": (("-1.0 if code & 0x80 else 1.0", "-1.0 if code & 0x40 else 1.0"), None),
    "e4m3_mantissa_width": (("(1.0 + mant / 8.0)", "(1.0 + mant / 16.0)"), None),
    "bf16_shift": (("<< np.uint32(16)", "<< np.uint32(15)"), None),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name):
    f_edit, a_edit = MUTATIONS[name]
    assert not _pins_pass(*_load(f_edit, a_edit)), f"mutation {name} slipped through the pins"
