"""Plant plausible mistakes in oracle/prefill.py (on the CPU) and check the pins catch each one.

Each mutation is a textual edit of the prefill oracle: a top-left instead of bottom-right
causal mask, an off-by-one in the reach, a wrong GQA head, a dropped descale, a log-sum-exp
in the wrong base or without its maximum, the wrong value rows, a wrong normalisation, the
wrong default scale.  The mutated source runs in a fresh namespace (the real oracle is
untouched) through a compact copy of the pins of tests/test_oracle_prefill_pins.py.
"""
from __future__ import annotations

import math
import os
import types

import numpy as np
import pytest

from oracle.formats import E4M3_TABLE
from tests.test_oracle_prefill_pins import GOLDEN, _batch, _brute, _code_of, _merge

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "prefill.py")


def _load(edit=None):
    with open(SRC) as f:
        src = f.read()
    if edit is not None:
        old, new = edit
        assert src.count(old) >= 1, f"mutation target not found: {old!r}"
        src = src.replace(old, new)
    src = src.replace("from .formats import E4M3_TABLE", "")
    mod = types.ModuleType("prefill_mut")
    mod.__dict__["E4M3_TABLE"] = E4M3_TABLE
    exec(compile(src, "prefill_mut.py", "exec"), mod.__dict__)
    return mod


def _pins(mod) -> None:
    """Raises AssertionError when any compact pin fails."""
    f = mod.varlen_prefill_attention
    # brute force, causal and not, with GQA, unequal lengths and an empty key set
    for causal in (False, True):
        q, k, v, cq, ck = _batch([9, 14, 3], [20, 6, 0], 4, 2, seed=71 + int(causal))
        out, lse = f(q, k, v, cq, ck, 0.75, 1.5, 2.0, 0.0625, causal, return_lse=True)
        ref, ref_lse, seen = _brute(q, k, v, cq, ck, 0.75, 1.5, 2.0, 0.0625, causal)
        assert np.allclose(out[seen], ref[seen], rtol=1e-11, atol=1e-12)
        assert np.allclose(lse[:, seen], ref_lse[:, seen], rtol=1e-12, atol=1e-12)
        assert not out[~seen].any() and np.all(np.isneginf(lse[:, ~seen]))
    # default scale and the page's printed value (a smaller key count keeps it quick; the
    # closed form is checked at the printed size in the pins file)
    rows = [line.split() for line in open(GOLDEN) if line.strip() and not line.startswith("#")]
    _, keys, q00, k00, printed, decimals = rows[0]
    keys = int(keys)
    q = np.zeros((2, 1, 192), np.uint8)
    k = np.zeros((keys, 1, 192), np.uint8)
    v = np.full((keys, 1, 128), _code_of(-1.0), np.uint8)
    q[:, 0, 0] = _code_of(float(q00))
    k[0, 0, 0] = _code_of(float(k00))
    v[0] = _code_of(1.0)
    out = f(q, k, v, [0, 2], [0, keys], 1.0, 1.0, 1.0)
    assert np.all(np.round(out, int(decimals)) == float(printed))
    # chunked-prefill merge
    q, k, v, _, _ = _batch([8], [24], 2, 1, seed=73)
    args = (0.5, 1.25, 1.5, 0.07)
    full, lf = f(q, k, v, [0, 8], [0, 24], *args, causal=True, return_lse=True)
    o1, l1 = f(q, k[:16], v[:16], [0, 8], [0, 16], *args, causal=False, return_lse=True)
    o2, l2 = f(q, k[16:], v[16:], [0, 8], [0, 8], *args, causal=True, return_lse=True)
    om, lm = _merge(o1, l1, o2, l2)
    assert np.allclose(full, om, rtol=1e-12, atol=1e-13) and np.allclose(lf, lm, rtol=1e-13)


MUTANTS = {
    "top_left_causal": ("return max(0, min(lk, i + lk - lq + 1))", "return max(0, min(lk, i + 1))"),
    "reach_off_by_one": ("return max(0, min(lk, i + lk - lq + 1))", "return max(0, min(lk, i + lk - lq))"),
    "gqa_modulo": ("g = h // ratio", "g = h % hkv"),
    "q_descale_dropped": ("logit_scale = scale * float(q_descale) * float(k_descale)",
                          "logit_scale = scale * float(k_descale)"),
    "v_descale_dropped": ("out[q0 + i, h, :] = float(v_descale) * (p @ V[:n]) / den",
                          "out[q0 + i, h, :] = (p @ V[:n]) / den"),
    "lse_base_2": ("lse[h, q0 + i] = m + math.log(den)", "lse[h, q0 + i] = m + math.log2(den)"),
    "lse_without_max": ("lse[h, q0 + i] = m + math.log(den)", "lse[h, q0 + i] = math.log(den)"),
    "last_value_rows": ("(p @ V[:n])", "(p @ V[lk - n:])"),
    "mean_not_softmax": ("(p @ V[:n]) / den", "(p @ V[:n]) / n"),
    "default_scale_dv": ("1.0 / math.sqrt(HEAD_DIM_QK)", "1.0 / math.sqrt(HEAD_DIM_V)"),
    "empty_row_nan": ("                    continue                                 # output 0, lse -inf",
                      "                    out[q0 + i, h, :] = np.nan\n                    continue"),
}


def test_unmutated_prefill_oracle_passes_the_compact_pins():
    _pins(_load())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_prefill_mutation(name):
    mod = _load(MUTANTS[name])
    with pytest.raises(AssertionError):
        _pins(mod)
