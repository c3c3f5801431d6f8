"""Error measures used to compare a result with the oracle.

Test infrastructure only (see the package docstring).

The accuracy figure on the aiter PR #5190 page ("Output of
op_tests/test_mtp_verify_attn_asm.py", correctness table) is the largest
absolute error divided by the standard deviation of the output.  Here the
standard deviation is the population standard deviation over every element of
the reference output of the call.
"""
from __future__ import annotations

import numpy as np

from .formats import bf16_ulp


def max_err_over_std(result: np.ndarray, reference: np.ndarray) -> float:
    """max |result - reference| / std(reference), std over the whole tensor."""
    result = np.asarray(result, dtype=np.float64)
    reference = np.asarray(reference, dtype=np.float64)
    sd = float(reference.std())
    return float(np.abs(result - reference).max()) / sd if sd > 0 else float(
        np.abs(result - reference).max())


def excess_over_half_ulp(result: np.ndarray, reference: np.ndarray) -> float:
    """Like max_err_over_std, after granting each element half a bf16 ulp.

    A bf16 output cannot be closer to an exact value than half a bf16 ulp of
    that value, so that much of the error belongs to the output format, not to
    the computation: per element, max(0, |result - reference| - ulp/2).
    """
    result = np.asarray(result, dtype=np.float64)
    reference = np.asarray(reference, dtype=np.float64)
    excess = np.maximum(0.0, np.abs(result - reference) - 0.5 * bf16_ulp(reference))
    sd = float(reference.std())
    return float(excess.max()) / sd if sd > 0 else float(excess.max())
