"""The exp split's FMA-pipe exp2 (blockwise_common.cuh, ex2_fma): its
polynomial coefficients are those the Remez exchange in
sparse_mask_transformer_gb300/csrc/ex2_poly.py derives (relative minimax on
[-1/2, 1/2] with p(0) = 1), and their error bound holds.  The device
function itself is checked against exp2 in tests/test_gpu_attention_options.py."""
import os
import re
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "sparse_mask_transformer_gb300", "csrc")


def _header_coefficients():
    src = open(os.path.join(CSRC, "blockwise_common.cuh")).read()
    body = src[src.index("float ex2_fma(float x)"):]
    body = body[:body.index("\n}\n")]
    lits = [float.fromhex(h) for h in re.findall(r"(0x1\.[0-9a-f]+p-?\d+)f", body)]
    # Horner order in the source: c4, c3 in the first fma, then c2, c1, then 1
    c4, c3, c2, c1 = lits
    return [1.0, c1, c2, c3, c4]


def test_header_constants_are_the_remez_coefficients():
    pytest.importorskip("mpmath")
    sys.path.insert(0, CSRC)
    try:
        import ex2_poly
    finally:
        sys.path.remove(CSRC)
    coeffs, level = ex2_poly.remez_exp2()
    assert [np.float32(c) for c in coeffs] == [np.float32(c) for c in _header_coefficients()]
    err = ex2_poly.fp32_relative_error(coeffs)
    assert err <= 2.9e-6 and abs(err - level) < 0.05 * level   # levelled: the exchange converged


def test_polynomial_error_bound_and_its_value_at_zero():
    """Independent of the derivation: on [-1/2, 1/2] the fp32 polynomial is
    within 2.9e-6 of 2^f relative, and exactly 1 at 0."""
    c = _header_coefficients()
    f = np.linspace(-0.5, 0.5, 200001)
    p = np.zeros_like(f)
    for a in reversed(c):
        p = p * f + a
    assert np.max(np.abs(p - np.exp2(f)) / np.exp2(f)) <= 2.9e-6
    assert c[0] == 1.0
    # a plausible slip (a dropped or swapped coefficient) is far off
    assert np.max(np.abs((1 + f * (c[1] + f * (c[2] + f * c[3]))) - np.exp2(f))) > 1e-4
