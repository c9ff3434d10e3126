"""The polynomial exponential of the e4m3 forward's split-exponential option
(CPU checks of the committed coefficients).

"Kernels and Memory in LLM Inference", "FlashAttention-4: when the roof moves",
item 1: some exponentials run as a short polynomial on the CUDA cores.  The
coefficients in csrc/exp2_poly.h come from a Lawson minimax fit
(tiled_attention_fa2_gb300/exp2_poly.py); here they are re-derived, and the
float32 evaluation the kernel performs is checked against float64 exp2.
"""

import re

import numpy as np

from tiled_attention_fa2_gb300 import exp2_poly


def _header_coefficients():
    text = open(exp2_poly.HEADER).read()
    assert f"kExp2PolyFloor = {exp2_poly.EXP2_FLOOR!r}f" in text
    vals = re.findall(r"kExp2PolyC(\d) = ([0-9.eE+-]+)f;", text)
    return np.array([float(v) for _, v in sorted(vals)], dtype=np.float32)


def test_header_holds_the_fit():
    assert np.array_equal(_header_coefficients(), exp2_poly.coefficients32())


def test_fit_is_equal_ripple():
    """A minimax fit's relative error alternates in sign at degree + 2 points
    with (nearly) equal magnitude."""
    c = exp2_poly.lawson_fit()
    f = np.linspace(-0.5, 0.5, 200001)
    e = np.polynomial.polynomial.polyval(f, c) / np.exp2(f) - 1.0
    peak = np.abs(e).max()
    # local extrema of e (including the end points) that reach 99% of the peak
    ext = [0] + [i for i in range(1, len(e) - 1) if (e[i] - e[i - 1]) * (e[i + 1] - e[i]) <= 0] + [len(e) - 1]
    big = [e[i] for i in ext if abs(e[i]) >= 0.99 * peak]
    signs = np.sign(big)
    assert len(big) >= exp2_poly.DEGREE + 2
    assert np.all(signs[1:] != signs[:-1])


def test_float32_evaluation_error_bound():
    c32 = _header_coefficients()
    assert exp2_poly.max_rel_error(c32) < 8e-5


def test_reconstruction_over_the_kernel_range():
    """2^x = 2^round(x) * p(x - round(x)) for every x the softmax produces
    (scores minus the reference, at most 8 in log2 units) down to the floor."""
    c32 = _header_coefficients()
    x = np.concatenate([np.linspace(exp2_poly.EXP2_FLOOR, 8.0, 1 << 20, dtype=np.float32),
                        np.float32([-0.5, 0.5, -1.5, 1.5, 7.5, 8.0, 0.0, exp2_poly.EXP2_FLOOR])])
    got = exp2_poly.exp2_via_poly32(c32, x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.max(np.abs(got / ref - 1.0)) < 8e-5


def test_negative_infinity_gives_a_negligible_weight():
    """Masked keys carry -inf: the floor makes their weight about 2^-125, which
    e4m3 rounds to zero and which no row sum can notice next to the row's
    largest weight (>= 1)."""
    c32 = _header_coefficients()
    got = exp2_poly.exp2_via_poly32(c32, np.float32([-np.inf, -1e30, -127.0]))
    assert np.all(np.isfinite(got)) and np.all(got > 0) and np.all(got < 2.0 ** -124)
