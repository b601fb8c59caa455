"""The polynomial tanh of the softcap (csrc/softcap_math.cuh) against
float64 tanh: the coefficients in the header, evaluated the way the kernels
evaluate them in fp32, stay within 1e-7 of tanh on |u| <= 1, and the fitting
script reproduces them. Needs no GPU."""
import os
import re
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "flashattention_attention_backward_gb300", "csrc")
sys.path.insert(0, CSRC)

import tanh_poly_fit  # noqa: E402


def header_coefficients():
    text = open(os.path.join(CSRC, "softcap_math.cuh")).read()
    found = dict(re.findall(r"constexpr float kC(\d) = ([-+0-9.eE]+)f;", text))
    return np.array([np.float32(found[str(i)]) for i in range(len(found))], dtype=np.float32)


def test_header_coefficients_within_bound():
    c = header_coefficients()
    assert len(c) == tanh_poly_fit.DEG + 1
    assert tanh_poly_fit.max_abs_error(c) < 1e-7
    # odd function, exact at 0, and the leading term is the Taylor one (-1/3)
    u = np.float32([0.0, 0.25, -0.25, 1.0, -1.0])
    t = tanh_poly_fit.eval_fp32(c, u)
    assert t[0] == 0.0 and t[1] == -t[2] and t[3] == -t[4]
    assert abs(float(c[0]) + 1.0 / 3.0) < 1e-4


def test_fit_reproduces_header():
    # to within two float32 ulps (the least-squares solve may round
    # differently on another machine)
    c = tanh_poly_fit.fit().astype(np.float32)
    h = header_coefficients()
    assert np.all(np.abs(c - h) <= 2 * np.spacing(np.abs(h)))


def test_wrong_coefficient_breaks_bound():
    c = header_coefficients().copy()
    c[2] *= np.float32(1.01)  # a 1 % error in one coefficient
    assert tanh_poly_fit.max_abs_error(c) > 1e-7
