"""The FMA-pipe exp2 used by the softmax warps: its coefficients come from a
committed Remez fit; check the header matches a fresh fit and that the fp32
evaluation scheme meets its accuracy bounds against fp64 exp2."""
import importlib.util
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_attention_99_gb300", "csrc")


def load_fit():
    spec = importlib.util.spec_from_file_location("fit_exp2", os.path.join(CSRC, "fit_exp2.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def header_coeffs():
    text = open(os.path.join(CSRC, "exp2_poly.h")).read()
    return np.array([float(v) for v in re.findall(r"#define FA_EXP2_C\d ([-0-9.e]+)f", text)], dtype=np.float32)


def test_header_matches_fit():
    fit = load_fit()
    c = fit.remez().astype(np.float32)
    np.testing.assert_array_equal(c, header_coeffs())


def test_relative_error_and_bias():
    fit = load_fit()
    c = header_coeffs()
    x = np.linspace(-100.0, 0.0, 3_000_001, dtype=np.float32)
    y = fit.fp32_eval(c, x).astype(np.float64)
    rel = y / np.exp2(x.astype(np.float64)) - 1.0
    assert np.abs(rel).max() < 1e-4
    assert abs(rel.mean()) < 2e-5


def test_underflow_and_exact_points():
    fit = load_fit()
    c = header_coeffs()
    assert fit.fp32_eval(c, np.array([-127.0, -200.0, -np.inf], dtype=np.float32)).tolist() == [0.0, 0.0, 0.0]
    y = fit.fp32_eval(c, np.array([0.0, -1.0, -10.0], dtype=np.float32)).astype(np.float64)
    np.testing.assert_allclose(y, [1.0, 0.5, 2.0 ** -10], rtol=1e-4)
