"""The polynomial in the kernels' softplus comes from fit_log1p.py: the header
holds exactly the fitted fp32 coefficients, and they meet the stated error."""
import importlib.util
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "selective_state_space_118_b300", "csrc")


def load_fit():
    spec = importlib.util.spec_from_file_location("fit_log1p", os.path.join(CSRC, "fit_log1p.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def header_coefficients():
    src = open(os.path.join(CSRC, "ssm_math.cuh")).read()
    named = {int(k): float(v) for k, v in re.findall(r"constexpr float kLp(\d) = (-?\d+\.\d+(?:e-?\d+)?)f;", src)}
    assert sorted(named) == [1, 2, 3, 4, 5], named
    # the constant term is the 1 of Estrin's first term (1 + a1 e)
    assert "__fmaf_rn(e, kLp1, 1.0f)" in src
    return np.array([1.0] + [named[k] for k in range(1, 6)], dtype=np.float32)


def test_header_holds_the_fitted_coefficients():
    fit = load_fit()
    np.testing.assert_array_equal(header_coefficients(), fit.fit())


def test_polynomial_error_bound():
    fit = load_fit()
    assert fit.max_rel_error(header_coefficients()) < 1.5e-7
