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
    body = src[src.index("float softplus_small(float e)"):src.index("constexpr float kSoftplusSmallE")]
    vals = [float(v) for v in re.findall(r"(-?\d+\.\d+(?:e-?\d+)?)f", body)]
    # Estrin's terms in source order: (c1, c0), (c3, c2), (c5, c4)
    c1, c0, c3, c2, c5, c4 = vals[0], vals[1], vals[2], vals[3], vals[4], vals[5]
    return np.array([c0, c1, c2, c3, c4, c5], dtype=np.float32)


def test_header_holds_the_fitted_coefficients():
    fit = load_fit()
    np.testing.assert_array_equal(header_coefficients(), fit.fit())


def test_polynomial_error_bound():
    fit = load_fit()
    assert fit.max_rel_error(header_coefficients()) < 1.5e-7
