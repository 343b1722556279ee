"""Convex verify-cost fit of the cost-aware tree budget ("Cost-Aware Diffusion
Draft Trees for Speculative Decoding", Method item 5): the fit must be convex
and non-decreasing in the node count, reproduce convex data exactly, and
interpolate between context lengths."""

import numpy as np
import pytest

pytest.importorskip("scipy")

from tree_speculative_decoding_tsd_gb300 import costmodel


def _convex_ok(c, rel=1e-9):
    tol = rel * float(np.max(np.abs(c)))
    d = np.diff(c)
    return np.all(d >= -tol) and np.all(np.diff(d) >= -tol)


def test_fit_reproduces_convex_piecewise_linear_data():
    n = np.array([1, 2, 4, 8, 16, 32, 64], np.float64)
    y = 20.0 + 0.5 * n + 0.3 * np.maximum(0, n - 8) + 1.0 * np.maximum(0, n - 32)
    fit = costmodel.fit_convex_nondecreasing(n, y)
    np.testing.assert_allclose(costmodel.eval_fit(fit, n), y, rtol=1e-9, atol=1e-9)


def test_fit_of_noisy_data_is_convex_and_monotone():
    rng = np.random.default_rng(0)
    n = np.repeat(np.array([1, 2, 4, 8, 16, 32, 64], np.float64), 3)
    y = 25.0 + 0.02 * n * n + rng.normal(0, 2.0, n.size)
    fit = costmodel.fit_convex_nondecreasing(n, y)
    c = costmodel.eval_fit(fit, np.arange(65))
    assert _convex_ok(c)
    # a projection onto a convex cone never does worse than a member of it
    ref = 25.0 + 0.02 * n * n
    assert np.sum((costmodel.eval_fit(fit, n) - y) ** 2) <= np.sum((ref - y) ** 2) + 1e-6


def test_model_tables_interpolate_between_context_lengths():
    samples = {1024: ([1, 8, 64], [10.0, 12.0, 30.0]), 4096: ([1, 8, 64], [20.0, 24.0, 60.0])}
    m = costmodel.CostModel.from_samples(5.0, samples)
    lo, hi = m.verify_cost(1024, 64), m.verify_cost(4096, 64)
    mid = m.verify_cost(2560, 64)
    np.testing.assert_allclose(mid, 0.5 * lo + 0.5 * hi, rtol=1e-6)
    np.testing.assert_allclose(m.verify_cost(100, 64), lo)
    np.testing.assert_allclose(m.verify_cost(1 << 20, 64), hi)
    # convex up to the fp32 rounding of the returned table
    assert _convex_ok(mid.astype(np.float64), rel=1e-6)
    cd, cv = m.tables([1024, 2560, 4096], 16)
    assert cd.dtype == np.float32 and cv.shape == (3, 17) and cv.dtype == np.float32
