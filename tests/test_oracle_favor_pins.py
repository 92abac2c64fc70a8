"""Pins for the oracle's positive random features ("Linear Attention Math",
"Feature maps: elu+1 and positive random features"):
phi(x)_r = exp(w_r . x - |x|^2 / 2) / sqrt(m).

Each check ties the oracle to something other than its own formula: the
closed form at W = 0, the unbiasedness the page states (E[phi(x).phi(y)] =
exp(x.y) for Gaussian projections, checked by Monte Carlo within a bound
from the estimator's variance), positivity, the scaling in m, and the
causal read with these features against the softmax-style average it
approximates when m is large."""
import numpy as np
import pytest

import oracle


def _rng(seed):
    return np.random.default_rng(seed)


def test_zero_projections_give_the_gaussian_factor():
    x = _rng(1).standard_normal((5, 7)) * 0.6
    m = 16
    out = oracle.favor_features(x, np.zeros((m, 7)))
    expect = np.exp(-0.5 * np.sum(x * x, axis=1))[:, None] / np.sqrt(m)
    np.testing.assert_allclose(out, np.broadcast_to(expect, (5, m)), rtol=1e-14)


def test_one_projection_along_a_basis_vector():
    # w = e_1: phi(x) = exp(x_1 - |x|^2 / 2) (m = 1)
    x = _rng(2).standard_normal((4, 3))
    W = np.array([[1.0, 0.0, 0.0]])
    np.testing.assert_allclose(oracle.favor_features(x, W)[:, 0], np.exp(x[:, 0] - 0.5 * np.sum(x * x, axis=1)),
                               rtol=1e-14)


@pytest.mark.parametrize("scale", [0.3, 0.6])
def test_unbiased_for_the_exponential_kernel(scale):
    d, m = 8, 1 << 16
    rng = _rng(3)
    x, y = rng.standard_normal(d) * scale, rng.standard_normal(d) * scale
    W = rng.standard_normal((m, d))
    est = float(oracle.favor_features(x, W) @ oracle.favor_features(y, W))
    exact = np.exp(x @ y)
    # Z = m phi_r(x) phi_r(y) = exp(w.(x+y) - (|x|^2+|y|^2)/2): E[Z] = exp(x.y) and
    # E[Z^2] = exp(2|x+y|^2 - |x|^2 - |y|^2), so the mean of m draws has variance Var[Z] / m
    var = np.exp(2 * np.sum((x + y) ** 2) - x @ x - y @ y) - np.exp(2 * (x @ y))
    assert abs(est - exact) <= 5 * np.sqrt(var / m)


def test_positive_and_scaled_by_one_over_sqrt_m():
    rng = _rng(4)
    x = rng.standard_normal((6, 5))
    W = rng.standard_normal((32, 5))
    a = oracle.favor_features(x, W)
    assert np.all(a > 0)
    # repeating every projection 4 times: each feature is divided by 2 and there are 4 copies
    b = oracle.favor_features(x, np.repeat(W, 4, axis=0))
    np.testing.assert_allclose(b[:, ::4], a / 2, rtol=1e-14)
    np.testing.assert_allclose(np.sum(b * b, axis=1), np.sum(a * a, axis=1), rtol=1e-13)


def test_causal_read_with_many_features_approaches_the_softmax_average():
    # with m large, phi(q_t).phi(k_j) ~ exp(q_t.k_j), so the normalized causal read
    # approaches the softmax-weighted average of v_1..v_t
    rng = _rng(5)
    N, d, dv, m = 6, 4, 3, 1 << 15
    q, k, v = rng.standard_normal((N, d)) * 0.4, rng.standard_normal((N, d)) * 0.4, rng.standard_normal((N, dv))
    W = rng.standard_normal((m, d))
    out, _, _ = oracle.causal(oracle.favor_features(q, W), oracle.favor_features(k, W), v, eps=0.0, phi="identity")
    for t in range(N):
        w = np.exp(q[t] @ k[: t + 1].T)
        np.testing.assert_allclose(out[t], w @ v[: t + 1] / w.sum(), atol=3e-2)
