"""Pins for the oracle's causal backward pass.

The pages describe training through the chunked causal form but write no
backward pass, so the oracle's gradient is the plain derivative of the
causal definition (o_t = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps), inclusive
state).  Each check ties it to something other than its own formulas:
central finite differences of the forward oracle for every input (q, k, v,
the initial state and the final-state gradients), closed forms where the
output does not depend on q and k, linearity in the upstream gradient, and
thread splits."""
import numpy as np
import pytest

import oracle


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _away_from_zero(x, gap=0.05):
    # phi is not twice differentiable at 0; keep finite differences off the kink
    return np.where(np.abs(x) < gap, np.sign(x + 1e-12) * gap, x)


def _loss(q, k, v, dO, eps, phi, S0, z0, dS, dz):
    out, S, z = oracle.causal(q, k, v, eps=eps, phi=phi, S0=S0, z0=z0)
    L = np.sum(dO * out)
    if dS is not None:
        L += np.sum(dS * S) + np.sum(dz * z)
    return L


def _fd(f, x, h=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        xp, xm = x.copy(), x.copy()
        xp[i] += h
        xm[i] -= h
        g[i] = (f(xp) - f(xm)) / (2 * h)
    return g


@pytest.mark.parametrize("phi", ["elu1", "identity"])
@pytest.mark.parametrize("with_state", [False, True])
@pytest.mark.parametrize("eps", [0.0, 1e-6, 0.3])
def test_matches_finite_differences(phi, with_state, eps):
    H, N, dk, dv = 2, 5, 3, 2
    q = _away_from_zero(_rand((H, N, dk), 1))
    k = _away_from_zero(_rand((H, N, dk), 2))
    v = _rand((H, N, dv), 3)
    if phi == "identity":  # keep the denominators positive: positive features
        q, k = np.abs(q) + 0.1, np.abs(k) + 0.1
    dO = _rand((H, N, dv), 4)
    S0 = z0 = dS = dz = None
    if with_state:
        S0, z0 = _rand((H, dk, dv), 5), np.abs(_rand((H, dk), 6)) + 1.0
        dS, dz = _rand((H, dk, dv), 7), _rand((H, dk), 8)
    args = dict(eps=eps, phi=phi, S0=S0, z0=z0, dS=dS, dz=dz)
    dq, dkk, dvv, dS0, dz0 = oracle.causal_backward(q, k, v, dO, **args)
    L = lambda **kw: _loss(kw.get("q", q), kw.get("k", k), kw.get("v", v), dO, eps, phi, kw.get("S0", S0),
                           kw.get("z0", z0), dS, dz)
    tol = dict(rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(dq, _fd(lambda x: L(q=x), q), **tol)
    np.testing.assert_allclose(dkk, _fd(lambda x: L(k=x), k), **tol)
    np.testing.assert_allclose(dvv, _fd(lambda x: L(v=x), v), **tol)
    if with_state:
        np.testing.assert_allclose(dS0, _fd(lambda x: L(S0=x), S0), **tol)
        np.testing.assert_allclose(dz0, _fd(lambda x: L(z0=x), z0), **tol)


def test_single_token_without_eps_depends_only_on_v():
    # N = 1, eps = 0: o_0 = phi(q).phi(k) v_0 / phi(q).phi(k) = v_0 exactly
    q, k, v, dO = _rand((4, 1, 6), 10), _rand((4, 1, 6), 11), _rand((4, 1, 3), 12), _rand((4, 1, 3), 13)
    dq, dkk, dvv, dS0, dz0 = oracle.causal_backward(q, k, v, dO, eps=0.0)
    np.testing.assert_allclose(dq, 0.0, atol=1e-14)
    np.testing.assert_allclose(dkk, 0.0, atol=1e-14)
    np.testing.assert_allclose(dvv, dO, rtol=1e-13)


def test_equal_values_without_eps_give_no_query_or_key_gradient():
    # every v_j equal: each output is that common value, whatever q and k are
    q, k = _rand((2, 9, 4), 14), _rand((2, 9, 4), 15)
    v = np.broadcast_to(_rand((2, 1, 3), 16), (2, 9, 3)).copy()
    dO = _rand((2, 9, 3), 17)
    dq, dkk, dvv, _, _ = oracle.causal_backward(q, k, v, dO, eps=0.0)
    np.testing.assert_allclose(dq, 0.0, atol=1e-12)
    np.testing.assert_allclose(dkk, 0.0, atol=1e-12)
    # the values' gradients: each output is a convex combination of the v_j
    np.testing.assert_allclose(dvv.sum(axis=1), dO.sum(axis=1), rtol=1e-11)


def test_linear_in_the_upstream_gradient():
    q, k, v = _rand((3, 7, 4), 18), _rand((3, 7, 4), 19), _rand((3, 7, 5), 20)
    a, b = _rand((3, 7, 5), 21), _rand((3, 7, 5), 22)
    ga = oracle.causal_backward(q, k, v, a)
    gb = oracle.causal_backward(q, k, v, b)
    gab = oracle.causal_backward(q, k, v, 2 * a - 0.5 * b)
    for x, y, z in zip(ga, gb, gab):
        np.testing.assert_allclose(z, 2 * x - 0.5 * y, rtol=1e-10, atol=1e-12)
    zero = oracle.causal_backward(q, k, v, np.zeros_like(a))
    for x in zero:
        assert np.all(x == 0.0)


def test_initial_state_gradient_is_the_suffix_sum_at_the_start():
    # with only a final-state gradient, every token's key and value see it, and dS0 = dS_N, dz0 = dz_N
    q, k, v = _rand((2, 6, 3), 23), _rand((2, 6, 3), 24), _rand((2, 6, 2), 25)
    dS, dz = _rand((2, 3, 2), 26), _rand((2, 3), 27)
    dq, dkk, dvv, dS0, dz0 = oracle.causal_backward(q, k, v, np.zeros_like(v), dS=dS, dz=dz)
    np.testing.assert_allclose(dS0, dS, rtol=1e-15)
    np.testing.assert_allclose(dz0, dz, rtol=1e-15)
    assert np.all(dq == 0.0)
    phik = oracle.phi(k)
    np.testing.assert_allclose(dvv, np.einsum("hid,hti->htd", dS, phik), rtol=1e-12)


def test_threads_and_empty_sequence():
    q, k, v, dO = _rand((5, 8, 3), 28), _rand((5, 8, 3), 29), _rand((5, 8, 2), 30), _rand((5, 8, 2), 31)
    g1 = oracle.causal_backward(q, k, v, dO, nthreads=1)
    g3 = oracle.causal_backward(q, k, v, dO, nthreads=3)
    for x, y in zip(g1, g3):
        assert np.array_equal(x, y)
    e = np.zeros((2, 0, 3))
    dq, dkk, dvv, dS0, dz0 = oracle.causal_backward(e, e, e, e)
    assert dq.shape == (2, 0, 3) and np.all(dS0 == 0.0) and np.all(dz0 == 0.0)
