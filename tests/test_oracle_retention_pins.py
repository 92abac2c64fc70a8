"""Pins for the oracle's retention form ("Linear Attention Math", "The kernel
cousins: SSMs and RetNet": S_t = gamma S_{t-1} + k_t v_t^T, the read taken
after the update and without a denominator).

Each check ties the token-serial recurrence in oracle/la_oracle.c to
something other than itself: the pairwise definition written out by brute
force, a closed-form geometric series, the special cases gamma = 1 (the
causal state of the existing oracle) and gamma = 0 (a single-token read),
state continuation and linearity."""
import numpy as np
import pytest

import oracle


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _pairwise(q, k, v, gamma):
    """out_i = sum_{j <= i} gamma^(i - j) (q_i . k_j) v_j, by explicit loops."""
    N = q.shape[-2]
    out = np.zeros(q.shape[:-1] + (v.shape[-1],))
    for i in range(N):
        for j in range(i + 1):
            w = gamma ** (i - j) * np.einsum("...d,...d->...", q[..., i, :], k[..., j, :])
            out[..., i, :] += w[..., None] * v[..., j, :]
    return out


@pytest.mark.parametrize("gamma", [0.0, 0.5, 0.9, 0.97, 1.0])
@pytest.mark.parametrize("dk,dv", [(1, 1), (3, 2), (8, 5)])
def test_recurrence_equals_the_pairwise_definition(gamma, dk, dv):
    q, k, v = _rand((2, 9, dk), 1), _rand((2, 9, dk), 2), _rand((2, 9, dv), 3)
    out, S = oracle.retention(q, k, v, gamma)
    np.testing.assert_allclose(out, _pairwise(q, k, v, gamma), rtol=1e-12, atol=1e-12)
    # the final state is the decayed sum of outer products
    N = q.shape[-2]
    w = np.array([gamma ** (N - 1 - j) for j in range(N)])
    np.testing.assert_allclose(S, np.einsum("j,hjd,hje->hde", w, k, v), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("gamma", [0.3, 0.9, 0.999])
def test_constant_inputs_give_the_geometric_series(gamma):
    N = 40
    e = np.zeros((1, N, 2))
    e[..., 0] = 1.0
    v = np.ones((1, N, 1))
    out, _ = oracle.retention(e, e, v, gamma)
    t = np.arange(N)
    np.testing.assert_allclose(out[0, :, 0], (1 - gamma ** (t + 1)) / (1 - gamma), rtol=1e-12)


def test_gamma_one_is_the_undecayed_causal_state():
    q, k, v = np.abs(_rand((3, 12, 4), 4)), np.abs(_rand((3, 12, 4), 5)), _rand((3, 12, 3), 6)
    out, S = oracle.retention(q, k, v, 1.0)
    o_c, S_c, z_c = oracle.causal(q, k, v, eps=0.0, phi="identity")
    np.testing.assert_allclose(S, S_c, rtol=1e-12)
    # the normalized causal read times its denominator is the undecayed retention read
    den = np.einsum("hd,hd->h", q[:, -1], z_c)
    np.testing.assert_allclose(out[:, -1], o_c[:, -1] * den[:, None], rtol=1e-11)


def test_gamma_zero_reads_only_the_current_token():
    q, k, v = _rand((2, 7, 3), 7), _rand((2, 7, 3), 8), _rand((2, 7, 4), 9)
    out, _ = oracle.retention(q, k, v, 0.0)
    np.testing.assert_allclose(out, np.einsum("htd,htd->ht", q, k)[..., None] * v, rtol=1e-12, atol=1e-14)


def test_per_head_gamma():
    q, k, v = _rand((3, 6, 2), 10), _rand((3, 6, 2), 11), _rand((3, 6, 2), 12)
    g = np.array([0.2, 0.7, 1.0])
    out, _ = oracle.retention(q, k, v, g)
    for h in range(3):
        np.testing.assert_allclose(out[h], _pairwise(q[h], k[h], v[h], g[h]), rtol=1e-12, atol=1e-12)


def test_state_continues_the_prefix():
    q, k, v = _rand((2, 20, 4), 13), _rand((2, 20, 4), 14), _rand((2, 20, 3), 15)
    full, S_full = oracle.retention(q, k, v, 0.8)
    a, S_a = oracle.retention(q[:, :8], k[:, :8], v[:, :8], 0.8)
    b, S_b = oracle.retention(q[:, 8:], k[:, 8:], v[:, 8:], 0.8, S0=S_a)
    np.testing.assert_allclose(np.concatenate([a, b], 1), full, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S_b, S_full, rtol=1e-12, atol=1e-12)


def test_linear_in_v_and_in_q():
    q, k, v = _rand((1, 10, 3), 16), _rand((1, 10, 3), 17), _rand((1, 10, 2), 18)
    v2 = _rand((1, 10, 2), 19)
    o1, _ = oracle.retention(q, k, v, 0.95)
    o2, _ = oracle.retention(q, k, v2, 0.95)
    o12, _ = oracle.retention(q, k, 2 * v - 3 * v2, 0.95)
    np.testing.assert_allclose(o12, 2 * o1 - 3 * o2, rtol=1e-11, atol=1e-12)
    o3, _ = oracle.retention(-0.5 * q, k, v, 0.95)
    np.testing.assert_allclose(o3, -0.5 * o1, rtol=1e-12, atol=1e-14)


def test_threads_and_empty_input():
    q, k, v = _rand((5, 11, 3), 20), _rand((5, 11, 3), 21), _rand((5, 11, 2), 22)
    o1, S1 = oracle.retention(q, k, v, 0.9, nthreads=1)
    o4, S4 = oracle.retention(q, k, v, 0.9, nthreads=4)
    assert np.array_equal(o1, o4) and np.array_equal(S1, S4)
    out, S = oracle.retention(np.zeros((2, 0, 3)), np.zeros((2, 0, 3)), np.zeros((2, 0, 2)), 0.9)
    assert out.shape == (2, 0, 2) and np.array_equal(S, np.zeros((2, 3, 2)))
