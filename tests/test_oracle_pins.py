"""Pins for the fp64 oracle against what the pages and the mathematics fix.

Each check ties the oracle to something other than itself: the pages'
worked examples (tests/golden, each with its citation), closed forms, the
pairwise O(N^2) definition evaluated by brute force, the matrix form through
numpy's matmul, and invariants the pages state.  No GPU is used.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import golden

IDENT = dict(phi="identity", eps=0.0)


# --- worked examples --------------------------------------------------------

def test_two_token_exact_read():
    g = golden("two_token_exact.json")
    k = np.array(g["k"], float)
    v = np.array(g["v"], float)
    q = np.array([g["q_read"], g["q_read"]], float)
    out1, S1, z1 = oracle.causal(q[:1], k[:1], v[:1], **IDENT)
    np.testing.assert_array_equal(S1, g["S_after_1"])
    np.testing.assert_array_equal(z1, g["z_after_1"])
    out2, S2, z2 = oracle.causal(q, k, v, **IDENT)
    np.testing.assert_array_equal(S2, g["S_after_2"])
    np.testing.assert_array_equal(z2, g["z_after_2"])
    assert out2[1, 0] == pytest.approx(g["output_num"] / g["output_den"], rel=1e-15)
    # the same number from the pairwise weights the page lists
    w = np.array(g["pairwise_weights"], float)
    assert out2[1, 0] == pytest.approx((w @ v[:, 0]) / w.sum(), rel=1e-15)


def test_three_token_states_reads_and_output():
    g = golden("three_token_2x2.json")
    k = np.array(g["k"], float)
    v = np.array(g["v"], float)
    q = np.array([[1, 0], [1, 0], g["q2"]], float)
    for n, key in ((1, "S1"), (2, "S2"), (3, "S3")):
        _, S, _ = oracle.causal(q[:n], k[:n], v[:n], **IDENT)
        np.testing.assert_array_equal(S, g[key])
    out, S3, z3 = oracle.causal(q, k, v, **IDENT)
    np.testing.assert_array_equal(z3, g["z3"])
    np.testing.assert_allclose(out[2], g["y2"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(out[2] * g["y2_denominator"], g["y2_numerator"], atol=1e-14)
    # reads of the updated state through the decode step: update with token p2,
    # then read with each query; numerator = output * (q . z3)
    _, S2, z2 = oracle.causal(q[:2], k[:2], v[:2], **IDENT)
    reads = g["unnormalized_reads_of_S3"]
    for qr, num in zip(reads["q"], reads["numerator"]):
        o, Sn, zn = oracle.decode_step(np.array(qr, float), k[2], v[2], S2, z2, **IDENT)
        np.testing.assert_array_equal(Sn, g["S3"])
        den = float(np.dot(qr, g["z3"]))
        np.testing.assert_allclose(o * den, num, atol=1e-14)


def test_global_worked_example():
    g = golden("global_worked_example.json")
    phk = np.array(g["phi_k"], float)
    v = np.array(g["v"], float)
    q = np.array([g["phi_q"], g["phi_q"]], float)
    out, S, z = oracle.global_(q, phk, v, **IDENT)
    np.testing.assert_array_equal(S, g["S"])
    np.testing.assert_array_equal(z, g["z"])
    np.testing.assert_allclose(out, [g["output"], g["output"]], atol=1e-15)


def test_outer_products():
    for c in golden("outer_products.json")["cases"]:
        k = np.array([c["k"]], float)
        v = np.array([c["v"]], float)
        _, S, z = oracle.causal(k, k, v, **IDENT)
        np.testing.assert_allclose(S, c["kvT"], atol=1e-15)
        np.testing.assert_allclose(z, c["k"], atol=1e-15)


def test_associativity_example():
    g = golden("associativity_fig2.json")
    q, k, v = (np.array(g[n], float) for n in ("q", "k", "v"))
    out, S, z = oracle.global_(q, k, v, **IDENT)
    np.testing.assert_allclose(out, g["normalized"], atol=1e-15)
    den = q @ z
    np.testing.assert_allclose(out * den[:, None], g["unnormalized"], atol=1e-14)


def test_state_size_count():
    g = golden("state_size.json")
    s = g["state_scalars_per_head"]
    assert oracle.state_scalars(s["r"], s["d_v"]) == s["count"]
    c = g["softmax_vs_state"]
    assert c["N"] ** 2 == c["softmax_entries_per_head"]
    assert abs(oracle.state_scalars(c["d"], c["d"]) - c["state_scalars_approx"]) < 1000


# --- feature map ------------------------------------------------------------

def test_phi_closed_form():
    assert oracle.phi(0.0) == 1.0
    assert oracle.phi(2.0) == 3.0
    assert oracle.phi(0.5) == 1.5
    assert oracle.phi(-1.0) == pytest.approx(math.exp(-1.0), rel=1e-16)
    assert oracle.phi(-30.0) == pytest.approx(math.exp(-30.0), rel=1e-16)
    assert oracle.phi(-3.0, "identity") == -3.0


def test_phi_matches_library_elu_plus_one():
    x = np.random.default_rng(0).normal(size=2000) * 4
    ref = (torch.nn.functional.elu(torch.tensor(x, dtype=torch.float64), alpha=1.0) + 1.0).numpy()
    # the library forms expm1(x) + 1 for x <= 0, exact to about one ulp of 1.0
    np.testing.assert_allclose(oracle.phi(x), ref, rtol=1e-15, atol=2.3e-16)
    assert np.all(oracle.phi(np.linspace(-700, 50, 1001)) > 0)


# --- brute force pairwise definition ----------------------------------------

def _phi_lib(x):
    return (torch.nn.functional.elu(torch.tensor(x, dtype=torch.float64)) + 1.0).numpy()


def _pairwise(q, k, v, eps, causal):
    """o_i = sum_j sim(q_i,k_j) v_j / (sum_j sim(q_i,k_j) + eps), pair by pair."""
    fq, fk = _phi_lib(q), _phi_lib(k)
    N = q.shape[0]
    out = np.zeros((N, v.shape[1]))
    for i in range(N):
        num = np.zeros(v.shape[1])
        den = 0.0
        for j in range(N):
            if causal and j > i:
                continue
            w = float(np.dot(fq[i], fk[j]))
            num += w * v[j]
            den += w
        out[i] = num / (den + eps)
    return out


@pytest.mark.parametrize("N,dk,dv", [(1, 1, 1), (5, 2, 3), (17, 3, 1), (33, 8, 8), (64, 8, 3)])
@pytest.mark.parametrize("causal", [True, False])
def test_recurrence_equals_pairwise_bruteforce(N, dk, dv, causal):
    rng = np.random.default_rng(N * 100 + dk * 10 + dv)
    q, k = rng.normal(size=(N, dk)) * 1.5, rng.normal(size=(N, dk)) * 1.5
    v = rng.normal(size=(N, dv))
    fn = oracle.causal if causal else oracle.global_
    out, _, _ = fn(q, k, v, eps=1e-6)
    np.testing.assert_allclose(out, _pairwise(q, k, v, 1e-6, causal), rtol=1e-12, atol=1e-14)


def test_global_matches_matrix_form_with_library_matmul():
    """Matrix form: O = phi(Q)(phi(K)^T V) / (phi(Q)(phi(K)^T 1) + eps), and the
    other association (phi(Q)phi(K)^T)V, both through numpy matmul."""
    rng = np.random.default_rng(7)
    q, k, v = rng.normal(size=(40, 6)), rng.normal(size=(40, 6)), rng.normal(size=(40, 5))
    fq, fk = _phi_lib(q), _phi_lib(k)
    num1 = fq @ (fk.T @ v)
    num2 = (fq @ fk.T) @ v
    den = fq @ (fk.T @ np.ones(40))
    out, S, z = oracle.global_(q, k, v, eps=1e-6)
    np.testing.assert_allclose(out, num1 / (den[:, None] + 1e-6), rtol=1e-12)
    np.testing.assert_allclose(out, num2 / (den[:, None] + 1e-6), rtol=1e-12)
    np.testing.assert_allclose(S, fk.T @ v, rtol=1e-12)
    np.testing.assert_allclose(z, fk.sum(0), rtol=1e-12)


def test_causal_matches_masked_matrix_form():
    rng = np.random.default_rng(8)
    q, k, v = rng.normal(size=(30, 4)), rng.normal(size=(30, 4)), rng.normal(size=(30, 7))
    fq, fk = _phi_lib(q), _phi_lib(k)
    A = np.tril(fq @ fk.T)
    out, _, _ = oracle.causal(q, k, v, eps=1e-6)
    np.testing.assert_allclose(out, (A @ v) / (A.sum(1)[:, None] + 1e-6), rtol=1e-12)


# --- epsilon ----------------------------------------------------------------

def test_eps_only_in_denominator():
    # q.z = 1e-6, so the read is 1e-6 / (1e-6 + eps); with eps = 1e-6 it is 1/2
    q = np.array([[1e-6]])
    k = np.array([[1.0]])
    v = np.array([[1.0]])
    out, _, _ = oracle.causal(q, k, v, eps=1e-6, phi="identity")
    assert out[0, 0] == pytest.approx(0.5, rel=1e-12)
    out, _, _ = oracle.causal(q, k, v, eps=0.0, phi="identity")
    assert out[0, 0] == pytest.approx(1.0, rel=1e-15)


def test_worked_examples_with_small_eps():
    g = golden("three_token_2x2.json")
    k, v = np.array(g["k"], float), np.array(g["v"], float)
    q = np.array([[1, 0], [1, 0], g["q2"]], float)
    out, _, _ = oracle.causal(q, k, v, eps=1e-6, phi="identity")
    np.testing.assert_allclose(out[2], g["y2"], rtol=1e-6)


# --- invariants ---------------------------------------------------------------

def _rand(seed, BH, N, dk, dv, scale=1.0):
    rng = np.random.default_rng(seed)
    return (rng.normal(size=(BH, N, dk)) * scale, rng.normal(size=(BH, N, dk)) * scale,
            rng.normal(size=(BH, N, dv)))


def test_last_causal_row_equals_global_and_states_agree():
    q, k, v = _rand(1, 3, 50, 8, 5)
    oc, Sc, zc = oracle.causal(q, k, v)
    og, Sg, zg = oracle.global_(q, k, v)
    np.testing.assert_allclose(oc[:, -1], og[:, -1], rtol=1e-12)
    np.testing.assert_allclose(Sc, Sg, rtol=1e-12)
    np.testing.assert_allclose(zc, zg, rtol=1e-12)


def test_weighted_average_properties():
    q, k, v = _rand(2, 2, 40, 6, 4)
    out, _, _ = oracle.causal(q, k, v, eps=0.0)
    for h in range(2):
        for t in range(40):
            lo, hi = v[h, : t + 1].min(0), v[h, : t + 1].max(0)
            assert np.all(out[h, t] >= lo - 1e-12) and np.all(out[h, t] <= hi + 1e-12)
    # constant values read back unchanged (weights sum to one)
    vc = np.full_like(v, 3.25)
    out, _, _ = oracle.causal(q, k, vc, eps=0.0)
    np.testing.assert_allclose(out, 3.25, rtol=1e-13)
    # and the denominator is positive: with eps > 0 the read shrinks by den/(den+eps) < 1
    out_e, _, _ = oracle.causal(q, k, vc, eps=1e-3)
    assert np.all(out_e < 3.25) and np.all(out_e > 0)


def test_normalizer_dot_query_is_the_sum_of_scores():
    # "Linear Attention: Accumulating KV in a Fixed-Size State", "Divide by the sum of scores",
    # Figure 6: q's dot with the normalizer z is the sum of its similarity scores with every key
    # read so far
    q, k, v = _rand(5, 2, 30, 6, 3)
    _, S, z = oracle.global_(q, k, v)
    pq, pk = _phi_lib(q), _phi_lib(k)
    for h in range(2):
        np.testing.assert_allclose(pq[h] @ z[h], (pq[h] @ pk[h].T).sum(1), rtol=1e-12)
        # and S is the sum of the outer products phi(k_j) v_j^T
        np.testing.assert_allclose(S[h], sum(np.outer(pk[h, j], v[h, j]) for j in range(30)), rtol=1e-12)


def test_duplicating_every_pair_leaves_global_read_unchanged():
    q, k, v = _rand(3, 1, 20, 5, 3)
    out, _, _ = oracle.global_(q, k, v, eps=0.0)
    out2, _, _ = oracle.global_(np.concatenate([q, q], 1), np.concatenate([k, k], 1),
                                np.concatenate([v, v], 1), eps=0.0)
    np.testing.assert_allclose(out2[:, :20], out, rtol=1e-13)


def test_linear_in_v():
    q, k, v = _rand(4, 2, 30, 4, 6)
    v2 = np.random.default_rng(9).normal(size=v.shape)
    a, _, _ = oracle.causal(q, k, v)
    b, _, _ = oracle.causal(q, k, v2)
    c, _, _ = oracle.causal(q, k, 2.0 * v - 0.5 * v2)
    np.testing.assert_allclose(c, 2.0 * a - 0.5 * b, rtol=1e-11, atol=1e-13)


def test_causal_then_decode_steps_equal_longer_causal():
    q, k, v = _rand(5, 2, 24, 8, 8)
    full, Sf, zf = oracle.causal(q, k, v)
    _, S, z = oracle.causal(q[:, :16], k[:, :16], v[:, :16])
    for t in range(16, 24):
        o, S, z = oracle.decode_step(q[:, t], k[:, t], v[:, t], S, z)
        np.testing.assert_allclose(o, full[:, t], rtol=1e-12)
    np.testing.assert_allclose(S, Sf, rtol=1e-12)
    np.testing.assert_allclose(z, zf, rtol=1e-12)


def test_initial_state_continues_the_prefix():
    q, k, v = _rand(6, 2, 40, 4, 3)
    full, Sf, zf = oracle.causal(q, k, v)
    _, S1, z1 = oracle.causal(q[:, :25], k[:, :25], v[:, :25])
    tail, S2, z2 = oracle.causal(q[:, 25:], k[:, 25:], v[:, 25:], S0=S1, z0=z1)
    np.testing.assert_allclose(tail, full[:, 25:], rtol=1e-12)
    np.testing.assert_allclose(S2, Sf, rtol=1e-12)


def test_state_size_is_independent_of_sequence_length():
    for N in (1, 10, 300):
        q, k, v = _rand(N, 1, N, 6, 2)
        _, S, z = oracle.causal(q, k, v)
        assert S.shape == (1, 6, 2) and z.shape == (1, 6)


def test_threads_split_heads_consistently():
    q, k, v = _rand(10, 7, 33, 4, 5)
    a, Sa, za = oracle.causal(q, k, v, nthreads=1)
    b, Sb, zb = oracle.causal(q, k, v, nthreads=3)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(Sa, Sb)
    for h in range(7):
        o1, _, _ = oracle.causal(q[h], k[h], v[h])
        np.testing.assert_array_equal(o1, a[h])


def test_empty_sequence():
    q = np.zeros((2, 0, 4))
    v = np.zeros((2, 0, 3))
    out, S, z = oracle.causal(q, q, v)
    assert out.shape == (2, 0, 3)
    np.testing.assert_array_equal(S, 0)
    np.testing.assert_array_equal(z, 0)
