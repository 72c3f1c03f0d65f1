"""Pins of the oracle's backward (the gradient of the plain definition, the
training use of the forward named in the abstract of "Kernelized Linear
Attention: Breaking the Capacity Wall with Symmetric Cones", arXiv 2607.17419;
the pages give no backward algorithm, so the oracle takes the chain rule
through the definition).  Pinned by central finite differences of the pinned
forward and by what the definition's symmetries force on any gradient."""
import numpy as np
import pytest

import oracle


def _rand(B, H, T, p, dv, seed):
    r = np.random.default_rng(seed)
    return (r.standard_normal((B, H, T, p)), r.standard_normal((B, H, T, p)), r.standard_normal((B, H, T, dv)),
            r.standard_normal((B, H, T, dv)))


def _loss(q, k, v, G):
    return float((G * oracle.forward_plain(q, k, v)).sum())


def test_every_coordinate_against_central_differences():
    q, k, v, G = _rand(1, 2, 7, 4, 3, seed=1)
    dq, dk, dv = oracle.backward_plain(q, k, v, G)
    h = 1e-6
    for x, grad, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which], args_m[which] = xp, xm
            num[idx] = (_loss(*args_p, G) - _loss(*args_m, G)) / (2 * h)
        np.testing.assert_allclose(grad, num, atol=2e-8, rtol=1e-6)


@pytest.mark.parametrize("T,p,dv", [(40, 16, 8), (33, 5, 2)])
def test_directional_derivatives(T, p, dv):
    q, k, v, G = _rand(2, 1, T, p, dv, seed=T)
    dq, dk, dv_ = oracle.backward_plain(q, k, v, G)
    r = np.random.default_rng(T + 1)
    h = 1e-6
    for _ in range(3):
        eq, ek, ev = r.standard_normal(q.shape), r.standard_normal(k.shape), r.standard_normal(v.shape)
        num = (_loss(q + h * eq, k + h * ek, v + h * ev, G) - _loss(q - h * eq, k - h * ek, v - h * ev, G)) / (2 * h)
        ana = float((dq * eq).sum() + (dk * ek).sum() + (dv_ * ev).sum())
        assert abs(num - ana) <= 1e-6 * max(1.0, abs(ana))


def test_gradients_are_orthogonal_to_q_and_k():
    """o does not change when a q_t or k_s is rescaled, so each dq_t is
    orthogonal to q_t and each dk_s to k_s."""
    q, k, v, G = _rand(1, 2, 30, 8, 4, seed=3)
    dq, dk, _ = oracle.backward_plain(q, k, v, G)
    assert np.abs((q * dq).sum(-1)).max() < 1e-12
    assert np.abs((k * dk).sum(-1)).max() < 1e-12


def test_value_shift_and_value_gradient_sum():
    """o_t(v + c) = o_t(v) + c: dq and dk do not depend on a common shift of the
    values; dv does not depend on v at all; and the weights of a row sum to one,
    so sum_s dv_s = sum_t dO_t."""
    q, k, v, G = _rand(1, 1, 25, 6, 3, seed=5)
    dq, dk, dv = oracle.backward_plain(q, k, v, G)
    dq2, dk2, dv2 = oracle.backward_plain(q, k, v + np.array([1.5, -2.0, 0.25]), G)
    np.testing.assert_allclose(dq2, dq, atol=1e-12)
    np.testing.assert_allclose(dk2, dk, atol=1e-12)
    np.testing.assert_allclose(dv2, dv, atol=1e-13)
    np.testing.assert_allclose(dv.sum(axis=2), G.sum(axis=2), atol=1e-12)


def test_rotation_equivariance():
    """Rotating every q and k by R leaves o unchanged, so dq and dk rotate by R
    and dv stays."""
    q, k, v, G = _rand(1, 1, 20, 5, 3, seed=7)
    R, _ = np.linalg.qr(np.random.default_rng(8).standard_normal((5, 5)))
    dq, dk, dv = oracle.backward_plain(q, k, v, G)
    dqr, dkr, dvr = oracle.backward_plain(q @ R, k @ R, v, G)
    np.testing.assert_allclose(dqr, dq @ R, atol=1e-12)
    np.testing.assert_allclose(dkr, dk @ R, atol=1e-12)
    np.testing.assert_allclose(dvr, dv, atol=1e-12)


def test_single_token_and_zero_vectors():
    """T = 1 returns v_1: dv = dO, no gradient to q or k.  A zero key receives
    no gradient; a zero query's row has a zero denominator and passes none."""
    q, k, v, G = _rand(1, 1, 1, 4, 3, seed=9)
    dq, dk, dv = oracle.backward_plain(q, k, v, G)
    assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14
    np.testing.assert_allclose(dv, G, atol=1e-15)
    q, k, v, G = _rand(1, 1, 6, 4, 3, seed=10)
    k[0, 0, 2] = 0.0
    q[0, 0, 4] = 0.0
    dq, dk, dv = oracle.backward_plain(q, k, v, G)
    assert np.all(dk[0, 0, 2] == 0) and np.all(dq[0, 0, 4] == 0)
    G2 = G.copy()
    G2[0, 0, 4] += 10.0  # the zero query's row: no effect on any gradient
    dq2, dk2, dv2 = oracle.backward_plain(q, k, v, G2)
    np.testing.assert_allclose(dq2, dq, atol=1e-14)
    np.testing.assert_allclose(dk2, dk, atol=1e-14)
    np.testing.assert_allclose(dv2, dv, atol=1e-14)
