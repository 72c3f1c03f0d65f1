"""Pins of the oracle's gated prefix (the Gated variant: "a Gated prefix adds the
learned gate" in "Kernelized Linear Attention: Breaking the Capacity Wall with
Symmetric Cones", arXiv 2607.17419, HTML page; its recurrence sits in an
appendix the pages do not contain, so the oracle takes the plainest reading: a
scalar gate per head and token scaling the running state before the token's
own term is added).  Pinned by the reductions and closed forms that reading
fixes, and by the associativity of the gated scan."""
import math

import numpy as np
import pytest

import oracle


def _rand(B, H, T, p, dv, seed, lo=0.3):
    r = np.random.default_rng(seed)
    return (r.standard_normal((B, H, T, p)), r.standard_normal((B, H, T, p)), r.standard_normal((B, H, T, dv)),
            r.uniform(lo, 1.0, (B, H, T)))


def test_unit_gate_is_the_ungated_forward():
    q, k, v, _ = _rand(2, 1, 30, 5, 3, seed=1)
    ones = np.ones((2, 1, 30))
    ref = oracle.forward_plain(q, k, v)
    np.testing.assert_allclose(oracle.forward_plain_gated(q, k, v, ones), ref, atol=1e-13)
    np.testing.assert_allclose(oracle.forward_recurrent_gated(q, k, v, ones)[0], ref, atol=1e-12)
    np.testing.assert_allclose(oracle.forward_chunked_gated(q, k, v, ones, 8, oracle.SCAN_TREE)[0], ref, atol=1e-12)


@pytest.mark.parametrize("r0", [1, 9, 16, 29])
def test_zero_gate_restarts_the_sequence(r0):
    """gate_r0 = 0 forgets everything before r0: from r0 on, the outputs are the
    ungated forward of the suffix starting at r0 (gates after r0 equal to 1)."""
    q, k, v, _ = _rand(1, 2, 30, 4, 3, seed=r0)
    gate = np.ones((1, 2, 30))
    gate[..., r0] = 0.0
    suffix = oracle.forward_plain(q[:, :, r0:], k[:, :, r0:], v[:, :, r0:])
    for o in (oracle.forward_plain_gated(q, k, v, gate), oracle.forward_recurrent_gated(q, k, v, gate)[0],
              oracle.forward_chunked_gated(q, k, v, gate, 8, oracle.SCAN_SEQUENTIAL)[0]):
        np.testing.assert_allclose(o[:, :, r0:], suffix, atol=1e-12)
        np.testing.assert_allclose(o[:, :, :r0], oracle.forward_plain(q[:, :, :r0], k[:, :, :r0], v[:, :, :r0]),
                                   atol=1e-12)


def test_constant_gate_identical_keys_is_the_moving_average():
    """All keys identical and a constant gate g: o_t = sum_s g^(t-s) v_s /
    sum_s g^(t-s), the exponentially weighted moving average, whatever the
    queries (the squared score is common to every term)."""
    T, g = 25, 0.8
    r = np.random.default_rng(3)
    key = r.standard_normal(6)
    k = np.broadcast_to(key, (1, 1, T, 6)).copy()
    q = r.standard_normal((1, 1, T, 6))
    v = r.standard_normal((1, 1, T, 2))
    gate = np.full((1, 1, T), g)
    ema = np.zeros((T, 2))
    for t in range(T):
        wts = g ** (t - np.arange(t + 1))
        ema[t] = wts @ v[0, 0, :t + 1] / wts.sum()
    for o in (oracle.forward_plain_gated(q, k, v, gate), oracle.forward_recurrent_gated(q, k, v, gate)[0],
              oracle.forward_chunked_gated(q, k, v, gate, 4, oracle.SCAN_TREE)[0]):
        np.testing.assert_allclose(o[0, 0], ema, atol=1e-12)


@pytest.mark.parametrize("T,C,p", [(37, 8, 4), (64, 16, 3), (5, 32, 5), (33, 1, 2)])
@pytest.mark.parametrize("mode", [0, 1])
def test_gated_forms_agree(T, C, p, mode):
    q, k, v, gate = _rand(2, 2, T, p, 3, seed=T + C + mode)
    ref = oracle.forward_plain_gated(q, k, v, gate)
    o_r, S_r, z_r = oracle.forward_recurrent_gated(q, k, v, gate)
    o_c, S_c, z_c = oracle.forward_chunked_gated(q, k, v, gate, C, mode)
    np.testing.assert_allclose(o_r, ref, atol=1e-12)
    np.testing.assert_allclose(o_c, ref, atol=1e-12)
    np.testing.assert_allclose(S_c, S_r, atol=1e-12)
    np.testing.assert_allclose(z_c, z_r, atol=1e-12)


@pytest.mark.parametrize("NC", [1, 2, 3, 7, 8, 33])
def test_gated_scan_is_associative(NC):
    """(a1, x1) then (a2, x2) = (a1 a2, a2 x1 + x2) is associative, so the
    log-depth scan equals the step-by-step one, in ceil(log2 NC) rounds; the
    step-by-step prefix is the plain gated recurrence."""
    r = np.random.default_rng(NC)
    a = r.uniform(0.0, 1.0, (2, NC))
    x = r.standard_normal((2, NC, 5))
    seq, rs = oracle.scan_exclusive_gated(a, x, oracle.SCAN_SEQUENTIAL)
    tree, rt = oracle.scan_exclusive_gated(a, x, oracle.SCAN_TREE)
    np.testing.assert_allclose(tree, seq, atol=1e-12)
    assert rs == NC and rt == (math.ceil(math.log2(NC)) if NC > 1 else 0)
    run = np.zeros((2, 5))
    for c in range(NC):
        np.testing.assert_allclose(seq[:, c], run, atol=1e-13)
        run = a[:, c, None] * run + x[:, c]


@pytest.mark.parametrize("T1", [1, 13, 24])
def test_gated_split_call_with_carried_state(T1):
    """forward(T) = forward(T1) then forward(T - T1) from the carried state, for
    both the recurrent and the chunked gated forms."""
    q, k, v, gate = _rand(1, 2, 31, 4, 3, seed=50 + T1)
    o_ref, S_ref, z_ref = oracle.forward_recurrent_gated(q, k, v, gate)
    for fwd in (lambda *a, **kw: oracle.forward_recurrent_gated(*a, **kw),
                lambda *a, **kw: oracle.forward_chunked_gated(*a[:4], 8, 1, **kw)):
        o1, S1, z1 = fwd(q[:, :, :T1], k[:, :, :T1], v[:, :, :T1], gate[:, :, :T1])
        o2, S2, z2 = fwd(q[:, :, T1:], k[:, :, T1:], v[:, :, T1:], gate[:, :, T1:], S0=S1, z0=z1)
        np.testing.assert_allclose(np.concatenate([o1, o2], axis=2), o_ref, atol=1e-12)
        np.testing.assert_allclose(S2, S_ref, atol=1e-12)
        np.testing.assert_allclose(z2, z_ref, atol=1e-12)


def test_gated_outputs_inside_the_hull():
    """Gates in [0, 1] keep every weight nonnegative: outputs stay between the
    smallest and largest value seen."""
    q, k, v, gate = _rand(1, 2, 40, 6, 3, seed=60, lo=0.0)
    o = oracle.forward_plain_gated(q, k, v, gate)
    assert np.all(o >= np.minimum.accumulate(v, axis=2) - 1e-12)
    assert np.all(o <= np.maximum.accumulate(v, axis=2) + 1e-12)


def test_sampled_gated_rows_equal_the_full_definition():
    q, k, v, gate = _rand(2, 2, 40, 6, 3, seed=70, lo=0.0)
    bh = np.array([0, 3, 1, 2, 3])
    t = np.array([0, 39, 17, 5, 20])
    full = oracle.forward_plain_gated(q, k, v, gate).reshape(4, 40, 3)
    np.testing.assert_array_equal(oracle.forward_plain_gated_rows(q, k, v, gate, bh, t), full[bh, t])
