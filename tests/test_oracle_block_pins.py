"""Pins of the oracle's block lifts (KATA-Sigma-g and KATA-M-g, the "two reduced
PSD families" paragraph of "Kernelized Linear Attention: Breaking the Capacity
Wall with Symmetric Cones", arXiv 2607.17419, HTML page) against what the
paragraph and the mathematics fix: its state-size formulas, the block outer
products, its two inner-product identities (computed here from numpy block
products, not through the lift), the reduction to the full lift at g = 1, and
special cases with closed answers."""
import itertools

import numpy as np
import pytest

import oracle

SIGMA, MULTI = oracle.LIFT_SIGMA, oracle.LIFT_MULTI


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _rand_qkv(B, H, T, p, dv, seed=0):
    r = np.random.default_rng(seed)
    return r.standard_normal((B, H, T, p)), r.standard_normal((B, H, T, p)), r.standard_normal((B, H, T, dv))


def _unpack(psi, m):
    """Packed m x m upper triangle (off-diagonals carry sqrt 2) -> symmetric matrix."""
    M = np.zeros((m, m))
    iu = np.triu_indices(m)
    M[iu] = psi
    off = ~np.eye(m, dtype=bool)
    M[off] /= np.sqrt(2.0)
    return np.triu(M) + np.triu(M, 1).T


@pytest.mark.parametrize("p,g", [(64, 1), (64, 2), (64, 4), (32, 2), (16, 4), (12, 3), (8, 8)])
def test_state_sizes_follow_the_paragraph(p, g):
    """Dominant state sizes: Sigma-g (d/g)(d/g+1)/2 d_v and M-g d(d/g+1)/2 d_v."""
    assert oracle.block_dim(p, SIGMA, g) * 2 == (p // g) * (p // g + 1)
    assert oracle.block_dim(p, MULTI, g) * 2 == p * (p // g + 1)
    if g == 1:
        assert oracle.block_dim(p, SIGMA, 1) == oracle.block_dim(p, MULTI, 1) == oracle.packed_dim(p)


def test_state_sizes_at_d64():
    # Sigma-2 at d = 64: m = 32 -> 528; M-2: 1056; the full lift 2080
    assert [oracle.block_dim(64, SIGMA, 2), oracle.block_dim(64, MULTI, 2), oracle.packed_dim(64)] == [528, 1056, 2080]
    assert oracle.block_dim(64, SIGMA, 3) == -1 and oracle.block_dim(10, MULTI, 4) == -1
    assert oracle.block_dim(64, oracle.LIFT_FULL, 2) == -1


@pytest.mark.parametrize("p,g", [(8, 2), (12, 3), (16, 4), (6, 6)])
def test_lifts_are_the_block_outer_products(p, g):
    m = p // g
    u = np.random.default_rng(p + g).standard_normal(p)
    blocks = u.reshape(g, m)
    sig = _unpack(oracle.lift_block(u, SIGMA, g), m)
    np.testing.assert_allclose(sig, sum(np.outer(b, b) for b in blocks), atol=1e-14)
    mul = oracle.lift_block(u, MULTI, g).reshape(g, -1)
    for a in range(g):
        np.testing.assert_allclose(_unpack(mul[a], m), np.outer(blocks[a], blocks[a]), atol=1e-14)


@pytest.mark.parametrize("p,g", [(8, 2), (16, 4), (12, 3), (64, 2)])
def test_inner_product_identities(p, g):
    """<psi_Sigma(q), psi_Sigma(k)> = sum_{a,b} (q_a.k_b)^2 and
    <psi_M(q), psi_M(k)> = sum_a (q_a.k_a)^2 (the paragraph's two identities)."""
    r = np.random.default_rng(3 * p + g)
    for _ in range(5):
        q, k = _unit(r.standard_normal(p)), _unit(r.standard_normal(p))
        Q, K = q.reshape(g, -1), k.reshape(g, -1)
        cross = Q @ K.T
        assert abs(oracle.lift_block(q, SIGMA, g) @ oracle.lift_block(k, SIGMA, g) - np.sum(cross ** 2)) < 1e-14
        assert abs(oracle.lift_block(q, MULTI, g) @ oracle.lift_block(k, MULTI, g) - np.sum(np.diag(cross) ** 2)) < 1e-14


@pytest.mark.parametrize("p", [4, 16, 64])
def test_g1_is_the_full_lift(p):
    u = _unit(np.random.default_rng(p).standard_normal(p))
    np.testing.assert_allclose(oracle.lift_block(u, SIGMA, 1), oracle.lift(u), rtol=0, atol=1e-15)
    np.testing.assert_allclose(oracle.lift_block(u, MULTI, 1), oracle.lift(u), rtol=0, atol=1e-15)
    q, k, v = _rand_qkv(1, 2, 17, p, 3, seed=p)
    full = oracle.forward_plain(q, k, v)
    for fam in (SIGMA, MULTI):
        np.testing.assert_allclose(oracle.forward_plain_block(q, k, v, fam, 1), full, atol=1e-13)
        np.testing.assert_allclose(oracle.forward_recurrent_block(q, k, v, fam, 1)[0], full, atol=1e-12)


@pytest.mark.parametrize("fam,p,g,T", [(SIGMA, 8, 2, 23), (MULTI, 8, 2, 23), (SIGMA, 12, 3, 9),
                                       (MULTI, 12, 4, 30), (SIGMA, 16, 4, 1), (MULTI, 6, 6, 12)])
def test_definition_and_lifted_recurrence_agree(fam, p, g, T):
    """Two routes to the same result: block dot products squared (the kernel)
    and the packed-lift state recurrence."""
    q, k, v = _rand_qkv(2, 1, T, p, 5, seed=T + g)
    o_plain = oracle.forward_plain_block(q, k, v, fam, g)
    o_rec, S, z = oracle.forward_recurrent_block(q, k, v, fam, g)
    np.testing.assert_allclose(o_rec, o_plain, atol=1e-12)
    assert S.shape == (2, 1, oracle.block_dim(p, fam, g), 5)


def test_sigma_with_scalar_blocks_is_the_running_mean():
    """Sigma-p (m = 1): psi(u) = sum_a u_a^2 = 1 for every unit u, so every
    weight is 1 and o_t is the mean of v_1..v_t whatever q and k are."""
    q, k, v = _rand_qkv(1, 1, 20, 6, 4, seed=7)
    mean = np.cumsum(v, axis=2) / np.arange(1, 21)[None, None, :, None]
    np.testing.assert_allclose(oracle.forward_plain_block(q, k, v, SIGMA, 6), mean, atol=1e-13)
    np.testing.assert_allclose(oracle.forward_recurrent_block(q, k, v, SIGMA, 6)[0], mean, atol=1e-13)


def test_disjoint_blocks_separate_the_families():
    """A query living in block 1 and keys living in block 2: M-g sees no match
    (zero denominator, zero rows), Sigma-g matches them across blocks as the
    full kernel would if the blocks were overlaid."""
    p, g, T = 8, 2, 6
    r = np.random.default_rng(11)
    q = np.zeros((1, 1, T, p))
    k = np.zeros((1, 1, T, p))
    q[..., :4] = r.standard_normal((T, 4))
    k[..., 4:] = r.standard_normal((T, 4))
    v = r.standard_normal((1, 1, T, 3))
    assert np.all(oracle.forward_plain_block(q, k, v, MULTI, g) == 0.0)
    assert np.all(oracle.forward_recurrent_block(q, k, v, MULTI, g)[0] == 0.0)
    overlaid = oracle.forward_plain(q[..., :4], k[..., 4:], v)
    np.testing.assert_allclose(oracle.forward_plain_block(q, k, v, SIGMA, g), overlaid, atol=1e-13)


def test_block_permutations():
    """Sigma-g sums over every block pair: permuting the blocks of the keys
    alone changes nothing.  M-g pairs block a with block a: the same
    permutation of q's and k's blocks changes nothing, one of k's alone does."""
    p, g, T = 12, 3, 15
    q, k, v = _rand_qkv(1, 1, T, p, 4, seed=13)
    perm = [2, 0, 1]
    kp = k.reshape(1, 1, T, g, p // g)[..., perm, :].reshape(1, 1, T, p)
    qp = q.reshape(1, 1, T, g, p // g)[..., perm, :].reshape(1, 1, T, p)
    np.testing.assert_allclose(oracle.forward_plain_block(q, kp, v, SIGMA, g),
                               oracle.forward_plain_block(q, k, v, SIGMA, g), atol=1e-13)
    np.testing.assert_allclose(oracle.forward_plain_block(qp, kp, v, MULTI, g),
                               oracle.forward_plain_block(q, k, v, MULTI, g), atol=1e-13)
    assert np.abs(oracle.forward_plain_block(q, kp, v, MULTI, g) - oracle.forward_plain_block(q, k, v, MULTI, g)).max() > 1e-3


@pytest.mark.parametrize("fam,g", list(itertools.product([SIGMA, MULTI], [2, 4])))
def test_block_outputs_inside_the_hull_and_single_token(fam, g):
    """Nonnegative weights: every output coordinate lies between the smallest
    and largest value seen so far; T = 1 returns v_1."""
    q, k, v = _rand_qkv(1, 2, 25, 8, 3, seed=17 + g)
    o = oracle.forward_plain_block(q, k, v, fam, g)
    lo = np.minimum.accumulate(v, axis=2)
    hi = np.maximum.accumulate(v, axis=2)
    assert np.all(o >= lo - 1e-12) and np.all(o <= hi + 1e-12)
    np.testing.assert_allclose(oracle.forward_plain_block(q[:, :, :1], k[:, :, :1], v[:, :, :1], fam, g),
                               v[:, :, :1], atol=1e-14)


@pytest.mark.parametrize("fam,T1", [(SIGMA, 1), (SIGMA, 12), (MULTI, 7), (MULTI, 20)])
def test_block_split_call_with_carried_state(fam, T1):
    q, k, v = _rand_qkv(1, 2, 21, 8, 3, seed=19)
    o_ref, S_ref, z_ref = oracle.forward_recurrent_block(q, k, v, fam, 2)
    o1, S1, z1 = oracle.forward_recurrent_block(q[:, :, :T1], k[:, :, :T1], v[:, :, :T1], fam, 2)
    o2, S2, z2 = oracle.forward_recurrent_block(q[:, :, T1:], k[:, :, T1:], v[:, :, T1:], fam, 2, S0=S1, z0=z1)
    np.testing.assert_allclose(np.concatenate([o1, o2], axis=2), o_ref, atol=1e-12)
    np.testing.assert_allclose(S2, S_ref, atol=1e-12)
    np.testing.assert_allclose(z2, z_ref, atol=1e-12)


def test_sampled_block_rows_equal_the_full_definition():
    q, k, v = _rand_qkv(2, 2, 40, 8, 3, seed=23)
    bh = np.array([0, 3, 1, 2, 3])
    t = np.array([0, 39, 17, 5, 20])
    for fam in (SIGMA, MULTI):
        full = oracle.forward_plain_block(q, k, v, fam, 2).reshape(4, 40, 3)
        np.testing.assert_array_equal(oracle.forward_plain_block_rows(q, k, v, fam, 2, bh, t), full[bh, t])
