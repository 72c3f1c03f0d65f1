"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these compares the oracle with a re-typed copy of itself: each check is
a closed form, an identity, an invariant or a special case with a textbook
answer (see the docstrings for the passage each follows).  Citations are to
"Kernelized Linear Attention: Breaking the Capacity Wall with Symmetric Cones"
(arXiv 2607.17419), HTML page.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def _rng(seed=0):
    return np.random.default_rng(seed)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _rand_qkv(B, H, T, p, dv, seed=0, scale=1.0):
    r = _rng(seed)
    return (scale * r.standard_normal((B, H, T, p)), scale * r.standard_normal((B, H, T, p)),
            r.standard_normal((B, H, T, dv)))


def _unpack(psi, p):
    """Packed upper triangle (off-diagonals carry sqrt 2) -> symmetric p x p matrix."""
    M = np.zeros((p, p))
    a = 0
    for i in range(p):
        for j in range(i, p):
            val = psi[a] if i == j else psi[a] / math.sqrt(2.0)
            M[i, j] = M[j, i] = val
            a += 1
    return M


# ---------------------------------------------------------------- lift (Eq. 8, rank-one lift)

def test_packed_dim_matches_eq8_and_state_size_paragraph():
    """n = p(p+1)/2 (Eq. 8); at d = 64 the direct and packed widths are 4096 and 2080."""
    for p in (1, 2, 3, 16, 32, 64):
        assert oracle.packed_dim(p) == p * (p + 1) // 2
    assert oracle.packed_dim(64) == 2080 and 64 * 64 == 4096
    assert oracle.packed_dim(32) == 528 and oracle.packed_dim(16) == 136


def test_lift_golden_values():
    """Hand-derived packed lifts, including the coordinate order."""
    cases = {c["name"]: c for c in json.load(open(GOLDEN))["cases"]}
    for name in ("lift_3_4_5", "lift_1_2_2_order"):
        c = cases[name]
        np.testing.assert_allclose(oracle.lift(np.array(c["u"])), c["psi"], rtol=0, atol=1e-15)


@pytest.mark.parametrize("p", [2, 3, 16, 64])
def test_lift_is_packed_outer_product(p):
    """psi(u) unpacks to u u^T (rank-one lift paragraph after Eq. 8)."""
    u = _unit(_rng(p).standard_normal(p))
    np.testing.assert_allclose(_unpack(oracle.lift(u), p), np.outer(u, u), rtol=0, atol=1e-15)


@pytest.mark.parametrize("p", [2, 3, 16, 64])
def test_lift_identities(p):
    """||uu^T||_F = 1 and <uu^T, vv^T>_F = (u.v)^2 for unit u, v."""
    r = _rng(100 + p)
    for _ in range(20):
        u, v = _unit(r.standard_normal(p)), _unit(r.standard_normal(p))
        pu, pv = oracle.lift(u), oracle.lift(v)
        assert abs(np.linalg.norm(pu) - 1.0) < 1e-14
        assert abs(pu @ pv - (u @ v) ** 2) < 1e-14
        assert pu @ pv >= 0.0


def test_normalize_unit_sphere_and_zero():
    x = _rng(3).standard_normal((5, 7)) * 4.0
    u = oracle.normalize(x)
    np.testing.assert_allclose(np.linalg.norm(u, axis=-1), 1.0, atol=1e-15)
    np.testing.assert_allclose(u, x / np.linalg.norm(x, axis=-1, keepdims=True), atol=1e-15)
    assert np.all(oracle.normalize(np.zeros(4)) == 0.0)


# ---------------------------------------------------------------- forms agree

FORM_CASES = [
    # B, H, T, p, dv, C
    (1, 1, 1, 2, 1, 1),
    (1, 1, 7, 2, 3, 2),
    (1, 2, 16, 3, 2, 4),
    (2, 1, 37, 4, 5, 8),
    (1, 1, 64, 16, 4, 16),
    (1, 1, 64, 16, 4, 64),
    (1, 1, 50, 16, 3, 64),  # one partial chunk
]


@pytest.mark.parametrize("B,H,T,p,dv,C", FORM_CASES)
def test_quadratic_recurrent_chunked_agree(B, H, T, p, dv, C):
    """The plain definition, the token-recurrent state form and the chunked form
    (both prefix modes) give one result; chunked needs exclusive prefix + local
    inclusive part (chunked-scan paragraph), recurrent needs the lift identity."""
    q, k, v = _rand_qkv(B, H, T, p, dv, seed=T * 7 + p, scale=2.5)
    o_plain = oracle.forward_plain(q, k, v)
    o_rec, S_rec, z_rec = oracle.forward_recurrent(q, k, v)
    np.testing.assert_allclose(o_rec, o_plain, rtol=0, atol=1e-12)
    for mode in (oracle.SCAN_SEQUENTIAL, oracle.SCAN_TREE):
        o_ch, S_ch, z_ch = oracle.forward_chunked(q, k, v, C, mode)
        np.testing.assert_allclose(o_ch, o_plain, rtol=0, atol=1e-12)
        np.testing.assert_allclose(S_ch, S_rec, rtol=0, atol=1e-11)
        np.testing.assert_allclose(z_ch, z_rec, rtol=0, atol=1e-11)


def test_chunk_size_independence():
    """The chunked form is exact, so C in {32, 64, 128} and a ragged C agree."""
    q, k, v = _rand_qkv(1, 2, 256, 8, 4, seed=11)
    ref = oracle.forward_plain(q, k, v)
    for C in (32, 64, 128, 48):
        o, _, _ = oracle.forward_chunked(q, k, v, C, oracle.SCAN_TREE)
        np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def test_plain_rows_match_full():
    q, k, v = _rand_qkv(2, 2, 40, 4, 3, seed=5)
    full = oracle.forward_plain(q, k, v)
    bh = np.array([0, 1, 2, 3, 3, 2])
    t = np.array([0, 39, 17, 1, 38, 0])
    rows = oracle.forward_plain_rows(q, k, v, bh, t)
    np.testing.assert_allclose(rows, full.reshape(4, 40, 3)[bh, t], rtol=0, atol=0)


# ---------------------------------------------------------------- special cases

def test_worked_examples():
    cases = {c["name"]: c for c in json.load(open(GOLDEN))["cases"]}
    c = cases["two_tokens_60deg"]
    o = oracle.forward_plain(np.array(c["q"])[None, None], np.array(c["k"])[None, None],
                             np.array(c["v"])[None, None])[0, 0]
    np.testing.assert_allclose(o, c["o"], rtol=0, atol=1e-15)
    c = cases["triangle_code_V_identity"]
    o = oracle.forward_plain(np.array(c["q"])[None, None], np.array(c["k"])[None, None],
                             np.array(c["v"])[None, None])[0, 0]
    np.testing.assert_allclose(o[-1], c["o_last"], rtol=0, atol=1e-15)
    a = o[-1]
    assert abs(a[0] ** 2 / (a[1] ** 2 + a[2] ** 2) - c["psnr"]) < 1e-12


def test_single_token_returns_its_value():
    """T = 1: the only weight is on v_1, so o_1 = v_1."""
    q, k, v = _rand_qkv(2, 3, 1, 5, 4, seed=9)
    np.testing.assert_allclose(oracle.forward_plain(q, k, v), v, rtol=0, atol=1e-15)
    o, _, _ = oracle.forward_chunked(q, k, v, 32)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-15)


def test_identical_keys_give_prefix_mean():
    """All keys equal: every weight is (q.k)^2, so o_t is the running mean of v."""
    r = _rng(21)
    T, p, dv = 30, 6, 3
    kk = r.standard_normal(p)
    k = np.broadcast_to(kk, (1, 1, T, p)).copy()
    q = kk + 0.3 * r.standard_normal((1, 1, T, p))
    v = r.standard_normal((1, 1, T, dv))
    mean = np.cumsum(v[0, 0], axis=0) / np.arange(1, T + 1)[:, None]
    for o in (oracle.forward_plain(q, k, v), oracle.forward_chunked(q, k, v, 8, 1)[0]):
        np.testing.assert_allclose(o[0, 0], mean, rtol=0, atol=1e-13)


def test_orthonormal_keys_exact_recall():
    """p >= T orthonormal keys, q_t = k_j with j <= t: weights are delta_{js}, o_t = v_j."""
    r = _rng(22)
    p = T = 16
    Qm, _ = np.linalg.qr(r.standard_normal((p, p)))
    k = Qm.T[None, None].copy()                         # rows orthonormal
    j = np.array([int(r.integers(0, t + 1)) for t in range(T)])
    q = k[:, :, j, :] * 2.0
    v = r.standard_normal((1, 1, T, 5))
    for o in (oracle.forward_plain(q, k, v), oracle.forward_recurrent(q, k, v)[0],
              oracle.forward_chunked(q, k, v, 4, 1)[0]):
        np.testing.assert_allclose(o[0, 0], v[0, 0, j], rtol=0, atol=1e-12)


def test_weights_visible_nonnegative_convex_causal():
    """With V = I_T (orthogonal unit values, d_v >= T) row t is the weight
    vector: nonnegative, zero after t (causal), summing to 1 -- the convex
    output gate of the normalised readout."""
    T, p = 24, 4
    q, k, _ = _rand_qkv(1, 2, T, p, 1, seed=31)
    V = np.broadcast_to(np.eye(T), (1, 2, T, T)).copy()
    W = oracle.forward_plain(q, k, V)
    assert np.all(W >= 0.0)
    np.testing.assert_allclose(W.sum(-1), 1.0, atol=1e-13)
    assert np.all(np.triu(W[0, 0], 1) == 0.0) and np.all(np.triu(W[0, 1], 1) == 0.0)
    # the weight pattern is that of squared cosines: w_ts / w_tt = cos^2(q_t,k_s)/cos^2(q_t,k_t)
    qu, ku = _unit(q[0, 0]), _unit(k[0, 0])
    t, s = T - 1, 3
    ratio = (qu[t] @ ku[s]) ** 2 / (qu[t] @ ku[t]) ** 2
    assert abs(W[0, 0, t, s] / W[0, 0, t, t] - ratio) < 1e-10


def test_outputs_inside_hull_of_seen_values():
    """Every o_t coordinate lies within [min_{s<=t} v_s, max_{s<=t} v_s]."""
    q, k, v = _rand_qkv(2, 2, 80, 8, 6, seed=41, scale=5.0)
    o = oracle.forward_chunked(q, k, v, 16, 1)[0]
    lo = np.minimum.accumulate(v, axis=2)
    hi = np.maximum.accumulate(v, axis=2)
    assert np.all(o >= lo - 1e-12) and np.all(o <= hi + 1e-12)


def test_convex_gate_identity():
    """o_t = (1 - a_t) * o_{t-1}(q_t) + a_t v_t with a_t = w_tt / sum_{s<=t} w_ts:
    the readout interpolates between the previous state's readout (with the new
    query) and the current value."""
    T, p, dv = 20, 5, 3
    q, k, v = _rand_qkv(1, 1, T, p, dv, seed=51)
    o = oracle.forward_plain(q, k, v)[0, 0]
    W = oracle.forward_plain(q, k, np.eye(T)[None, None])[0, 0]
    for t in range(1, T):
        qp = q.copy()
        qp[0, 0, t - 1] = q[0, 0, t]                      # previous state, new query
        prev = oracle.forward_plain(qp[:, :, :t], k[:, :, :t], v[:, :, :t])[0, 0, t - 1]
        a = W[t, t]
        np.testing.assert_allclose(o[t], (1 - a) * prev + a * v[0, 0, t], rtol=0, atol=1e-12)


@pytest.mark.parametrize("p", [2, 3, 8, 16])
def test_psnr_regular_simplex_welch_bound(p):
    """T = p + 1 keys forming a regular simplex meet the Welch bound: squared
    correlation eps* = (T-p)/(p(T-1)) = 1/p^2 with the matched query, and the
    readout through orthogonal values has pSNR_PSD = p^2 (T-1)/(T-p)^2 = p^3
    (Eqs. 10-12)."""
    T = p + 1
    E = np.eye(T) - 1.0 / T
    basis, _ = np.linalg.qr(E[:, :p])            # orthonormal basis of the hyperplane
    keys = _unit(E @ basis)                      # T unit vectors in R^p
    G = keys @ keys.T
    eps = (T - p) / (p * (T - 1))
    off = G[~np.eye(T, dtype=bool)] ** 2
    np.testing.assert_allclose(off, eps, atol=1e-14)
    r = _rng(p)
    order = r.permutation(T)                     # matched key at a random position
    k = keys[order][None, None]
    star = int(np.where(order == 0)[0][0])
    q = np.broadcast_to(keys[0], (1, 1, T, p)).copy()
    a = oracle.forward_plain(q, k, np.eye(T)[None, None])[0, 0, -1]
    psnr = a[star] ** 2 / (np.sum(a ** 2) - a[star] ** 2)
    assert abs(psnr - p ** 2 * (T - 1) / (T - p) ** 2) < 1e-9 * psnr
    assert abs(psnr - p ** 3) < 1e-9 * psnr


@pytest.mark.parametrize("p,T", [(4, 9), (16, 40), (32, 100)])
def test_psnr_equal_interference_closed_form(p, T):
    """T-1 distractors each with squared correlation eps* to the query give
    pSNR_PSD = 1/((T-1) eps*^2) = p^2(T-1)/(T-p)^2 (Eq. 12)."""
    eps = (T - p) / (p * (T - 1))
    r = _rng(T)
    e1 = np.zeros(p)
    e1[0] = 1.0
    keys = [e1]
    for _ in range(T - 1):
        w = r.standard_normal(p)
        w[0] = 0.0
        w /= np.linalg.norm(w)
        keys.append(math.sqrt(eps) * e1 + math.sqrt(1 - eps) * w)
    keys = np.array(keys)[r.permutation(T)]
    star = int(np.argmax(keys[:, 0]))
    q = np.broadcast_to(e1, (1, 1, T, p)).copy()
    a = oracle.forward_plain(q, keys[None, None], np.eye(T)[None, None])[0, 0, -1]
    psnr = a[star] ** 2 / (np.sum(a ** 2) - a[star] ** 2)
    assert abs(psnr - p ** 2 * (T - 1) / (T - p) ** 2) < 1e-9 * psnr


def test_rotation_and_scale_invariance():
    """An orthogonal map of q and k (isometric invariance, Assumption 2) and any
    nonzero rescaling of individual rows (unit-sphere projection, squared
    scores) leave the output unchanged."""
    q, k, v = _rand_qkv(1, 2, 33, 6, 4, seed=61)
    ref = oracle.forward_plain(q, k, v)
    U, _ = np.linalg.qr(_rng(62).standard_normal((6, 6)))
    np.testing.assert_allclose(oracle.forward_plain(q @ U.T, k @ U.T, v), ref, atol=1e-13)
    sq = _rng(63).uniform(-4, 4, size=(1, 2, 33, 1))
    sk = _rng(64).uniform(-4, 4, size=(1, 2, 33, 1))
    np.testing.assert_allclose(oracle.forward_chunked(q * sq, k * sk, v, 8, 1)[0], ref, atol=1e-12)


def test_zero_key_and_zero_query():
    """A zero key contributes nothing; a zero query has a zero denominator and
    a zero output row."""
    q, k, v = _rand_qkv(1, 1, 12, 4, 3, seed=71)
    k2 = k.copy()
    k2[0, 0, 5] = 0.0
    o = oracle.forward_plain(q, k2, v)
    keep = [i for i in range(12) if i != 5]
    o_drop = oracle.forward_plain(q[:, :, keep], k[:, :, keep], v[:, :, keep])
    np.testing.assert_allclose(o[:, :, keep], o_drop, atol=1e-13)
    q2 = q.copy()
    q2[0, 0, 7] = 0.0
    for o in (oracle.forward_plain(q2, k, v), oracle.forward_recurrent(q2, k, v)[0],
              oracle.forward_chunked(q2, k, v, 4)[0]):
        assert np.all(o[0, 0, 7] == 0.0)


# ---------------------------------------------------------------- state, scan, split calls

def test_state_readout_identity():
    """psi(u)^T S_T = sum_s (u.kh_s)^2 v_s and psi(u)^T z_T = sum_s (u.kh_s)^2 for
    any unit u: the exported state is Psi(K)^T V in the packed layout."""
    q, k, v = _rand_qkv(1, 1, 25, 5, 3, seed=81)
    _, S, z = oracle.forward_recurrent(q, k, v)
    ku = _unit(k[0, 0])
    for s in range(5):
        u = _unit(_rng(82 + s).standard_normal(5))
        w = (ku @ u) ** 2
        np.testing.assert_allclose(oracle.lift(u) @ S[0, 0], w @ v[0, 0], atol=1e-13)
        assert abs(oracle.lift(u) @ z[0, 0] - w.sum()) < 1e-13


@pytest.mark.parametrize("NC", [1, 2, 3, 5, 8, 64, 100])
def test_scan_tree_equals_sequential(NC):
    """(S_loc, Z_loc) is a vector-space cumulative sum, so any bracketing gives
    the sequential prefix; the log-depth scan takes ceil(log2 N_C) rounds."""
    r = _rng(NC)
    S = r.standard_normal((2, 1, NC, 3, 2))
    z = r.standard_normal((2, 1, NC, 3))
    Ss, zs, rs = oracle.scan_exclusive(S, z, oracle.SCAN_SEQUENTIAL)
    St, zt, rt = oracle.scan_exclusive(S, z, oracle.SCAN_TREE)
    np.testing.assert_allclose(St, Ss, atol=1e-12)
    np.testing.assert_allclose(zt, zs, atol=1e-12)
    assert np.all(Ss[:, :, 0] == 0.0)
    np.testing.assert_allclose(Ss[:, :, 1:], np.cumsum(S, axis=2)[:, :, :-1], atol=1e-12)
    assert rs == NC and rt == (math.ceil(math.log2(NC)) if NC > 1 else 0)


def test_scan_depth_at_T2048_C32():
    """At T = 2048, C = 32: N_C = 64 sequential steps shrink to 6 rounds."""
    NC = 2048 // 32
    S = np.ones((1, 1, NC, 1, 1))
    z = np.ones((1, 1, NC, 1))
    assert oracle.scan_exclusive(S, z, oracle.SCAN_TREE)[2] == 6
    assert oracle.scan_exclusive(S, z, oracle.SCAN_SEQUENTIAL)[2] == 64


def test_chunk_states_sum_to_final_state():
    q, k, v = _rand_qkv(1, 2, 45, 4, 3, seed=91)
    Sl, zl = oracle.chunk_states(k, v, 8)
    _, S, z = oracle.forward_recurrent(q, k, v)
    np.testing.assert_allclose(Sl.sum(axis=2), S, atol=1e-12)
    np.testing.assert_allclose(zl.sum(axis=2), z, atol=1e-12)


@pytest.mark.parametrize("T1", [1, 16, 21, 40])
def test_split_call_with_carried_state(T1):
    """forward(T) equals forward(T1) followed by forward(T - T1) seeded with the
    carried (S, z): the state update is commutative and additive."""
    q, k, v = _rand_qkv(1, 2, 41, 4, 3, seed=101)
    o_ref, S_ref, z_ref = oracle.forward_recurrent(q, k, v)
    for fwd in (lambda *a, **kw: oracle.forward_recurrent(*a, **kw),
                lambda *a, **kw: oracle.forward_chunked(*a[:3], 8, 1, **kw)):
        o1, S1, z1 = fwd(q[:, :, :T1], k[:, :, :T1], v[:, :, :T1])
        o2, S2, z2 = fwd(q[:, :, T1:], k[:, :, T1:], v[:, :, T1:], S0=S1, z0=z1)
        np.testing.assert_allclose(np.concatenate([o1, o2], axis=2), o_ref, atol=1e-12)
        np.testing.assert_allclose(S2, S_ref, atol=1e-12)
        np.testing.assert_allclose(z2, z_ref, atol=1e-12)


def test_empty_sequence_passes_state_through():
    q, k, v = _rand_qkv(1, 1, 0, 3, 2)
    S0 = _rng(1).standard_normal((1, 1, 6, 2))
    z0 = _rng(2).standard_normal((1, 1, 6))
    o, S, z = oracle.forward_chunked(q, k, v, 4, 0, S0=S0, z0=z0)
    assert o.shape == (1, 1, 0, 2)
    np.testing.assert_array_equal(S, S0)
    np.testing.assert_array_equal(z, z0)


def test_decode_steps_from_carried_states_equal_the_definition():
    """The decode step is the recurrence taken one token at a time (constant-
    time recurrent inference, abstract): T one-token calls, each seeded with the
    previous call's state, give the definition's rows, and one step adds exactly
    psi(kh) v^T, read back through any unit u as (u.kh)^2 v."""
    B, H, T, p, dv = 2, 1, 19, 5, 4
    q, k, v = _rand_qkv(B, H, T, p, dv, seed=111)
    n = p * (p + 1) // 2
    S, z = np.zeros((B, H, n, dv)), np.zeros((B, H, n))
    rows = []
    for t in range(T):
        S_prev = S
        o, S, z = oracle.forward_recurrent(q[:, :, t:t + 1], k[:, :, t:t + 1], v[:, :, t:t + 1], S0=S, z0=z)
        rows.append(o)
        u = _unit(_rng(200 + t).standard_normal(p))
        kh = _unit(k[0, 0, t])
        np.testing.assert_allclose(oracle.lift(u) @ (S - S_prev)[0, 0], (u @ kh) ** 2 * v[0, 0, t], atol=1e-13)
    np.testing.assert_allclose(np.concatenate(rows, axis=2), oracle.forward_plain(q, k, v), atol=1e-12)
