"""GPU parity of the gated prefix (kata_forward_chunked_gated,
kata_decode_step_gated) against the fp64 oracle's gated forms."""
import numpy as np
import pytest
import torch

import oracle
from kernelized_linear_attention_03_b300 import binding as kb
from kernelized_linear_attention_03_b300 import inputs
from tests.parity import TOL, assert_close, f64

pytestmark = pytest.mark.gpu
DNAME = {torch.float32: "fp32", torch.bfloat16: "bf16"}


def _case(B, H, T, p, dv, dtype, seed, lo=0.5):
    q, k, v = inputs.make(inputs.small(B, H, T, p, dv, 32, DNAME[dtype], "raw", seed), "cuda")
    gate = torch.from_numpy(np.random.default_rng(seed).uniform(lo, 1.0, (B, H, T))).float().cuda()
    return q, k, v, gate


def _rel(a, b):
    return float(np.abs(np.asarray(a) - b).max() / max(np.abs(b).max(), 1e-300))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("p,dv", [(16, 16), (32, 64), (64, 64)])
@pytest.mark.parametrize("C", [32, 128])
def test_gated_chunked_matches_the_definition(dtype, p, dv, C):
    q, k, v, gate = _case(1, 2, 200, p, dv, dtype, seed=p + dv + C)
    o = kb.kata_forward_chunked_gated(q, k, v, gate, C)
    torch.cuda.synchronize()
    if dtype == torch.bfloat16:
        # bf16 chunk states are sums of bf16 unit-key lifts: rows held to the
        # tolerance where the readout is well conditioned, all rows to the hull
        _check_gated_rows(q, k, v, gate, o, p, "gated chunked")
        return
    ref = oracle.forward_plain_gated(f64(q), f64(k), f64(v), f64(gate))
    assert_close(f64(o), ref, dtype, "gated chunked")


def test_gated_zero_gates_and_unit_gates():
    q, k, v, gate = _case(1, 2, 150, 32, 32, torch.float32, seed=3)
    gate[:, :, 40] = 0.0
    gate[:, :, 97] = 0.0
    o = kb.kata_forward_chunked_gated(q, k, v, gate, 32)
    ones = torch.ones_like(gate)
    o1 = kb.kata_forward_chunked_gated(q, k, v, ones, 64)
    torch.cuda.synchronize()
    assert_close(f64(o), oracle.forward_plain_gated(f64(q), f64(k), f64(v), f64(gate)), torch.float32, "zero gates")
    assert_close(f64(o1), oracle.forward_plain(f64(q), f64(k), f64(v)), torch.float32, "unit gates")


def test_gated_states_and_split_calls():
    dtype, p, dv, C = torch.float32, 16, 32, 32
    B, H, T1, T2 = 1, 2, 77, 50
    q, k, v, gate = _case(B, H, T1 + T2, p, dv, dtype, seed=9)
    n = p * (p + 1) // 2
    S, z = torch.empty(B, H, n, dv, device="cuda"), torch.empty(B, H, n, device="cuda")
    S2, z2 = torch.empty_like(S), torch.empty_like(z)
    part = lambda x, a, b: x[:, :, a:b].contiguous()  # noqa: E731
    o1, _, _ = kb.kata_forward_chunked_gated(part(q, 0, T1), part(k, 0, T1), part(v, 0, T1), part(gate, 0, T1), C,
                                             S_final=S, z_final=z)
    o2, _, _ = kb.kata_forward_chunked_gated(part(q, T1, T1 + T2), part(k, T1, T1 + T2), part(v, T1, T1 + T2),
                                             part(gate, T1, T1 + T2), C, S0=S, z0=z, S_final=S2, z_final=z2)
    torch.cuda.synchronize()
    ref = oracle.forward_plain_gated(f64(q), f64(k), f64(v), f64(gate))
    assert_close(np.concatenate([f64(o1), f64(o2)], axis=2), ref, dtype, "gated split")
    _, S_ref, z_ref = oracle.forward_recurrent_gated(f64(q), f64(k), f64(v), f64(gate))
    assert _rel(f64(S2), S_ref) <= TOL[dtype] and _rel(f64(z2), z_ref) <= TOL[dtype]


def _readout_condition(q, k, gate):
    """kappa_t = tr(Z_t) / (qh_t^T Z_t qh_t) with Z_t = sum_s d_ts kh_s kh_s^T and
    d_ts = prod_{r=s+1..t} gate_r: the factor by which the recurrent readout's
    lifted denominator psi(qh_t)^T z_t (a sum of terms of either sign whose
    magnitudes add up to at most tr(Z_t)) amplifies rounding.  Large when the
    query is nearly orthogonal to every key the gates have left alive."""
    qh = q / np.maximum(np.linalg.norm(q, axis=-1, keepdims=True), 1e-300)
    kh = k / np.maximum(np.linalg.norm(k, axis=-1, keepdims=True), 1e-300)
    B, H, T, _ = q.shape
    kappa = np.empty((B, H, T))
    for b in range(B):
        for h in range(H):
            for t in range(T):
                d = np.array([np.prod(gate[b, h, s + 1:t + 1]) for s in range(t + 1)])
                den = float(np.sum(d * (kh[b, h, :t + 1] @ qh[b, h, t]) ** 2))
                kappa[b, h, t] = np.sum(d) / max(den, 1e-300)
    return kappa


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("p,dv", [(16, 16), (64, 64)])
def test_gated_decode_steps(dtype, p, dv):
    """Decode steps against the gated definition, row by row: each row may
    differ by the dtype's tolerance of the head's largest output plus the
    fp32 rounding of the lifted denominator amplified by the row's
    condition kappa_t (gates in [0.5, 1] leave few keys alive, and a query
    nearly orthogonal to all of them has a denominator of 1e-5 or less)."""
    B, H, T = 2, 3, 20
    q, k, v, gate = _case(B, H, T, p, dv, dtype, seed=p * dv)
    n = p * (p + 1) // 2
    S, z = torch.zeros(B, H, n, dv, device="cuda"), torch.zeros(B, H, n, device="cuda")
    rows = [kb.kata_decode_step_gated(q[:, :, t].contiguous(), k[:, :, t].contiguous(), v[:, :, t].contiguous(),
                                      gate[:, :, t].contiguous(), S, z) for t in range(T)]
    torch.cuda.synchronize()
    qq, kk, vv, gg = f64(q), f64(k), f64(v), f64(gate)
    ref = oracle.forward_plain_gated(qq, kk, vv, gg)
    got = f64(torch.stack(rows, dim=2))
    kappa = _readout_condition(qq, kk, gg)
    scale = np.abs(ref).max(axis=(2, 3), keepdims=True)
    vmax = np.abs(vv).max(axis=(2, 3), keepdims=True)
    allowed = TOL[dtype] * scale + 16 * np.finfo(np.float32).eps * kappa[..., None] * vmax
    assert np.all(np.abs(got - ref) <= allowed), "gated decode rows outside the conditioned bound"
    # rows whose denominator is well conditioned (kappa within ten times its
    # typical size p for random directions) meet the plain tolerance
    good = kappa <= 10 * p
    assert good.mean() > 0.75
    d = np.where(good[..., None], np.abs(got - ref), 0.0).max(axis=(2, 3), keepdims=True)
    assert np.all(d <= TOL[dtype] * scale), "well-conditioned gated decode rows"


@pytest.mark.slow
def test_gated_full_size_sampled_rows():
    """The 16384-token, 16-head, p = dv = 64 bf16 workload (C = 64) with gates in
    [0.9, 1], against the oracle's gated definition on sampled rows."""
    from tests.parity import rows_error, sample_rows
    w = inputs.WORKLOADS[2]
    q, k, v = inputs.make(w, "cuda")
    gate = torch.from_numpy(np.random.default_rng(3).uniform(0.9, 1.0, (w.B, w.H, w.T))).float().cuda()
    o = kb.kata_forward_chunked_gated(q, k, v, gate, w.C)
    torch.cuda.synchronize()
    bh, t = sample_rows(w.B, w.H, w.T, w.C, per_head=6, seed=2)
    ref = oracle.forward_plain_gated_rows(f64(q), f64(k), f64(v), f64(gate), bh, t)
    got = f64(o).reshape(w.B * w.H, w.T, w.dv)[bh, t]
    assert rows_error(got, ref) <= TOL[torch.bfloat16]


# ---------------------------------------------------------------- gated flash-style form (tensor cores)

def _traced_names(fn):
    kb.kata_trace_start(4096)
    try:
        out = fn()
        torch.cuda.synchronize()
    finally:
        names = {name for name, _ in kb.kata_trace_stop()}
    return out, names


def _decays(gate):
    """d[b, h, t, s] = prod_{r=s+1..t} gate_r for s <= t (0 above the diagonal)."""
    B, H, T = gate.shape
    d = np.zeros((B, H, T, T))
    for t in range(T):
        d[:, :, t, t] = 1.0
        if t:
            d[:, :, t, :t] = np.flip(np.cumprod(np.flip(gate[:, :, 1:t + 1], axis=-1), axis=-1), axis=-1)
    return d


def _check_gated_rows(q, k, v, gate, o, p, what, min_good=0.9):
    """Rows against the oracle's gated definition at the bf16 tolerance where
    the readout is well conditioned, and every row inside the hull of the
    values its weights can reach.  The condition kappa_t = sum_s d_ts /
    sum_s d_ts (qh_t.kh_s)^2 (1 for a query parallel to every live key, about p
    for random directions) is the factor by which the rounding of the unit
    keys to bf16 is amplified in the ratio of the weights: a query nearly
    orthogonal to the few keys the gates leave alive has a large kappa, and its
    output is only bound by the convex hull (nonnegative weights)."""
    qq, kk, vv, gg = f64(q), f64(k), f64(v), f64(gate)
    ref = oracle.forward_plain_gated(qq, kk, vv, gg)
    got = f64(o)
    qh = qq / np.maximum(np.linalg.norm(qq, axis=-1, keepdims=True), 1e-300)
    kh = kk / np.maximum(np.linalg.norm(kk, axis=-1, keepdims=True), 1e-300)
    d = _decays(gg)
    cos2 = np.einsum("bhtp,bhsp->bhts", qh, kh) ** 2
    kappa = d.sum(-1) / np.maximum((d * cos2).sum(-1), 1e-300)
    good = kappa <= 10 * p
    # (most rows are well conditioned: a check that would pass vacuously is not one)
    assert good.size < 50 or good.mean() > min_good, f"{what}: {good.mean():.2f} of the rows well conditioned"
    scale = np.abs(ref).max(axis=(2, 3), keepdims=True)
    err = np.abs(got - ref)
    worst = float(np.where(good[..., None], err / scale, 0.0).max())
    assert worst <= TOL[torch.bfloat16], f"{what}: well-conditioned rows {worst:.3e}"
    # convex hull: the values at or after the last zero gate up to t (what a
    # nonnegative weight can reach), with the output's bf16 rounding as slack
    # (the live keys of row t are the window [a_t, t]: d_ts only shrinks with
    # distance, and a zero gate ends it)
    first = np.argmax(d > 0, axis=-1)
    B, H, T, _ = vv.shape
    slack = 1e-2 * np.abs(vv).max()
    for b in range(B):
        for h in range(H):
            for t in range(T):
                win = vv[b, h, first[b, h, t]:t + 1]
                assert np.all(got[b, h, t] >= win.min(axis=0) - slack) and np.all(got[b, h, t] <= win.max(axis=0) + slack), \
                    f"{what}: row {t} of head {h} outside the convex hull"


@pytest.mark.parametrize("p,dv,C", [(32, 32, 32), (64, 64, 64), (16, 64, 128)])
def test_gated_chunked_bf16_states_on_tensor_cores(p, dv, C):
    """bf16 chunk states from the tensor-core chunk-state kernel, each token's
    key lift weighted by its decay to its chunk's end (gate_decay): zero gates
    inside a chunk and on a chunk's last and first tokens, ragged tails, and a
    second call that carries the state; outputs and the final state against
    the oracle's gated definition and recurrence."""
    B, H, T1, T2 = 1, 2, 3 * C + 5, 2 * C - 3
    q, k, v, gate = _case(B, H, T1 + T2, p, dv, torch.bfloat16, seed=3 * p + C)
    gate[0, 0, C // 2] = 0.0
    gate[0, 1, C - 1] = 0.0
    gate[0, 1, 2 * C] = 0.0
    n = p * (p + 1) // 2
    S, z = torch.empty(B, H, n, dv, device="cuda"), torch.empty(B, H, n, device="cuda")
    S2, z2 = torch.empty_like(S), torch.empty_like(z)
    part = lambda x, a, b: x[:, :, a:b].contiguous()  # noqa: E731
    (o1, _, _), names = _traced_names(lambda: kb.kata_forward_chunked_gated(
        part(q, 0, T1), part(k, 0, T1), part(v, 0, T1), part(gate, 0, T1), C, S_final=S, z_final=z))
    assert {"gate_decay", "states_tc"} <= names and "gated_states_simt" not in names, names
    o2, _, _ = kb.kata_forward_chunked_gated(part(q, T1, T1 + T2), part(k, T1, T1 + T2), part(v, T1, T1 + T2),
                                             part(gate, T1, T1 + T2), C, S0=S, z0=z, S_final=S2, z_final=z2)
    kb.kata_get_device_status()
    o = torch.cat([o1, o2], dim=2)
    _check_gated_rows(q, k, v, gate, o, p, "gated chunked, tensor-core states", min_good=0.75)
    _, S_ref, z_ref = oracle.forward_recurrent_gated(f64(q), f64(k), f64(v), f64(gate))
    assert _rel(f64(S2), S_ref) <= TOL[torch.bfloat16] and _rel(f64(z2), z_ref) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("p,dv", [(16, 16), (32, 64), (64, 64), (64, 32)])
@pytest.mark.parametrize("T", [1, 127, 300, 600])
def test_gated_quadratic_matches_the_definition(p, dv, T):
    """Gates in [0.5, 1]: every query tile's decay is moderate, so its weights
    take the keys' factors; against the oracle's gated definition."""
    q, k, v, gate = _case(1, 3, T, p, dv, torch.bfloat16, seed=11 * p + dv + T)
    o, names = _traced_names(lambda: kb.kata_forward_quadratic_gated(q, k, v, gate))
    kb.kata_get_device_status()
    assert "quadratic_gated_tc" in names and "gate_prefix" in names, names
    _check_gated_rows(q, k, v, gate, o, p, "gated quadratic")


@pytest.mark.parametrize("p,dv", [(32, 32), (64, 64)])
def test_gated_quadratic_strong_decay_and_zero_gates(p, dv):
    """Gates in [0.015, 0.3] (a query tile's decay far past the key-factor
    range, so every weight takes its own exponential) and zero gates inside
    query tiles and on a tile edge; against the oracle."""
    q, k, v, gate = _case(1, 2, 420, p, dv, torch.bfloat16, seed=p + 5, lo=0.05)
    gate = gate * 0.3
    gate[0, 0, 40] = 0.0
    gate[0, 0, 128] = 0.0
    gate[0, 1, 300] = 0.0
    o = kb.kata_forward_quadratic_gated(q, k, v, gate)
    kb.kata_get_device_status()
    assert np.isfinite(f64(o)).all()
    # (with one to three keys alive per row, fewer rows are well conditioned)
    _check_gated_rows(q, k, v, gate, o, p, "gated quadratic, strong decay and zero gates", min_good=0.75)


def test_gated_quadratic_unit_gates_are_the_ungated_form():
    """All gates 1: every decay factor is exactly 1, so the gated kernel's
    weights and output are those of the ungated flash-style form, bit for bit."""
    q, k, v, gate = _case(2, 2, 333, 64, 64, torch.bfloat16, seed=21)
    gate = torch.ones_like(gate)
    o = kb.kata_forward_quadratic_gated(q, k, v, gate)
    ref = kb.kata_forward_quadratic(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(o, ref)


def test_gated_quadratic_refuses_fp32():
    q, k, v, gate = _case(1, 1, 64, 16, 16, torch.float32, seed=1)
    with pytest.raises(kb.KataError):
        kb.kata_forward_quadratic_gated(q, k, v, gate)


@pytest.mark.slow
def test_gated_quadratic_full_size_sampled_rows():
    """The 16384-token, 16-head, p = dv = 64 bf16 workload with gates in [0.9, 1]
    through the gated flash-style form, against the oracle's gated definition on
    sampled rows (32 per head in the last quarter), gated per head and row by row."""
    from tests.parity import row_errors, rows_error, sample_rows
    w = inputs.WORKLOADS[2]
    q, k, v = inputs.make(w, "cuda")
    gate = torch.from_numpy(np.random.default_rng(3).uniform(0.9, 1.0, (w.B, w.H, w.T))).float().cuda()
    o = kb.kata_forward_quadratic_gated(q, k, v, gate)
    kb.kata_get_device_status()
    bh, t = sample_rows(w.B, w.H, w.T, w.C, per_head=6, seed=2)
    ref = oracle.forward_plain_gated_rows(f64(q), f64(k), f64(v), f64(gate), bh, t)
    got = f64(o).reshape(w.B * w.H, w.T, w.dv)[bh, t]
    assert rows_error(got, ref) <= TOL[torch.bfloat16]
    assert row_errors(got, ref).max() <= TOL[torch.bfloat16]
