"""GPU parity of the block-lift forwards (KATA-Sigma-g, KATA-M-g) against the
fp64 oracle's block-lift definition and recurrence, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from kernelized_linear_attention_03_b300 import binding as kb
from kernelized_linear_attention_03_b300 import inputs
from tests.parity import TOL, assert_close, f64

pytestmark = pytest.mark.gpu
DNAME = {torch.float32: "fp32", torch.bfloat16: "bf16"}
SIGMA, MULTI = kb.KATA_LIFT_SIGMA, kb.KATA_LIFT_MULTI
assert (SIGMA, MULTI) == (oracle.LIFT_SIGMA, oracle.LIFT_MULTI)


def _tokens(B, H, T, p, dv, dtype, seed):
    return inputs.make(inputs.small(B, H, T, p, dv, 32, DNAME[dtype], "raw", seed), "cuda")


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


CASES = [(SIGMA, 2, 64, 64), (MULTI, 2, 64, 64), (SIGMA, 4, 32, 16), (MULTI, 4, 16, 32), (SIGMA, 8, 64, 32),
         (MULTI, 16, 16, 16)]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("fam,g,p,dv", CASES)
@pytest.mark.parametrize("C", [32, 128])
def test_chunked_block_matches_the_definition(dtype, fam, g, p, dv, C):
    q, k, v = _tokens(1, 2, 150, p, dv, dtype, seed=g + p + C)
    o = kb.kata_forward_chunked_block(q, k, v, C, fam, g)
    torch.cuda.synchronize()
    assert_close(f64(o), oracle.forward_plain_block(f64(q), f64(k), f64(v), fam, g), dtype, "chunked block")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("fam,g,p,dv", CASES[:4])
def test_quadratic_block_matches_the_definition(dtype, fam, g, p, dv):
    q, k, v = _tokens(2, 1, 130, p, dv, dtype, seed=3 * g + p)
    o = kb.kata_forward_quadratic_block(q, k, v, fam, g)
    torch.cuda.synchronize()
    assert_close(f64(o), oracle.forward_plain_block(f64(q), f64(k), f64(v), fam, g), dtype, "quadratic block")


@pytest.mark.parametrize("mode", [kb.KATA_SCAN_SEQUENTIAL, kb.KATA_SCAN_TREE])
@pytest.mark.parametrize("fam,g,p,dv", CASES[:2])
def test_chunked_block_states_and_split_calls(mode, fam, g, p, dv):
    """forward(T1) -> (S, z) -> forward(T2) seeded with it: the rows equal the
    definition over the whole sequence and the final state the oracle's."""
    dtype = torch.float32
    B, H, T1, T2, C = 1, 2, 70, 61, 32
    q, k, v = _tokens(B, H, T1 + T2, p, dv, dtype, seed=41)
    n = kb.kata_lift_dim(fam, p, g)
    S = torch.empty(B, H, n, dv, device="cuda")
    z = torch.empty(B, H, n, device="cuda")
    S2, z2 = torch.empty_like(S), torch.empty_like(z)
    part = lambda x, a, b: x[:, :, a:b].contiguous()  # noqa: E731
    o1, _, _ = kb.kata_forward_chunked_block(part(q, 0, T1), part(k, 0, T1), part(v, 0, T1), C, fam, g, mode,
                                             S_final=S, z_final=z)
    o2, _, _ = kb.kata_forward_chunked_block(part(q, T1, T1 + T2), part(k, T1, T1 + T2), part(v, T1, T1 + T2), C,
                                             fam, g, mode, S0=S, z0=z, S_final=S2, z_final=z2)
    torch.cuda.synchronize()
    ref = oracle.forward_plain_block(f64(q), f64(k), f64(v), fam, g)
    assert_close(np.concatenate([f64(o1), f64(o2)], axis=2), ref, dtype, "split block")
    _, S_ref, z_ref = oracle.forward_recurrent_block(f64(q), f64(k), f64(v), fam, g)
    assert _rel(f64(S2), S_ref) <= TOL[dtype] and _rel(f64(z2), z_ref) <= TOL[dtype]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("fam,g,p,dv", CASES)
def test_decode_block_from_a_prefix_state(dtype, fam, g, p, dv):
    B, H, T0 = 2, 3, 12
    q, k, v = _tokens(B, H, T0 + 1, p, dv, dtype, seed=g * p + dv)
    _, S0, z0 = oracle.forward_recurrent_block(f64(q[:, :, :T0]), f64(k[:, :, :T0]), f64(v[:, :, :T0]), fam, g)
    S = torch.from_numpy(S0).float().cuda()
    z = torch.from_numpy(z0).float().cuda()
    S_in, z_in = f64(S), f64(z)
    qt, kt, vt = (x[:, :, T0].contiguous() for x in (q, k, v))
    o = kb.kata_decode_step_block(qt, kt, vt, S, z, fam, g)
    torch.cuda.synchronize()
    o_ref, S_ref, z_ref = oracle.forward_recurrent_block(f64(qt)[:, :, None], f64(kt)[:, :, None],
                                                         f64(vt)[:, :, None], fam, g, S_in, z_in)
    assert_close(f64(o)[:, :, None], o_ref, dtype, "decode block o")
    assert _rel(f64(S), S_ref) <= 1e-6 and _rel(f64(z), z_ref) <= 1e-6


def test_block_forward_decode_round_trip_bf16():
    """Chunked block forward -> its final state -> a decode step -> the state
    seeding the next forward: all rows equal the definition."""
    fam, g, p, dv, C = SIGMA, 2, 64, 64, 64
    B, H, T0, T1 = 1, 2, 100, 40
    T = T0 + 1 + T1
    q, k, v = _tokens(B, H, T, p, dv, torch.bfloat16, seed=77)
    n = kb.kata_lift_dim(fam, p, g)
    S = torch.empty(B, H, n, dv, device="cuda")
    z = torch.empty(B, H, n, device="cuda")
    part = lambda x, a, b: x[:, :, a:b].contiguous()  # noqa: E731
    o0, _, _ = kb.kata_forward_chunked_block(part(q, 0, T0), part(k, 0, T0), part(v, 0, T0), C, fam, g,
                                             S_final=S, z_final=z)
    o1 = kb.kata_decode_step_block(q[:, :, T0].contiguous(), k[:, :, T0].contiguous(), v[:, :, T0].contiguous(),
                                   S, z, fam, g)
    o2 = kb.kata_forward_chunked_block(part(q, T0 + 1, T), part(k, T0 + 1, T), part(v, T0 + 1, T), C, fam, g,
                                       S0=S, z0=z)
    torch.cuda.synchronize()
    o = torch.cat([o0, o1[:, :, None], o2], dim=2)
    assert_close(f64(o), oracle.forward_plain_block(f64(q), f64(k), f64(v), fam, g), torch.bfloat16, "round trip")


def test_full_family_through_the_block_path_is_the_forward():
    q, k, v = _tokens(1, 2, 90, 32, 32, torch.float32, seed=5)
    o = kb.kata_forward_chunked_block(q, k, v, 32, kb.KATA_LIFT_FULL, 1)
    torch.cuda.synchronize()
    assert_close(f64(o), oracle.forward_plain(f64(q), f64(k), f64(v)), torch.float32, "full via block")


def test_block_argument_errors():
    q, k, v = _tokens(1, 1, 8, 16, 16, torch.float32, seed=1)
    with pytest.raises(kb.KataError) as e:
        kb.kata_forward_quadratic_block(q, k, v, 7, 2)
    assert e.value.status == kb.KATA_ERR_INVALID_ARG
    with pytest.raises(kb.KataError) as e:
        kb.kata_forward_quadratic_block(q, k, v, SIGMA, 3)
    assert e.value.status == kb.KATA_ERR_UNSUPPORTED
    with pytest.raises(kb.KataError) as e:
        kb.kata_forward_quadratic_block(q, k, v, kb.KATA_LIFT_FULL, 2)
    assert e.value.status == kb.KATA_ERR_UNSUPPORTED


# ---------------------------------------------------------------- KATA-Sigma-g on the tensor cores
# bf16 KATA-Sigma-g with blocks of 16 or 32 runs on the fused tensor-core
# forward (the lift of one block sets the state's width; the key and query
# lifts sum the g block lifts, Z sums the g block Gram matrices, and the
# intra-chunk scores sum the squares of every block pair's dot products).

def _traced(fn):
    kb.kata_trace_start(1024)
    try:
        out = fn()
        torch.cuda.synchronize()
    finally:
        names = {name for name, _ in kb.kata_trace_stop()}
    return out, names


TC_SIGMA = [(2, 64, 64), (2, 64, 16), (4, 64, 32), (2, 32, 64)]


@pytest.mark.parametrize("g,p,dv", TC_SIGMA)
@pytest.mark.parametrize("T", [1, 127, 129, 600])
def test_sigma_tensor_core_forward(g, p, dv, T):
    q, k, v = _tokens(1, 3, T, p, dv, torch.bfloat16, seed=7 * g + p + T)
    o, names = _traced(lambda: kb.kata_forward_chunked_block(q, k, v, 128, SIGMA, g))
    assert "chunked_tc" in names and "intra_tc" in names, names
    # three heads leave CTAs free, so a sequence of more than one 128-token
    # chunk is cut into segments whose start states come from the chunk-state
    # kernel's segment totals (block lift) and the scan
    if T > 128:
        assert "states_tc" in names, names
    assert_close(f64(o), oracle.forward_plain_block(f64(q), f64(k), f64(v), SIGMA, g), torch.bfloat16,
                 "Sigma tensor cores")


@pytest.mark.parametrize("g,p,dv", TC_SIGMA[:2])
def test_sigma_tensor_core_states_and_split_calls(g, p, dv):
    """The carried state of the tensor-core path (KATA-Sigma-g packing, sqrt(2)
    off the diagonal) continues a forward and matches the oracle's recurrence."""
    B, H, T1, T2 = 1, 2, 300, 222
    q, k, v = _tokens(B, H, T1 + T2, p, dv, torch.bfloat16, seed=5 + g)
    n = kb.kata_lift_dim(SIGMA, p, g)
    S, z = torch.empty(B, H, n, dv, device="cuda"), torch.empty(B, H, n, device="cuda")
    S2, z2 = torch.empty_like(S), torch.empty_like(z)
    part = lambda x, a, b: x[:, :, a:b].contiguous()  # noqa: E731
    o1, _, _ = kb.kata_forward_chunked_block(part(q, 0, T1), part(k, 0, T1), part(v, 0, T1), 64, SIGMA, g,
                                             S_final=S, z_final=z)
    o2, _, _ = kb.kata_forward_chunked_block(part(q, T1, T1 + T2), part(k, T1, T1 + T2), part(v, T1, T1 + T2), 64,
                                             SIGMA, g, S0=S, z0=z, S_final=S2, z_final=z2)
    torch.cuda.synchronize()
    ref = oracle.forward_plain_block(f64(q), f64(k), f64(v), SIGMA, g)
    assert_close(np.concatenate([f64(o1), f64(o2)], axis=2), ref, torch.bfloat16, "Sigma split")
    _, S_ref, z_ref = oracle.forward_recurrent_block(f64(q), f64(k), f64(v), SIGMA, g)
    assert _rel(f64(S2), S_ref) <= TOL[torch.bfloat16] and _rel(f64(z2), z_ref) <= TOL[torch.bfloat16]


def test_sigma_tensor_core_zero_vectors():
    q, k, v = _tokens(1, 2, 260, 64, 64, torch.bfloat16, seed=3)
    q[0, 0, 7] = 0
    k[0, 1, 0] = 0
    k[0, 0, 128] = 0
    o = kb.kata_forward_chunked_block(q, k, v, 128, SIGMA, 2)
    torch.cuda.synchronize()
    assert torch.count_nonzero(o[0, 0, 7]) == 0
    assert_close(f64(o), oracle.forward_plain_block(f64(q), f64(k), f64(v), SIGMA, 2), torch.bfloat16, "zero")


@pytest.mark.slow
def test_chunked_block_full_size_sampled_rows():
    """KATA-Sigma-2 on the 131072-token, 8-head, p = dv = 64 bf16 workload (C = 128)
    -- the fused tensor-core forward -- against the oracle's definition on
    sampled rows (first, last, chunk edges, random and late positions) of every
    head, gated per head and row by row."""
    from tests.parity import row_errors, rows_error, sample_rows
    w = inputs.WORKLOADS[3]
    q, k, v = inputs.make(w, "cuda")
    o, names = _traced(lambda: kb.kata_forward_chunked_block(q, k, v, w.C, SIGMA, 2))
    assert "chunked_tc" in names
    bh, t = sample_rows(w.B, w.H, w.T, w.C, per_head=6, seed=1)
    ref = oracle.forward_plain_block_rows(f64(q), f64(k), f64(v), SIGMA, 2, bh, t)
    got = f64(o).reshape(w.B * w.H, w.T, w.dv)[bh, t]
    assert rows_error(got, ref) <= TOL[torch.bfloat16]
    per_row = row_errors(got, ref)
    print(f"Sigma-2 full size: worst per-row error {per_row.max():.3e}")
    assert per_row.max() <= TOL[torch.bfloat16]
