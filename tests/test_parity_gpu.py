"""GPU parity of every libkata entry point against the fp64 oracle.

Small cases compare every output element; the full-size workloads (in the
launch configuration the benchmark times) compare sampled rows against the
plain definition plus properties that hold at any size.  All calls go
through the C ABI (binding = argument marshalling only).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from kernelized_linear_attention_03_b300 import binding as kb
from kernelized_linear_attention_03_b300 import inputs
from tests.parity import TOL, assert_close, f64, head_errors, row_errors, rows_error, sample_rows

pytestmark = pytest.mark.gpu
DTYPES = [torch.float32, torch.bfloat16]
DNAME = {torch.float32: "fp32", torch.bfloat16: "bf16"}


def _inputs(B, H, T, p, dv, dtype, kind="raw", seed=0, C=32):
    w = inputs.small(B, H, T, p, dv, C, DNAME[dtype], kind, seed)
    return inputs.make(w, "cuda")


def _state_tol(dtype):
    return TOL[dtype]


def _state_err(S_gpu, S_ref):
    S_gpu = f64(S_gpu)
    return float(np.abs(S_gpu - S_ref).max() / max(np.abs(S_ref).max(), 1e-300))


# ---------------------------------------------------------------- quadratic form

@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("p,dv", [(16, 16), (16, 64), (32, 32), (32, 64), (64, 16), (64, 64)])
@pytest.mark.parametrize("T", [1, 37, 200])
def test_quadratic_small(dtype, p, dv, T):
    q, k, v = _inputs(2, 1, T, p, dv, dtype, seed=T + p)
    o = kb.kata_forward_quadratic(q, k, v)
    torch.cuda.synchronize()
    assert_close(f64(o), oracle.forward_plain(f64(q), f64(k), f64(v)), dtype, "quadratic")


@pytest.mark.parametrize("C", [0, 32, 64, 128])
def test_quadratic_tile_hint_does_not_change_results(C):
    q, k, v = _inputs(1, 2, 300, 32, 32, torch.bfloat16, seed=3)
    o = kb.kata_forward_quadratic(q, k, v, C=C)
    assert_close(f64(o), oracle.forward_plain(f64(q), f64(k), f64(v)), torch.bfloat16, "quadratic")


@pytest.mark.parametrize("B,H", [(1, 2), (4, 10)])
@pytest.mark.parametrize("T", [129, 600, 1000])
def test_quadratic_key_split_and_whole_pairs(B, H, T):
    """bf16 flash-style form where two CTAs a pair of query tiles fit in one
    wave (two heads, and 40 heads of 129 tokens: each pair's key tiles split
    over a cluster of two CTAs whose partial sums add) and where they do not
    (40 heads of 600 or 1000 tokens: one CTA a pair); 129 tokens puts one key
    tile in each part, 600 an odd tile count (a last pair with one query tile)."""
    q, k, v = _inputs(B, H, T, 64, 64, torch.bfloat16, seed=B * H + T)
    o = kb.kata_forward_quadratic(q, k, v)
    kb.kata_get_device_status()
    assert_close(f64(o), oracle.forward_plain(f64(q), f64(k), f64(v)), torch.bfloat16, "quadratic, key split")


# ---------------------------------------------------------------- chunked form

@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("p,dv", [(16, 16), (32, 64), (64, 32), (64, 64)])
@pytest.mark.parametrize("T,C", [(1, 32), (31, 32), (33, 32), (100, 64), (300, 128), (257, 64)])
@pytest.mark.parametrize("mode", [kb.KATA_SCAN_SEQUENTIAL, kb.KATA_SCAN_TREE])
def test_chunked_small(dtype, p, dv, T, C, mode):
    q, k, v = _inputs(1, 2, T, p, dv, dtype, seed=T * 3 + p + dv)
    n = kb.kata_packed_dim(p)
    Sf = torch.empty(1, 2, n, dv, dtype=torch.float32, device="cuda")
    zf = torch.empty(1, 2, n, dtype=torch.float32, device="cuda")
    o, Sf, zf = kb.kata_forward_chunked(q, k, v, C, mode, S_final=Sf, z_final=zf)
    kb.kata_get_device_status()
    qq, kk, vv = f64(q), f64(k), f64(v)
    assert_close(f64(o), oracle.forward_plain(qq, kk, vv), dtype, "chunked")
    _, S_ref, z_ref = oracle.forward_recurrent(qq, kk, vv)
    assert _state_err(Sf, S_ref) <= _state_tol(dtype)
    assert _state_err(zf, z_ref) <= _state_tol(dtype)


@pytest.mark.parametrize("dtype", DTYPES)
def test_chunked_initial_state_and_split_call(dtype):
    """forward(T) == forward(T1) then forward(T - T1) seeded with the carried
    state (the multi-call / sequence-sharding hook), against the oracle."""
    T, T1, p, dv, C = 290, 97, 32, 64, 64
    q, k, v = _inputs(2, 2, T, p, dv, dtype, seed=5)
    n = kb.kata_packed_dim(p)
    S1 = torch.empty(2, 2, n, dv, device="cuda")
    z1 = torch.empty(2, 2, n, device="cuda")
    o1, _, _ = kb.kata_forward_chunked(q[:, :, :T1].contiguous(), k[:, :, :T1].contiguous(),
                                       v[:, :, :T1].contiguous(), C, S_final=S1, z_final=z1)
    S2 = torch.empty_like(S1)
    z2 = torch.empty_like(z1)
    o2, _, _ = kb.kata_forward_chunked(q[:, :, T1:].contiguous(), k[:, :, T1:].contiguous(),
                                       v[:, :, T1:].contiguous(), C, S0=S1, z0=z1, S_final=S2,
                                       z_final=z2)
    qq, kk, vv = f64(q), f64(k), f64(v)
    ref = oracle.forward_plain(qq, kk, vv)
    assert_close(np.concatenate([f64(o1), f64(o2)], axis=2), ref, dtype, "split call")
    _, S_ref, z_ref = oracle.forward_recurrent(qq, kk, vv)
    assert _state_err(S2, S_ref) <= _state_tol(dtype)
    assert _state_err(z2, z_ref) <= _state_tol(dtype)
    # the state may be updated in place (S_final aliases S0)
    o3, S1b, z1b = kb.kata_forward_chunked(q[:, :, T1:].contiguous(), k[:, :, T1:].contiguous(),
                                           v[:, :, T1:].contiguous(), C, S0=S1, z0=z1,
                                           S_final=S1, z_final=z1)
    assert _state_err(S1, S_ref) <= _state_tol(dtype)


def _traced_kernels(fn):
    kb.kata_trace_start(4096)
    try:
        out = fn()
        torch.cuda.synchronize()
    finally:
        names = [name for name, _ in kb.kata_trace_stop()]
    return out, names


def test_segmented_forward_with_parts_and_initial_state():
    """One head of 4096 tokens leaves most CTAs free, so the bf16 forward is cut
    into segments whose start states are exclusive prefixes over parts of the
    segments (the chunk-state kernel builds two parts per segment here),
    seeded with the initial state: the full lift and KATA-Sigma-2 against the
    oracle, the output and the carried state."""
    T1, T = 300, 300 + 4096
    q, k, v = _inputs(1, 1, T, 64, 64, torch.bfloat16, seed=31)
    qq, kk, vv = f64(q), f64(k), f64(v)
    part = lambda x, a, b: x[:, :, a:b].contiguous()  # noqa: E731
    # the full lift
    n = kb.kata_packed_dim(64)
    S1, z1 = torch.empty(1, 1, n, 64, device="cuda"), torch.empty(1, 1, n, device="cuda")
    o1, _, _ = kb.kata_forward_chunked(part(q, 0, T1), part(k, 0, T1), part(v, 0, T1), 128, S_final=S1, z_final=z1)
    S2, z2 = torch.empty_like(S1), torch.empty_like(z1)
    (o2, _, _), names = _traced_kernels(lambda: kb.kata_forward_chunked(
        part(q, T1, T), part(k, T1, T), part(v, T1, T), 128, S0=S1, z0=z1, S_final=S2, z_final=z2))
    assert names.count("states_tc") == 1 and "chunked_tc" in names, names
    ref = oracle.forward_plain(qq, kk, vv)
    assert_close(np.concatenate([f64(o1), f64(o2)], axis=2), ref, torch.bfloat16, "segments with parts")
    _, S_ref, z_ref = oracle.forward_recurrent(qq, kk, vv)
    assert _state_err(S2, S_ref) <= _state_tol(torch.bfloat16)
    assert _state_err(z2, z_ref) <= _state_tol(torch.bfloat16)
    # KATA-Sigma-2
    nb = kb.kata_lift_dim(kb.KATA_LIFT_SIGMA, 64, 2)
    B1, y1 = torch.empty(1, 1, nb, 64, device="cuda"), torch.empty(1, 1, nb, device="cuda")
    p1, _, _ = kb.kata_forward_chunked_block(part(q, 0, T1), part(k, 0, T1), part(v, 0, T1), 128, kb.KATA_LIFT_SIGMA, 2,
                                             S_final=B1, z_final=y1)
    B2, y2 = torch.empty_like(B1), torch.empty_like(y1)
    (p2, _, _), names = _traced_kernels(lambda: kb.kata_forward_chunked_block(
        part(q, T1, T), part(k, T1, T), part(v, T1, T), 128, kb.KATA_LIFT_SIGMA, 2, S0=B1, z0=y1, S_final=B2,
        z_final=y2))
    assert names.count("states_tc") == 1, names
    refb = oracle.forward_plain_block(qq, kk, vv, oracle.LIFT_SIGMA, 2)
    assert_close(np.concatenate([f64(p1), f64(p2)], axis=2), refb, torch.bfloat16, "Sigma-2 segments with parts")
    _, B_ref, y_ref = oracle.forward_recurrent_block(qq, kk, vv, oracle.LIFT_SIGMA, 2)
    assert _state_err(B2, B_ref) <= _state_tol(torch.bfloat16)
    assert _state_err(y2, y_ref) <= _state_tol(torch.bfloat16)


def test_chunked_empty_sequence_passes_state_through():
    S0 = torch.randn(1, 3, 136, 16, device="cuda")
    z0 = torch.rand(1, 3, 136, device="cuda")
    Sf = torch.full_like(S0, 7.0)
    zf = torch.full_like(z0, 7.0)
    e = torch.empty(1, 3, 0, 16, dtype=torch.bfloat16, device="cuda")
    kb.kata_forward_chunked(torch.empty(1, 3, 0, 16, dtype=torch.bfloat16, device="cuda"),
                            torch.empty(1, 3, 0, 16, dtype=torch.bfloat16, device="cuda"), e, 32,
                            S0=S0, z0=z0, S_final=Sf, z_final=zf)
    torch.cuda.synchronize()
    assert torch.equal(Sf, S0) and torch.equal(zf, z0)
    kb.kata_forward_chunked(torch.empty(1, 3, 0, 16, dtype=torch.bfloat16, device="cuda"),
                            torch.empty(1, 3, 0, 16, dtype=torch.bfloat16, device="cuda"), e, 32,
                            S_final=Sf, z_final=zf)
    torch.cuda.synchronize()
    assert torch.count_nonzero(Sf) == 0 and torch.count_nonzero(zf) == 0


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("p,dv", [(16, 16), (32, 64), (64, 64)])
def test_degenerate_zero_query_and_key(dtype, p, dv):
    """A zero key drops out of every row (its lift is zero); a zero query
    row has a zero denominator and is written as 0.  Also a query that is
    zero at t = 0 and a zero key at a chunk edge.  Both forms, both dtypes
    (the bf16 forms run on the tensor cores)."""
    T = 300
    q, k, v = _inputs(1, 2, T, p, dv, dtype, seed=8 + p)
    q[0, 0, 10] = 0.0
    q[0, 1, 0] = 0.0
    k[0, 0, 5] = 0.0
    k[0, 1, 128] = 0.0
    k[0, 1, 0] = 0.0
    ref = oracle.forward_plain(f64(q), f64(k), f64(v))
    for C in (32, 128):
        for name, o in (("quadratic", kb.kata_forward_quadratic(q, k, v)), ("chunked", kb.kata_forward_chunked(q, k, v, C))):
            kb.kata_get_device_status()
            assert torch.count_nonzero(o[0, 0, 10]) == 0, name
            assert torch.count_nonzero(o[0, 1, 0]) == 0, name
            assert np.isfinite(f64(o)).all(), name
            assert_close(f64(o), ref, dtype, f"zero rows {name}")


# ---------------------------------------------------------------- chunk states and scans

@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("p,dv,T,C", [(16, 16, 100, 32), (32, 64, 256, 64), (64, 32, 300, 128)])
@pytest.mark.parametrize("mode", [kb.KATA_SCAN_SEQUENTIAL, kb.KATA_SCAN_TREE])
def test_chunk_state_scan(dtype, p, dv, T, C, mode):
    q, k, v = _inputs(1, 2, T, p, dv, dtype, seed=p + T)
    Sp, zp = kb.kata_chunk_state_scan(k, v, C, mode)
    torch.cuda.synchronize()
    Sl, zl = oracle.chunk_states(f64(k), f64(v), C)
    Sr, zr, _ = oracle.scan_exclusive(Sl, zl, oracle.SCAN_SEQUENTIAL)
    scale_S = np.abs(Sl).sum(axis=2).max()
    scale_z = np.abs(zl).sum(axis=2).max()
    assert np.abs(f64(Sp) - Sr).max() <= TOL[dtype] * scale_S
    assert np.abs(f64(zp) - zr).max() <= TOL[dtype] * scale_z
    assert torch.count_nonzero(Sp[:, :, 0]) == 0


@pytest.mark.parametrize("NC", [1, 2, 7, 64, 1000, 1025, 2500])
@pytest.mark.parametrize("n,dv", [(3, 2), (136, 16), (5, 7)])
@pytest.mark.parametrize("mode", [kb.KATA_SCAN_SEQUENTIAL, kb.KATA_SCAN_TREE])
@pytest.mark.parametrize("inplace", [False, True])
def test_scan_states(NC, n, dv, mode, inplace):
    g = torch.Generator(device="cpu").manual_seed(NC + n)
    S = torch.randn(2, 1, NC, n, dv, generator=g).cuda()
    z = torch.rand(2, 1, NC, n, generator=g).cuda()
    Sr, zr, _ = oracle.scan_exclusive(f64(S), f64(z), oracle.SCAN_SEQUENTIAL)
    if inplace:
        Sp, zp = kb.kata_scan_states(S, z, mode, S_prefix=S, z_prefix=z)
    else:
        Sp, zp = kb.kata_scan_states(S, z, mode)
    torch.cuda.synchronize()
    scale = max(1.0, float(np.abs(Sr).max()))
    assert np.abs(f64(Sp) - Sr).max() <= 1e-5 * scale
    assert np.abs(f64(zp) - zr).max() <= 1e-5 * max(1.0, float(zr.max()))


# ---------------------------------------------------------------- host-side rejection on a GPU machine

def test_host_and_short_buffers_rejected():
    lib = kb.load()
    host = np.zeros(4096, dtype=np.float32)
    hp = host.ctypes.data
    assert lib.kata_forward_quadratic(hp, hp, hp, hp, kb.KATA_FP32, 1, 1, 8, 16, 16, 0, None) == \
        kb.KATA_ERR_INVALID_ARG
    cudart = ctypes.CDLL("libcudart.so.13")
    ptr = ctypes.c_void_p()
    assert cudart.cudaMalloc(ctypes.byref(ptr), ctypes.c_size_t(1024)) == 0
    try:
        # 1 x 1 x 64 x 16 fp32 needs 4 KiB per operand; the allocation holds 1 KiB.
        st = lib.kata_forward_quadratic(ptr, ptr, ptr, ptr, kb.KATA_FP32, 1, 1, 64, 16, 16, 0, None)
        assert st == kb.KATA_ERR_INVALID_ARG
    finally:
        cudart.cudaFree(ptr)
    q, k, v = _inputs(1, 1, 64, 16, 16, torch.float32)  # the fp32 path keeps per-chunk states
    assert kb.kata_chunked_workspace_bytes(torch.float32, 1, 1, 64, 16, 16, 32) > 16
    with pytest.raises(kb.KataError) as ei:
        kb.kata_forward_chunked(q, k, v, 32, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert ei.value.status == kb.KATA_ERR_WORKSPACE


# ---------------------------------------------------------------- the five workloads

_CACHE = {}


def _workload(i):
    w = inputs.WORKLOADS[i]
    if w.name not in _CACHE:
        _CACHE.clear()
        _CACHE[w.name] = inputs.make(w, "cuda")
    return w, _CACHE[w.name]


def test_workload_c1_all_forms():
    w, (q, k, v) = _workload(0)
    qq, kk, vv = f64(q), f64(k), f64(v)
    ref = oracle.forward_plain(qq, kk, vv)
    np.testing.assert_allclose(oracle.forward_recurrent(qq, kk, vv)[0], ref, atol=1e-12)
    np.testing.assert_allclose(oracle.forward_chunked(qq, kk, vv, w.C, 1)[0], ref, atol=1e-12)
    assert_close(f64(kb.kata_forward_quadratic(q, k, v, C=w.C)), ref, torch.float32, "c1 quadratic")
    for mode in (0, 1):
        assert_close(f64(kb.kata_forward_chunked(q, k, v, w.C, mode)), ref, torch.float32, "c1 chunked")


def test_workload_c2_quadratic_and_chunked():
    w, (q, k, v) = _workload(1)
    ref = oracle.forward_plain(f64(q), f64(k), f64(v))
    oq = kb.kata_forward_quadratic(q, k, v, C=w.C)
    oc = kb.kata_forward_chunked(q, k, v, w.C, kb.KATA_SCAN_TREE)
    assert_close(f64(oq), ref, torch.bfloat16, "c2 quadratic")
    assert_close(f64(oc), ref, torch.bfloat16, "c2 chunked")


def _check_sampled(w, q, k, v, o, what):
    """Sampled rows (32 per head in the last quarter of T among them) against
    the plain definition, gated per head and row by row; then the convex
    output gate at every position, with a slack of the row's own size."""
    bh, t = sample_rows(w.B, w.H, w.T, w.C)
    ref = oracle.forward_plain_rows(f64(q), f64(k), f64(v), bh, t)
    got = f64(o).reshape(w.B * w.H, w.T, w.dv)[bh, t]
    err = rows_error(got, ref)
    assert err <= TOL[torch.bfloat16], f"{what}: sampled-row error {err:.3e}"
    per_row = row_errors(got, ref)
    worst = int(np.argmax(per_row))
    print(f"{what}: worst per-row error {per_row[worst]:.3e} at head {bh[worst]} t {t[worst]}; "
          f"worst over the last quarter {per_row[t >= w.T - w.T // 4].max():.3e}")
    assert per_row[worst] <= TOL[torch.bfloat16], \
        f"{what}: row t={t[worst]} of head {bh[worst]} has error {per_row[worst]:.3e}"
    # convex output gate at every position: o_t within the hull of v_{<=t},
    # up to the tolerance of the row's own largest output
    vf = v.float()
    lo = torch.cummin(vf, dim=2).values
    hi = torch.cummax(vf, dim=2).values
    of = o.float()
    slack = TOL[torch.bfloat16] * of.abs().amax(dim=-1, keepdim=True)
    assert bool(((of >= lo - slack) & (of <= hi + slack)).all()), f"{what}: outside the convex hull"
    return err


def _traced(fn):
    """Run fn() under the library's launch trace; return (result, kernel names)."""
    kb.kata_trace_start(4096)
    try:
        out = fn()
        torch.cuda.synchronize()
    finally:
        names = [name for name, _ in kb.kata_trace_stop()]
    return out, names


def test_workload_c3_sequential_vs_tree_and_chunk_sizes():
    """The 16-head workload as one call per head: a single head leaves
    clusters free, so the forward cuts the sequence into segments whose start
    states come from the selected inter-chunk prefix (sequential or
    log-depth).  Both modes are checked against the plain definition, and
    the launch trace shows that they ran different scan kernels."""
    w, (q, k, v) = _workload(2)
    outs, scans = {}, {}
    for mode in (kb.KATA_SCAN_SEQUENTIAL, kb.KATA_SCAN_TREE):
        o = torch.empty_like(v)

        def run():
            for h in range(w.H):
                kb.kata_forward_chunked(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1], w.C, mode, o=o[:, h:h + 1])
            return o

        _, names = _traced(run)
        scans[mode] = sorted({n for n in names if n.startswith("scan")})
        assert any(n.startswith("chunk_states") or n.startswith("states") for n in names), names
        _check_sampled(w, q, k, v, o, f"c3 per-head mode {mode}")
        outs[mode] = o
    assert scans[kb.KATA_SCAN_SEQUENTIAL] and scans[kb.KATA_SCAN_TREE]
    assert scans[kb.KATA_SCAN_SEQUENTIAL] != scans[kb.KATA_SCAN_TREE], scans
    o_all = kb.kata_forward_chunked(q, k, v, w.C, kb.KATA_SCAN_TREE)
    _check_sampled(w, q, k, v, o_all, "c3 all heads")
    for C in (32, 128):
        o_c = kb.kata_forward_chunked(q, k, v, C, kb.KATA_SCAN_TREE)
        assert head_errors(f64(o_c), f64(o_all)).max() <= TOL[torch.bfloat16]
    oq = kb.kata_forward_quadratic(q, k, v)
    _check_sampled(w, q, k, v, oq, "c3 quadratic")


def test_workload_c4_headline():
    w, (q, k, v) = _workload(3)
    o = kb.kata_forward_chunked(q, k, v, w.C, kb.KATA_SCAN_TREE)
    kb.kata_get_device_status()
    _check_sampled(w, q, k, v, o, "c4 chunked")


def test_workload_c5_codebook():
    w, (q, k, v) = _workload(4)
    o = kb.kata_forward_chunked(q, k, v, w.C, kb.KATA_SCAN_TREE)
    kb.kata_get_device_status()
    _check_sampled(w, q, k, v, o, "c5 chunked")


def test_workload_c3_chunk_state_scan_modes():
    w, (q, k, v) = _workload(2)
    Sa, za = kb.kata_chunk_state_scan(k, v, w.C, kb.KATA_SCAN_SEQUENTIAL)
    Sb, zb = kb.kata_chunk_state_scan(k, v, w.C, kb.KATA_SCAN_TREE)
    torch.cuda.synchronize()
    assert torch.count_nonzero(Sa[:, :, 0]) == 0
    rel = ((Sa - Sb).abs().amax() / Sa.abs().amax()).item()
    assert rel <= 1e-5
    # last prefix + last chunk state == full state: check one head against the oracle
    kk = f64(k[:, :1, : w.T - w.C])
    vv = f64(v[:, :1, : w.T - w.C])
    _, S_ref, z_ref = oracle.forward_recurrent(kk, kk, vv)
    assert _state_err(Sa[:, :1, -1], S_ref) <= TOL[torch.bfloat16]
    assert _state_err(za[:, :1, -1], z_ref) <= TOL[torch.bfloat16]


def test_chunked_calls_on_concurrent_streams():
    # single-head calls issued back to back on separate streams (the library's
    # second stream and its events are shared by all of them) match one call
    # over all heads and the plain definition
    q, k, v = _inputs(1, 4, 1000, 64, 64, torch.bfloat16, seed=11)
    whole = kb.kata_forward_chunked(q, k, v, 128, kb.KATA_SCAN_TREE)
    o = torch.empty_like(v)
    streams = [torch.cuda.Stream() for _ in range(4)]
    cur = torch.cuda.current_stream()
    for h, s in enumerate(streams):
        s.wait_stream(cur)
        kb.kata_forward_chunked(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1], 128, kb.KATA_SCAN_TREE,
                                o=o[:, h:h + 1], stream=s)
    for s in streams:
        cur.wait_stream(s)
    torch.cuda.synchronize()
    ref = oracle.forward_plain(f64(q), f64(k), f64(v))
    assert_close(f64(o), ref, torch.bfloat16, "per-head calls")
    assert_close(f64(whole), ref, torch.bfloat16, "one call")


def test_chunked_calls_from_host_threads():
    # the same single-head calls issued from four host threads at once
    import threading
    q, k, v = _inputs(1, 4, 700, 64, 64, torch.bfloat16, seed=12)
    ref = oracle.forward_plain(f64(q), f64(k), f64(v))
    o = torch.empty_like(v)
    streams = [torch.cuda.Stream() for _ in range(4)]
    torch.cuda.synchronize()
    errors = []

    def run(h):
        try:
            for _ in range(3):
                kb.kata_forward_chunked(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1], 128, kb.KATA_SCAN_TREE,
                                        o=o[:, h:h + 1], stream=streams[h])
            streams[h].synchronize()
        except Exception as exc:  # noqa: BLE001 - reported below
            errors.append(exc)

    threads = [threading.Thread(target=run, args=(h,)) for h in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    assert_close(f64(o), ref, torch.bfloat16, "calls from host threads")
