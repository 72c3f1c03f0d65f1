"""GPU parity of the backward (kata_backward) against the fp64 oracle's
gradient of the plain definition."""
import numpy as np
import pytest
import torch

import oracle
from kernelized_linear_attention_03_b300 import binding as kb
from kernelized_linear_attention_03_b300 import inputs
from tests.parity import f64

pytestmark = pytest.mark.gpu
DNAME = {torch.float32: "fp32", torch.bfloat16: "bf16"}
# fp32: the gradient sums cancel (dO.v_s - dO.o_t); bf16: output rounding 2^-8 plus that
GRAD_TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def _case(B, H, T, p, dv, dtype, seed):
    q, k, v = inputs.make(inputs.small(B, H, T, p, dv, 32, DNAME[dtype], "raw", seed), "cuda")
    g = torch.Generator(device="cpu").manual_seed(seed)
    dO = torch.randn(v.shape, generator=g, dtype=torch.float64).to(dtype).cuda()
    return q, k, v, dO


def _term_scale(x, y, v, dO, rows_are_queries):
    """Per-row size of one gradient term, |dO| |v| / (||x_r|| c_r), with c_r the
    largest |qh_t . kh_s| the row r takes part in (x = q, y = k for dq rows;
    x = k, y = q for dk rows).  The chain rule's dc_ts = 2 c (dO.v_s - dO.o_t)/D_t
    is of that size, and where the exact gradient cancels (T = 1: o = v
    whatever q and k, so dq = dk = 0) rounding leaves noise of that order."""
    B, H, T, _ = x.shape
    xh = x / np.maximum(np.linalg.norm(x, axis=-1, keepdims=True), 1e-300)
    yh = y / np.maximum(np.linalg.norm(y, axis=-1, keepdims=True), 1e-300)
    c = np.abs(np.einsum("bhtp,bhsp->bhts", xh, yh))
    mask = np.tril(np.ones((T, T), bool)) if rows_are_queries else np.triu(np.ones((T, T), bool))
    cmax = np.where(mask, c, 0.0).max(axis=-1)
    g = np.abs(dO).max(axis=(2, 3))[..., None] * np.abs(v).max(axis=(2, 3))[..., None]
    nrm = np.linalg.norm(x, axis=-1)
    return g / np.maximum(nrm * cmax, 1e-300)


def grad_errors(got, ref, row_floor):
    """Per head: max over rows of |got - ref| / max(max |ref| of the head,
    the row's term size)."""
    B, H = ref.shape[:2]
    d = np.abs(got - ref).max(axis=-1)
    m = np.abs(ref).reshape(B, H, -1).max(axis=-1)[..., None]
    return (d / np.maximum(m, row_floor)).reshape(B * H, -1).max(axis=1)


def _check(q, k, v, dO, dtype, form="chunked"):
    dq, dk, dv = kb.kata_backward(q, k, v, dO, form=form)
    torch.cuda.synchronize()
    qq, kk, vv, gg = f64(q), f64(k), f64(v), f64(dO)
    ref = oracle.backward_plain(qq, kk, vv, gg)
    floors = (_term_scale(qq, kk, vv, gg, True), _term_scale(kk, qq, vv, gg, False),
              np.zeros(vv.shape[:3]))
    for name, got, r, fl in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, floors):
        err = float(grad_errors(f64(got), r, fl).max())
        assert err <= GRAD_TOL[dtype], f"{name}: worst-head relative error {err:.3e}"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("p,dv", [(16, 16), (32, 64), (64, 32), (64, 64)])
@pytest.mark.parametrize("T", [1, 37, 130])
@pytest.mark.parametrize("form", ["chunked", "quadratic"])
def test_backward_matches_the_oracle(dtype, p, dv, T, form):
    _check(*_case(1, 2, T, p, dv, dtype, seed=T + p + dv), dtype, form)


@pytest.mark.parametrize("form", ["chunked", "quadratic"])
def test_backward_zero_vectors(form):
    q, k, v, dO = _case(1, 1, 90, 16, 16, torch.float32, seed=4)
    k[0, 0, 3] = 0
    q[0, 0, 70] = 0
    dq, dk, dv = kb.kata_backward(q, k, v, dO, form=form)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dk[0, 0, 3]) == 0 and torch.count_nonzero(dq[0, 0, 70]) == 0
    _check(q, k, v, dO, torch.float32, form)


def test_chunked_backward_long_sequence():
    """Many backward chunks (the reverse prefix over 33 chunks) on several heads."""
    _check(*_case(2, 2, 2100, 32, 32, torch.float32, seed=8), torch.float32, "chunked")


def test_chunked_backward_bf16_prefix_states_on_tensor_cores():
    """bf16: the forward's prefix states at the backward's 64-token chunks come
    from the tensor-core chunk-state kernel in prefix mode (every chunk's
    exclusive prefix in one pass, no scan); 33 chunks on several heads, a
    ragged last chunk, against the oracle's gradients."""
    kb.kata_trace_start(4096)
    try:
        _check(*_case(2, 2, 2100, 32, 32, torch.bfloat16, seed=8), torch.bfloat16, "chunked")
    finally:
        names = {name for name, _ in kb.kata_trace_stop()}
    assert "states_tc" in names and "chunk_states_simt" not in names, names
