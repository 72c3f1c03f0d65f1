"""GPU parity of the recurrent decode step (kata_decode_step) against the fp64
oracle's token recurrence, taken one token at a time from a given state.

The start states come from the oracle (its recurrence over a prefix of the
same seeded tokens, rounded to fp32) or from the library's own forward; the
expected values always come from the oracle alone.
"""
import numpy as np
import pytest
import torch

import oracle
from kernelized_linear_attention_03_b300 import binding as kb
from kernelized_linear_attention_03_b300 import inputs
from tests.parity import TOL, assert_close, f64

pytestmark = pytest.mark.gpu
DTYPES = [torch.float32, torch.bfloat16]
DNAME = {torch.float32: "fp32", torch.bfloat16: "bf16"}
STATE_TOL = 1e-6  # fp32 state: one rounded FMA per element on top of the start state


def _tokens(B, H, T, p, dv, dtype, seed, kind="raw"):
    return inputs.make(inputs.small(B, H, T, p, dv, 32, DNAME[dtype], kind, seed), "cuda")


def _oracle_state(q, k, v, T0):
    """The oracle's (S, z) after the first T0 tokens, as fp32 CUDA tensors."""
    B, H, _, p = q.shape
    dv, n = v.shape[-1], p * (p + 1) // 2
    if T0 == 0:
        return (torch.zeros(B, H, n, dv, device="cuda"), torch.zeros(B, H, n, device="cuda"))
    _, S, z = oracle.forward_recurrent(f64(q[:, :, :T0]), f64(k[:, :, :T0]), f64(v[:, :, :T0]))
    return torch.from_numpy(S).float().cuda(), torch.from_numpy(z).float().cuda()


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


def _step_and_check(q, k, v, T0, dtype):
    """Decode token T0 from the oracle's state after T0 tokens; compare o, S, z."""
    S, z = _oracle_state(q, k, v, T0)
    S_in, z_in = f64(S), f64(z)
    qt, kt, vt = (x[:, :, T0].contiguous() for x in (q, k, v))
    o = kb.kata_decode_step(qt, kt, vt, S, z)
    torch.cuda.synchronize()
    o_ref, S_ref, z_ref = oracle.forward_recurrent(f64(qt)[:, :, None], f64(kt)[:, :, None],
                                                   f64(vt)[:, :, None], S_in, z_in)
    assert_close(f64(o)[:, :, None], o_ref, dtype, "decode o")
    assert _rel(f64(S), S_ref) <= STATE_TOL
    assert _rel(f64(z), z_ref) <= STATE_TOL


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("p", [16, 32, 64])
@pytest.mark.parametrize("dv", [16, 32, 64])
def test_decode_step_from_a_prefix_state(dtype, p, dv):
    # one head (the head's rows split over the most CTAs) and a few heads
    for B, H, T0 in ((1, 1, 9), (2, 3, 20)):
        q, k, v = _tokens(B, H, T0 + 1, p, dv, dtype, seed=p + dv + T0)
        _step_and_check(q, k, v, T0, dtype)


@pytest.mark.parametrize("dtype", DTYPES)
def test_decode_step_many_heads(dtype):
    # enough heads that every head runs on a single CTA
    q, k, v = _tokens(8, 40, 5, 32, 64, dtype, seed=11)
    _step_and_check(q, k, v, 4, dtype)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("p,dv", [(16, 16), (32, 64), (64, 64)])
def test_decode_steps_from_zero_equal_the_plain_definition(dtype, p, dv):
    B, H, T = 2, 2, 24
    q, k, v = _tokens(B, H, T, p, dv, dtype, seed=5 * p + dv)
    n = p * (p + 1) // 2
    S = torch.zeros(B, H, n, dv, device="cuda")
    z = torch.zeros(B, H, n, device="cuda")
    rows = [kb.kata_decode_step(q[:, :, t].contiguous(), k[:, :, t].contiguous(), v[:, :, t].contiguous(), S, z)
            for t in range(T)]
    o = torch.stack(rows, dim=2)
    torch.cuda.synchronize()
    assert_close(f64(o), oracle.forward_plain(f64(q), f64(k), f64(v)), dtype, "decode steps")


@pytest.mark.parametrize("dtype,p,dv,C", [(torch.float32, 16, 32, 32), (torch.bfloat16, 64, 64, 128),
                                          (torch.bfloat16, 32, 32, 64)])
def test_decode_continues_a_forward_and_seeds_the_next(dtype, p, dv, C):
    """forward(T0) -> S_final -> decode token T0 -> state as S0 of forward(T1):
    every output row equals the plain definition over the whole sequence."""
    B, H, T0, T1 = 1, 2, 200, 70
    T = T0 + 1 + T1
    q, k, v = _tokens(B, H, T, p, dv, dtype, seed=p + C)
    n = p * (p + 1) // 2
    S = torch.empty(B, H, n, dv, device="cuda")
    z = torch.empty(B, H, n, device="cuda")
    part = lambda x, a, b: x[:, :, a:b].contiguous()  # noqa: E731
    o0, _, _ = kb.kata_forward_chunked(part(q, 0, T0), part(k, 0, T0), part(v, 0, T0), C, S_final=S, z_final=z)
    o1 = kb.kata_decode_step(q[:, :, T0].contiguous(), k[:, :, T0].contiguous(), v[:, :, T0].contiguous(), S, z)
    o2 = kb.kata_forward_chunked(part(q, T0 + 1, T), part(k, T0 + 1, T), part(v, T0 + 1, T), C, S0=S, z0=z)
    torch.cuda.synchronize()
    o = torch.cat([o0, o1[:, :, None], o2], dim=2)
    assert_close(f64(o), oracle.forward_plain(f64(q), f64(k), f64(v)), dtype, "forward/decode/forward")


@pytest.mark.parametrize("dtype", DTYPES)
def test_decode_degenerate_tokens(dtype):
    B, H, p, dv = 1, 3, 32, 32
    n = p * (p + 1) // 2
    q, k, v = _tokens(B, H, 1, p, dv, dtype, seed=2)
    q, k, v = q[:, :, 0].contiguous(), k[:, :, 0].contiguous(), v[:, :, 0].contiguous()
    k[:, 0] = 0  # head 0: zero key on an empty state -> nothing added, zero denominator
    q[:, 1] = 0  # head 1: zero query -> zero row, state still updated
    S = torch.zeros(B, H, n, dv, device="cuda")
    z = torch.zeros(B, H, n, device="cuda")
    o = kb.kata_decode_step(q, k, v, S, z)
    torch.cuda.synchronize()
    assert torch.count_nonzero(S[:, 0]) == 0 and torch.count_nonzero(z[:, 0]) == 0
    assert torch.count_nonzero(o[:, 0]) == 0 and torch.count_nonzero(o[:, 1]) == 0
    assert torch.count_nonzero(z[:, 1]) > 0
    # head 2: one token on an empty state reads back its own value (T = 1 gives o = v)
    assert_close(f64(o[:, 2])[:, None, None], f64(v[:, 2])[:, None, None], dtype, "o = v")


def test_decode_empty_and_bad_arguments():
    assert kb.load().kata_decode_step(None, None, None, None, kb.KATA_FP32, 0, 2, 16, 16, None, None, None) == kb.KATA_OK
    q = torch.randn(1, 1, 16, device="cuda")
    v = torch.randn(1, 1, 16, device="cuda")
    buf = torch.zeros(136 * 16 + 136, device="cuda")
    lib = kb.load()
    # z inside S: rejected before launch
    st = lib.kata_decode_step(q.data_ptr(), q.data_ptr(), v.data_ptr(), v.data_ptr(), kb.KATA_FP32, 1, 1, 16, 16,
                              buf.data_ptr(), buf.data_ptr() + 64, None)
    assert st == kb.KATA_ERR_INVALID_ARG
    # misaligned state pointer
    st = lib.kata_decode_step(q.data_ptr(), q.data_ptr(), v.data_ptr(), v.data_ptr(), kb.KATA_FP32, 1, 1, 16, 16,
                              buf.data_ptr() + 4, buf.data_ptr() + 136 * 16 * 4, None)
    assert st == kb.KATA_ERR_INVALID_ARG


@pytest.mark.slow
def test_decode_full_batch_p64_bf16():
    """A serving-size decode batch (B = 64, H = 16, p = dv = 64, bf16; 545 MB of
    state, above L2), in the launch configuration the benchmark times."""
    B, H, p, dv, T0 = 64, 16, 64, 64, 3
    q, k, v = _tokens(B, H, T0 + 1, p, dv, torch.bfloat16, seed=21, kind="gaussian")
    _step_and_check(q, k, v, T0, torch.bfloat16)
