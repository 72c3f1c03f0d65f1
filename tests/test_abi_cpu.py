"""The C-ABI library builds, loads and exports every symbol include/kata.h
declares, and rejects bad arguments on the host before touching a GPU.
No compute call is made here (no GPU in this process)."""
import ctypes
import os
import re
import subprocess

import pytest

from kernelized_linear_attention_03_b300 import build as kbuild
from kernelized_linear_attention_03_b300 import binding as kb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kata.h")


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kb.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"KATA_API\s+[\w\s\*]+?\b(kata_\w+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_symbols() == sorted(kb.SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", kb.LIB_PATH], check=True,
                         capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(kata_\w+)", out))
    for name in declared_symbols():
        assert name in exported, name
        assert hasattr(lib, name)


def test_library_is_built_for_sm103a(lib):
    assert "arch=compute_103a,code=sm_103a" in " ".join(kbuild.FLAGS)


def test_packed_dim_and_status_strings(lib):
    assert [kb.kata_packed_dim(p) for p in (16, 32, 64)] == [136, 528, 2080]
    assert kb.kata_packed_dim(-1) == -1
    for code in range(6):
        assert kb.kata_status_string(code).startswith("KATA_")
    assert kb.kata_status_string(99) == "KATA_ERR_UNKNOWN"


def test_workspace_query(lib):
    # fp32 states per chunk: n*dv + n floats, each region 256-byte aligned.
    got = kb.kata_chunked_workspace_bytes(kb.KATA_FP32, 1, 1, 256, 16, 16, 32)
    nc, n = 8, 136
    expect = ((nc * n * 16 * 4 + 255) // 256) * 256 + ((nc * n * 4 + 255) // 256) * 256
    assert got >= expect
    assert kb.kata_chunked_workspace_bytes(kb.KATA_BF16, 1, 1, 256, 17, 16, 32) == 0
    assert kb.kata_chunked_workspace_bytes(kb.KATA_BF16, 0, 1, 256, 16, 16, 32) == 0


NULL = None
MISALIGNED = ctypes.c_void_p(0x1001)


def _quad(lib, dt=kb.KATA_BF16, B=1, H=1, T=8, p=16, dv=16, C=0, ptr=NULL):
    return lib.kata_forward_quadratic(ptr, ptr, ptr, ptr, dt, B, H, T, p, dv, C, None)


def test_quadratic_argument_errors(lib):
    assert _quad(lib, dt=7) == kb.KATA_ERR_INVALID_ARG
    assert _quad(lib, T=-1) == kb.KATA_ERR_INVALID_ARG
    assert _quad(lib, p=8) == kb.KATA_ERR_UNSUPPORTED
    assert _quad(lib, dv=128) == kb.KATA_ERR_UNSUPPORTED
    assert _quad(lib, C=48) == kb.KATA_ERR_UNSUPPORTED
    assert _quad(lib, B=300, H=300) == kb.KATA_ERR_UNSUPPORTED
    assert _quad(lib, ptr=NULL) == kb.KATA_ERR_INVALID_ARG
    assert _quad(lib, ptr=MISALIGNED) == kb.KATA_ERR_INVALID_ARG
    # empty input: nothing to do, pointers unused
    assert _quad(lib, T=0) == kb.KATA_OK
    assert _quad(lib, B=0) == kb.KATA_OK


def _chunked(lib, mode=1, C=32, T=64, S0=NULL, z0=NULL, Sf=NULL, zf=NULL, ptr=NULL, ws=NULL,
             ws_bytes=0, B=1, p=16, dv=16):
    return lib.kata_forward_chunked(ptr, ptr, ptr, ptr, kb.KATA_BF16, B, 1, T, p, dv, C, mode, S0,
                                    z0, Sf, zf, ws, ws_bytes, None)


def test_chunked_argument_errors(lib):
    assert _chunked(lib, C=16) == kb.KATA_ERR_UNSUPPORTED
    assert _chunked(lib, C=0) == kb.KATA_ERR_UNSUPPORTED
    assert _chunked(lib, mode=2) == kb.KATA_ERR_INVALID_ARG
    assert _chunked(lib, S0=MISALIGNED) == kb.KATA_ERR_INVALID_ARG   # S0 without z0
    assert _chunked(lib, Sf=MISALIGNED) == kb.KATA_ERR_INVALID_ARG   # S_final without z_final
    assert _chunked(lib, S0=MISALIGNED, z0=MISALIGNED) == kb.KATA_ERR_INVALID_ARG
    assert _chunked(lib, ptr=NULL) == kb.KATA_ERR_INVALID_ARG
    assert _chunked(lib, p=48) == kb.KATA_ERR_UNSUPPORTED
    assert _chunked(lib, B=0) == kb.KATA_OK
    assert _chunked(lib, T=0) == kb.KATA_OK                        # no final state asked


def test_state_scan_and_scan_argument_errors(lib):
    f = lib.kata_chunk_state_scan
    assert f(NULL, NULL, kb.KATA_BF16, 1, 1, 64, 16, 16, 32, 1, NULL, NULL, None) == kb.KATA_ERR_INVALID_ARG
    assert f(NULL, NULL, kb.KATA_BF16, 1, 1, 64, 16, 16, 40, 1, NULL, NULL, None) == kb.KATA_ERR_UNSUPPORTED
    assert f(NULL, NULL, kb.KATA_BF16, 1, 1, 64, 16, 16, 32, 3, NULL, NULL, None) == kb.KATA_ERR_INVALID_ARG
    assert f(NULL, NULL, kb.KATA_BF16, 1, 1, 0, 16, 16, 32, 1, NULL, NULL, None) == kb.KATA_OK
    g = lib.kata_scan_states
    assert g(NULL, NULL, NULL, NULL, 1, 1, 4, 3, 2, 0, None) == kb.KATA_ERR_INVALID_ARG
    assert g(NULL, NULL, NULL, NULL, 1, 1, -4, 3, 2, 0, None) == kb.KATA_ERR_INVALID_ARG
    assert g(NULL, NULL, NULL, NULL, 1, 1, 4, 3, 2, 5, None) == kb.KATA_ERR_INVALID_ARG
    assert g(NULL, NULL, NULL, NULL, 1, 1, 0, 3, 2, 0, None) == kb.KATA_OK


def test_binding_rejects_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 1, 4, 16, dtype=torch.bfloat16)
    v = torch.zeros(1, 1, 4, 16, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        kb.kata_forward_quadratic(q, q, v, o=v.clone())


def _dec(lib, dt=kb.KATA_BF16, B=1, H=1, p=16, dv=16, ptr=NULL):
    return lib.kata_decode_step(ptr, ptr, ptr, ptr, dt, B, H, p, dv, ptr, ptr, None)


def test_decode_argument_errors(lib):
    assert _dec(lib, dt=3) == kb.KATA_ERR_INVALID_ARG
    assert _dec(lib, B=-1) == kb.KATA_ERR_INVALID_ARG
    assert _dec(lib, p=48) == kb.KATA_ERR_UNSUPPORTED
    assert _dec(lib, dv=8) == kb.KATA_ERR_UNSUPPORTED
    assert _dec(lib, B=256, H=512) == kb.KATA_ERR_UNSUPPORTED
    assert _dec(lib, ptr=NULL) == kb.KATA_ERR_INVALID_ARG
    assert _dec(lib, ptr=MISALIGNED) == kb.KATA_ERR_INVALID_ARG
    # no heads: nothing to do, pointers unused
    assert _dec(lib, B=0) == kb.KATA_OK


def test_lift_dims_and_block_workspace(lib):
    L = kb
    assert kb.kata_lift_dim(L.KATA_LIFT_SIGMA, 64, 2) == 528
    assert kb.kata_lift_dim(L.KATA_LIFT_MULTI, 64, 2) == 1056
    assert kb.kata_lift_dim(L.KATA_LIFT_SIGMA, 16, 4) == 10
    assert kb.kata_lift_dim(L.KATA_LIFT_FULL, 64, 1) == 2080
    assert kb.kata_lift_dim(L.KATA_LIFT_FULL, 64, 2) == -1
    assert kb.kata_lift_dim(L.KATA_LIFT_SIGMA, 64, 3) == -1
    assert kb.kata_lift_dim(5, 64, 2) == -1
    # chunk states [BH, NC, n, dv] and [BH, NC, n] fp32, each 256-byte aligned
    got = kb.kata_chunked_block_workspace_bytes(kb.KATA_FP32, L.KATA_LIFT_MULTI, 2, 1, 2, 100, 16, 16, 32)
    nc, n = 4, 72
    assert got == ((2 * nc * n * 16 * 4 + 255) // 256) * 256 + ((2 * nc * n * 4 + 255) // 256) * 256
    assert kb.kata_chunked_block_workspace_bytes(kb.KATA_FP32, L.KATA_LIFT_SIGMA, 3, 1, 1, 64, 16, 16, 32) == 0


def test_block_argument_errors(lib):
    P = None
    f = lib.kata_forward_chunked_block
    args = lambda fam, g, B=1: (P, P, P, P, kb.KATA_FP32, B, 1, 8, 16, 16, 32, fam, g, 0, P, P, P, P, P, 0, P)  # noqa
    assert f(*args(9, 2)) == kb.KATA_ERR_INVALID_ARG
    assert f(*args(kb.KATA_LIFT_SIGMA, 0)) == kb.KATA_ERR_INVALID_ARG
    assert f(*args(kb.KATA_LIFT_SIGMA, 3)) == kb.KATA_ERR_UNSUPPORTED
    assert f(*args(kb.KATA_LIFT_FULL, 2)) == kb.KATA_ERR_UNSUPPORTED
    assert f(*args(kb.KATA_LIFT_MULTI, 2)) == kb.KATA_ERR_INVALID_ARG  # null pointers
    assert f(*args(kb.KATA_LIFT_MULTI, 2, B=0)) == kb.KATA_OK
    q = lib.kata_forward_quadratic_block
    assert q(P, P, P, P, kb.KATA_BF16, 1, 1, 8, 16, 16, kb.KATA_LIFT_SIGMA, 32, P) == kb.KATA_ERR_UNSUPPORTED
    assert q(P, P, P, P, kb.KATA_BF16, 0, 1, 8, 16, 16, kb.KATA_LIFT_SIGMA, 2, P) == kb.KATA_OK
    d = lib.kata_decode_step_block
    assert d(P, P, P, P, kb.KATA_BF16, 1, 1, 16, 16, 4, 2, P, P, P) == kb.KATA_ERR_INVALID_ARG
    assert d(P, P, P, P, kb.KATA_BF16, 1, 1, 16, 16, kb.KATA_LIFT_MULTI, 2, P, P, P) == kb.KATA_ERR_INVALID_ARG
    assert d(P, P, P, P, kb.KATA_BF16, 0, 1, 16, 16, kb.KATA_LIFT_MULTI, 2, P, P, P) == kb.KATA_OK


def test_backward_workspace_and_argument_errors(lib):
    assert kb.load().kata_backward_quadratic_workspace_bytes(1, 2, 100) == 2 * ((2 * 100 * 4 + 255) // 256) * 256
    assert kb.load().kata_backward_quadratic_workspace_bytes(0, 2, 100) == 0
    r = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert kb.load().kata_backward_chunked_workspace_bytes(1, 2, 100, 16, 16) == (
        r(2 * 2 * 136 * 16 * 4) + r(2 * 2 * 136 * 4) + 2 * r(2 * 100 * 4))
    f = lib.kata_backward_quadratic
    P = None
    assert f(P, P, P, P, P, P, P, 7, 1, 1, 8, 16, 16, P, 0, P) == kb.KATA_ERR_INVALID_ARG
    assert f(P, P, P, P, P, P, P, kb.KATA_FP32, 1, 1, 8, 24, 16, P, 0, P) == kb.KATA_ERR_UNSUPPORTED
    assert f(P, P, P, P, P, P, P, kb.KATA_FP32, 1, 1, 8, 16, 16, P, 0, P) == kb.KATA_ERR_INVALID_ARG
    assert f(P, P, P, P, P, P, P, kb.KATA_FP32, 1, 1, 0, 16, 16, P, 0, P) == kb.KATA_OK


def test_gated_argument_errors(lib):
    P = None
    f = lib.kata_forward_chunked_gated
    assert f(P, P, P, P, P, 9, 1, 1, 8, 16, 16, 32, P, P, P, P, P, 0, P) == kb.KATA_ERR_INVALID_ARG
    assert f(P, P, P, P, P, kb.KATA_FP32, 1, 1, 8, 16, 16, 48, P, P, P, P, P, 0, P) == kb.KATA_ERR_UNSUPPORTED
    assert f(P, P, P, P, P, kb.KATA_FP32, 1, 1, 8, 16, 16, 32, P, P, P, P, P, 0, P) == kb.KATA_ERR_INVALID_ARG
    assert f(P, P, P, P, P, kb.KATA_FP32, 0, 1, 8, 16, 16, 32, P, P, P, P, P, 0, P) == kb.KATA_OK
    d = lib.kata_decode_step_gated
    assert d(P, P, P, P, P, kb.KATA_FP32, 1, 1, 16, 16, P, P, P) == kb.KATA_ERR_INVALID_ARG
    assert d(P, P, P, P, P, kb.KATA_FP32, 0, 1, 16, 16, P, P, P) == kb.KATA_OK
    # states [BH, NC, n, dv] + [BH, NC, n] + chunk decays [BH, NC] + token decays [BH, T], each 256-byte aligned
    got = lib.kata_chunked_gated_workspace_bytes(kb.KATA_FP32, 1, 2, 100, 16, 16, 32)
    r = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert got == r(2 * 4 * 136 * 16 * 4) + r(2 * 4 * 136 * 4) + r(2 * 4 * 4) + r(2 * 100 * 4)
