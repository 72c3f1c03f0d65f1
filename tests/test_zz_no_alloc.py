"""kata_forward_chunked_noalloc: the chunked forward for callers that cannot
allocate device memory (a plugin inside a runtime that owns every allocation,
code under a fixed start-up memory budget, a real-time loop that must not enter
the allocator).  Its scratch is a fixed array inside libkata.so, so the only
thing to check is that it computes what the allocating entry point computes,
call after call, and that it refuses sizes its array cannot hold.

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import numpy as np
import pytest
import torch

import oracle
from kernelized_linear_attention_03_b300 import binding as kb
from kernelized_linear_attention_03_b300 import inputs
from tests.parity import TOL, f64, head_errors

SCRATCH_BYTES = 32 << 20  # KATA_NOALLOC_SCRATCH_BYTES in include/kata.h


def _case(dtype, seed, T=300, p=32, dv=64, C=64):
    w = inputs.small(2, 2, T, p, dv, C, dtype, "raw", seed)
    return w, inputs.make(w, "cuda")


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_noalloc_matches_allocating_forward_on_two_calls(dtype):
    tdt = {"fp32": torch.float32, "bf16": torch.bfloat16}[dtype]
    for call, seed in enumerate((11, 12)):          # two calls in a row, different inputs
        w, (q, k, v) = _case(dtype, seed)
        assert kb.kata_chunked_workspace_bytes(tdt, w.B, w.H, w.T, w.p, w.dv, w.C) <= SCRATCH_BYTES
        S = torch.empty(w.B, w.H, w.n, w.dv, device="cuda")
        z = torch.empty(w.B, w.H, w.n, device="cuda")
        ref, S_ref, z_ref = kb.kata_forward_chunked(q, k, v, w.C, kb.KATA_SCAN_TREE,
                                                    S_final=S.clone(), z_final=z.clone())
        o = torch.full_like(v, float("nan"))
        o, S, z = kb.kata_forward_chunked_noalloc(q, k, v, w.C, kb.KATA_SCAN_TREE, o=o,
                                                  S_final=S, z_final=z)
        kb.kata_get_device_status()
        err = head_errors(f64(o), f64(ref)).max()
        assert err <= TOL[tdt], f"call {call}: {err:.3e}"
        # and, on its own, what the plain definition gives
        err = head_errors(f64(o), oracle.forward_plain(f64(q), f64(k), f64(v))).max()
        assert err <= TOL[tdt], f"call {call}: against the oracle {err:.3e}"
        for a, b in ((S, S_ref), (z, z_ref)):
            rel = float((a - b).abs().max() / b.abs().max())
            assert rel <= TOL[tdt], f"call {call}: state {rel:.3e}"


def test_noalloc_refuses_sizes_beyond_its_scratch():
    lib = kb.load()
    # p = dv = 64 needs n (dv+1) 4 bytes ~ 0.54 MB per chunk and head: 64 chunks exceed 32 MiB.
    B, H, T, p, dv, C = 1, 1, 64 * 128, 64, 64, 128
    assert kb.kata_chunked_workspace_bytes(kb.KATA_BF16, B, H, T, p, dv, C) > SCRATCH_BYTES
    st = lib.kata_forward_chunked_noalloc(None, None, None, None, kb.KATA_BF16, B, H, T, p, dv, C,
                                          kb.KATA_SCAN_TREE, None, None, None, None, None)
    assert st == kb.KATA_ERR_UNSUPPORTED
