"""The full-size parity gate can fail: a planted error in late rows, of the
kind a chunked kernel could make, is rejected by the per-row gate although
the per-sample normwise gate alone would accept it.

The planted mistake is made in the oracle's own rows, on the CPU: for rows
past T/2 the inter-chunk part of the numerator (every key before the row's
chunk) is scaled by 0.9 while the denominator is kept, which is what a
kernel that lost a tenth of its running state in the readout would give.
"""
import numpy as np
import torch

import oracle
from kernelized_linear_attention_03_b300 import inputs
from tests.parity import TOL, row_errors, rows_error, sample_rows


def _planted_rows(q, k, v, bh, t, C, T):
    """Rows (bh, t) with the inter-chunk numerator of rows past T/2 scaled by 0.9."""
    out = oracle.forward_plain_rows(q, k, v, bh, t)
    for r in np.nonzero(t > T // 2)[0]:
        start = (int(t[r]) // C) * C
        h = int(bh[r])
        vh = v[:, h:h + 1].copy()
        vh[:, :, :start] *= 0.9  # every key before the row's chunk
        out[r] = oracle.forward_plain_rows(q[:, h:h + 1], k[:, h:h + 1], vh, np.array([0]), t[r:r + 1])[0]
    return out


def test_per_row_gate_rejects_a_scaled_inter_chunk_part():
    w = inputs.WORKLOADS[2]  # 16384 tokens, p = dv = 64, bf16, C = 64
    q, k, v = (x[:, :2].contiguous() for x in inputs.make(w, "cpu"))
    q, k, v = (x.double().numpy() for x in (q, k, v))
    H = 2
    bh, t = sample_rows(1, H, w.T, w.C, per_head=4, seed=1, late=12)
    ref = oracle.forward_plain_rows(q, k, v, bh, t)
    # the correct rows, rounded to the output dtype, pass both gates
    good = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    assert rows_error(good, ref) <= TOL[torch.bfloat16]
    assert row_errors(good, ref).max() <= TOL[torch.bfloat16]
    bad = _planted_rows(q, k, v, bh, t, 128, w.T)
    late = t > w.T // 2
    assert late.sum() >= 12
    # the per-sample normwise gate cannot see it: the sample's largest output
    # is an early row, about 50 times larger than the late rows ...
    assert rows_error(bad, ref) <= TOL[torch.bfloat16]
    # ... but every late row is off by about 10 % of its own size
    per_row = row_errors(bad, ref)
    assert per_row[late].min() > 4 * TOL[torch.bfloat16]
    assert per_row[~late].max() == 0.0
