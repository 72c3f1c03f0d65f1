"""Shared helpers of the GPU parity tests: tolerance metric and conversions.

Tolerance (per head, as the benchmark definition states "max relative
error"): err_h = max_i |o_i - r_i| / max_i |r_i| over the head's outputs,
gated at 1e-5 for fp32 inputs and 2e-2 for bf16 inputs (fp32 accumulate,
bf16 output rounding included); the worst head is reported.

At long T the outputs shrink like 1/sqrt(t) (a convex combination of ever
more values), so a head's largest output comes from its first rows and the
per-head gate alone cannot see a late row that is wrong.  Sampled rows at
full size are therefore also gated row by row: for every row,
max_j |o_tj - r_tj| / max_j |r_tj| within the same tolerance.
"""
import numpy as np
import torch

TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-2}


def f64(t):
    """Exact fp64 copy of a (CPU or CUDA) tensor's values."""
    return t.detach().to("cpu", torch.float64).numpy()


def head_errors(o, ref):
    """Per-head normwise max relative error of o against ref, both [B,H,T,dv]."""
    o = np.asarray(o, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    B, H = ref.shape[:2]
    d = np.abs(o - ref).reshape(B * H, -1).max(axis=1)
    m = np.abs(ref).reshape(B * H, -1).max(axis=1)
    return d / np.where(m > 0, m, 1.0)


def assert_close(o, ref, dtype, what=""):
    err = head_errors(o, ref)
    worst = float(err.max()) if err.size else 0.0
    assert worst <= TOL[dtype], f"{what}: worst-head max relative error {worst:.3e} > {TOL[dtype]:.0e}"
    return worst


def rows_error(o_rows, ref_rows):
    """Normwise error of sampled rows: max |o - r| / max |r| over the sample."""
    o_rows = np.asarray(o_rows, dtype=np.float64)
    ref_rows = np.asarray(ref_rows, dtype=np.float64)
    return float(np.abs(o_rows - ref_rows).max() / max(np.abs(ref_rows).max(), 1e-300))


def row_errors(o_rows, ref_rows):
    """Per-row normwise error: max_j |o - r| / max_j |r| for every row of [R, dv]."""
    o_rows = np.asarray(o_rows, dtype=np.float64)
    ref_rows = np.asarray(ref_rows, dtype=np.float64)
    m = np.abs(ref_rows).max(axis=-1)
    return np.abs(o_rows - ref_rows).max(axis=-1) / np.where(m > 0, m, 1.0)


def sample_rows(B, H, T, C, per_head=8, seed=0, max_heads=16, late=32):
    """(bh, t) sample covering first/last positions, chunk edges, random t and
    `late` random positions in the last quarter of the sequence, on every head
    or on `max_heads` heads spread over B*H (always the first and the last)."""
    rng = np.random.default_rng(seed)
    heads = np.arange(B * H)
    if B * H > max_heads:
        heads = np.unique(np.concatenate([[0, B * H - 1], rng.choice(B * H, max_heads - 2, replace=False)]))
    bh, ts = [], []
    for h in heads:
        cand = {0, T - 1, min(C - 1, T - 1), min(C, T - 1), T // 2}
        cand.update(int(x) for x in rng.integers(0, T, size=per_head))
        if late > 0:
            cand.update(int(x) for x in rng.integers(T - T // 4 - 1, T, size=late))
        for t in sorted(cand):
            bh.append(int(h))
            ts.append(t)
    return np.array(bh, dtype=np.int64), np.array(ts, dtype=np.int64)
