"""Seeded synthetic inputs for the KATA forward: the five workloads and small cases.

This module only draws random numbers; it holds none of the attention
arithmetic, so both the fp64 oracle (through the tests) and the CUDA path can
use it.  Draws are numpy PCG64 (``default_rng(seed)``) in fp64, then rounded
to the workload dtype with torch (round-to-nearest-even for bf16).

Recipes (one seed per workload, 0 unless given):
* "gaussian" workloads: q, k, v drawn in that order, each i.i.d. N(0, 1);
  q and k rows are then put on the unit sphere (x / ||x||), which is how one
  samples uniformly from S^{p-1}; v stays N(0, 1).
* "codebook" workload (repeated-key overwrite shape): a codebook of 256
  N(0, I_p) vectors put on the sphere; key indices uniform with replacement;
  for t >= 1 the query copies the key at a uniform earlier position s < t
  (t = 0 copies k_0) plus N(0, 0.01) noise (sigma = 0.1), then is put back
  on the sphere; v ~ N(0, 1).
* "raw" small cases: q, k, v all i.i.d. N(0, 1) scaled by 3, not
  normalised, so the forward's own unit-sphere step is exercised.
"""
from dataclasses import dataclass, asdict

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    p: int
    dv: int
    C: int
    dtype: str          # "fp32" or "bf16"
    kind: str = "gaussian"
    seed: int = 0

    @property
    def n(self) -> int:
        return self.p * (self.p + 1) // 2

    @property
    def NC(self) -> int:
        return (self.T + self.C - 1) // self.C

    def as_dict(self):
        d = asdict(self)
        d["n"] = self.n
        return d


# The five workloads of the benchmark definition, in order.
WORKLOADS = [
    Workload("c1_tiny_fp32", 1, 1, 256, 16, 16, 32, "fp32"),
    Workload("c2_T2048_p32_bf16", 2, 8, 2048, 32, 64, 64, "bf16"),
    Workload("c3_T16384_p64_bf16", 1, 16, 16384, 64, 64, 64, "bf16"),
    Workload("c4_T131072_p64_bf16", 1, 8, 131072, 64, 64, 128, "bf16"),
    Workload("c5_codebook_B64_bf16", 64, 16, 4096, 32, 32, 64, "bf16", kind="codebook"),
]
HEADLINE = WORKLOADS[3]


def torch_dtype(dtype: str):
    return {"fp32": torch.float32, "bf16": torch.bfloat16}[dtype]


def _unit_rows(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def draw_fp64(w: Workload):
    """Return q, k, v as fp64 numpy arrays (before rounding to the dtype)."""
    rng = np.random.default_rng(w.seed)
    shp_qk = (w.B, w.H, w.T, w.p)
    shp_v = (w.B, w.H, w.T, w.dv)
    if w.kind == "gaussian":
        q = _unit_rows(rng.standard_normal(shp_qk))
        k = _unit_rows(rng.standard_normal(shp_qk))
        v = rng.standard_normal(shp_v)
    elif w.kind == "raw":
        q = 3.0 * rng.standard_normal(shp_qk)
        k = 3.0 * rng.standard_normal(shp_qk)
        v = 3.0 * rng.standard_normal(shp_v)
    elif w.kind == "codebook":
        book = _unit_rows(rng.standard_normal((256, w.p)))
        key_idx = rng.integers(0, 256, size=(w.B, w.H, w.T))
        k = book[key_idx]
        pos = np.maximum(np.arange(w.T), 1)
        src = np.floor(rng.random((w.B, w.H, w.T)) * pos).astype(np.int64)
        src[..., 0] = 0
        q = np.take_along_axis(k, src[..., None], axis=2)
        q = _unit_rows(q + 0.1 * rng.standard_normal(shp_qk))
        v = rng.standard_normal(shp_v)
    else:
        raise ValueError(w.kind)
    return q, k, v


def make(w: Workload, device="cpu"):
    """Inputs rounded to the workload dtype, as torch tensors on `device`."""
    dt = torch_dtype(w.dtype)
    return tuple(torch.from_numpy(x).to(dt).to(device).contiguous() for x in draw_fp64(w))


def small(B, H, T, p, dv, C=32, dtype="fp32", kind="gaussian", seed=0, name="small"):
    return Workload(name, B, H, T, p, dv, C, dtype, kind, seed)
