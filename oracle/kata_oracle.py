"""ctypes front end of the fp64 CPU oracle (``kata_oracle.cpp``).

TEST INFRASTRUCTURE ONLY: the oracle restates, slowly and in fp64, what the
KATA causal normalised linear-attention forward computes, so that the CUDA
library can be checked against it.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import this module; the product path never
does.  It shares no code with the CUDA library.

All arrays are numpy float64, C-contiguous, in the documented layouts:
q, k [B,H,T,p]; v, o [B,H,T,dv]; S [B,H,n,dv]; z [B,H,n]; n = p(p+1)/2.
Anything that is not already float64 (e.g. bf16 values held in float32) is
widened exactly before the call.

Parity status of each function (pins live in tests/test_oracle_pins.py):
  packed_dim, normalize, lift       pinned (closed forms, lift identities)
  forward_plain, forward_plain_rows pinned (special cases, pSNR closed form,
                                     rotation/scale invariance, convexity)
  forward_recurrent                 pinned (agrees with plain; split calls; one-token
                                     decode steps chained through their states)
  forward_chunked, chunk_states     pinned (agrees with plain for every C,
                                     ragged T; split calls; state identity)
  scan_exclusive                    pinned (tree == sequential; depth)
  block_dim, lift_block             pinned (page's state sizes, block outer products,
                                     kernel identities, g = 1 is the full lift)
  forward_plain_block,              pinned (agree with each other; g = 1 is the full
  forward_recurrent_block            forward; Sigma-p running mean; disjoint blocks;
                                     block-permutation behaviour; split calls)
  forward_plain_block_rows,         pinned (equal the full-row definitions they
  forward_plain_gated_rows           sample)
  forward_plain_gated,              pinned (gate 1 is the ungated forward; a zero
  forward_recurrent_gated,           gate restarts; constant gate with identical
  forward_chunked_gated,             keys is the moving average; the three forms
  scan_exclusive_gated               agree; tree = sequential; split calls)
  backward_plain                    pinned (central finite differences of the
                                     definition; orthogonality to q and k; value
                                     shifts; rotations; T = 1; zero vectors)
"""
import ctypes

import numpy as np

from . import build as _build

_lib = None
_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.POINTER(ctypes.c_int64)
SCAN_SEQUENTIAL = 0
SCAN_TREE = 1
LIFT_FULL = 0
LIFT_SIGMA = 1
LIFT_MULTI = 2


def _bind(lib):
    """Declare the C signatures on a loaded oracle library."""
    i = ctypes.c_int
    lib.kor_packed_dim.argtypes = [i]
    lib.kor_packed_dim.restype = i
    lib.kor_normalize.argtypes = [_D, i, _D]
    lib.kor_normalize.restype = None
    lib.kor_lift.argtypes = [_D, i, _D]
    lib.kor_lift.restype = None
    lib.kor_forward_plain.argtypes = [_D, _D, _D, i, i, i, i, i, _D, i]
    lib.kor_forward_plain.restype = i
    lib.kor_forward_plain_rows.argtypes = [_D, _D, _D, i, i, i, i, i, _I64, _I64,
                                           ctypes.c_int64, _D, i]
    lib.kor_forward_plain_rows.restype = i
    lib.kor_forward_recurrent.argtypes = [_D, _D, _D, i, i, i, i, i, _D, _D, _D, _D, _D, i]
    lib.kor_forward_recurrent.restype = i
    lib.kor_chunk_states.argtypes = [_D, _D, i, i, i, i, i, i, _D, _D, i]
    lib.kor_chunk_states.restype = i
    lib.kor_scan_exclusive.argtypes = [_D, _D, i, i, i, i, i, i, _D, _D, i]
    lib.kor_scan_exclusive.restype = i
    lib.kor_forward_chunked.argtypes = [_D, _D, _D, i, i, i, i, i, i, i, _D, _D, _D, _D, _D, i]
    lib.kor_forward_chunked.restype = i
    lib.kor_block_dim.argtypes = [i, i, i]
    lib.kor_block_dim.restype = i
    lib.kor_lift_block.argtypes = [_D, i, i, i, _D]
    lib.kor_lift_block.restype = None
    lib.kor_forward_plain_block.argtypes = [_D, _D, _D, i, i, i, i, i, i, i, _D, i]
    lib.kor_forward_plain_block.restype = i
    lib.kor_forward_recurrent_block.argtypes = [_D, _D, _D, i, i, i, i, i, i, i, _D, _D, _D, _D, _D, i]
    lib.kor_forward_recurrent_block.restype = i
    lib.kor_backward_plain.argtypes = [_D, _D, _D, _D, i, i, i, i, i, _D, _D, _D, i]
    lib.kor_backward_plain.restype = i
    lib.kor_forward_plain_gated.argtypes = [_D, _D, _D, _D, i, i, i, i, i, _D, i]
    lib.kor_forward_plain_gated.restype = i
    lib.kor_forward_recurrent_gated.argtypes = [_D, _D, _D, _D, i, i, i, i, i, _D, _D, _D, _D, _D, i]
    lib.kor_forward_recurrent_gated.restype = i
    lib.kor_scan_exclusive_gated.argtypes = [_D, _D, i, i, i, i, _D, i]
    lib.kor_scan_exclusive_gated.restype = i
    lib.kor_forward_chunked_gated.argtypes = [_D, _D, _D, _D, i, i, i, i, i, i, i, _D, _D, _D, _D, _D, i]
    lib.kor_forward_chunked_gated.restype = i
    lib.kor_forward_plain_block_rows.argtypes = [_D, _D, _D, i, i, i, i, i, i, i, _I64, _I64, ctypes.c_int64, _D, i]
    lib.kor_forward_plain_block_rows.restype = i
    lib.kor_forward_plain_gated_rows.argtypes = [_D, _D, _D, _D, i, i, i, i, i, _I64, _I64, ctypes.c_int64, _D, i]
    lib.kor_forward_plain_gated_rows.restype = i
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(_build.build()))
    return _lib


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_D)


def _shape4(q, k, v):
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim != 4 or k.shape != q.shape or v.ndim != 4 or v.shape[:3] != q.shape[:3]:
        raise ValueError("expected q, k [B,H,T,p] and v [B,H,T,dv]")
    return q, k, v


def packed_dim(p: int) -> int:
    return _load().kor_packed_dim(p)


def normalize(x):
    """Row-wise unit-sphere projection of an [..., p] array."""
    x = _f64(x)
    p = x.shape[-1]
    flat = x.reshape(-1, p)
    u = np.empty_like(flat)
    for r in range(flat.shape[0]):
        _load().kor_normalize(_ptr(flat[r]), p, _ptr(u[r]))
    return u.reshape(x.shape)


def lift(u):
    u = _f64(u)
    p = u.shape[-1]
    out = np.empty(packed_dim(p))
    _load().kor_lift(_ptr(u), p, _ptr(out))
    return out


def forward_plain(q, k, v, nthreads=0):
    q, k, v = _shape4(q, k, v)
    B, H, T, p = q.shape
    dv = v.shape[-1]
    o = np.empty((B, H, T, dv))
    _load().kor_forward_plain(_ptr(q), _ptr(k), _ptr(v), B, H, T, p, dv, _ptr(o), nthreads)
    return o


def forward_plain_rows(q, k, v, bh, t, nthreads=0):
    """Plain-definition outputs for rows (bh[r], t[r]); bh = b*H + h. Returns [R, dv]."""
    q, k, v = _shape4(q, k, v)
    B, H, T, p = q.shape
    dv = v.shape[-1]
    bh = np.ascontiguousarray(np.asarray(bh, dtype=np.int64))
    t = np.ascontiguousarray(np.asarray(t, dtype=np.int64))
    if bh.shape != t.shape or (bh.size and (bh.min() < 0 or bh.max() >= B * H or t.min() < 0
                                            or t.max() >= T)):
        raise ValueError("row index out of range")
    out = np.empty((bh.size, dv))
    _load().kor_forward_plain_rows(_ptr(q), _ptr(k), _ptr(v), B, H, T, p, dv,
                                   bh.ctypes.data_as(_I64), t.ctypes.data_as(_I64), bh.size,
                                   _ptr(out), nthreads)
    return out


def forward_recurrent(q, k, v, S0=None, z0=None, nthreads=0):
    """Token-recurrent form. Returns (o, S_final, z_final)."""
    q, k, v = _shape4(q, k, v)
    B, H, T, p = q.shape
    dv = v.shape[-1]
    n = packed_dim(p)
    S0 = None if S0 is None else _f64(S0).reshape(B, H, n, dv)
    z0 = None if z0 is None else _f64(z0).reshape(B, H, n)
    o = np.empty((B, H, T, dv))
    S = np.empty((B, H, n, dv))
    z = np.empty((B, H, n))
    _load().kor_forward_recurrent(_ptr(q), _ptr(k), _ptr(v), B, H, T, p, dv, _ptr(S0), _ptr(z0),
                                  _ptr(o), _ptr(S), _ptr(z), nthreads)
    return o, S, z


def chunk_states(k, v, C, nthreads=0):
    """Per-chunk local states. Returns (S_loc [B,H,NC,n,dv], z_loc [B,H,NC,n])."""
    k, v = _f64(k), _f64(v)
    B, H, T, p = k.shape
    dv = v.shape[-1]
    n = packed_dim(p)
    NC = (T + C - 1) // C
    S = np.empty((B, H, NC, n, dv))
    z = np.empty((B, H, NC, n))
    _load().kor_chunk_states(_ptr(k), _ptr(v), B, H, T, p, dv, C, _ptr(S), _ptr(z), nthreads)
    return S, z


def scan_exclusive(S_loc, z_loc, mode=SCAN_SEQUENTIAL, nthreads=0):
    """Exclusive prefix over the chunk axis. Returns (S_prefix, z_prefix, rounds)."""
    S_loc, z_loc = _f64(S_loc), _f64(z_loc)
    B, H, NC, n, dv = S_loc.shape
    Sp = np.empty_like(S_loc)
    zp = np.empty_like(z_loc)
    rounds = _load().kor_scan_exclusive(_ptr(S_loc), _ptr(z_loc), B, H, NC, n, dv, mode,
                                        _ptr(Sp), _ptr(zp), nthreads)
    return Sp, zp, rounds


def forward_chunked(q, k, v, C, mode=SCAN_SEQUENTIAL, S0=None, z0=None, nthreads=0):
    """Chunked form. Returns (o, S_final, z_final)."""
    q, k, v = _shape4(q, k, v)
    B, H, T, p = q.shape
    dv = v.shape[-1]
    n = packed_dim(p)
    S0 = None if S0 is None else _f64(S0).reshape(B, H, n, dv)
    z0 = None if z0 is None else _f64(z0).reshape(B, H, n)
    o = np.empty((B, H, T, dv))
    S = np.empty((B, H, n, dv))
    z = np.empty((B, H, n))
    _load().kor_forward_chunked(_ptr(q), _ptr(k), _ptr(v), B, H, T, p, dv, C, mode, _ptr(S0),
                                _ptr(z0), _ptr(o), _ptr(S), _ptr(z), nthreads)
    return o, S, z


# ---------------------------------------------------------------- block lifts

def block_dim(p: int, family: int, g: int) -> int:
    """Width of the lift: full p(p+1)/2 (g = 1), Sigma-g m(m+1)/2, M-g g m(m+1)/2
    with m = p/g; -1 if (family, g) does not fit p."""
    return _load().kor_block_dim(int(p), int(family), int(g))


def _check_block(p, family, g):
    n = block_dim(p, family, g)
    if n < 0:
        raise ValueError(f"lift family {family} with g={g} does not fit p={p}")
    return n


def lift_block(u, family, g):
    """Packed block lift of one vector (used as given, not normalised)."""
    u = _f64(u)
    n = _check_block(u.shape[-1], family, g)
    out = np.empty(n)
    _load().kor_lift_block(_ptr(u), u.shape[-1], int(family), int(g), _ptr(out))
    return out


def forward_plain_block(q, k, v, family, g, nthreads=0):
    """The definition with a block-lift kernel (block dot products squared)."""
    q, k, v = _shape4(q, k, v)
    B, H, T, p = q.shape
    dv = v.shape[-1]
    _check_block(p, family, g)
    o = np.empty((B, H, T, dv))
    _load().kor_forward_plain_block(_ptr(q), _ptr(k), _ptr(v), B, H, T, p, dv, int(family), int(g), _ptr(o),
                                    nthreads)
    return o


def forward_recurrent_block(q, k, v, family, g, S0=None, z0=None, nthreads=0):
    """Token recurrence in the packed block lift. Returns (o, S_final, z_final)."""
    q, k, v = _shape4(q, k, v)
    B, H, T, p = q.shape
    dv = v.shape[-1]
    n = _check_block(p, family, g)
    S0 = None if S0 is None else _f64(S0).reshape(B, H, n, dv)
    z0 = None if z0 is None else _f64(z0).reshape(B, H, n)
    o = np.empty((B, H, T, dv))
    S = np.empty((B, H, n, dv))
    z = np.empty((B, H, n))
    _load().kor_forward_recurrent_block(_ptr(q), _ptr(k), _ptr(v), B, H, T, p, dv, int(family), int(g),
                                        _ptr(S0), _ptr(z0), _ptr(o), _ptr(S), _ptr(z), nthreads)
    return o, S, z


# ---------------------------------------------------------------- backward

def backward_plain(q, k, v, dO, nthreads=0):
    """Gradients (dq, dk, dv) of L = sum(dO * o) through the plain definition."""
    q, k, v = _shape4(q, k, v)
    dO = _f64(dO)
    if dO.shape != v.shape:
        raise ValueError("dO must have v's shape [B,H,T,dv]")
    B, H, T, p = q.shape
    dv = v.shape[-1]
    dq, dk, dvv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    _load().kor_backward_plain(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), B, H, T, p, dv, _ptr(dq), _ptr(dk), _ptr(dvv),
                               nthreads)
    return dq, dk, dvv


# ---------------------------------------------------------------- gated prefix

def _gate(gate, q):
    gate = _f64(gate)
    if gate.shape != q.shape[:3]:
        raise ValueError("gate must be [B,H,T]")
    return gate


def forward_plain_gated(q, k, v, gate, nthreads=0):
    """Definition of the gated forward: weights (qh_t.kh_s)^2 prod_{r=s+1..t} gate_r."""
    q, k, v = _shape4(q, k, v)
    gate = _gate(gate, q)
    B, H, T, p = q.shape
    dv = v.shape[-1]
    o = np.empty((B, H, T, dv))
    _load().kor_forward_plain_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(gate), B, H, T, p, dv, _ptr(o), nthreads)
    return o


def forward_recurrent_gated(q, k, v, gate, S0=None, z0=None, nthreads=0):
    """Gated token recurrence S_t = gate_t S_{t-1} + psi(kh_t) v_t^T. Returns (o, S, z)."""
    q, k, v = _shape4(q, k, v)
    gate = _gate(gate, q)
    B, H, T, p = q.shape
    dv = v.shape[-1]
    n = packed_dim(p)
    S0 = None if S0 is None else _f64(S0).reshape(B, H, n, dv)
    z0 = None if z0 is None else _f64(z0).reshape(B, H, n)
    o = np.empty((B, H, T, dv))
    S = np.empty((B, H, n, dv))
    z = np.empty((B, H, n))
    _load().kor_forward_recurrent_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(gate), B, H, T, p, dv, _ptr(S0), _ptr(z0),
                                        _ptr(o), _ptr(S), _ptr(z), nthreads)
    return o, S, z


def scan_exclusive_gated(a, x, mode=SCAN_SEQUENTIAL, nthreads=0):
    """Exclusive gated prefix of items (a [heads, NC], x [heads, NC, W]):
    prefix_0 = 0, prefix_{c+1} = a_c prefix_c + x_c.  Returns (prefix, rounds)."""
    a, x = _f64(a), _f64(x)
    heads, NC, W = x.shape
    if a.shape != (heads, NC):
        raise ValueError("a must be [heads, NC]")
    out = np.empty_like(x)
    rounds = _load().kor_scan_exclusive_gated(_ptr(a), _ptr(x), heads, NC, W, mode, _ptr(out), nthreads)
    return out, rounds


def forward_chunked_gated(q, k, v, gate, C, mode=SCAN_SEQUENTIAL, S0=None, z0=None, nthreads=0):
    """Gated chunked form (decayed local states, gated prefix scan, decayed
    readout plus the local causal part). Returns (o, S_final, z_final)."""
    q, k, v = _shape4(q, k, v)
    gate = _gate(gate, q)
    B, H, T, p = q.shape
    dv = v.shape[-1]
    n = packed_dim(p)
    S0 = None if S0 is None else _f64(S0).reshape(B, H, n, dv)
    z0 = None if z0 is None else _f64(z0).reshape(B, H, n)
    o = np.empty((B, H, T, dv))
    S = np.empty((B, H, n, dv))
    z = np.empty((B, H, n))
    _load().kor_forward_chunked_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(gate), B, H, T, p, dv, C, mode, _ptr(S0),
                                      _ptr(z0), _ptr(o), _ptr(S), _ptr(z), nthreads)
    return o, S, z


# ---------------------------------------------------------------- sampled rows

def _rows(q, bh, t):
    B, H, T = q.shape[:3]
    bh = np.ascontiguousarray(np.asarray(bh, dtype=np.int64))
    t = np.ascontiguousarray(np.asarray(t, dtype=np.int64))
    if bh.shape != t.shape or (bh.size and (bh.min() < 0 or bh.max() >= B * H or t.min() < 0 or t.max() >= T)):
        raise ValueError("row index out of range")
    return bh, t


def forward_plain_block_rows(q, k, v, family, g, bh, t, nthreads=0):
    """Block-lift definition for rows (bh[r], t[r]). Returns [R, dv]."""
    q, k, v = _shape4(q, k, v)
    B, H, T, p = q.shape
    dv = v.shape[-1]
    _check_block(p, family, g)
    bh, t = _rows(q, bh, t)
    out = np.empty((bh.size, dv))
    _load().kor_forward_plain_block_rows(_ptr(q), _ptr(k), _ptr(v), B, H, T, p, dv, int(family), int(g),
                                         bh.ctypes.data_as(_I64), t.ctypes.data_as(_I64), bh.size, _ptr(out),
                                         nthreads)
    return out


def forward_plain_gated_rows(q, k, v, gate, bh, t, nthreads=0):
    """Gated definition for rows (bh[r], t[r]). Returns [R, dv]."""
    q, k, v = _shape4(q, k, v)
    gate = _gate(gate, q)
    B, H, T, p = q.shape
    dv = v.shape[-1]
    bh, t = _rows(q, bh, t)
    out = np.empty((bh.size, dv))
    _load().kor_forward_plain_gated_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(gate), B, H, T, p, dv,
                                         bh.ctypes.data_as(_I64), t.ctypes.data_as(_I64), bh.size, _ptr(out),
                                         nthreads)
    return out


def library_path() -> str:
    return _build.LIB

