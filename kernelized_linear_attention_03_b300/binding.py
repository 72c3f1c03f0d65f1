"""Python binding of ``libkata.so``: the names of ``include/kata.h``, argument
marshalling only (torch tensors -> pointers, sizes and the current stream).
Every step of the forward runs in the library's CUDA kernels; if the library
is missing this module raises instead of computing anything itself.

Tensors must be contiguous CUDA tensors: q, k [B,H,T,p]; v [B,H,T,dv] of one
dtype (float32 or bfloat16); states are float32 [B,H,n,dv] / [B,H,n].
"""
import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkata.so")

KATA_OK = 0
KATA_ERR_INVALID_ARG = 1
KATA_ERR_UNSUPPORTED = 2
KATA_ERR_WORKSPACE = 3
KATA_ERR_CUDA = 4
KATA_ERR_TIMEOUT = 5
KATA_FP32 = 0
KATA_BF16 = 1
KATA_SCAN_SEQUENTIAL = 0
KATA_SCAN_TREE = 1
KATA_LIFT_FULL = 0
KATA_LIFT_SIGMA = 1
KATA_LIFT_MULTI = 2

SYMBOLS = ("kata_packed_dim", "kata_status_string", "kata_forward_quadratic",
           "kata_chunked_workspace_bytes", "kata_forward_chunked", "kata_chunk_state_scan",
           "kata_scan_states", "kata_get_device_status", "kata_trace_start", "kata_trace_stop",
           "kata_trace_get", "kata_forward_chunked_noalloc", "kata_decode_step", "kata_lift_dim",
           "kata_chunked_block_workspace_bytes", "kata_forward_chunked_block", "kata_forward_quadratic_block",
           "kata_decode_step_block", "kata_backward_quadratic_workspace_bytes",
           "kata_backward_quadratic", "kata_backward_chunked_workspace_bytes", "kata_backward_chunked",
           "kata_chunked_gated_workspace_bytes", "kata_forward_chunked_gated", "kata_decode_step_gated",
           "kata_quadratic_gated_workspace_bytes", "kata_forward_quadratic_gated")


class KataError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {kata_status_string(status)}")


_lib = None


def load():
    """Load libkata.so (once) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise FileNotFoundError(f"libkata.so not built at {LIB_PATH}; run "
                                "python -m kernelized_linear_attention_03_b300.build")
    lib = ctypes.CDLL(LIB_PATH)
    I, P, Z = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
    lib.kata_packed_dim.argtypes = [I]
    lib.kata_packed_dim.restype = I
    lib.kata_status_string.argtypes = [I]
    lib.kata_status_string.restype = ctypes.c_char_p
    lib.kata_forward_quadratic.argtypes = [P, P, P, P, I, I, I, I, I, I, I, P]
    lib.kata_forward_quadratic.restype = I
    lib.kata_chunked_workspace_bytes.argtypes = [I, I, I, I, I, I, I]
    lib.kata_chunked_workspace_bytes.restype = Z
    lib.kata_forward_chunked.argtypes = [P, P, P, P, I, I, I, I, I, I, I, I, P, P, P, P, P, Z, P]
    lib.kata_forward_chunked.restype = I
    lib.kata_chunk_state_scan.argtypes = [P, P, I, I, I, I, I, I, I, I, P, P, P]
    lib.kata_chunk_state_scan.restype = I
    lib.kata_scan_states.argtypes = [P, P, P, P, I, I, I, I, I, I, P]
    lib.kata_scan_states.restype = I
    lib.kata_get_device_status.argtypes = [P]
    lib.kata_get_device_status.restype = I
    lib.kata_forward_chunked_noalloc.argtypes = [P, P, P, P, I, I, I, I, I, I, I, I, P, P, P, P, P]
    lib.kata_forward_chunked_noalloc.restype = I
    lib.kata_decode_step.argtypes = [P, P, P, P, I, I, I, I, I, P, P, P]
    lib.kata_decode_step.restype = I
    lib.kata_lift_dim.argtypes = [I, I, I]
    lib.kata_lift_dim.restype = I
    lib.kata_chunked_block_workspace_bytes.argtypes = [I, I, I, I, I, I, I, I, I]
    lib.kata_chunked_block_workspace_bytes.restype = Z
    lib.kata_forward_chunked_block.argtypes = [P, P, P, P, I, I, I, I, I, I, I, I, I, I, P, P, P, P, P, Z, P]
    lib.kata_forward_chunked_block.restype = I
    lib.kata_forward_quadratic_block.argtypes = [P, P, P, P, I, I, I, I, I, I, I, I, P]
    lib.kata_forward_quadratic_block.restype = I
    lib.kata_decode_step_block.argtypes = [P, P, P, P, I, I, I, I, I, I, I, P, P, P]
    lib.kata_decode_step_block.restype = I
    lib.kata_backward_quadratic_workspace_bytes.argtypes = [I, I, I]
    lib.kata_backward_quadratic_workspace_bytes.restype = Z
    lib.kata_backward_quadratic.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, P, Z, P]
    lib.kata_backward_quadratic.restype = I
    lib.kata_backward_chunked_workspace_bytes.argtypes = [I, I, I, I, I]
    lib.kata_backward_chunked_workspace_bytes.restype = Z
    lib.kata_backward_chunked.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, P, Z, P]
    lib.kata_backward_chunked.restype = I
    lib.kata_chunked_gated_workspace_bytes.argtypes = [I, I, I, I, I, I, I]
    lib.kata_chunked_gated_workspace_bytes.restype = Z
    lib.kata_forward_chunked_gated.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, P, P, P, P, P, Z, P]
    lib.kata_forward_chunked_gated.restype = I
    lib.kata_quadratic_gated_workspace_bytes.argtypes = [I, I, I, I]
    lib.kata_quadratic_gated_workspace_bytes.restype = Z
    lib.kata_forward_quadratic_gated.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P, Z, P]
    lib.kata_forward_quadratic_gated.restype = I
    lib.kata_decode_step_gated.argtypes = [P, P, P, P, P, I, I, I, I, I, P, P, P]
    lib.kata_decode_step_gated.restype = I
    lib.kata_trace_start.argtypes = [I]
    lib.kata_trace_start.restype = I
    lib.kata_trace_stop.argtypes = []
    lib.kata_trace_stop.restype = I
    lib.kata_trace_get.argtypes = [I, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float)]
    lib.kata_trace_get.restype = I
    _lib = lib
    return lib


def _check(status, where):
    if status != KATA_OK:
        raise KataError(status, where)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _used_on(t, stream):
    """Tell torch's caching allocator that `t`, allocated here, is used on
    `stream` (so its memory is not handed out again before that stream has
    passed this call)."""
    if t is None or stream is None:
        return
    s = stream if isinstance(stream, torch.cuda.Stream) else torch.cuda.ExternalStream(int(stream))
    t.record_stream(s)


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor")
    return t.data_ptr()


def _dtype_code(t):
    if t.dtype == torch.float32:
        return KATA_FP32
    if t.dtype == torch.bfloat16:
        return KATA_BF16
    raise ValueError(f"unsupported dtype {t.dtype}")


def _shapes(q, k, v):
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or v.shape[:3] != q.shape[:3]:
        raise ValueError("expected q, k [B,H,T,p] and v [B,H,T,dv]")
    if not (q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k, v must share one dtype")
    B, H, T, p = q.shape
    return B, H, T, p, v.shape[-1]


def kata_packed_dim(p):
    return load().kata_packed_dim(int(p))


def kata_status_string(status):
    return load().kata_status_string(int(status)).decode()


def kata_forward_quadratic(q, k, v, o=None, C=0, stream=None):
    """o = flash-style causal KATA forward of (q, k, v); returns o."""
    B, H, T, p, dv = _shapes(q, k, v)
    if o is None:
        o = torch.empty_like(v)
    _check(load().kata_forward_quadratic(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _dtype_code(q), B, H,
                                         T, p, dv, int(C), _stream(stream)),
           "kata_forward_quadratic")
    return o


def kata_chunked_workspace_bytes(dtype, B, H, T, p, dv, C):
    code = dtype if isinstance(dtype, int) else (KATA_FP32 if dtype == torch.float32 else KATA_BF16)
    return int(load().kata_chunked_workspace_bytes(code, B, H, T, p, dv, C))


def kata_forward_chunked(q, k, v, C, mode=KATA_SCAN_TREE, S0=None, z0=None, o=None,
                         S_final=None, z_final=None, workspace=None, stream=None):
    """Chunked-state forward; returns o, or (o, S_final, z_final) when state
    buffers are given.  `workspace` is a CUDA uint8 tensor of at least
    kata_chunked_workspace_bytes() bytes (allocated through torch when None)."""
    B, H, T, p, dv = _shapes(q, k, v)
    if o is None:
        o = torch.empty_like(v)
    need = kata_chunked_workspace_bytes(_dtype_code(q), B, H, T, p, dv, C)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        _used_on(workspace, stream)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().kata_forward_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _dtype_code(q), B, H, T,
                                       p, dv, int(C), int(mode), _ptr(S0), _ptr(z0), _ptr(S_final),
                                       _ptr(z_final), _ptr(workspace), ws_bytes, _stream(stream)),
           "kata_forward_chunked")
    return o if S_final is None else (o, S_final, z_final)


def kata_forward_chunked_noalloc(q, k, v, C, mode=KATA_SCAN_TREE, S0=None, z0=None, o=None,
                                 S_final=None, z_final=None, stream=None):
    """Chunked forward using the library's fixed device scratch instead of a
    workspace, for callers that must not allocate device memory.  The caller
    passes every input and output (pass `o` to avoid the torch allocation made
    here for convenience).  Returns o, or (o, S_final, z_final)."""
    B, H, T, p, dv = _shapes(q, k, v)
    if o is None:
        o = torch.empty_like(v)
    _check(load().kata_forward_chunked_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _dtype_code(q), B,
                                               H, T, p, dv, int(C), int(mode), _ptr(S0), _ptr(z0),
                                               _ptr(S_final), _ptr(z_final), _stream(stream)),
           "kata_forward_chunked_noalloc")
    return o if S_final is None else (o, S_final, z_final)


def kata_chunk_state_scan(k, v, C, mode=KATA_SCAN_TREE, S_prefix=None, z_prefix=None, stream=None):
    """Exclusive per-chunk state prefixes; returns (S_prefix, z_prefix)."""
    B, H, T, p, dv = _shapes(k, k, v)
    n = kata_packed_dim(p)
    NC = (T + C - 1) // C
    if S_prefix is None:
        S_prefix = torch.empty((B, H, NC, n, dv), dtype=torch.float32, device=k.device)
    if z_prefix is None:
        z_prefix = torch.empty((B, H, NC, n), dtype=torch.float32, device=k.device)
    _check(load().kata_chunk_state_scan(_ptr(k), _ptr(v), _dtype_code(k), B, H, T, p, dv, int(C),
                                        int(mode), _ptr(S_prefix), _ptr(z_prefix), _stream(stream)),
           "kata_chunk_state_scan")
    return S_prefix, z_prefix


def kata_scan_states(S_loc, z_loc, mode=KATA_SCAN_TREE, S_prefix=None, z_prefix=None, stream=None):
    """Exclusive prefix over the chunk axis of S_loc [B,H,NC,n,dv], z_loc [B,H,NC,n]."""
    if S_loc.dim() != 5 or z_loc.shape != S_loc.shape[:4]:
        raise ValueError("expected S_loc [B,H,NC,n,dv] and z_loc [B,H,NC,n]")
    if S_loc.dtype != torch.float32 or z_loc.dtype != torch.float32:
        raise ValueError("states are float32")
    B, H, NC, n, dv = S_loc.shape
    if S_prefix is None:
        S_prefix = torch.empty_like(S_loc)
    if z_prefix is None:
        z_prefix = torch.empty_like(z_loc)
    _check(load().kata_scan_states(_ptr(S_loc), _ptr(z_loc), _ptr(S_prefix), _ptr(z_prefix), B, H,
                                   NC, n, dv, int(mode), _stream(stream)),
           "kata_scan_states")
    return S_prefix, z_prefix


def kata_decode_step(q, k, v, S, z, o=None, stream=None):
    """One recurrent decode step: q, k [B,H,p], v [B,H,dv] (one dtype); S
    [B,H,n,dv] and z [B,H,n] float32, updated in place.  Returns o [B,H,dv]."""
    if q.dim() != 3 or k.shape != q.shape or v.dim() != 3 or v.shape[:2] != q.shape[:2]:
        raise ValueError("expected q, k [B,H,p] and v [B,H,dv]")
    if not (q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k, v must share one dtype")
    B, H, p = q.shape
    dv = v.shape[-1]
    n = kata_packed_dim(p)
    if S.shape != (B, H, n, dv) or z.shape != (B, H, n) or S.dtype != torch.float32 or z.dtype != torch.float32:
        raise ValueError("expected float32 S [B,H,n,dv] and z [B,H,n]")
    if o is None:
        o = torch.empty_like(v)
    _check(load().kata_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _dtype_code(q), B, H, p, dv,
                                   _ptr(S), _ptr(z), _stream(stream)),
           "kata_decode_step")
    return o


def kata_lift_dim(family, p, g):
    return load().kata_lift_dim(int(family), int(p), int(g))


def kata_chunked_block_workspace_bytes(dtype, family, g, B, H, T, p, dv, C):
    code = dtype if isinstance(dtype, int) else (KATA_FP32 if dtype == torch.float32 else KATA_BF16)
    return int(load().kata_chunked_block_workspace_bytes(code, int(family), int(g), B, H, T, p, dv, C))


def kata_forward_chunked_block(q, k, v, C, family, g, mode=KATA_SCAN_TREE, S0=None, z0=None, o=None,
                               S_final=None, z_final=None, workspace=None, stream=None):
    """Chunked forward with a block lift (KATA-Sigma-g / KATA-M-g); returns o,
    or (o, S_final, z_final) when state buffers are given."""
    B, H, T, p, dv = _shapes(q, k, v)
    if o is None:
        o = torch.empty_like(v)
    need = kata_chunked_block_workspace_bytes(_dtype_code(q), family, g, B, H, T, p, dv, C)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        _used_on(workspace, stream)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().kata_forward_chunked_block(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _dtype_code(q), B, H, T, p, dv,
                                             int(C), int(family), int(g), int(mode), _ptr(S0), _ptr(z0),
                                             _ptr(S_final), _ptr(z_final), _ptr(workspace), ws_bytes,
                                             _stream(stream)),
           "kata_forward_chunked_block")
    return o if S_final is None else (o, S_final, z_final)


def kata_forward_quadratic_block(q, k, v, family, g, o=None, stream=None):
    """Flash-style forward with a block lift's kernel; returns o."""
    B, H, T, p, dv = _shapes(q, k, v)
    if o is None:
        o = torch.empty_like(v)
    _check(load().kata_forward_quadratic_block(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _dtype_code(q), B, H, T, p, dv,
                                               int(family), int(g), _stream(stream)),
           "kata_forward_quadratic_block")
    return o


def kata_decode_step_block(q, k, v, S, z, family, g, o=None, stream=None):
    """Decode step with a block lift: S [B,H,n,dv], z [B,H,n] float32 with
    n = kata_lift_dim(family, p, g), updated in place.  Returns o [B,H,dv]."""
    if q.dim() != 3 or k.shape != q.shape or v.dim() != 3 or v.shape[:2] != q.shape[:2]:
        raise ValueError("expected q, k [B,H,p] and v [B,H,dv]")
    if not (q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k, v must share one dtype")
    B, H, p = q.shape
    dv = v.shape[-1]
    n = kata_lift_dim(family, p, g)
    if S.shape != (B, H, n, dv) or z.shape != (B, H, n) or S.dtype != torch.float32 or z.dtype != torch.float32:
        raise ValueError("expected float32 S [B,H,n,dv] and z [B,H,n] for the lift")
    if o is None:
        o = torch.empty_like(v)
    _check(load().kata_decode_step_block(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _dtype_code(q), B, H, p, dv,
                                         int(family), int(g), _ptr(S), _ptr(z), _stream(stream)),
           "kata_decode_step_block")
    return o


def kata_forward_chunked_gated(q, k, v, gate, C, S0=None, z0=None, o=None, S_final=None, z_final=None,
                               workspace=None, stream=None):
    """Gated chunked forward; gate [B,H,T] float32.  Returns o, or (o, S_final,
    z_final) when state buffers are given."""
    B, H, T, p, dv = _shapes(q, k, v)
    if gate.shape != (B, H, T) or gate.dtype != torch.float32:
        raise ValueError("expected a float32 gate [B,H,T]")
    if o is None:
        o = torch.empty_like(v)
    need = int(load().kata_chunked_gated_workspace_bytes(_dtype_code(q), B, H, T, p, dv, int(C)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        _used_on(workspace, stream)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().kata_forward_chunked_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(o), _dtype_code(q), B, H,
                                             T, p, dv, int(C), _ptr(S0), _ptr(z0), _ptr(S_final), _ptr(z_final),
                                             _ptr(workspace), ws_bytes, _stream(stream)),
           "kata_forward_chunked_gated")
    return o if S_final is None else (o, S_final, z_final)


def kata_forward_quadratic_gated(q, k, v, gate, o=None, workspace=None, stream=None):
    """Gated flash-style forward (bf16, gates in [0, 1]); gate [B,H,T] float32.
    Returns o."""
    B, H, T, p, dv = _shapes(q, k, v)
    if gate.shape != (B, H, T) or gate.dtype != torch.float32:
        raise ValueError("expected a float32 gate [B,H,T]")
    if o is None:
        o = torch.empty_like(v)
    need = int(load().kata_quadratic_gated_workspace_bytes(_dtype_code(q), B, H, T))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        _used_on(workspace, stream)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().kata_forward_quadratic_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(o), _dtype_code(q), B, H,
                                               T, p, dv, _ptr(workspace), ws_bytes, _stream(stream)),
           "kata_forward_quadratic_gated")
    return o


def kata_decode_step_gated(q, k, v, gate, S, z, o=None, stream=None):
    """Gated decode step; gate [B,H] float32; S, z updated in place.  Returns o."""
    if q.dim() != 3 or k.shape != q.shape or v.dim() != 3 or v.shape[:2] != q.shape[:2]:
        raise ValueError("expected q, k [B,H,p] and v [B,H,dv]")
    B, H, p = q.shape
    dv = v.shape[-1]
    if gate.shape != (B, H) or gate.dtype != torch.float32:
        raise ValueError("expected a float32 gate [B,H]")
    if o is None:
        o = torch.empty_like(v)
    _check(load().kata_decode_step_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(o), _dtype_code(q), B, H, p,
                                         dv, _ptr(S), _ptr(z), _stream(stream)),
           "kata_decode_step_gated")
    return o


def kata_backward(q, k, v, dO, dq=None, dk=None, dv=None, workspace=None, stream=None, form="chunked"):
    """Gradients (dq, dk, dv) of sum(dO * o) for the forward of (q, k, v),
    through the chunked form (O(T), default) or the quadratic form."""
    B, H, T, p, dv_dim = _shapes(q, k, v)
    if dO.shape != v.shape or dO.dtype != v.dtype:
        raise ValueError("dO must match v's shape and dtype")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    lib = load()
    if form == "chunked":
        need, fn = int(lib.kata_backward_chunked_workspace_bytes(B, H, T, p, dv_dim)), lib.kata_backward_chunked
    elif form == "quadratic":
        need, fn = int(lib.kata_backward_quadratic_workspace_bytes(B, H, T)), lib.kata_backward_quadratic
    else:
        raise ValueError(f"unknown backward form {form!r}")
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        _used_on(workspace, stream)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv), _dtype_code(q), B, H, T, p, dv_dim,
              _ptr(workspace), ws_bytes, _stream(stream)),
           f"kata_backward_{form}")
    return dq, dk, dv


def kata_get_device_status(stream=None):
    """Synchronise the stream; raise KataError if a device-side wait expired."""
    _check(load().kata_get_device_status(_stream(stream)), "kata_get_device_status")


def kata_trace_start(capacity):
    """Record an event pair around each kernel the library launches from now on."""
    _check(load().kata_trace_start(int(capacity)), "kata_trace_start")


def kata_trace_stop():
    """Stop tracing; return [(kernel_name, ms), ...] for the recorded launches."""
    lib = load()
    count = lib.kata_trace_stop()
    if count < 0:
        raise KataError(KATA_ERR_CUDA, "kata_trace_stop")
    out = []
    name = ctypes.c_char_p()
    ms = ctypes.c_float()
    for i in range(count):
        _check(lib.kata_trace_get(i, ctypes.byref(name), ctypes.byref(ms)), "kata_trace_get")
        out.append((name.value.decode(), float(ms.value)))
    return out
