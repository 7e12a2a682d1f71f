"""Thin torch binding of libla.so (argument marshalling only).

Each function takes torch CUDA tensors, checks their dtype/shape/contiguity,
allocates the outputs with torch, and calls the C entry point of the same name
on the current torch stream.  Every step of the computation runs in the
library's kernels; there is no CPU or PyTorch fallback: if libla.so is missing
or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libla.so")

LA_OK, LA_ERR_INVALID_ARG, LA_ERR_UNSUPPORTED, LA_ERR_CUDA, LA_ERR_TIMEOUT = range(5)
LA_F32, LA_BF16 = 0, 1
LA_MODE_CAUSAL, LA_MODE_READ_BEFORE_WRITE, LA_MODE_NONCAUSAL = 0, 1, 2

SYMBOLS = ("la_prefill", "la_prefill_workspace_bytes", "la_decode_step",
           "delta_prefill", "la_state_bytes", "la_status_string",
           "la_read_device_status", "delta_read_device_status",
           "la_prefill_variant", "la_prefill_variant_workspace_bytes", "gated_delta_prefill",
           "la_prefill_backward", "la_prefill_backward_workspace_bytes")


class LAError(RuntimeError):
    """A non-LA_OK status from libla.so."""

    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load libla.so (once) and declare the C signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"libla.so not found at {p}; build it with "
                "`python -m fixed_state_recurrent_gb300.build`")
        lib = ctypes.CDLL(p)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.la_prefill.argtypes = [vp, vp, vp, i, i, i, i, i, i, f, vp, vp, vp, vp,
                                   vp, i, vp, sz, vp]
        lib.la_prefill.restype = i
        lib.la_prefill_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
        lib.la_prefill_workspace_bytes.restype = sz
        lib.la_decode_step.argtypes = [vp, vp, vp, i, i, i, i, i, f, vp, vp, vp, vp]
        lib.la_decode_step.restype = i
        lib.delta_prefill.argtypes = [vp, vp, i, vp, i, i, i, i, i, vp, vp, vp, vp]
        lib.delta_prefill.restype = i
        lib.la_state_bytes.argtypes = [i, i]
        lib.la_state_bytes.restype = sz
        lib.la_status_string.argtypes = [i]
        lib.la_status_string.restype = ctypes.c_char_p
        lib.la_read_device_status.argtypes = [vp, vp]
        lib.la_read_device_status.restype = i
        lib.delta_read_device_status.argtypes = [vp]
        lib.delta_read_device_status.restype = i
        lib.la_prefill_variant.argtypes = [vp, vp, vp, i, i, i, i, i, i, f, vp, i, vp, vp,
                                           vp, vp, vp, vp, sz, vp]
        lib.la_prefill_variant.restype = i
        lib.la_prefill_variant_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i]
        lib.la_prefill_variant_workspace_bytes.restype = sz
        lib.gated_delta_prefill.argtypes = [vp, vp, i, vp, vp, i, i, i, i, i, vp, vp, vp, vp]
        lib.gated_delta_prefill.restype = i
        lib.la_prefill_backward.argtypes = [vp, vp, vp, i, i, i, i, i, i, f, vp, vp, vp, vp, vp,
                                            vp, vp, vp, vp, vp, vp, sz, vp]
        lib.la_prefill_backward.restype = i
        lib.la_prefill_backward_workspace_bytes.argtypes = [i, i, i, i, i, i]
        lib.la_prefill_backward_workspace_bytes.restype = sz
        _lib = lib
        return lib


def __getattr__(name):
    if name == "lib":
        return load()
    raise AttributeError(name)


def status_string(status: int) -> str:
    return load().la_status_string(int(status)).decode()


def _check(fn, status):
    if status != LA_OK:
        raise LAError(fn, status)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return LA_BF16
    if t.dtype == torch.float32:
        return LA_F32
    raise TypeError(f"unsupported input dtype {t.dtype} (float32 or bfloat16)")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, name, shape, dtype, device):
    if t is None:
        return
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be on {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def state_bytes(dk: int, dv: int) -> int:
    return int(load().la_state_bytes(dk, dv))


def prefill_workspace_bytes(B, H, N, dk, dv, dtype=torch.bfloat16, chunk=0) -> int:
    code = LA_BF16 if dtype == torch.bfloat16 else LA_F32
    return int(load().la_prefill_workspace_bytes(B, H, N, dk, dv, code, chunk))


_ws_cache: dict = {}


def workspace(B, H, N, dk, dv, dtype, chunk=0, device=None) -> torch.Tensor:
    """A zero-filled workspace large enough for these arguments, cached per
    device and grown on demand (the kernels leave it ready for reuse)."""
    device = torch.device(device or "cuda")
    if device.index is None:
        device = torch.device("cuda", torch.cuda.current_device())
    need = prefill_workspace_bytes(B, H, N, dk, dv, dtype, chunk)
    if need == 0:
        raise ValueError("invalid prefill arguments")
    ws = _ws_cache.get(device)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(max(need, 1 << 16), dtype=torch.uint8, device=device)
        _ws_cache[device] = ws
    return ws


def prefill(q, k, v, eps=1e-6, S0=None, z0=None, *, o=None, S_N=None, z_N=None,
            chunk=0, ws=None):
    """Causal prefill: returns (o, S_N, z_N); see la_prefill in include/la.h."""
    B, H, N, dk = q.shape
    dv = v.shape[3]
    dev = q.device
    dt = q.dtype
    code = _dtype_code(q)
    _need(q, "q", (B, H, N, dk), dt, dev)
    _need(k, "k", (B, H, N, dk), dt, dev)
    _need(v, "v", (B, H, N, dv), dt, dev)
    _need(S0, "S0", (B, H, dk, dv), torch.float32, dev)
    _need(z0, "z0", (B, H, dk), torch.float32, dev)
    if o is None:
        o = torch.empty((B, H, N, dv), dtype=torch.float32, device=dev)
    if S_N is None:
        S_N = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    if z_N is None:
        z_N = torch.empty((B, H, dk), dtype=torch.float32, device=dev)
    _need(o, "o", (B, H, N, dv), torch.float32, dev)
    _need(S_N, "S_N", (B, H, dk, dv), torch.float32, dev)
    _need(z_N, "z_N", (B, H, dk), torch.float32, dev)
    if ws is None:
        ws = workspace(B, H, N, dk, dv, dt, chunk, dev)
    st = load().la_prefill(_ptr(q), _ptr(k), _ptr(v), code, B, H, N, dk, dv,
                           float(eps), _ptr(S0), _ptr(z0), _ptr(o), _ptr(S_N),
                           _ptr(z_N), int(chunk), _ptr(ws), ws.numel(), _stream(dev))
    _check("la_prefill", st)
    return o, S_N, z_N


def decode_step(q, k, v, S, z, eps=1e-6, *, o=None):
    """One decode step in place on (S, z); returns o.  See la_decode_step."""
    B, H, dk = q.shape
    dv = v.shape[2]
    dev = q.device
    code = _dtype_code(q)
    _need(k, "k", (B, H, dk), q.dtype, dev)
    _need(v, "v", (B, H, dv), q.dtype, dev)
    _need(S, "S", (B, H, dk, dv), torch.float32, dev)
    _need(z, "z", (B, H, dk), torch.float32, dev)
    if o is None:
        o = torch.empty((B, H, dv), dtype=torch.float32, device=dev)
    _need(o, "o", (B, H, dv), torch.float32, dev)
    st = load().la_decode_step(_ptr(q), _ptr(k), _ptr(v), code, B, H, dk, dv,
                               float(eps), _ptr(S), _ptr(z), _ptr(o), _stream(dev))
    _check("la_decode_step", st)
    return o


def delta_prefill(k, v, beta, S0=None, *, reads=None, S_N=None):
    """Delta-rule memory: returns (reads, S_N).  See delta_prefill in la.h."""
    B, H, N, dk = k.shape
    dv = v.shape[3]
    dev = k.device
    code = _dtype_code(k)
    _need(v, "v", (B, H, N, dv), k.dtype, dev)
    _need(beta, "beta", (B, H, N), torch.float32, dev)
    _need(S0, "S0", (B, H, dk, dv), torch.float32, dev)
    if reads is None:
        reads = torch.empty((B, H, N, dv), dtype=torch.float32, device=dev)
    if S_N is None:
        S_N = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    _need(reads, "reads", (B, H, N, dv), torch.float32, dev)
    _need(S_N, "S_N", (B, H, dk, dv), torch.float32, dev)
    st = load().delta_prefill(_ptr(k), _ptr(v), code, _ptr(beta), B, H, N, dk, dv,
                              _ptr(S0), _ptr(reads), _ptr(S_N), _stream(dev))
    _check("delta_prefill", st)
    return reads, S_N


def gated_delta_prefill(k, v, beta, alpha=None, S0=None, *, reads=None, S_N=None):
    """Gated delta rule: returns (reads, S_N).  See gated_delta_prefill in la.h."""
    B, H, N, dk = k.shape
    dv = v.shape[3]
    dev = k.device
    code = _dtype_code(k)
    _need(v, "v", (B, H, N, dv), k.dtype, dev)
    _need(beta, "beta", (B, H, N), torch.float32, dev)
    _need(alpha, "alpha", (B, H, N), torch.float32, dev)
    _need(S0, "S0", (B, H, dk, dv), torch.float32, dev)
    if reads is None:
        reads = torch.empty((B, H, N, dv), dtype=torch.float32, device=dev)
    if S_N is None:
        S_N = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    _need(reads, "reads", (B, H, N, dv), torch.float32, dev)
    _need(S_N, "S_N", (B, H, dk, dv), torch.float32, dev)
    st = load().gated_delta_prefill(_ptr(k), _ptr(v), code, _ptr(beta), _ptr(alpha), B, H,
                                    N, dk, dv, _ptr(S0), _ptr(reads), _ptr(S_N), _stream(dev))
    _check("gated_delta_prefill", st)
    return reads, S_N


_vws_cache: dict = {}


def _cached_scratch(dev, need):
    """A device uint8 scratch of at least `need` bytes, cached per device and
    grown on demand (shared by the optional-workspace calls; they run in
    stream order on the current stream).  None when need is 0."""
    if need <= 0:
        return None
    key = dev if dev.index is not None else torch.device("cuda", torch.cuda.current_device())
    ws = _vws_cache.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
        _vws_cache[key] = ws
    return ws


def _ws_args(ws):
    if ws is False or ws is None:
        return None, 0
    return _ptr(ws), ws.numel() * ws.element_size()


def variant_workspace_bytes(B, H, N, dk, dv, dtype=torch.bfloat16, mode=LA_MODE_CAUSAL,
                            decay=True) -> int:
    """la_prefill_variant_workspace_bytes (0: the call uses no workspace)."""
    code = LA_BF16 if dtype == torch.bfloat16 else LA_F32
    return int(load().la_prefill_variant_workspace_bytes(B, H, N, dk, dv, code, int(mode),
                                                         int(bool(decay))))


def prefill_variant(q, k, v, alpha=None, mode=LA_MODE_CAUSAL, eps=1e-6, S0=None, z0=None, *,
                    o=None, S_N=None, z_N=None, ws=None):
    """la_prefill_variant: decayed state and/or another read order; returns
    (o, S_N, z_N).  See la_prefill_variant in la.h.  ws: a device uint8
    tensor for the workspace; None uses a scratch cached per device, grown on
    demand; False passes none (the one-block-per-head form)."""
    B, H, N, dk = q.shape
    dv = v.shape[3]
    dev = q.device
    code = _dtype_code(q)
    _need(k, "k", (B, H, N, dk), q.dtype, dev)
    _need(v, "v", (B, H, N, dv), q.dtype, dev)
    _need(alpha, "alpha", (B, H, N), torch.float32, dev)
    _need(S0, "S0", (B, H, dk, dv), torch.float32, dev)
    _need(z0, "z0", (B, H, dk), torch.float32, dev)
    if o is None:
        o = torch.empty((B, H, N, dv), dtype=torch.float32, device=dev)
    if S_N is None:
        S_N = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    if z_N is None:
        z_N = torch.empty((B, H, dk), dtype=torch.float32, device=dev)
    _need(o, "o", (B, H, N, dv), torch.float32, dev)
    _need(S_N, "S_N", (B, H, dk, dv), torch.float32, dev)
    _need(z_N, "z_N", (B, H, dk), torch.float32, dev)
    if ws is None:
        ws = _cached_scratch(dev, variant_workspace_bytes(B, H, N, dk, dv, q.dtype, mode,
                                                          alpha is not None))
    ws_ptr, ws_bytes = _ws_args(ws)
    st = load().la_prefill_variant(_ptr(q), _ptr(k), _ptr(v), code, B, H, N, dk, dv,
                                   ctypes.c_float(eps), _ptr(alpha), int(mode), _ptr(S0),
                                   _ptr(z0), _ptr(o), _ptr(S_N), _ptr(z_N), ws_ptr, ws_bytes,
                                   _stream(dev))
    _check("la_prefill_variant", st)
    return o, S_N, z_N


def backward_workspace_bytes(B, H, N, dk, dv, dtype=torch.bfloat16) -> int:
    """la_prefill_backward_workspace_bytes (0: the call uses no workspace)."""
    code = LA_BF16 if dtype == torch.bfloat16 else LA_F32
    return int(load().la_prefill_backward_workspace_bytes(B, H, N, dk, dv, code))


def prefill_backward(q, k, v, dO, eps=1e-6, S0=None, z0=None, dS_N=None, dz_N=None, *,
                     want_state_grads=True, ws=None):
    """la_prefill_backward: returns (dq, dk, dv, dS0, dz0) (the last two None
    unless want_state_grads).  See la_prefill_backward in la.h.  ws as for
    prefill_variant: None uses the cached per-device scratch, False none (one
    block per head), else a device uint8 tensor."""
    B, H, N, dk = q.shape
    dv = v.shape[3]
    dev = q.device
    code = _dtype_code(q)
    _need(k, "k", (B, H, N, dk), q.dtype, dev)
    _need(v, "v", (B, H, N, dv), q.dtype, dev)
    _need(dO, "dO", (B, H, N, dv), torch.float32, dev)
    _need(S0, "S0", (B, H, dk, dv), torch.float32, dev)
    _need(z0, "z0", (B, H, dk), torch.float32, dev)
    _need(dS_N, "dS_N", (B, H, dk, dv), torch.float32, dev)
    _need(dz_N, "dz_N", (B, H, dk), torch.float32, dev)
    dq = torch.empty((B, H, N, dk), dtype=torch.float32, device=dev)
    dk_ = torch.empty((B, H, N, dk), dtype=torch.float32, device=dev)
    dv_ = torch.empty((B, H, N, dv), dtype=torch.float32, device=dev)
    dS0 = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev) if want_state_grads else None
    dz0 = torch.empty((B, H, dk), dtype=torch.float32, device=dev) if want_state_grads else None
    if ws is None:
        ws = _cached_scratch(dev, backward_workspace_bytes(B, H, N, dk, dv, q.dtype))
    ws_ptr, ws_bytes = _ws_args(ws)
    st = load().la_prefill_backward(_ptr(q), _ptr(k), _ptr(v), code, B, H, N, dk, dv,
                                    ctypes.c_float(eps), _ptr(S0), _ptr(z0), _ptr(dO),
                                    _ptr(dS_N), _ptr(dz_N), _ptr(dq), _ptr(dk_), _ptr(dv_),
                                    _ptr(dS0), _ptr(dz0), ws_ptr, ws_bytes, _stream(dev))
    _check("la_prefill_backward", st)
    return dq, dk_, dv_, dS0, dz0


def read_device_status(ws, stream=None) -> int:
    """Synchronize and return/clear the device status word of a workspace."""
    s = ctypes.c_void_p(stream.cuda_stream) if stream is not None else _stream(ws.device)
    return int(load().la_read_device_status(_ptr(ws), s))


def delta_read_device_status(stream=None) -> int:
    """Synchronize and return/clear the tensor-core delta kernel's status word
    (current device)."""
    import torch
    s = ctypes.c_void_p(stream.cuda_stream) if stream is not None else \
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return int(load().delta_read_device_status(s))


def prefill_noalloc(q, k, v, eps=1e-6, S0=None, z0=None, *, o=None, S_N=None, z_N=None,
                    chunk=0):
    """la_prefill_noalloc: the same computation as prefill() for callers that
    cannot allocate device memory; the library uses its own fixed 16 MiB
    device scratch instead of a workspace (see include/la.h)."""
    lib = load()
    fn = lib.la_prefill_noalloc
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp, vp, vp, i, i, i, i, i, i, f, vp, vp, vp, vp, vp, i, vp]
    fn.restype = i
    B, H, N, dk = q.shape
    dv = v.shape[3]
    dev = q.device
    dt = q.dtype
    code = _dtype_code(q)
    _need(k, "k", (B, H, N, dk), dt, dev)
    _need(v, "v", (B, H, N, dv), dt, dev)
    _need(S0, "S0", (B, H, dk, dv), torch.float32, dev)
    _need(z0, "z0", (B, H, dk), torch.float32, dev)
    if o is None:
        o = torch.empty((B, H, N, dv), dtype=torch.float32, device=dev)
    if S_N is None:
        S_N = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    if z_N is None:
        z_N = torch.empty((B, H, dk), dtype=torch.float32, device=dev)
    st = fn(_ptr(q), _ptr(k), _ptr(v), code, B, H, N, dk, dv, float(eps), _ptr(S0),
            _ptr(z0), _ptr(o), _ptr(S_N), _ptr(z_N), int(chunk), _stream(dev))
    _check("la_prefill_noalloc", st)
    return o, S_N, z_N
