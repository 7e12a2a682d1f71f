"""fp64 CPU oracle for normalized causal linear attention and the delta rule.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``fixed_state_recurrent_gb300``) never imports it, and it imports nothing from
the product library: the two share no code.

The arithmetic lives in ``la_oracle.c`` (plain C, double precision).  This
module only compiles it with gcc and marshals numpy arrays through ctypes.
Every entry takes float64 numpy arrays in the layouts documented in
``la_oracle.h`` ([B,H,N,d] tokens, [B,H,dk,dv] state) and returns new arrays.

Definitions followed (page "AIGC 基本功|线性、循环与记忆架构-LinearMem",
section 03; page "sequence-models" practice notes, "Delta-rule fast weight";
page "线性注意力与SSM", sections 1.3 and 3):

* ``phi(u) = u + 1 if u > 0 else exp(u)``
* ``la_recurrent``: S_t = S_{t-1} + phi(k_t) v_t^T, z_t = z_{t-1} + phi(k_t),
  o_t = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps)   (write, then read)
* ``la_quadratic``: the same outputs from explicit masked phi(Q) phi(K)^T
* ``la_chunked``: the same outputs chunk by chunk, carrying only (S, z)
* ``la_decode_step``: one step of the recurrence on a given state
* ``delta``: reads_t = k_t^T S_{t-1}; S_t = S_{t-1} + beta_t k_t (v_t - reads_t)^T
* ``gated_delta``: D = alpha_t S_{t-1}; reads_t = k_t^T D;
  S_t = D + beta_t k_t (v_t - reads_t)^T   (forget, then correct)
* ``la_variant``: the recurrence with a scalar decay alpha_t of the old (S, z)
  (mode 0, write then read), read-then-write (mode 1, strictly past), or
  non-causal (mode 2: the state over all tokens, then every query reads it)
* ``la_variant_quadratic``: the same outputs from explicit weights
* ``la_backward``: the exact gradient of ``la_recurrent`` (states recomputed)
* ``outer_read``: additive identity-feature memory S = sum k v^T, read q^T S
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "la_oracle.c")
_HDR = os.path.join(_HERE, "la_oracle.h")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liblaoracle.so")

_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile la_oracle.c into a shared library (gcc, -O2, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= newest_src):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-Wall", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i, d, p = ctypes.c_int, ctypes.c_double, _D
        lib.orc_phi.argtypes = [p, p, ctypes.c_int64]
        lib.orc_la_recurrent.argtypes = [p, p, p, i, i, i, i, i, d, p, p, p, p, p, i]
        lib.orc_la_quadratic.argtypes = [p, p, p, i, i, i, i, i, d, p, p, p, i]
        lib.orc_la_chunked.argtypes = [p, p, p, i, i, i, i, i, d, p, p, i, p, p, p, i]
        lib.orc_la_decode_step.argtypes = [p, p, p, i, i, i, i, d, p, p, p, i]
        lib.orc_delta.argtypes = [p, p, p, i, i, i, i, i, p, p, p, i]
        lib.orc_outer_read.argtypes = [p, p, i, i, i, p, i, p]
        lib.orc_gated_delta.argtypes = [p, p, p, p, i, i, i, i, i, p, p, p, i]
        lib.orc_la_variant.argtypes = [p, p, p, p, i, i, i, i, i, d, i, p, p, p, p, p, i]
        lib.orc_la_variant_quadratic.argtypes = [p, p, p, p, i, i, i, i, i, d, i, p, p, p, i]
        lib.orc_la_backward.argtypes = [p, p, p, i, i, i, i, i, d, p, p, p, p, p, p, p, p, p, p, i]
        for name in ("orc_phi", "orc_la_recurrent", "orc_la_quadratic",
                     "orc_la_chunked", "orc_la_decode_step", "orc_delta",
                     "orc_outer_read", "orc_default_threads", "orc_gated_delta",
                     "orc_la_variant", "orc_la_variant_quadratic", "orc_la_backward"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def default_threads() -> int:
    return _load().orc_default_threads()


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(_D)


def _shape4(q, v):
    if q.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    B, H, N, dk = q.shape
    dv = v.shape[3]
    return B, H, N, dk, dv


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name}: invalid arguments")


def phi(u):
    u = _f64(u)
    out = np.empty_like(u)
    _check(_load().orc_phi(_ptr(u), _ptr(out), u.size), "phi")
    return out


def la_recurrent(q, k, v, eps=1e-6, S0=None, z0=None, threads=0):
    """Returns (o, S_N, z_N) from the token-by-token recurrence."""
    q, k, v, S0, z0 = map(_f64, (q, k, v, S0, z0))
    B, H, N, dk, dv = _shape4(q, v)
    o = np.empty((B, H, N, dv))
    S = np.empty((B, H, dk, dv))
    z = np.empty((B, H, dk))
    _check(_load().orc_la_recurrent(_ptr(q), _ptr(k), _ptr(v), B, H, N, dk, dv,
                                    eps, _ptr(S0), _ptr(z0), _ptr(o), _ptr(S),
                                    _ptr(z), threads), "la_recurrent")
    return o, S, z


def la_quadratic(q, k, v, eps=1e-6, S0=None, z0=None, threads=0):
    """Returns o from the explicit causal-masked weights (small N only)."""
    q, k, v, S0, z0 = map(_f64, (q, k, v, S0, z0))
    B, H, N, dk, dv = _shape4(q, v)
    o = np.empty((B, H, N, dv))
    _check(_load().orc_la_quadratic(_ptr(q), _ptr(k), _ptr(v), B, H, N, dk, dv,
                                    eps, _ptr(S0), _ptr(z0), _ptr(o), threads),
           "la_quadratic")
    return o


def la_chunked(q, k, v, C, eps=1e-6, S0=None, z0=None, threads=0):
    """Returns (o, S_N, z_N) from the chunkwise form with chunk length C."""
    q, k, v, S0, z0 = map(_f64, (q, k, v, S0, z0))
    B, H, N, dk, dv = _shape4(q, v)
    o = np.empty((B, H, N, dv))
    S = np.empty((B, H, dk, dv))
    z = np.empty((B, H, dk))
    _check(_load().orc_la_chunked(_ptr(q), _ptr(k), _ptr(v), B, H, N, dk, dv,
                                  eps, _ptr(S0), _ptr(z0), int(C), _ptr(o),
                                  _ptr(S), _ptr(z), threads), "la_chunked")
    return o, S, z


def la_decode_step(q, k, v, S, z, eps=1e-6, threads=0):
    """One decode step.  q,k [B,H,dk], v [B,H,dv], S [B,H,dk,dv], z [B,H,dk].
    Returns (o, S_new, z_new); the inputs are not modified."""
    q, k, v = map(_f64, (q, k, v))
    S = np.array(S, dtype=np.float64, copy=True, order="C")
    z = np.array(z, dtype=np.float64, copy=True, order="C")
    B, H, dk = q.shape
    dv = v.shape[2]
    o = np.empty((B, H, dv))
    _check(_load().orc_la_decode_step(_ptr(q), _ptr(k), _ptr(v), B, H, dk, dv,
                                      eps, _ptr(S), _ptr(z), _ptr(o), threads),
           "la_decode_step")
    return o, S, z


def delta(k, v, beta, S0=None, threads=0):
    """Returns (reads, S_N) of the delta-rule memory."""
    k, v, beta, S0 = map(_f64, (k, v, beta, S0))
    B, H, N, dk, dv = _shape4(k, v)
    if beta.shape != (B, H, N):
        raise ValueError("beta must be [B, H, N]")
    reads = np.empty((B, H, N, dv))
    S = np.empty((B, H, dk, dv))
    _check(_load().orc_delta(_ptr(k), _ptr(v), _ptr(beta), B, H, N, dk, dv,
                             _ptr(S0), _ptr(reads), _ptr(S), threads), "delta")
    return reads, S


def gated_delta(k, v, beta, alpha=None, S0=None, threads=0):
    """Returns (reads, S_N) of the gated delta rule (alpha None = 1)."""
    k, v, beta, alpha, S0 = map(_f64, (k, v, beta, alpha, S0))
    B, H, N, dk, dv = _shape4(k, v)
    if beta.shape != (B, H, N) or (alpha is not None and alpha.shape != (B, H, N)):
        raise ValueError("beta and alpha must be [B, H, N]")
    reads = np.empty((B, H, N, dv))
    S = np.empty((B, H, dk, dv))
    _check(_load().orc_gated_delta(_ptr(k), _ptr(v), _ptr(beta), _ptr(alpha), B, H, N,
                                   dk, dv, _ptr(S0), _ptr(reads), _ptr(S), threads),
           "gated_delta")
    return reads, S


MODE_CAUSAL, MODE_READ_BEFORE_WRITE, MODE_NONCAUSAL = 0, 1, 2


def la_variant(q, k, v, alpha=None, mode=MODE_CAUSAL, eps=1e-6, S0=None, z0=None,
               threads=0):
    """Returns (o, S_N, z_N) of a variant of the recurrence (see la_oracle.h)."""
    q, k, v, alpha, S0, z0 = map(_f64, (q, k, v, alpha, S0, z0))
    B, H, N, dk, dv = _shape4(q, v)
    if alpha is not None and alpha.shape != (B, H, N):
        raise ValueError("alpha must be [B, H, N]")
    o = np.empty((B, H, N, dv))
    S = np.empty((B, H, dk, dv))
    z = np.empty((B, H, dk))
    _check(_load().orc_la_variant(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), B, H, N, dk,
                                  dv, eps, int(mode), _ptr(S0), _ptr(z0), _ptr(o),
                                  _ptr(S), _ptr(z), threads), "la_variant")
    return o, S, z


def la_variant_quadratic(q, k, v, alpha=None, mode=MODE_CAUSAL, eps=1e-6, S0=None,
                         z0=None, threads=0):
    """Returns o of a variant from its explicit weights (small N only)."""
    q, k, v, alpha, S0, z0 = map(_f64, (q, k, v, alpha, S0, z0))
    B, H, N, dk, dv = _shape4(q, v)
    o = np.empty((B, H, N, dv))
    _check(_load().orc_la_variant_quadratic(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), B, H,
                                            N, dk, dv, eps, int(mode), _ptr(S0), _ptr(z0),
                                            _ptr(o), threads), "la_variant_quadratic")
    return o


def la_backward(q, k, v, dO, eps=1e-6, S0=None, z0=None, dS_N=None, dz_N=None, threads=0):
    """Returns (dq, dk, dv, dS0, dz0): the gradient of la_recurrent's
    (o, S_N, z_N) against dO, dS_N, dz_N (None = zero)."""
    q, k, v, dO, S0, z0, dS_N, dz_N = map(_f64, (q, k, v, dO, S0, z0, dS_N, dz_N))
    B, H, N, dk, dv = _shape4(q, v)
    dq = np.empty((B, H, N, dk))
    dk_ = np.empty((B, H, N, dk))
    dv_ = np.empty((B, H, N, dv))
    dS0 = np.empty((B, H, dk, dv))
    dz0 = np.empty((B, H, dk))
    _check(_load().orc_la_backward(_ptr(q), _ptr(k), _ptr(v), B, H, N, dk, dv, eps, _ptr(S0),
                                   _ptr(z0), _ptr(dO), _ptr(dS_N), _ptr(dz_N), _ptr(dq),
                                   _ptr(dk_), _ptr(dv_), _ptr(dS0), _ptr(dz0), threads),
           "la_backward")
    return dq, dk_, dv_, dS0, dz0


def outer_read(keys, values, queries):
    """Additive identity-feature memory: reads = queries @ (sum_m k_m v_m^T)."""
    keys, values, queries = map(_f64, (keys, values, queries))
    M, dk = keys.shape
    dv = values.shape[1]
    P = queries.shape[0]
    reads = np.empty((P, dv))
    _check(_load().orc_outer_read(_ptr(keys), _ptr(values), M, dk, dv,
                                  _ptr(queries), P, _ptr(reads)), "outer_read")
    return reads
