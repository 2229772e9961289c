"""Float64 CPU oracle of the gated delta rule -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline and
reference arm import this package.  The product path (the CUDA library and its
Python binding) never does, and shares no code with it.

The arithmetic lives in ``gdn_oracle.c`` (plain C, float64, OpenMP over the
independent (batch, head) streams); this module only marshals numpy arrays:

* :func:`gated_delta_fwd` -- the token-by-token recurrence
  ``S_t = alpha_t S_{t-1}(I - beta_t k_t k_t^T) + beta_t v_t k_t^T``,
  ``o_t = S_t q_t`` ("Sparse Delta Memory: layer and kernels", "What the layer
  computes" and its dense-limit paragraph; shapes and streaming contract from
  "OpenGDN", "Core operator reference").
* :func:`gated_delta_bwd` -- the chain rule through the same loop, in reverse,
  for ``L = sum(d_o * o) + sum(d_final_state * final_state)``.

Shapes: q, k ``[B,T,H,K]``; v, o ``[B,T,H,V]``; alpha, beta ``[B,T,H]``;
states ``[B,H,V,K]``.  Every array is converted to contiguous float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gdn_oracle.c`` into ``liboracle.so`` with gcc (-O2, OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
           "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        d = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        lib.oracle_gdn_fwd.argtypes = [i64] * 5 + [d] * 8 + [ctypes.c_int]
        lib.oracle_gdn_fwd.restype = ctypes.c_int
        lib.oracle_gdn_bwd.argtypes = ([i64] * 5 + [d] * 6 + [d] * 2 + [d] * 6
                                       + [i64, ctypes.c_int])
        lib.oracle_gdn_bwd.restype = ctypes.c_int
        lib.oracle_threads.argtypes = [ctypes.c_int]
        lib.oracle_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def threads(n: int = 0) -> int:
    """Number of OpenMP threads a call with ``threads=n`` uses."""
    return int(_load().oracle_threads(int(n)))


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # a torch tensor
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a):
    if a is None:
        return ctypes.cast(None, ctypes.POINTER(ctypes.c_double))
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _dims(q, v):
    B, T, H, K = q.shape
    V = v.shape[-1]
    return B, T, H, K, V


def gated_delta_fwd(q, k, v, alpha, beta, initial_state=None, threads: int = 0):
    """Token-by-token forward.  Returns ``(o [B,T,H,V], final_state [B,H,V,K])``."""
    q, k, v, alpha, beta = map(_f64, (q, k, v, alpha, beta))
    s0 = _f64(initial_state)
    B, T, H, K, V = _dims(q, v)
    assert k.shape == q.shape and v.shape[:3] == q.shape[:3]
    assert alpha.shape == (B, T, H) and beta.shape == (B, T, H)
    if s0 is not None:
        assert s0.shape == (B, H, V, K)
    o = np.zeros((B, T, H, V))
    sT = np.zeros((B, H, V, K))
    rc = _load().oracle_gdn_fwd(B, T, H, K, V, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                                _ptr(beta), _ptr(s0), _ptr(o), _ptr(sT), int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_gdn_fwd failed with code {rc}")
    return o, sT


def gated_delta_bwd(q, k, v, alpha, beta, initial_state, d_o, d_final_state=None,
                    seg: int = 64, threads: int = 0):
    """Reverse recurrence.  Returns a dict with dq, dk, dv, dalpha, dbeta and
    d_initial_state (``[B,H,V,K]``), the gradients of
    ``sum(d_o * o) + sum(d_final_state * final_state)``."""
    q, k, v, alpha, beta, d_o = map(_f64, (q, k, v, alpha, beta, d_o))
    s0 = _f64(initial_state)
    dsT = _f64(d_final_state)
    B, T, H, K, V = _dims(q, v)
    assert d_o.shape == v.shape
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v),
               dalpha=np.zeros_like(alpha), dbeta=np.zeros_like(beta),
               d_initial_state=np.zeros((B, H, V, K)))
    rc = _load().oracle_gdn_bwd(
        B, T, H, K, V, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(s0),
        _ptr(d_o), _ptr(dsT), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
        _ptr(out["dalpha"]), _ptr(out["dbeta"]), _ptr(out["d_initial_state"]),
        int(seg), int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_gdn_bwd failed with code {rc}")
    return out
