"""Python binding of libgdn.so (the C ABI declared in include/gdn.h).

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, device buffers (outputs, workspace, saved states) are allocated with
torch, and the call goes through ctypes to the C entry point of the same name on
torch's current CUDA stream.  Every step of the computation runs in the
library's CUDA kernels; there is no CPU or Python fallback -- if the library is
missing, importing or calling raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_WORKSPACE, GDN_ERR_CUDA = range(5)
GDN_F32, GDN_BF16 = 0, 1


class GdnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"gdn status {status}: {message}")
        self.status = status


class gdn_problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("T", ctypes.c_int64), ("H", ctypes.c_int64),
                ("K", ctypes.c_int64), ("V", ctypes.c_int64), ("chunk", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


_lib = None
_vp = ctypes.c_void_p


def load_library():
    """Load libgdn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(gdn_problem)
    lib.gdn_version.restype = ctypes.c_int
    lib.gdn_status_string.argtypes = [ctypes.c_int]
    lib.gdn_status_string.restype = ctypes.c_char_p
    lib.gdn_last_error.restype = ctypes.c_char_p
    for fn in ("gdn_fwd_workspace_bytes", "gdn_saved_bytes", "gdn_bwd_workspace_bytes"):
        getattr(lib, fn).argtypes = [P]
        getattr(lib, fn).restype = ctypes.c_size_t
    lib.gdn_fwd.argtypes = [P] + [_vp] * 10 + [ctypes.c_size_t, _vp]
    lib.gdn_fwd.restype = ctypes.c_int
    lib.gdn_bwd.argtypes = [P] + [_vp] * 16 + [ctypes.c_size_t, _vp]
    lib.gdn_bwd.restype = ctypes.c_int
    for fn in ("gdn_raw_saved_bytes", "gdn_raw_fwd_workspace_bytes", "gdn_raw_bwd_workspace_bytes"):
        getattr(lib, fn).argtypes = [P]
        getattr(lib, fn).restype = ctypes.c_size_t
    lib.gdn_fwd_raw.argtypes = [P] + [_vp] * 10 + [ctypes.c_size_t, _vp]
    lib.gdn_fwd_raw.restype = ctypes.c_int
    lib.gdn_bwd_raw.argtypes = [P] + [_vp] * 16 + [ctypes.c_size_t, _vp]
    lib.gdn_bwd_raw.restype = ctypes.c_int
    for fn in ("gdn_reset_saved_bytes", "gdn_reset_fwd_workspace_bytes", "gdn_reset_bwd_workspace_bytes"):
        getattr(lib, fn).argtypes = [P, ctypes.c_int64]
        getattr(lib, fn).restype = ctypes.c_size_t
    lib.gdn_reset_fwd.argtypes = [P, ctypes.c_int64] + [_vp] * 11 + [ctypes.c_size_t, _vp]
    lib.gdn_reset_fwd.restype = ctypes.c_int
    lib.gdn_reset_bwd.argtypes = [P, ctypes.c_int64] + [_vp] * 17 + [ctypes.c_size_t, _vp]
    lib.gdn_reset_bwd.restype = ctypes.c_int
    lib.gdn_fwd_noalloc.argtypes = [P] + [_vp] * 8 + [_vp]
    lib.gdn_fwd_noalloc.restype = ctypes.c_int
    lib.gdn_decode.argtypes = [P] + [_vp] * 7 + [_vp]
    lib.gdn_decode.restype = ctypes.c_int
    lib.gdn_prologue_fwd.argtypes = [P] + [_vp] * 8 + [_vp]
    lib.gdn_prologue_fwd.restype = ctypes.c_int
    lib.gdn_prologue_bwd.argtypes = [P] + [_vp] * 12 + [_vp]
    lib.gdn_prologue_bwd.restype = ctypes.c_int
    for fn in ("gdn_varlen_fwd_workspace_bytes", "gdn_varlen_bwd_workspace_bytes", "gdn_varlen_saved_bytes"):
        getattr(lib, fn).argtypes = [P, ctypes.c_int64]
        getattr(lib, fn).restype = ctypes.c_size_t
    lib.gdn_varlen_fwd.argtypes = [P, ctypes.c_int64] + [_vp] * 11 + [ctypes.c_size_t, _vp]
    lib.gdn_varlen_fwd.restype = ctypes.c_int
    lib.gdn_varlen_bwd.argtypes = [P, ctypes.c_int64] + [_vp] * 17 + [ctypes.c_size_t, _vp]
    lib.gdn_varlen_bwd.restype = ctypes.c_int
    lib.gdn_count_nonfinite.argtypes = [_vp, ctypes.c_int64, ctypes.c_int, _vp, _vp]
    lib.gdn_count_nonfinite.restype = ctypes.c_int
    lib.gdn_set_sequence_split.argtypes = [ctypes.c_int]
    lib.gdn_set_sequence_split.restype = ctypes.c_int
    lib.gdn_test_set_wait_limit.argtypes = [ctypes.c_uint32]
    lib.gdn_test_set_wait_limit.restype = ctypes.c_int
    lib.gdn_get_sequence_split.restype = ctypes.c_int
    lib.gdn_num_kernels.restype = ctypes.c_int
    lib.gdn_kernel_name.argtypes = [ctypes.c_int]
    lib.gdn_kernel_name.restype = ctypes.c_char_p
    lib.gdn_profiler_start.argtypes = [ctypes.c_int]
    lib.gdn_profiler_start.restype = ctypes.c_int
    lib.gdn_profiler_stop.restype = ctypes.c_int
    lib.gdn_profiler_summary.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                         ctypes.POINTER(ctypes.c_double)]
    lib.gdn_profiler_summary.restype = ctypes.c_int
    lib.gdn_profiler_release.restype = None
    _lib = lib
    return lib


EXPORTED = ("gdn_version", "gdn_status_string", "gdn_last_error", "gdn_fwd_workspace_bytes",
            "gdn_saved_bytes", "gdn_bwd_workspace_bytes", "gdn_fwd", "gdn_bwd",
            "gdn_num_kernels", "gdn_kernel_name", "gdn_profiler_start", "gdn_profiler_stop",
            "gdn_profiler_summary", "gdn_profiler_release", "gdn_fwd_noalloc", "gdn_decode",
            "gdn_prologue_fwd", "gdn_prologue_bwd", "gdn_varlen_fwd_workspace_bytes",
            "gdn_varlen_bwd_workspace_bytes", "gdn_varlen_saved_bytes", "gdn_varlen_fwd", "gdn_varlen_bwd",
            "gdn_set_sequence_split", "gdn_get_sequence_split", "gdn_count_nonfinite",
            "gdn_test_set_wait_limit")


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return GDN_F32
    if dt == torch.bfloat16:
        return GDN_BF16
    raise GdnError(GDN_ERR_UNSUPPORTED, f"dtype {dt} (use float32 or bfloat16)")


def make_problem(B, T, H, K, V, chunk=64, dtype=torch.bfloat16) -> gdn_problem:
    code = dtype if isinstance(dtype, int) else _dtype_code(dtype)
    return gdn_problem(int(B), int(T), int(H), int(K), int(V), int(chunk), int(code))


def gdn_version() -> int:
    return int(load_library().gdn_version())


def gdn_status_string(status: int) -> str:
    return load_library().gdn_status_string(int(status)).decode()


def gdn_last_error() -> str:
    return load_library().gdn_last_error().decode()


def gdn_fwd_workspace_bytes(p: gdn_problem) -> int:
    return int(load_library().gdn_fwd_workspace_bytes(ctypes.byref(p)))


def gdn_saved_bytes(p: gdn_problem) -> int:
    return int(load_library().gdn_saved_bytes(ctypes.byref(p)))


def gdn_bwd_workspace_bytes(p: gdn_problem) -> int:
    return int(load_library().gdn_bwd_workspace_bytes(ctypes.byref(p)))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(status: int):
    if status != GDN_OK:
        raise GdnError(status, gdn_last_error() or gdn_status_string(status))


def _need(t, name, shape, dtype, device):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise GdnError(GDN_ERR_INVALID_ARG, f"{name} is on {t.device}, expected {device}")
    if tuple(t.shape) != tuple(shape):
        raise GdnError(GDN_ERR_INVALID_ARG, f"{name} has shape {tuple(t.shape)}, expected {shape}")
    if t.dtype != dtype:
        raise GdnError(GDN_ERR_INVALID_ARG, f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise GdnError(GDN_ERR_INVALID_ARG, f"{name} must be contiguous")


def _stream_handle(device, stream):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def gdn_fwd(q, k, v, alpha, beta, initial_state=None, *, chunk: int = 64, o=None,
            final_state=True, saved=False, workspace=None, stream=None):
    """Chunkwise gated delta rule forward.

    q, k [B,T,H,K]; v [B,T,H,V]; alpha, beta [B,T,H] (all float32 or all bf16,
    contiguous, on one CUDA device); initial_state float32 [B,H,V,K] or None.
    ``final_state``: True (allocate), a float32 tensor to fill (may be
    initial_state itself), or False/None (not written).  ``saved``: True to
    allocate and return the chunk-boundary states for :func:`gdn_bwd`, or a
    uint8/float tensor of at least gdn_saved_bytes() bytes.
    Returns ``(o, final_state or None, saved or None)``.
    """
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise GdnError(GDN_ERR_INVALID_ARG, "inputs must be CUDA tensors")
    B, T, H, K = q.shape
    V = v.shape[-1]
    dt = q.dtype
    p = make_problem(B, T, H, K, V, chunk, dt)
    _need(k, "k", (B, T, H, K), dt, dev)
    _need(v, "v", (B, T, H, V), dt, dev)
    _need(q, "q", (B, T, H, K), dt, dev)
    _need(alpha, "alpha", (B, T, H), dt, dev)
    _need(beta, "beta", (B, T, H), dt, dev)
    _need(initial_state, "initial_state", (B, H, V, K), torch.float32, dev)
    if o is None:
        o = torch.empty((B, T, H, V), dtype=dt, device=dev)
    _need(o, "o", (B, T, H, V), dt, dev)
    if final_state is True:
        final_state = torch.empty((B, H, V, K), dtype=torch.float32, device=dev)
    elif final_state is False:
        final_state = None
    _need(final_state, "final_state", (B, H, V, K), torch.float32, dev)
    if saved is True:
        saved = torch.empty(max(gdn_saved_bytes(p), 1), dtype=torch.uint8, device=dev)
    elif saved is False:
        saved = None
    ws_need = gdn_fwd_workspace_bytes(p)
    if workspace is None:
        workspace = torch.empty(max(ws_need, 1), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.gdn_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                     _ptr(initial_state), _ptr(o), _ptr(final_state), _ptr(saved),
                     _ptr(workspace), ws_bytes, _stream_handle(dev, stream))
    _check(st)
    return o, final_state, saved


def gdn_bwd(q, k, v, alpha, beta, initial_state, d_o, d_final_state=None, *, saved=None,
            chunk: int = 64, grads=None, d_initial_state=True, workspace=None, stream=None):
    """Gradients of ``sum(d_o * o) + sum(d_final_state * final_state)``.

    ``saved`` is the buffer returned by ``gdn_fwd(..., saved=True)`` with the same
    inputs, or None (the chunk-boundary states are then recomputed).
    Returns ``(dq, dk, dv, dalpha, dbeta, d_initial_state or None)``.
    """
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise GdnError(GDN_ERR_INVALID_ARG, "inputs must be CUDA tensors")
    B, T, H, K = q.shape
    V = v.shape[-1]
    dt = q.dtype
    p = make_problem(B, T, H, K, V, chunk, dt)
    for t, n, s in ((k, "k", (B, T, H, K)), (v, "v", (B, T, H, V)), (q, "q", (B, T, H, K)),
                    (alpha, "alpha", (B, T, H)), (beta, "beta", (B, T, H)),
                    (d_o, "d_o", (B, T, H, V))):
        _need(t, n, s, dt, dev)
    _need(initial_state, "initial_state", (B, H, V, K), torch.float32, dev)
    _need(d_final_state, "d_final_state", (B, H, V, K), torch.float32, dev)
    if saved is not None and saved.numel() * saved.element_size() < gdn_saved_bytes(p):
        raise GdnError(GDN_ERR_INVALID_ARG, "saved buffer is smaller than gdn_saved_bytes()")
    if grads is None:
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
                 torch.empty_like(alpha), torch.empty_like(beta))
    dq, dk, dv, da, db = grads
    if d_initial_state is True:
        d_initial_state = torch.empty((B, H, V, K), dtype=torch.float32, device=dev)
    elif d_initial_state is False:
        d_initial_state = None
    ws_need = gdn_bwd_workspace_bytes(p)
    if workspace is None:
        workspace = torch.empty(max(ws_need, 1), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.gdn_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                     _ptr(initial_state), _ptr(saved), _ptr(d_o), _ptr(d_final_state),
                     _ptr(dq), _ptr(dk), _ptr(dv), _ptr(da), _ptr(db), _ptr(d_initial_state),
                     _ptr(workspace), ws_bytes, _stream_handle(dev, stream))
    _check(st)
    return dq, dk, dv, da, db, d_initial_state


def gdn_raw_saved_bytes(p: gdn_problem) -> int:
    return int(load_library().gdn_raw_saved_bytes(ctypes.byref(p)))


def gdn_raw_fwd_workspace_bytes(p: gdn_problem) -> int:
    return int(load_library().gdn_raw_fwd_workspace_bytes(ctypes.byref(p)))


def gdn_raw_bwd_workspace_bytes(p: gdn_problem) -> int:
    return int(load_library().gdn_raw_bwd_workspace_bytes(ctypes.byref(p)))


def gdn_fwd_raw(q_raw, k_raw, v, a_logit, b_logit, initial_state=None, *, chunk: int = 64, o=None,
                final_state=True, saved=False, workspace=None, stream=None):
    """The forward with its prologue folded in (``gdn_fwd_raw``): q_raw, k_raw are
    normalised to unit length per row and the gates come from the logits
    (alpha = exp(-softplus(a_logit)), beta = sigmoid(b_logit)).  Shapes and
    arguments as :func:`gdn_fwd`; ``saved`` (True or a buffer of
    gdn_raw_saved_bytes()) feeds :func:`gdn_bwd_raw`.  Returns
    ``(o, final_state or None, saved or None)``."""
    lib = load_library()
    dev = q_raw.device
    if dev.type != "cuda":
        raise GdnError(GDN_ERR_INVALID_ARG, "inputs must be CUDA tensors")
    B, T, H, K = q_raw.shape
    V = v.shape[-1]
    dt = q_raw.dtype
    p = make_problem(B, T, H, K, V, chunk, dt)
    for t, n, sh in ((q_raw, "q_raw", (B, T, H, K)), (k_raw, "k_raw", (B, T, H, K)), (v, "v", (B, T, H, V)),
                     (a_logit, "a_logit", (B, T, H)), (b_logit, "b_logit", (B, T, H))):
        _need(t, n, sh, dt, dev)
    _need(initial_state, "initial_state", (B, H, V, K), torch.float32, dev)
    if o is None:
        o = torch.empty((B, T, H, V), dtype=dt, device=dev)
    _need(o, "o", (B, T, H, V), dt, dev)
    if final_state is True:
        final_state = torch.empty((B, H, V, K), dtype=torch.float32, device=dev)
    elif final_state is False:
        final_state = None
    _need(final_state, "final_state", (B, H, V, K), torch.float32, dev)
    if saved is True:
        saved = torch.empty(max(gdn_raw_saved_bytes(p), 1), dtype=torch.uint8, device=dev)
    elif saved is False:
        saved = None
    if workspace is None:
        workspace = torch.empty(max(gdn_raw_fwd_workspace_bytes(p), 1), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.gdn_fwd_raw(ctypes.byref(p), _ptr(q_raw), _ptr(k_raw), _ptr(v), _ptr(a_logit), _ptr(b_logit),
                         _ptr(initial_state), _ptr(o), _ptr(final_state), _ptr(saved), _ptr(workspace), ws_bytes,
                         _stream_handle(dev, stream))
    _check(st)
    return o, final_state, saved


def gdn_bwd_raw(q_raw, k_raw, v, a_logit, b_logit, initial_state, d_o, d_final_state=None, *, saved=None,
                chunk: int = 64, grads=None, d_initial_state=True, workspace=None, stream=None):
    """Backward of :func:`gdn_fwd_raw` (``gdn_bwd_raw``): the gradients with respect
    to the raw inputs.  Returns ``(dq_raw, dk_raw, dv, da_logit, db_logit,
    d_initial_state or None)``."""
    lib = load_library()
    dev = q_raw.device
    if dev.type != "cuda":
        raise GdnError(GDN_ERR_INVALID_ARG, "inputs must be CUDA tensors")
    B, T, H, K = q_raw.shape
    V = v.shape[-1]
    dt = q_raw.dtype
    p = make_problem(B, T, H, K, V, chunk, dt)
    for t, n, sh in ((q_raw, "q_raw", (B, T, H, K)), (k_raw, "k_raw", (B, T, H, K)), (v, "v", (B, T, H, V)),
                     (a_logit, "a_logit", (B, T, H)), (b_logit, "b_logit", (B, T, H)),
                     (d_o, "d_o", (B, T, H, V))):
        _need(t, n, sh, dt, dev)
    _need(initial_state, "initial_state", (B, H, V, K), torch.float32, dev)
    _need(d_final_state, "d_final_state", (B, H, V, K), torch.float32, dev)
    if saved is not None and saved.numel() * saved.element_size() < gdn_raw_saved_bytes(p):
        raise GdnError(GDN_ERR_INVALID_ARG, "saved buffer is smaller than gdn_raw_saved_bytes()")
    if grads is None:
        grads = (torch.empty_like(q_raw), torch.empty_like(k_raw), torch.empty_like(v),
                 torch.empty_like(a_logit), torch.empty_like(b_logit))
    dq, dk, dv, da, db = grads
    if d_initial_state is True:
        d_initial_state = torch.empty((B, H, V, K), dtype=torch.float32, device=dev)
    elif d_initial_state is False:
        d_initial_state = None
    if workspace is None:
        workspace = torch.empty(max(gdn_raw_bwd_workspace_bytes(p), 1), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.gdn_bwd_raw(ctypes.byref(p), _ptr(q_raw), _ptr(k_raw), _ptr(v), _ptr(a_logit), _ptr(b_logit),
                         _ptr(initial_state), _ptr(saved), _ptr(d_o), _ptr(d_final_state), _ptr(dq), _ptr(dk),
                         _ptr(dv), _ptr(da), _ptr(db), _ptr(d_initial_state), _ptr(workspace), ws_bytes,
                         _stream_handle(dev, stream))
    _check(st)
    return dq, dk, dv, da, db, d_initial_state


def gdn_count_nonfinite(t, count=None, *, stream=None):
    """Adds the number of NaN / inf elements of the contiguous CUDA tensor ``t``
    (float32 or bfloat16) to ``count`` (a CUDA int64 tensor of one element;
    a new zero one when None) without synchronising, and returns ``count``."""
    lib = load_library()
    dev = t.device
    if dev.type != "cuda":
        raise GdnError(GDN_ERR_INVALID_ARG, "t must be a CUDA tensor")
    if not t.is_contiguous():
        raise GdnError(GDN_ERR_INVALID_ARG, "t must be contiguous")
    if count is None:
        count = torch.zeros(1, dtype=torch.int64, device=dev)
    if count.dtype != torch.int64 or count.device != dev or count.numel() < 1:
        raise GdnError(GDN_ERR_INVALID_ARG, "count must be an int64 tensor on t's device")
    _check(lib.gdn_count_nonfinite(_ptr(t), t.numel(), _dtype_code(t.dtype), _ptr(count),
                                   _stream_handle(dev, stream)))
    return count


def gdn_set_sequence_split(pieces: int) -> None:
    """Within-call sequence split policy for the calls that follow: 0 automatic
    (default), 1 never, n >= 2 pieces per sequence (see include/gdn.h)."""
    _check(load_library().gdn_set_sequence_split(int(pieces)))


def gdn_test_set_wait_limit(ns: int) -> None:
    """Test hook: limit, in nanoseconds, of the tensor-core kernels' bounded waits
    in the calls that follow (0 restores the default of 2 s); see include/gdn.h."""
    _check(load_library().gdn_test_set_wait_limit(int(ns)))


def gdn_get_sequence_split() -> int:
    return int(load_library().gdn_get_sequence_split())


def gdn_num_kernels() -> int:
    return int(load_library().gdn_num_kernels())


def gdn_kernel_name(i: int) -> str:
    return load_library().gdn_kernel_name(int(i)).decode()


def gdn_profiler_start(capacity: int) -> None:
    _check(load_library().gdn_profiler_start(int(capacity)))


def gdn_profiler_stop() -> None:
    _check(load_library().gdn_profiler_stop())


def gdn_profiler_summary() -> dict:
    """{kernel name: (launches, total ms)} for the launches timed since start."""
    lib = load_library()
    out = {}
    for i in range(gdn_num_kernels()):
        n = ctypes.c_int(0)
        ms = ctypes.c_double(0.0)
        _check(lib.gdn_profiler_summary(i, ctypes.byref(n), ctypes.byref(ms)))
        if n.value:
            out[gdn_kernel_name(i)] = (n.value, ms.value)
    return out


def gdn_profiler_release() -> None:
    load_library().gdn_profiler_release()


def _prologue_problem(q_raw, v_dim):
    B, T, H, K = q_raw.shape
    return make_problem(B, T, H, K, v_dim, 64, q_raw.dtype), (B, T, H, K)


def gdn_prologue_fwd(q_raw, k_raw, a_logit, b_logit, *, out=None, stream=None):
    """q/k L2 normalisation and gate activations through ``gdn_prologue_fwd``:
    returns ``(q, k, alpha, beta)`` with q = q_raw / sqrt(|q_raw|^2 + 1e-6) (same
    for k), alpha = exp(-softplus(a_logit)), beta = sigmoid(b_logit).  ``out`` may
    pass the four output tensors."""
    lib = load_library()
    dev = q_raw.device
    if dev.type != "cuda":
        raise GdnError(GDN_ERR_INVALID_ARG, "inputs must be CUDA tensors")
    p, (B, T, H, K) = _prologue_problem(q_raw, 16)
    dt = q_raw.dtype
    if out is None:
        out = (torch.empty_like(q_raw), torch.empty_like(q_raw), torch.empty(B, T, H, dtype=dt, device=dev),
               torch.empty(B, T, H, dtype=dt, device=dev))
    q, k, alpha, beta = out
    for t, n, sh in ((q_raw, "q_raw", (B, T, H, K)), (k_raw, "k_raw", (B, T, H, K)),
                     (a_logit, "a_logit", (B, T, H)), (b_logit, "b_logit", (B, T, H)),
                     (q, "q", (B, T, H, K)), (k, "k", (B, T, H, K)), (alpha, "alpha", (B, T, H)),
                     (beta, "beta", (B, T, H))):
        if t is None:
            raise GdnError(GDN_ERR_INVALID_ARG, f"{n} is required")
        _need(t, n, sh, dt, dev)
    st = lib.gdn_prologue_fwd(ctypes.byref(p), _ptr(q_raw), _ptr(k_raw), _ptr(a_logit), _ptr(b_logit),
                              _ptr(q), _ptr(k), _ptr(alpha), _ptr(beta), _stream_handle(dev, stream))
    _check(st)
    return q, k, alpha, beta


def gdn_prologue_bwd(q_raw, k_raw, a_logit, b_logit, dq, dk, dalpha, dbeta, *, out=None, stream=None):
    """Backward of :func:`gdn_prologue_fwd` through ``gdn_prologue_bwd``: returns
    ``(dq_raw, dk_raw, da_logit, db_logit)``."""
    lib = load_library()
    dev = q_raw.device
    if dev.type != "cuda":
        raise GdnError(GDN_ERR_INVALID_ARG, "inputs must be CUDA tensors")
    p, (B, T, H, K) = _prologue_problem(q_raw, 16)
    dt = q_raw.dtype
    if out is None:
        out = (torch.empty_like(q_raw), torch.empty_like(q_raw), torch.empty(B, T, H, dtype=dt, device=dev),
               torch.empty(B, T, H, dtype=dt, device=dev))
    dqr, dkr, da, db = out
    for t, n, sh in ((q_raw, "q_raw", (B, T, H, K)), (k_raw, "k_raw", (B, T, H, K)),
                     (a_logit, "a_logit", (B, T, H)), (b_logit, "b_logit", (B, T, H)),
                     (dq, "dq", (B, T, H, K)), (dk, "dk", (B, T, H, K)), (dalpha, "dalpha", (B, T, H)),
                     (dbeta, "dbeta", (B, T, H)), (dqr, "dq_raw", (B, T, H, K)), (dkr, "dk_raw", (B, T, H, K)),
                     (da, "da_logit", (B, T, H)), (db, "db_logit", (B, T, H))):
        if t is None:
            raise GdnError(GDN_ERR_INVALID_ARG, f"{n} is required")
        _need(t, n, sh, dt, dev)
    st = lib.gdn_prologue_bwd(ctypes.byref(p), _ptr(q_raw), _ptr(k_raw), _ptr(a_logit), _ptr(b_logit),
                              _ptr(dq), _ptr(dk), _ptr(dalpha), _ptr(dbeta), _ptr(dqr), _ptr(dkr), _ptr(da),
                              _ptr(db), _stream_handle(dev, stream))
    _check(st)
    return dqr, dkr, da, db


VARLEN_BAD_OFFSETS = 1 << 30  # bit of the varlen workspace's error word


def gdn_varlen_fwd_workspace_bytes(p: gdn_problem, total: int) -> int:
    return int(load_library().gdn_varlen_fwd_workspace_bytes(ctypes.byref(p), int(total)))


def gdn_varlen_bwd_workspace_bytes(p: gdn_problem, total: int) -> int:
    return int(load_library().gdn_varlen_bwd_workspace_bytes(ctypes.byref(p), int(total)))


def gdn_varlen_saved_bytes(p: gdn_problem, total: int) -> int:
    return int(load_library().gdn_varlen_saved_bytes(ctypes.byref(p), int(total)))


def _varlen_problem(q, v, cu_seqlens, max_len, chunk):
    if q.dim() != 3:
        raise GdnError(GDN_ERR_INVALID_ARG, "packed q must be [total, H, K]")
    total, H, K = q.shape
    V = v.shape[-1]
    if cu_seqlens is None or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1:
        raise GdnError(GDN_ERR_INVALID_ARG, "cu_seqlens must be a 1-d int32 tensor of S+1 offsets")
    _need(cu_seqlens, "cu_seqlens", tuple(cu_seqlens.shape), torch.int32, q.device)
    S = cu_seqlens.numel() - 1
    if max_len is None:
        if _flat_layout(q.dtype, K, V, chunk):
            # the tensor-core kernels read the packed tensors in place: the bound only
            # checks the offsets and guides the scans' slice width, and the packed total
            # bounds every length, so nothing is read back
            max_len = total
        else:  # the padded layout is sized by it: one device-to-host read (pass max_len to avoid it)
            max_len = int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()) if S > 0 else 0
    return make_problem(S, max_len, H, K, V, chunk, q.dtype), (total, S, H, K, V)


def _flat_layout(dtype, K, V, chunk) -> bool:
    """Whether the library runs this shape on its tensor-core kernels (bf16, 64-token
    chunks, K and V of 16, 32, 64 or 128), whose packed calls use the flat chunk layout."""
    dims = (16, 32, 64, 128)
    return dtype == torch.bfloat16 and chunk == 64 and K in dims and V in dims


def _varlen_error(workspace, stream, dev):
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    stream.synchronize()
    word = int(workspace[:4].view(torch.int32).item())
    if word & VARLEN_BAD_OFFSETS:
        raise GdnError(GDN_ERR_INVALID_ARG, "cu_seqlens is invalid (offsets must rise from 0 to total, "
                       "each length at most max_len)")
    if word:
        raise GdnError(GDN_ERR_CUDA, f"kernel error word {word:#x} (a bounded wait gave up)")


def gdn_varlen_fwd(q, k, v, alpha, beta, cu_seqlens, max_len=None, initial_state=None, *, chunk: int = 64,
                   o=None, final_state=True, saved=False, workspace=None, check=False, stream=None):
    """Forward over S packed sequences of different lengths (``gdn_varlen_fwd``).

    q, k [total,H,K]; v [total,H,V]; alpha, beta [total,H]; sequence s is rows
    ``cu_seqlens[s]:cu_seqlens[s+1]`` (int32 [S+1] on the device).  ``max_len``
    bounds every length; if None it is ``total`` on the tensor-core shapes (no
    read back) and is computed from cu_seqlens with one device-to-host read on
    the others, whose padded layout it sizes.  initial_state / final_state are float32 [S,H,V,K] as in
    :func:`gdn_fwd`.  ``check=True`` synchronises and raises if the kernels
    found cu_seqlens invalid.  Returns ``(o, final_state or None, saved or None)``;
    ``saved`` feeds :func:`gdn_varlen_bwd` with the same cu_seqlens and max_len.
    """
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise GdnError(GDN_ERR_INVALID_ARG, "inputs must be CUDA tensors")
    p, (total, S, H, K, V) = _varlen_problem(q, v, cu_seqlens, max_len, chunk)
    dt = q.dtype
    for t, n, sh in ((k, "k", (total, H, K)), (v, "v", (total, H, V)), (alpha, "alpha", (total, H)),
                     (beta, "beta", (total, H))):
        _need(t, n, sh, dt, dev)
    _need(initial_state, "initial_state", (S, H, V, K), torch.float32, dev)
    if o is None:
        o = torch.empty((total, H, V), dtype=dt, device=dev)
    _need(o, "o", (total, H, V), dt, dev)
    if final_state is True:
        final_state = torch.empty((S, H, V, K), dtype=torch.float32, device=dev)
    elif final_state is False:
        final_state = None
    _need(final_state, "final_state", (S, H, V, K), torch.float32, dev)
    if saved is True:
        saved = torch.empty(max(gdn_varlen_saved_bytes(p, total), 1), dtype=torch.uint8, device=dev)
    elif saved is False:
        saved = None
    if workspace is None:
        workspace = torch.empty(max(gdn_varlen_fwd_workspace_bytes(p, total), 4), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.gdn_varlen_fwd(ctypes.byref(p), total, _ptr(cu_seqlens), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                            _ptr(beta), _ptr(initial_state), _ptr(o), _ptr(final_state), _ptr(saved),
                            _ptr(workspace), ws_bytes, _stream_handle(dev, stream))
    _check(st)
    if check:
        _varlen_error(workspace, stream, dev)
    return o, final_state, saved


def gdn_varlen_bwd(q, k, v, alpha, beta, cu_seqlens, max_len, initial_state, d_o, d_final_state=None, *,
                   saved=None, chunk: int = 64, grads=None, d_initial_state=True, workspace=None,
                   check=False, stream=None):
    """Backward of :func:`gdn_varlen_fwd` (``gdn_varlen_bwd``), packed layouts as
    there.  Returns ``(dq, dk, dv, dalpha, dbeta, d_initial_state or None)``."""
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise GdnError(GDN_ERR_INVALID_ARG, "inputs must be CUDA tensors")
    p, (total, S, H, K, V) = _varlen_problem(q, v, cu_seqlens, max_len, chunk)
    dt = q.dtype
    for t, n, sh in ((k, "k", (total, H, K)), (v, "v", (total, H, V)), (alpha, "alpha", (total, H)),
                     (beta, "beta", (total, H)), (d_o, "d_o", (total, H, V))):
        _need(t, n, sh, dt, dev)
    _need(initial_state, "initial_state", (S, H, V, K), torch.float32, dev)
    _need(d_final_state, "d_final_state", (S, H, V, K), torch.float32, dev)
    if saved is not None and saved.numel() * saved.element_size() < gdn_varlen_saved_bytes(p, total):
        raise GdnError(GDN_ERR_INVALID_ARG, "saved buffer is smaller than gdn_varlen_saved_bytes()")
    if grads is None:
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(alpha),
                 torch.empty_like(beta))
    dq, dk, dv, da, db = grads
    for t, n, sh in ((dq, "dq", (total, H, K)), (dk, "dk", (total, H, K)), (dv, "dv", (total, H, V)),
                     (da, "dalpha", (total, H)), (db, "dbeta", (total, H))):
        _need(t, n, sh, dt, dev)
    if d_initial_state is True:
        d_initial_state = torch.empty((S, H, V, K), dtype=torch.float32, device=dev)
    elif d_initial_state is False:
        d_initial_state = None
    _need(d_initial_state, "d_initial_state", (S, H, V, K), torch.float32, dev)
    if workspace is None:
        workspace = torch.empty(max(gdn_varlen_bwd_workspace_bytes(p, total), 4), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.gdn_varlen_bwd(ctypes.byref(p), total, _ptr(cu_seqlens), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                            _ptr(beta), _ptr(initial_state), _ptr(saved), _ptr(d_o), _ptr(d_final_state),
                            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(da), _ptr(db), _ptr(d_initial_state),
                            _ptr(workspace), ws_bytes, _stream_handle(dev, stream))
    _check(st)
    if check:
        _varlen_error(workspace, stream, dev)
    return dq, dk, dv, da, db, d_initial_state


RESET_TOO_MANY_SEGMENTS = 1 << 29  # bit of the reset calls' error word


def _reset_mask(reset, B, T, dev):
    if reset is None or tuple(reset.shape) != (B, T):
        raise GdnError(GDN_ERR_INVALID_ARG, f"reset must be a [B, T] = [{B}, {T}] mask")
    if reset.device != dev or reset.dtype not in (torch.bool, torch.uint8) or not reset.is_contiguous():
        raise GdnError(GDN_ERR_INVALID_ARG, "reset must be a contiguous bool or uint8 tensor on the inputs' device")
    return reset.view(torch.uint8) if reset.dtype == torch.bool else reset


def reset_segment_count(reset) -> int:
    """The number of segments of a [B, T] reset mask: B plus the resets at t >= 1
    (one device-to-host read; pass ``max_segments`` to the reset calls instead
    when a bound is known)."""
    B, T = reset.shape
    return int(B + (int(reset[:, 1:].to(torch.int64).sum().item()) if T > 1 else 0))


def _reset_error(workspace, stream, dev):
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    stream.synchronize()
    word = int(workspace[:4].view(torch.int32).item())
    if word & RESET_TOO_MANY_SEGMENTS:
        raise GdnError(GDN_ERR_INVALID_ARG, "the reset mask has more segments than max_segments")
    if word:
        raise GdnError(GDN_ERR_CUDA, f"kernel error word {word:#x}")


def gdn_reset_fwd(q, k, v, alpha, beta, reset, initial_state=None, *, max_segments=None, chunk: int = 64, o=None,
                  final_state=True, saved=False, workspace=None, check=False, stream=None):
    """Forward over a dense batch (q, k [B,T,H,K]; v [B,T,H,V]; alpha, beta
    [B,T,H]) whose streams restart from the zero state at every position where
    ``reset`` ([B,T] bool or uint8, on the device) is set (``gdn_reset_fwd``: the
    segments are built from the mask by the library's kernels).
    ``max_segments`` bounds the number of segments (B plus the resets at t >= 1);
    if None it is counted with one device-to-host read.  ``check=True``
    synchronises and raises if the kernels found more segments than the bound.
    Returns ``(o, final_state or None, saved or None, max_segments)``; pass
    ``saved`` and ``max_segments`` on to :func:`gdn_reset_bwd`."""
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise GdnError(GDN_ERR_INVALID_ARG, "inputs must be CUDA tensors")
    B, T, H, K = q.shape
    V = v.shape[-1]
    dt = q.dtype
    mask = _reset_mask(reset, B, T, dev)
    if max_segments is None:
        max_segments = reset_segment_count(mask)
    p = make_problem(B, T, H, K, V, chunk, dt)
    for t, n, sh in ((k, "k", (B, T, H, K)), (v, "v", (B, T, H, V)), (q, "q", (B, T, H, K)),
                     (alpha, "alpha", (B, T, H)), (beta, "beta", (B, T, H))):
        _need(t, n, sh, dt, dev)
    _need(initial_state, "initial_state", (B, H, V, K), torch.float32, dev)
    if o is None:
        o = torch.empty((B, T, H, V), dtype=dt, device=dev)
    _need(o, "o", (B, T, H, V), dt, dev)
    if final_state is True:
        final_state = torch.empty((B, H, V, K), dtype=torch.float32, device=dev)
    elif final_state is False:
        final_state = None
    _need(final_state, "final_state", (B, H, V, K), torch.float32, dev)
    if saved is True:
        saved = torch.empty(max(int(lib.gdn_reset_saved_bytes(ctypes.byref(p), max_segments)), 1),
                            dtype=torch.uint8, device=dev)
    elif saved is False:
        saved = None
    if workspace is None:
        workspace = torch.empty(max(int(lib.gdn_reset_fwd_workspace_bytes(ctypes.byref(p), max_segments)), 4),
                                dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.gdn_reset_fwd(ctypes.byref(p), int(max_segments), _ptr(mask), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                           _ptr(beta), _ptr(initial_state), _ptr(o), _ptr(final_state), _ptr(saved),
                           _ptr(workspace), ws_bytes, _stream_handle(dev, stream))
    _check(st)
    if check and B * T * H:
        _reset_error(workspace, stream, dev)
    return o, final_state, saved, max_segments


def gdn_reset_bwd(q, k, v, alpha, beta, reset, initial_state, d_o, d_final_state=None, *, max_segments=None,
                  saved=None, chunk: int = 64, grads=None, d_initial_state=True, workspace=None, check=False,
                  stream=None):
    """Backward of :func:`gdn_reset_fwd` (``gdn_reset_bwd``): returns ``(dq, dk, dv,
    dalpha, dbeta, d_initial_state [B,H,V,K] or None)``; a row reset at t = 0
    gets a zero d_initial_state."""
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise GdnError(GDN_ERR_INVALID_ARG, "inputs must be CUDA tensors")
    B, T, H, K = q.shape
    V = v.shape[-1]
    dt = q.dtype
    mask = _reset_mask(reset, B, T, dev)
    if max_segments is None:
        max_segments = reset_segment_count(mask)
    p = make_problem(B, T, H, K, V, chunk, dt)
    for t, n, sh in ((k, "k", (B, T, H, K)), (v, "v", (B, T, H, V)), (q, "q", (B, T, H, K)),
                     (alpha, "alpha", (B, T, H)), (beta, "beta", (B, T, H)), (d_o, "d_o", (B, T, H, V))):
        _need(t, n, sh, dt, dev)
    _need(initial_state, "initial_state", (B, H, V, K), torch.float32, dev)
    _need(d_final_state, "d_final_state", (B, H, V, K), torch.float32, dev)
    if saved is not None and saved.numel() * saved.element_size() < int(
            lib.gdn_reset_saved_bytes(ctypes.byref(p), max_segments)):
        raise GdnError(GDN_ERR_INVALID_ARG, "saved buffer is smaller than gdn_reset_saved_bytes()")
    if grads is None:
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(alpha),
                 torch.empty_like(beta))
    dq, dk, dv, da, db = grads
    if d_initial_state is True:
        d_initial_state = torch.empty((B, H, V, K), dtype=torch.float32, device=dev)
    elif d_initial_state is False:
        d_initial_state = None
    _need(d_initial_state, "d_initial_state", (B, H, V, K), torch.float32, dev)
    if workspace is None:
        workspace = torch.empty(max(int(lib.gdn_reset_bwd_workspace_bytes(ctypes.byref(p), max_segments)), 4),
                                dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.gdn_reset_bwd(ctypes.byref(p), int(max_segments), _ptr(mask), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                           _ptr(beta), _ptr(initial_state), _ptr(saved), _ptr(d_o), _ptr(d_final_state), _ptr(dq),
                           _ptr(dk), _ptr(dv), _ptr(da), _ptr(db), _ptr(d_initial_state), _ptr(workspace), ws_bytes,
                           _stream_handle(dev, stream))
    _check(st)
    if check and B * T * H:
        _reset_error(workspace, stream, dev)
    return dq, dk, dv, da, db, d_initial_state


def gdn_decode(q, k, v, alpha, beta, state, *, o=None, stream=None):
    """Recurrent step through ``gdn_decode``: advances ``state`` ([B,H,V,K] fp32,
    updated in place) through the T tokens of q, k, v, alpha, beta (usually T=1)
    and writes their outputs.  Calls continue the stream exactly: T calls of one
    token equal one call of T tokens bit for bit.  Returns ``(o, state)``."""
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise GdnError(GDN_ERR_INVALID_ARG, "inputs must be CUDA tensors")
    B, T, H, K = q.shape
    V = v.shape[-1]
    dt = q.dtype
    p = make_problem(B, T, H, K, V, 64, dt)
    if o is None:
        o = torch.empty(B, T, H, V, dtype=dt, device=dev)
    for t, n, sh in ((k, "k", (B, T, H, K)), (v, "v", (B, T, H, V)), (q, "q", (B, T, H, K)),
                     (alpha, "alpha", (B, T, H)), (beta, "beta", (B, T, H)),
                     (o, "o", (B, T, H, V))):
        if t is None:
            raise GdnError(GDN_ERR_INVALID_ARG, f"{n} is required")
        _need(t, n, sh, dt, dev)
    if state is None:
        raise GdnError(GDN_ERR_INVALID_ARG, "state is required")
    _need(state, "state", (B, H, V, K), torch.float32, dev)
    st = lib.gdn_decode(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                        _ptr(state), _ptr(o), _stream_handle(dev, stream))
    _check(st)
    return o, state


# Size of the fixed scratch array gdn_fwd_noalloc runs on (GDN_FWD_NOALLOC_SCRATCH_BYTES).
GDN_FWD_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def gdn_fwd_noalloc(q, k, v, alpha, beta, initial_state, o, final_state=None, *,
                    chunk: int = 64, stream=None):
    """Forward through ``gdn_fwd_noalloc``: the same result as :func:`gdn_fwd`,
    for callers that cannot allocate device memory (a host framework that owns
    every byte of device memory, or a latency-critical path where cudaMalloc's
    device-wide synchronisation is not acceptable).  Its scratch is a fixed
    array in the library (``GDN_FWD_NOALLOC_SCRATCH_BYTES`` = 32 MiB per device);
    larger problems raise.  This wrapper allocates nothing either: the caller
    passes ``o`` and, optionally, ``final_state``.  Calls that overlap on the GPU
    share the array and race; the first call on a device must not be inside a
    stream capture.  Returns ``(o, final_state)``."""
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise GdnError(GDN_ERR_INVALID_ARG, "inputs must be CUDA tensors")
    B, T, H, K = q.shape
    V = v.shape[-1]
    dt = q.dtype
    p = make_problem(B, T, H, K, V, chunk, dt)
    for t, n, s in ((k, "k", (B, T, H, K)), (v, "v", (B, T, H, V)), (q, "q", (B, T, H, K)),
                    (alpha, "alpha", (B, T, H)), (beta, "beta", (B, T, H)),
                    (o, "o", (B, T, H, V))):
        if t is None:
            raise GdnError(GDN_ERR_INVALID_ARG, f"{n} is required")
        _need(t, n, s, dt, dev)
    _need(initial_state, "initial_state", (B, H, V, K), torch.float32, dev)
    _need(final_state, "final_state", (B, H, V, K), torch.float32, dev)
    with torch.cuda.device(dev):  # the library uses the current device's array
        st = lib.gdn_fwd_noalloc(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                                 _ptr(beta), _ptr(initial_state), _ptr(o), _ptr(final_state),
                                 _stream_handle(dev, stream))
    _check(st)
    return o, final_state
