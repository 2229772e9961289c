"""Helpers shared by the GPU parity tests: run the CUDA path (through the C ABI
binding) and the float64 oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

from gated_delta_rule_19_gb300 import gdn
from gated_delta_rule_19_gb300.inputs import Workload, custom, make_inputs

# Tolerances on relative L2 error, per output tensor: fp32 inputs 1e-5; bf16
# inputs with fp32 state and accumulation: 2e-2 for outputs / final state, 3e-2
# for gradients.
TOL = {"f32": dict(out=1e-5, grad=1e-5), "bf16": dict(out=2e-2, grad=3e-2)}


def rel_l2(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    den = np.linalg.norm(ref)
    num = np.linalg.norm(x - ref)
    if den == 0.0:
        return float(num)
    return float(num / den)


def to_np(t):
    return None if t is None else t.detach().float().cpu().double().numpy()


def poisoned(like, shape=None, dtype=None):
    """An output buffer filled with NaN, so that any element the kernels do not
    write shows up in the comparison."""
    return torch.full(like.shape if shape is None else shape, float("nan"),
                      dtype=like.dtype if dtype is None else dtype, device=like.device)


def gpu_run(w: Workload, inp: dict, backward: bool, saved_mode: str = "saved",
            device="cuda"):
    """Runs the CUDA path on NaN-filled outputs.  Returns a dict of numpy float64
    arrays."""
    d = {n: (t.to(device) if t is not None else None) for n, t in inp.items()}
    B, T, H, _ = d["q"].shape
    V = d["v"].shape[-1]
    K = d["q"].shape[-1]
    o, sT, saved = gdn.gdn_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"],
                               d["initial_state"], chunk=w.chunk,
                               o=poisoned(d["v"]),
                               final_state=poisoned(d["v"], (B, H, V, K), torch.float32),
                               saved=(backward and saved_mode == "saved"))
    out = dict(o=to_np(o), final_state=to_np(sT))
    if backward:
        grads = (poisoned(d["q"]), poisoned(d["k"]), poisoned(d["v"]), poisoned(d["alpha"]),
                 poisoned(d["beta"]))
        g = gdn.gdn_bwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["initial_state"],
                        d["d_o"], d["d_final_state"], saved=saved, chunk=w.chunk, grads=grads,
                        d_initial_state=poisoned(d["v"], (B, H, V, K), torch.float32))
        for n, t in zip(("dq", "dk", "dv", "dalpha", "dbeta", "d_initial_state"), g):
            out[n] = to_np(t)
    torch.cuda.synchronize()
    return out


def oracle_run(oracle, inp: dict, backward: bool, streams=None):
    """Runs the oracle on the (optionally sampled) streams.  `streams` is a list
    of (b, h) pairs; the returned arrays then have B'=1, H'=len(streams) layout
    [1, T, n, ...]."""
    q, k, v, a, be = (to_np(inp[n]) for n in ("q", "k", "v", "alpha", "beta"))
    s0 = to_np(inp["initial_state"])
    do = to_np(inp["d_o"])
    dsT = to_np(inp["d_final_state"])
    if streams is not None:
        q, k, v, a, be, do = (select_streams(x, streams) for x in (q, k, v, a, be, do))
        s0 = select_states(s0, streams) if s0 is not None else None
        dsT = select_states(dsT, streams) if dsT is not None else None
    o, sT = oracle.gated_delta_fwd(q, k, v, a, be, s0)
    out = dict(o=o, final_state=sT)
    if backward:
        out.update(oracle.gated_delta_bwd(q, k, v, a, be, s0, do, dsT))
    return out


def select_streams(x, streams):
    """[B,T,H,...] -> [1,T,n,...] for the listed (b,h) streams."""
    return np.stack([x[b, :, h] for b, h in streams], axis=1)[None]


def select_states(x, streams):
    """[B,H,...] -> [1,n,...]."""
    return np.stack([x[b, h] for b, h in streams], axis=0)[None]


def sample_gpu(out: dict, streams):
    res = {}
    for n, x in out.items():
        if x is None:
            continue
        if n in ("final_state", "d_initial_state"):
            res[n] = select_states(x, streams)
        else:
            res[n] = select_streams(x, streams)
    return res


# Tensors compared block by block as well as whole: token tensors [B,T,H,D] per
# (b, chunk of tokens, h); per-token gate gradients [B,T,H] and states [B,H,V,K]
# per (b, h).  A whole-tensor norm hides damage confined to one chunk or row
# (one wrong row of 128 values in a 6M-element o moves it by about 5e-3).
TOKEN_TENSORS = ("o", "dq", "dk", "dv", "dq_raw", "dk_raw", "q", "k")
GATE_TENSORS = ("dalpha", "dbeta", "da", "db", "alpha", "beta")
STATE_TENSORS = ("final_state", "d_initial_state")
LOCAL_FACTOR = 2.0   # a block may be this many times the whole-tensor tolerance
LOCAL_FLOOR = 0.1    # blocks normalised by at least this fraction of the RMS block norm


def block_errors(x, ref, name: str, chunk: int = 64):
    """Per-block relative L2 errors of x against ref, or None if the tensor has no
    block structure here.  Returns (errors, block shape description)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if x.shape != ref.shape:
        return None
    if name in TOKEN_TENSORS and x.ndim == 4:
        B, T, H, _ = x.shape
        if T == 0:
            return None
        d2 = ((x - ref) ** 2).sum(-1)            # [B, T, H]
        r2 = (ref ** 2).sum(-1)
        starts = np.arange(0, T, chunk)
        d2 = np.add.reduceat(d2, starts, axis=1)  # [B, NC, H]
        r2 = np.add.reduceat(r2, starts, axis=1)
        what = "(b, chunk, h)"
    elif name in GATE_TENSORS and x.ndim == 3:
        d2 = ((x - ref) ** 2).sum(1)             # [B, H]
        r2 = (ref ** 2).sum(1)
        what = "(b, h)"
    elif name in STATE_TENSORS and x.ndim == 4:
        d2 = ((x - ref) ** 2).sum((2, 3))        # [B, H]
        r2 = (ref ** 2).sum((2, 3))
        what = "(b, h)"
    else:
        return None
    if d2.size == 0:
        return None
    rms = np.sqrt(r2.sum() / r2.size)
    den = np.maximum(np.sqrt(r2), LOCAL_FLOOR * rms)
    with np.errstate(divide="ignore", invalid="ignore"):
        err = np.where(den > 0, np.sqrt(d2) / np.where(den > 0, den, 1.0), np.sqrt(d2))
    return err, what


def local_failure(x, ref, name: str, lim: float, chunk: int = 64, packed: bool = False):
    """None if every block of x is within LOCAL_FACTOR * lim of ref, else a
    message naming the worst block.  packed: x is one sequence of a packed batch
    ([T, H, ...], no batch axis)."""
    if packed:
        x, ref = np.asarray(x)[None], np.asarray(ref)[None]
    be = block_errors(x, ref, name, chunk)
    if be is None:
        return None
    err, what = be
    worst = np.unravel_index(int(np.argmax(np.where(np.isnan(err), np.inf, err))), err.shape)
    w = float(err[worst])
    if w <= LOCAL_FACTOR * lim:
        return None
    return f"{name}: block {what}={tuple(int(i) for i in worst)} rel_l2={w:.3e} > {LOCAL_FACTOR * lim:.0e}"


def compare(got: dict, ref: dict, dtype: str, names=None, chunk: int = 64):
    """Returns {name: rel_l2} and raises AssertionError listing failures: a tensor
    whose whole-tensor relative L2 exceeds its tolerance, or any block (see
    block_errors) whose relative L2 exceeds LOCAL_FACTOR times it; the worst
    block's index is named."""
    tol = TOL[dtype]
    errs, bad = {}, []
    for n in (names or ref.keys()):
        if n not in got or got[n] is None:
            continue
        e = rel_l2(got[n], ref[n])
        errs[n] = e
        lim = tol["out"] if n in ("o", "final_state") else tol["grad"]
        if not (e <= lim):
            bad.append(f"{n}: rel_l2={e:.3e} > {lim:.0e}")
        msg = local_failure(got[n], ref[n], n, lim, chunk)
        if msg:
            bad.append(msg)
    assert not bad, "; ".join(bad) + f" (all: {errs})"
    return errs


__all__ = ["TOL", "rel_l2", "gpu_run", "poisoned", "oracle_run", "compare", "block_errors", "local_failure", "custom", "make_inputs",
           "sample_gpu", "select_streams", "select_states", "to_np"]
