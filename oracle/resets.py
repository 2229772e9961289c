"""Float64 oracle of streams with reset positions -- TEST INFRASTRUCTURE (only the
tests import it; the product path never does).

"OpenGDN", Scope, names reset masks among what its operator does not support;
the pages give no formula for them.  Reading taken here: a reset at (b, t)
clears row b's state just before token t is applied, so the stream continues
from the zero state at t, exactly as a new sequence would.  A reset at t = 0
discards the row's initial state.  Each row is therefore a chain of independent
segments, and this module runs the token-recurrence oracle on every segment:

* :func:`fwd_resets` -- outputs and each row's final state;
* :func:`bwd_resets` -- gradients of ``sum(d_o * o) + sum(d_final_state *
  final_state)``; the row's d_final_state enters its last segment and its
  d_initial_state comes out of its first segment (zero after a reset at t = 0).

Shapes: q, k ``[B,T,H,K]``; v ``[B,T,H,V]``; alpha, beta ``[B,T,H]``; reset
``[B,T]`` bool; states ``[B,H,V,K]``.
"""
from __future__ import annotations

import numpy as np

from . import gated_delta_bwd, gated_delta_fwd


def segments(reset_row):
    """(start, end) of the segments of one row: a new one at t = 0 and at every reset."""
    T = len(reset_row)
    starts = [0] + [t for t in range(1, T) if reset_row[t]]
    return list(zip(starts, starts[1:] + [T])) if T else []


def fwd_resets(q, k, v, alpha, beta, reset, initial_state=None):
    B, T, H, K = q.shape
    V = v.shape[-1]
    o = np.zeros((B, T, H, V))
    sT = np.zeros((B, H, V, K))
    for b in range(B):
        state = None
        if initial_state is not None and not (T and reset[b, 0]):
            state = initial_state[b:b + 1]
        if T == 0:
            sT[b] = 0.0 if state is None else state[0]
        for i, (a, e) in enumerate(segments(reset[b])):
            sl = slice(a, e)
            # every segment after the first starts from the zero state
            ob, state = gated_delta_fwd(q[b:b + 1, sl], k[b:b + 1, sl], v[b:b + 1, sl], alpha[b:b + 1, sl],
                                        beta[b:b + 1, sl], state if i == 0 else None)
            o[b, sl] = ob[0]
        if T:
            sT[b] = state[0]
    return o, sT


def bwd_resets(q, k, v, alpha, beta, reset, initial_state, d_o, d_final_state=None):
    B, T, H, K = q.shape
    V = v.shape[-1]
    out = dict(dq=np.zeros(q.shape), dk=np.zeros(k.shape), dv=np.zeros(v.shape), dalpha=np.zeros(alpha.shape),
               dbeta=np.zeros(beta.shape), d_initial_state=np.zeros((B, H, V, K)))
    for b in range(B):
        segs = segments(reset[b])
        carry = initial_state is not None and not (T and reset[b, 0])
        if T == 0:
            if d_final_state is not None:
                out["d_initial_state"][b] = d_final_state[b]
            continue
        for i, (a, e) in enumerate(segs):
            sl = slice(a, e)
            # only the row's first segment can start from a non-zero state
            s0 = initial_state[b:b + 1] if (i == 0 and carry) else None
            dsT = d_final_state[b:b + 1] if (d_final_state is not None and i == len(segs) - 1) else None
            g = gated_delta_bwd(q[b:b + 1, sl], k[b:b + 1, sl], v[b:b + 1, sl], alpha[b:b + 1, sl],
                                beta[b:b + 1, sl], s0, d_o[b:b + 1, sl], dsT)
            for n in ("dq", "dk", "dv", "dalpha", "dbeta"):
                out[n][b, sl] = g[n][0]
            if i == 0 and not reset[b, 0]:  # after a reset at t = 0 it stays zero
                out["d_initial_state"][b] = g["d_initial_state"][0]
    return out
