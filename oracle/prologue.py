"""Float64 oracle of the prologue in front of the recurrence -- TEST INFRASTRUCTURE
(only the tests import it; the product path never does).

Every mixer the pages show feeds the recurrence L2-normalised keys and queries
and per-head gates ("OpenGDN", Mixer: the mixer normalises q and k to unit L2
length and computes one alpha and one beta per head; "Sparse Delta Memory: layer
and kernels", What the layer computes: l2-normalised read and write weights in
the dense limit).  This module writes
that step out in plain numpy:

* ``q = q_raw / sqrt(sum_K q_raw^2 + eps)`` and the same for k, per (b, t, h),
  with ``eps = 1e-6``;
* ``alpha = exp(-softplus(a))`` and ``beta = sigmoid(b)`` from the gate logits
  (the parameterisation of the synthetic workloads; ``exp(-softplus(a))``
  equals ``sigmoid(-a)``, so a mixer with ``alpha = sigmoid(a')`` passes
  ``a = -a'``).

:func:`prologue_bwd` is the chain rule of the same formulas.  Shapes: q_raw,
k_raw ``[B,T,H,K]``; a, b ``[B,T,H]``.
"""
from __future__ import annotations

import numpy as np

EPS = 1e-6


def _f64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def softplus(x):
    """log(1 + e^x), written so that neither branch overflows."""
    x = _f64(x)
    return np.where(x > 0, x + np.log1p(np.exp(-np.abs(x))), np.log1p(np.exp(np.minimum(x, 0.0))))


def sigmoid(x):
    x = _f64(x)
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def prologue_fwd(q_raw, k_raw, a, b):
    """Returns (q, k, alpha, beta) as float64 arrays."""
    q_raw, k_raw = _f64(q_raw), _f64(k_raw)
    rq = 1.0 / np.sqrt((q_raw * q_raw).sum(-1, keepdims=True) + EPS)
    rk = 1.0 / np.sqrt((k_raw * k_raw).sum(-1, keepdims=True) + EPS)
    alpha = np.exp(-softplus(a))
    beta = sigmoid(b)
    return q_raw * rq, k_raw * rk, alpha, beta


def prologue_bwd(q_raw, k_raw, a, b, dq, dk, dalpha, dbeta):
    """Gradients of L(q, k, alpha, beta) with respect to (q_raw, k_raw, a, b),
    given dL/dq, dL/dk, dL/dalpha, dL/dbeta.

    For y = x r with r = (x.x + eps)^(-1/2): dx = r (dy - y (y . dy)).
    alpha = exp(-softplus(a)) has d alpha / da = -alpha (1 - alpha);
    beta = sigmoid(b) has d beta / db = beta (1 - beta)."""
    q, k, alpha, beta = prologue_fwd(q_raw, k_raw, a, b)
    dq, dk = _f64(dq), _f64(dk)
    rq = 1.0 / np.sqrt((_f64(q_raw) ** 2).sum(-1, keepdims=True) + EPS)
    rk = 1.0 / np.sqrt((_f64(k_raw) ** 2).sum(-1, keepdims=True) + EPS)
    dq_raw = rq * (dq - q * (q * dq).sum(-1, keepdims=True))
    dk_raw = rk * (dk - k * (k * dk).sum(-1, keepdims=True))
    da = -_f64(dalpha) * alpha * (1.0 - alpha)
    db = _f64(dbeta) * beta * (1.0 - beta)
    return dq_raw, dk_raw, da, db
