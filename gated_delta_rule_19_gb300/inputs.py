"""Seeded synthetic inputs for the gated delta rule workloads.

This module only draws random tensors; it contains none of the recurrence's
arithmetic, so both the CUDA path's tests and the float64 oracle can consume
what it returns.

Recipe (the same for every workload):
  * a CPU ``torch.Generator`` seeded with the workload's seed;
  * draws, in float32 and in this order: q, k, v, alpha-logits, beta-logits,
    initial state, d_o, d_final_state (all drawn every time, so the stream of
    random numbers does not depend on which are used);
  * q, k ~ N(0,1) then divided by their L2 norm over the key dimension, per
    (b, t, h); v ~ N(0,1); alpha = exp(-softplus(x)); beta = sigmoid(x);
  * slow decay (``alpha_lo`` > 0): alpha = alpha_lo + (1 - alpha_lo) * alpha,
    gates in (alpha_lo, 1) whose state survives many chunks (with the default
    gates, about 0.5 on average, a chunk's decay is below float32 resolution);
  * initial state ~ N(0, init_std^2) (zero state when init_std == 0);
    d_o ~ N(0,1); d_final_state ~ N(0, dfinal_std^2) (absent when 0);
  * finally every tensor except the fp32 states is cast to the run dtype.
    The oracle receives exactly these cast values (upcast to float64).

The workloads are the five problem shapes the method is measured on: a tiny
fp32 case, a small bf16 forward, a medium and a large bf16 training shape, and a
long-context bf16 stream processed in four calls.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch
import torch.nn.functional as F


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    K: int
    V: int
    chunk: int
    dtype: str            # "f32" or "bf16"
    seed: int
    init_std: float = 0.0
    dfinal_std: float = 0.0
    backward: bool = False
    calls: int = 1        # streaming: the sequence is processed in this many calls
    extra: dict = field(default_factory=dict)
    alpha_lo: float = 0.0  # slow decay: alpha in (alpha_lo, 1)

    @property
    def token_heads(self) -> int:
        return self.B * self.T * self.H

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_f32_B1_T64_H2_K16_V16", 1, 64, 2, 16, 16, 16, "f32", seed=0,
                 backward=True),
        Workload("fwd_bf16_B2_T1024_H4_K64_V64", 2, 1024, 4, 64, 64, 64, "bf16", seed=1,
                 init_std=0.1),
        Workload("train_bf16_B4_T2048_H6_K128_V128", 4, 2048, 6, 128, 128, 64, "bf16",
                 seed=2, backward=True),
        Workload("train_bf16_B8_T4096_H6_K128_V128", 8, 4096, 6, 128, 128, 64, "bf16",
                 seed=3, dfinal_std=0.01, backward=True),
        Workload("stream_bf16_B1_T32768_H16_K128_V128_4calls", 1, 32768, 16, 128, 128, 64,
                 "bf16", seed=4, init_std=0.1, calls=4),
    ]
}

WORKLOAD_ORDER = list(WORKLOADS)

# The decode step (one token per call, the state carried between calls): a
# serving batch of 256 sequences with the long-stream shape's 16 heads and a
# warm state (256 MB of fp32 state, larger than L2).
DECODE_WORKLOADS = {
    w.name: w
    for w in [
        Workload("decode_bf16_B256_T1_H16_K128_V128", 256, 1, 16, 128, 128, 64, "bf16", seed=5,
                 init_std=0.1),
    ]
}


def torch_dtype(dtype: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]


def make_inputs(w: Workload, device="cpu") -> dict:
    """Draw the inputs of workload ``w`` (see the module docstring for the recipe).

    Returns a dict with q, k, v, alpha, beta in the run dtype, and
    initial_state, d_o (run dtype), d_final_state (fp32 or None)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed))
    B, T, H, K, V = w.B, w.T, w.H, w.K, w.V
    f32 = torch.float32
    q = torch.randn(B, T, H, K, generator=g, dtype=f32)
    k = torch.randn(B, T, H, K, generator=g, dtype=f32)
    v = torch.randn(B, T, H, V, generator=g, dtype=f32)
    a_logit = torch.randn(B, T, H, generator=g, dtype=f32)
    b_logit = torch.randn(B, T, H, generator=g, dtype=f32)
    s0 = torch.randn(B, H, V, K, generator=g, dtype=f32)
    d_o = torch.randn(B, T, H, V, generator=g, dtype=f32)
    dsT = torch.randn(B, H, V, K, generator=g, dtype=f32)

    q = q / q.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    alpha = torch.exp(-F.softplus(a_logit))
    if w.alpha_lo > 0:
        alpha = w.alpha_lo + (1.0 - w.alpha_lo) * alpha
    beta = torch.sigmoid(b_logit)
    dt = torch_dtype(w.dtype)
    out = dict(
        q=q.to(dt), k=k.to(dt), v=v.to(dt), alpha=alpha.to(dt), beta=beta.to(dt),
        initial_state=(s0 * w.init_std) if w.init_std > 0 else None,
        d_o=d_o.to(dt),
        d_final_state=(dsT * w.dfinal_std) if w.dfinal_std > 0 else None,
    )
    if device != "cpu":
        out = {n: (t.to(device) if t is not None else None) for n, t in out.items()}
    return out


def custom(name="custom", B=1, T=64, H=2, K=16, V=16, chunk=16, dtype="f32", seed=0,
           init_std=0.0, dfinal_std=0.0, backward=True, alpha_lo=0.0) -> Workload:
    """A workload of any shape with the same recipe (for edge-case tests)."""
    return Workload(name, B, T, H, K, V, chunk, dtype, seed, init_std, dfinal_std, backward,
                    alpha_lo=alpha_lo)


def make_prologue_inputs(B, T, H, K, dtype="f32", seed=0, scale=3.0, logit_scale=2.0) -> dict:
    """Raw inputs of the prologue (before q/k normalisation and the gate
    activations) and upstream gradients for its backward, drawn in this order
    from a CPU generator seeded with ``seed``: q_raw, k_raw ~ N(0, scale^2);
    a_logit, b_logit ~ N(0, logit_scale^2); dq, dk ~ N(0,1); dalpha, dbeta ~
    N(0,1); all cast to the run dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    f32 = torch.float32
    shape = (B, T, H, K)
    out = dict(
        q_raw=torch.randn(*shape, generator=g, dtype=f32) * scale,
        k_raw=torch.randn(*shape, generator=g, dtype=f32) * scale,
        a_logit=torch.randn(B, T, H, generator=g, dtype=f32) * logit_scale,
        b_logit=torch.randn(B, T, H, generator=g, dtype=f32) * logit_scale,
        dq=torch.randn(*shape, generator=g, dtype=f32),
        dk=torch.randn(*shape, generator=g, dtype=f32),
        dalpha=torch.randn(B, T, H, generator=g, dtype=f32),
        dbeta=torch.randn(B, T, H, generator=g, dtype=f32),
    )
    dt = torch_dtype(dtype)
    return {n: t.to(dt) for n, t in out.items()}


def varlen_lengths(total: int, lo: int, hi: int, seed: int) -> list:
    """Sequence lengths of a packed batch: drawn log-uniformly in [lo, hi] from a
    CPU generator seeded with ``seed`` until they sum to ``total`` (the last one
    is cut to fit)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    out, left = [], int(total)
    while left > 0:
        u = float(torch.rand(1, generator=g))
        n = int(round(lo * (hi / lo) ** u))
        n = max(1, min(n, left))
        out.append(n)
        left -= n
    return out


# Packed variable-length training batch: the large training shape's 32768 tokens
# split into sequences whose lengths are drawn log-uniformly in [128, 8192].
VARLEN_WORKLOADS = {
    "varlen_bf16_T32768_H6_K128_V128": dict(total=32768, lo=128, hi=8192, seed=6, H=6, K=128, V=128,
                                            dtype="bf16"),
}


def make_varlen_inputs(lengths, H, K, V, dtype="f32", seed=0, init_std=0.0, dfinal_std=0.0,
                       alpha_lo=0.0) -> dict:
    """Packed inputs of len(lengths) sequences with the recipe of
    :func:`make_inputs` (same distributions and draw order), but with q, k, v,
    alpha, beta, d_o laid out [total, H, ...] and one initial state and
    d_final_state per sequence ([S, H, V, K]).  ``cu_seqlens`` (int32 [S+1]) holds
    the offsets of the sequences."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    S, total = len(lengths), int(sum(lengths))
    f32 = torch.float32
    q = torch.randn(total, H, K, generator=g, dtype=f32)
    k = torch.randn(total, H, K, generator=g, dtype=f32)
    v = torch.randn(total, H, V, generator=g, dtype=f32)
    a_logit = torch.randn(total, H, generator=g, dtype=f32)
    b_logit = torch.randn(total, H, generator=g, dtype=f32)
    s0 = torch.randn(S, H, V, K, generator=g, dtype=f32)
    d_o = torch.randn(total, H, V, generator=g, dtype=f32)
    dsT = torch.randn(S, H, V, K, generator=g, dtype=f32)
    q = q / q.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    dt = torch_dtype(dtype)
    alpha = torch.exp(-F.softplus(a_logit))
    if alpha_lo > 0:
        alpha = alpha_lo + (1.0 - alpha_lo) * alpha
    cu = torch.zeros(S + 1, dtype=torch.int32)
    if S:
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    return dict(
        q=q.to(dt), k=k.to(dt), v=v.to(dt), alpha=alpha.to(dt),
        beta=torch.sigmoid(b_logit).to(dt),
        initial_state=(s0 * init_std) if init_std > 0 else None,
        d_o=d_o.to(dt),
        d_final_state=(dsT * dfinal_std) if dfinal_std > 0 else None,
        cu_seqlens=cu, lengths=list(lengths),
    )
