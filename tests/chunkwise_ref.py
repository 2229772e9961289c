"""Float64 numpy restatement of the chunkwise (extended-WY) gated delta rule.

Tests only.  It shares no code with the CUDA path or with the token-by-token
oracle; the tests compare it with the oracle at chunk sizes 16, 32 and 64, which
checks the chunk algebra that the CUDA kernels implement (forward and backward)
before any kernel is trusted.

Per chunk of C tokens with start state S0 ([V,K]):
  G_r = sum_{i<=r} log alpha_i (within the chunk), gamma_r = exp(G_r),
  Gam_ri = exp(G_r - G_i) for r >= i (0 above the diagonal)
  A   = strict_lower(diag(beta) (Gam * K K^T))          -- decay-weighted Gram
  T   = (I + A)^{-1}                                     -- WY solve
  Ut  = T diag(beta) V,   W = T diag(beta * gamma) K     -- recompute
  U   = Ut - W S0^T                                      -- corrected writes
  Mqk = lower(Gam * Q K^T)                               -- causal reads x writes
  O   = diag(gamma) Q S0^T + Mqk U                       -- readings
  S1  = gamma_C S0 + U^T diag(exp(G_C - G)) K            -- next chunk state
("Sparse Delta Memory: layer and kernels", "What the layer computes": Phase 1,
Solve, Phase 2; "OpenGDN", "Core operator reference": extended-WY chunk form.)

A ragged last chunk is padded with alpha=1, beta=0 and q=k=v=0, which leaves
the state unchanged; padded outputs are dropped.
"""
from __future__ import annotations

import numpy as np


def _pad(x, Tp, value=0.0):
    T = x.shape[0]
    if T == Tp:
        return x
    pad = np.full((Tp - T,) + x.shape[1:], value, dtype=x.dtype)
    return np.concatenate([x, pad], axis=0)


def _chunk_terms(Qc, Kc, Vc, a, be):
    C = a.shape[0]
    G = np.cumsum(np.log(a))
    gam = np.exp(G)
    low = np.tril(np.ones((C, C)))
    Gam = np.exp(np.where(low > 0, G[:, None] - G[None, :], -np.inf))
    KK = Kc @ Kc.T
    A = np.tril(be[:, None] * Gam * KK, -1)
    Tm = np.linalg.solve(np.eye(C) + A, np.eye(C))
    Ut = Tm @ (be[:, None] * Vc)
    W = Tm @ ((be * gam)[:, None] * Kc)
    Mqk = Gam * (Qc @ Kc.T)  # Gam is already zero above the diagonal
    eC = np.exp(G[-1] - G)
    Khat = eC[:, None] * Kc
    return dict(G=G, gam=gam, Gam=Gam, KK=KK, A=A, T=Tm, Ut=Ut, W=W, Mqk=Mqk, eC=eC,
                Khat=Khat)


def _stream_chunks(q, k, v, alpha, beta, C):
    T = q.shape[0]
    NC = -(-T // C)
    Tp = NC * C
    return (NC, _pad(q, Tp), _pad(k, Tp), _pad(v, Tp), _pad(alpha, Tp, 1.0),
            _pad(beta, Tp, 0.0))


def chunk_fwd(q, k, v, alpha, beta, s0=None, C=64, return_states=False):
    """Chunkwise forward; same signature/shapes as the oracle's forward."""
    B, T, H, K = q.shape
    V = v.shape[-1]
    o = np.zeros((B, T, H, V))
    sT = np.zeros((B, H, V, K))
    NC = -(-T // C) if T > 0 else 0
    states = np.zeros((B, H, NC, V, K))
    for b in range(B):
        for h in range(H):
            S = np.zeros((V, K)) if s0 is None else s0[b, h].copy()
            nc, qp, kp, vp, ap, bp = _stream_chunks(q[b, :, h], k[b, :, h], v[b, :, h],
                                                   alpha[b, :, h], beta[b, :, h], C)
            ob = np.zeros((nc * C, V))
            for c in range(nc):
                sl = slice(c * C, (c + 1) * C)
                states[b, h, c] = S
                t = _chunk_terms(qp[sl], kp[sl], vp[sl], ap[sl], bp[sl])
                U = t["Ut"] - t["W"] @ S.T
                ob[sl] = t["gam"][:, None] * (qp[sl] @ S.T) + t["Mqk"] @ U
                S = t["gam"][-1] * S + U.T @ t["Khat"]
            o[b, :, h] = ob[:T]
            sT[b, h] = S
    if return_states:
        return o, sT, states
    return o, sT


def chunk_bwd(q, k, v, alpha, beta, s0, d_o, d_final_state=None, C=64):
    """Chunkwise backward: a reverse walk over chunks carrying dS, plus the
    chunk-local gradients through T, A, the decay masks and the gates."""
    B, T, H, K = q.shape
    V = v.shape[-1]
    _, _, states = chunk_fwd(q, k, v, alpha, beta, s0, C, return_states=True)
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v),
               dalpha=np.zeros_like(alpha), dbeta=np.zeros_like(beta),
               d_initial_state=np.zeros((B, H, V, K)))
    for b in range(B):
        for h in range(H):
            nc, qp, kp, vp, ap, bp = _stream_chunks(q[b, :, h], k[b, :, h], v[b, :, h],
                                                   alpha[b, :, h], beta[b, :, h], C)
            dop = _pad(d_o[b, :, h], nc * C)
            dS = np.zeros((V, K)) if d_final_state is None else d_final_state[b, h].copy()
            dq = np.zeros((nc * C, K))
            dk = np.zeros((nc * C, K))
            dv = np.zeros((nc * C, V))
            da = np.zeros(nc * C)
            db = np.zeros(nc * C)
            for c in range(nc - 1, -1, -1):
                sl = slice(c * C, (c + 1) * C)
                Qc, Kc, Vc, a, be, dO = qp[sl], kp[sl], vp[sl], ap[sl], bp[sl], dop[sl]
                S0 = states[b, h, c]
                t = _chunk_terms(Qc, Kc, Vc, a, be)
                gam, Gam, Tm, W, Mqk, Khat = (t["gam"], t["Gam"], t["T"], t["W"], t["Mqk"],
                                              t["Khat"])
                U = t["Ut"] - W @ S0.T
                dS1 = dS
                # reverse scan step
                dU = Mqk.T @ dO + Khat @ dS1.T
                dS = gam[-1] * dS1 + dO.T @ (gam[:, None] * Qc) - dU.T @ W
                # chunk-local gradients
                QS = Qc @ S0.T
                dMqk = np.tril(dO @ U.T)
                dQK = Gam * dMqk
                dQ = gam[:, None] * (dO @ S0) + dQK @ Kc
                dK = dQK.T @ Qc
                dKhat = U @ dS1
                dK += t["eC"][:, None] * dKhat
                dW = -dU @ S0
                BV = be[:, None] * Vc
                BGK = (be * gam)[:, None] * Kc
                dT = dU @ BV.T + dW @ BGK.T
                TdU = Tm.T @ dU
                TdW = Tm.T @ dW
                dV = be[:, None] * TdU
                dK += (be * gam)[:, None] * TdW
                dA = np.tril(-(Tm.T @ dT @ Tm.T), -1)
                E = be[:, None] * Gam * dA
                dK += (E + E.T) @ Kc
                dbe = (TdU * Vc).sum(1) + gam * (TdW * Kc).sum(1) + (Gam * dA * t["KK"]).sum(1)
                dG = gam * (dO * QS).sum(1)
                dG += gam * be * (TdW * Kc).sum(1)
                E1 = dMqk * Mqk
                dG += E1.sum(1) - E1.sum(0)
                E2 = dA * t["A"]
                dG += E2.sum(1) - E2.sum(0)
                dG[-1] += gam[-1] * (dS1 * S0).sum()
                e = (dKhat * Khat).sum(1)
                dG[-1] += e.sum()
                dG -= e
                dloga = np.cumsum(dG[::-1])[::-1]
                dq[sl], dk[sl], dv[sl] = dQ, dK, dV
                da[sl] = dloga / a
                db[sl] = dbe
            out["dq"][b, :, h] = dq[:T]
            out["dk"][b, :, h] = dk[:T]
            out["dv"][b, :, h] = dv[:T]
            out["dalpha"][b, :, h] = da[:T]
            out["dbeta"][b, :, h] = db[:T]
            out["d_initial_state"][b, h] = dS
    return out
