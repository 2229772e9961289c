"""GPU parity of the fused prologue (gdn_prologue_fwd / gdn_prologue_bwd) against
the float64 prologue oracle, alone and composed with the recurrence: prologue ->
gdn_fwd -> gdn_bwd -> prologue backward against the same chain of oracles.
Relative L2 per tensor: 1e-5 for fp32, 2e-2 (outputs) / 3e-2 (gradients) for bf16."""
import numpy as np
import pytest
import torch

from gated_delta_rule_19_gb300 import gdn
from gated_delta_rule_19_gb300.inputs import custom, make_inputs, make_prologue_inputs
from gdn_testutil import TOL, local_failure, rel_l2, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_19_gb300 import _build

    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.fixture(scope="module")
def pro():
    from oracle import prologue

    return prologue


def _check(got, ref, lim, names):
    errs = {n: rel_l2(g, r) for n, g, r in zip(names, got, ref)}
    bad = [f"{n}: {e:.3e}" for n, e in errs.items() if not e <= lim]
    bad += [m for m in (local_failure(g, r, n, lim) for n, g, r in zip(names, got, ref)) if m]
    assert not bad, (bad, errs)


# Row tiles are 8 KB per tensor (16 to 256 rows, by K and dtype) and each CTA of
# the persistent grid walks several of them: the cases cover every K and dtype,
# ragged last tiles, and (the last two) more tiles than the grid has CTAs.
@pytest.mark.parametrize("B,T,H,K,dtype", [(2, 33, 3, 128, "f32"), (1, 17, 2, 64, "bf16"),
                                           (3, 5, 4, 16, "f32"), (2, 64, 6, 128, "bf16"),
                                           (1, 1000, 3, 32, "bf16"), (2, 777, 5, 16, "bf16"),
                                           (1, 50, 7, 64, "f32"), (1, 300, 3, 32, "f32"),
                                           (4, 4099, 6, 128, "bf16"), (3, 4097, 5, 32, "f32"),
                                           (8, 4096, 6, 128, "bf16")])  # the bench's workload
def test_prologue_matches_oracle(pro, B, T, H, K, dtype):
    x = make_prologue_inputs(B, T, H, K, dtype, seed=B * 100 + T + K)
    d = {n: t.cuda() for n, t in x.items()}
    got = gdn.gdn_prologue_fwd(d["q_raw"], d["k_raw"], d["a_logit"], d["b_logit"])
    ref = pro.prologue_fwd(*(to_np(x[n]) for n in ("q_raw", "k_raw", "a_logit", "b_logit")))
    _check([to_np(t) for t in got], ref, TOL[dtype]["out"], ("q", "k", "alpha", "beta"))
    gg = gdn.gdn_prologue_bwd(*(d[n] for n in ("q_raw", "k_raw", "a_logit", "b_logit", "dq", "dk", "dalpha",
                                                "dbeta")))
    rg = pro.prologue_bwd(*(to_np(x[n]) for n in ("q_raw", "k_raw", "a_logit", "b_logit", "dq", "dk",
                                                   "dalpha", "dbeta")))
    torch.cuda.synchronize()
    _check([to_np(t) for t in gg], rg, TOL[dtype]["grad"], ("dq_raw", "dk_raw", "da", "db"))


def test_prologue_extreme_logits_saturate():
    B, T, H, K = 1, 4, 1, 32
    a = torch.tensor([[[100.0], [-100.0], [0.0], [30.0]]], device="cuda")
    qr = torch.randn(B, T, H, K, device="cuda")
    q, k, alpha, beta = gdn.gdn_prologue_fwd(qr, qr, a, a)
    torch.cuda.synchronize()
    assert alpha[0, 0, 0].item() == 0.0 and alpha[0, 1, 0].item() == 1.0 and alpha[0, 2, 0].item() == 0.5
    assert beta[0, 0, 0].item() == 1.0 and beta[0, 1, 0].item() == 0.0 and beta[0, 2, 0].item() == 0.5
    ones = torch.ones_like(alpha)
    _, _, da, db = gdn.gdn_prologue_bwd(qr, qr, a, a, q, k, ones, ones)
    torch.cuda.synchronize()
    assert torch.isfinite(da).all() and torch.isfinite(db).all()


@pytest.mark.parametrize("B,T,H,K,V,C,dtype", [(1, 64, 2, 16, 16, 16, "f32"), (2, 128, 2, 128, 128, 64, "bf16")])
def test_prologue_composed_with_recurrence(oracle_mod, pro, B, T, H, K, V, C, dtype):
    """raw q/k and logits -> prologue -> gdn_fwd -> gdn_bwd -> prologue backward,
    against the oracles composed the same way."""
    x = make_prologue_inputs(B, T, H, K, dtype, seed=7 + K)
    w = custom(B=B, T=T, H=H, K=K, V=V, chunk=C, dtype=dtype, seed=70 + K, init_std=0.1)
    r = make_inputs(w)  # v, initial state and upstream gradients of the recurrence
    d = {n: t.cuda() for n, t in x.items()}
    v, s0, do = r["v"].cuda(), r["initial_state"].cuda(), r["d_o"].cuda()
    q, k, al, be = gdn.gdn_prologue_fwd(d["q_raw"], d["k_raw"], d["a_logit"], d["b_logit"])
    o, sT, saved = gdn.gdn_fwd(q, k, v, al, be, s0, chunk=C, saved=True)
    dq, dk, dv, dal, dbe, ds0 = gdn.gdn_bwd(q, k, v, al, be, s0, do, None, saved=saved, chunk=C)
    dqr, dkr, da, db = gdn.gdn_prologue_bwd(d["q_raw"], d["k_raw"], d["a_logit"], d["b_logit"], dq, dk, dal, dbe)
    torch.cuda.synchronize()
    # oracle chain (the oracle sees the prologue outputs cast to the run dtype, as the GPU path does)
    np_x = {n: to_np(t) for n, t in x.items()}
    rq, rk, ral, rbe = pro.prologue_fwd(np_x["q_raw"], np_x["k_raw"], np_x["a_logit"], np_x["b_logit"])
    cast = (lambda a: to_np(torch.from_numpy(a).to(torch.bfloat16))) if dtype == "bf16" else (lambda a: a)
    rq, rk, ral, rbe = cast(rq), cast(rk), cast(ral), cast(rbe)
    ro, rsT = oracle_mod.gated_delta_fwd(rq, rk, to_np(r["v"]), ral, rbe, to_np(r["initial_state"]))
    g = oracle_mod.gated_delta_bwd(rq, rk, to_np(r["v"]), ral, rbe, to_np(r["initial_state"]), to_np(r["d_o"]),
                                   None)
    rg = pro.prologue_bwd(np_x["q_raw"], np_x["k_raw"], np_x["a_logit"], np_x["b_logit"], g["dq"], g["dk"],
                          g["dalpha"], g["dbeta"])
    tol = TOL[dtype]
    _check([to_np(o), to_np(sT)], [ro, rsT], tol["out"], ("o", "final_state"))
    _check([to_np(t) for t in (dqr, dkr, da, db, dv)], list(rg) + [g["dv"]], tol["grad"],
           ("dq_raw", "dk_raw", "da", "db", "dv"))
