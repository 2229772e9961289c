"""GPU parity of the recurrence with its prologue folded in (gdn_fwd_raw /
gdn_bwd_raw) against the float64 chain of oracles: the prologue oracle (q, k
normalised to unit length, alpha = exp(-softplus(a)), beta = sigmoid(b);
"OpenGDN", Mixer), the token-loop oracle of the recurrence, and the prologue's
chain rule back to the raw inputs.  On the tensor-core shapes the prologue runs
inside the chunk and gradient kernels; other shapes run the prologue kernel
inside the call.  Tolerances as for gdn_fwd / gdn_bwd, checked per tensor and
per block."""
import numpy as np
import pytest
import torch

from gated_delta_rule_19_gb300 import gdn
from gated_delta_rule_19_gb300.inputs import custom, make_inputs, make_prologue_inputs
from gdn_testutil import compare, poisoned, to_np

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


def _inputs(B, T, H, K, V, C, dtype, seed, slow=False):
    x = make_prologue_inputs(B, T, H, K, dtype, seed=seed)
    if slow:  # alpha = sigmoid(-a) near 0.98: the state carries across many chunks
        g = torch.Generator().manual_seed(seed + 1)
        x["a_logit"] = (-4.0 + 0.5 * torch.randn(B, T, H, generator=g)).to(x["a_logit"].dtype)
    r = make_inputs(custom(B=B, T=T, H=H, K=K, V=V, chunk=C, dtype=dtype, seed=seed + 2, init_std=0.3,
                           dfinal_std=0.05))
    return x, r


def _oracle(oracle_mod, pro, x, r):
    nx = {n: to_np(t) for n, t in x.items()}
    q, k, al, be = pro.prologue_fwd(nx["q_raw"], nx["k_raw"], nx["a_logit"], nx["b_logit"])
    v, s0, do, dsT = (to_np(r[n]) for n in ("v", "initial_state", "d_o", "d_final_state"))
    o, sT = oracle_mod.gated_delta_fwd(q, k, v, al, be, s0)
    g = oracle_mod.gated_delta_bwd(q, k, v, al, be, s0, do, dsT)
    dq, dk, da, db = pro.prologue_bwd(nx["q_raw"], nx["k_raw"], nx["a_logit"], nx["b_logit"], g["dq"], g["dk"],
                                      g["dalpha"], g["dbeta"])
    return dict(o=o, final_state=sT, dq_raw=dq, dk_raw=dk, dv=g["dv"], da=da, db=db,
                d_initial_state=g["d_initial_state"])


def _gpu(x, r, C, saved=True):
    """Both calls on NaN-filled outputs (an element left unwritten shows up)."""
    d = {n: t.cuda() for n, t in x.items()}
    v, s0, do = r["v"].cuda(), r["initial_state"].cuda(), r["d_o"].cuda()
    dsT = r["d_final_state"].cuda() if r["d_final_state"] is not None else None
    args = (d["q_raw"], d["k_raw"], v, d["a_logit"], d["b_logit"], s0)
    o, sT, sv = gdn.gdn_fwd_raw(*args, chunk=C, saved=saved, o=poisoned(v), final_state=poisoned(s0))
    grads = tuple(poisoned(t) for t in (d["q_raw"], d["k_raw"], v, d["a_logit"], d["b_logit"]))
    g = gdn.gdn_bwd_raw(*args, do, dsT, saved=sv, chunk=C, grads=grads, d_initial_state=poisoned(s0))
    torch.cuda.synchronize()
    return dict(o=o, final_state=sT, **dict(zip(("dq_raw", "dk_raw", "dv", "da", "db", "d_initial_state"), g)))


# (B, T, H, K, V, chunk, dtype, slow decay): tensor-core shapes with a ragged tail,
# K or V below 128 (rows of 32 columns: the normalised rows' copies are written
# piece by piece), the within-call sequence split (B = 1, four streams of 64
# chunks), slow decay; then shapes that run the prologue kernel and the CUDA-core
# kernels
CASES = [
    (2, 300, 3, 128, 128, 64, "bf16", False),
    (2, 500, 2, 128, 128, 64, "bf16", True),
    (2, 256, 3, 64, 64, 64, "bf16", True),
    (1, 200, 2, 64, 128, 64, "bf16", False),
    (2, 130, 2, 32, 32, 64, "bf16", False),
    (1, 150, 3, 16, 64, 64, "bf16", True),
    (1, 4096, 4, 128, 128, 64, "bf16", False),
    (1, 100, 2, 32, 64, 32, "f32", True),
    (2, 130, 2, 32, 32, 32, "bf16", False),
]


@pytest.mark.parametrize("B,T,H,K,V,C,dtype,slow", CASES)
def test_raw_matches_oracle_chain(oracle_mod, pro, B, T, H, K, V, C, dtype, slow):
    x, r = _inputs(B, T, H, K, V, C, dtype, seed=800 + T + K, slow=slow)
    got = {n: to_np(t) for n, t in _gpu(x, r, C).items()}
    compare(got, _oracle(oracle_mod, pro, x, r), dtype, chunk=C)


def test_raw_backward_recompute_equals_saved():
    """gdn_bwd_raw without `saved` normalises the rows again and recomputes the
    chunk results with the same kernels: identical gradients."""
    x, r = _inputs(2, 256, 2, 128, 128, 64, "bf16", seed=901)
    a = _gpu(x, r, 64, saved=True)
    b = _gpu(x, r, 64, saved=False)
    for n in ("dq_raw", "dk_raw", "dv", "da", "db", "d_initial_state"):
        assert torch.equal(a[n], b[n]), n


def test_raw_equals_prologue_then_recurrence_within_tolerance():
    """The folded prologue computes the same function as gdn_prologue_fwd
    followed by gdn_fwd (they differ only in where alpha and beta are rounded)."""
    x, r = _inputs(2, 192, 2, 128, 128, 64, "bf16", seed=902)
    d = {n: t.cuda() for n, t in x.items()}
    v, s0 = r["v"].cuda(), r["initial_state"].cuda()
    o_raw, s_raw, _ = gdn.gdn_fwd_raw(d["q_raw"], d["k_raw"], v, d["a_logit"], d["b_logit"], s0, chunk=64)
    q, k, al, be = gdn.gdn_prologue_fwd(d["q_raw"], d["k_raw"], d["a_logit"], d["b_logit"])
    o, s, _ = gdn.gdn_fwd(q, k, v, al, be, s0, chunk=64)
    torch.cuda.synchronize()
    rel = lambda a, b: float((a.float() - b.float()).norm() / b.float().norm())
    assert rel(o_raw, o) < 1e-2 and rel(s_raw, s) < 1e-2
