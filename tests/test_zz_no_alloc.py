"""gdn_fwd_noalloc -- the forward for callers that cannot allocate device memory
(a host framework that owns all device memory, or a latency-critical path where
cudaMalloc's device-wide synchronisation is not acceptable).  Its scratch is a
fixed array inside the library instead of a caller-owned workspace.

The test calls it through the C ABI twice in a row, on two different problems
(so the second call runs on the scratch the first left behind), and checks each
result against the ordinary gdn_fwd within the parity tolerance.  This file is
named so that pytest collects it last."""
import pytest
import torch

from gated_delta_rule_19_gb300 import gdn
from gated_delta_rule_19_gb300.inputs import custom, make_inputs
from gdn_testutil import TOL, rel_l2, to_np

pytestmark = pytest.mark.gpu


def _run_pair(w):
    from gated_delta_rule_19_gb300 import _build

    _build.build()
    inp = make_inputs(w)
    d = {n: (t.cuda() if t is not None else None) for n, t in inp.items()}
    args = (d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["initial_state"])
    o_ref, s_ref, _ = gdn.gdn_fwd(*args, chunk=w.chunk)
    o = torch.full_like(o_ref, float("nan"))
    s = torch.full_like(s_ref, float("nan"))
    gdn.gdn_fwd_noalloc(*args, o, s, chunk=w.chunk)
    torch.cuda.synchronize()
    tol = TOL[w.dtype]["out"]
    assert rel_l2(to_np(o), to_np(o_ref)) <= tol
    assert rel_l2(to_np(s), to_np(s_ref)) <= tol


def test_fwd_noalloc_matches_fwd_two_calls_in_a_row():
    assert torch.cuda.is_available()
    # first call: bf16, K=V=64, 128 chunks of scratch
    _run_pair(custom(B=2, T=1024, H=4, K=64, V=64, chunk=64, dtype="bf16", seed=21,
                     init_std=0.1))
    # second call: another shape and dtype on the scratch the first call left
    _run_pair(custom(B=1, T=300, H=3, K=128, V=32, chunk=32, dtype="f32", seed=22,
                     init_std=0.1))


def test_fwd_noalloc_rejects_oversized_problem():
    w = custom(B=8, T=4096, H=6, K=128, V=128, chunk=64, dtype="bf16", seed=0)
    q = torch.zeros(w.B, w.T, w.H, w.K, dtype=torch.bfloat16, device="cuda")
    g = torch.zeros(w.B, w.T, w.H, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_fwd_noalloc(q, q, q, g, g, None, o, chunk=w.chunk)
    assert ei.value.status == gdn.GDN_ERR_UNSUPPORTED
    assert "scratch" in str(ei.value)
