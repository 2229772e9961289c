"""gdn_fwd_noalloc -- the forward for callers that cannot allocate device memory
(a host framework that owns all device memory, or a latency-critical path where
cudaMalloc's device-wide synchronisation is not acceptable).  Its scratch is a
fixed array inside the library instead of a caller-owned workspace.

The tests call it through the C ABI several times in a row on different
problems, so every call after the first runs on the scratch an earlier call left
behind: first the CUDA-core kernels (fp32 K=V=64, then fp32 K=128/V=32, chunk
32), then the tensor-core kernels, which keep an error word and the work
counters of their persistent kernels in the scratch (bf16 K=V=128, chunk 64:
one problem with the within-call sequence split, one with a ragged tail chunk).
The same kernels on the same inputs must give the same bits as gdn_fwd with its
own workspace, so results are compared with torch.equal.  This file is named so
that pytest collects it last."""
import pytest
import torch

from gated_delta_rule_19_gb300 import gdn
from gated_delta_rule_19_gb300.inputs import custom, make_inputs

pytestmark = pytest.mark.gpu


def _run_pair(w):
    from gated_delta_rule_19_gb300 import _build

    _build.build()
    p = gdn.make_problem(w.B, w.T, w.H, w.K, w.V, w.chunk,
                         torch.bfloat16 if w.dtype == "bf16" else torch.float32)
    assert 0 < gdn.gdn_fwd_workspace_bytes(p) <= gdn.GDN_FWD_NOALLOC_SCRATCH_BYTES
    inp = make_inputs(w)
    d = {n: (t.cuda() if t is not None else None) for n, t in inp.items()}
    args = (d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["initial_state"])
    o_ref, s_ref, _ = gdn.gdn_fwd(*args, chunk=w.chunk)
    o = torch.full_like(o_ref, float("nan"))
    s = torch.full_like(s_ref, float("nan"))
    gdn.gdn_fwd_noalloc(*args, o, s, chunk=w.chunk)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref)
    assert torch.equal(s, s_ref)


def test_fwd_noalloc_matches_fwd_calls_in_a_row():
    assert torch.cuda.is_available()
    # CUDA-core kernels: fp32 K=V=64 (128 chunks of scratch), then fp32 K=128/V=32
    _run_pair(custom(B=2, T=1024, H=4, K=64, V=64, chunk=64, dtype="f32", seed=21,
                     init_std=0.1))
    _run_pair(custom(B=1, T=300, H=3, K=128, V=32, chunk=32, dtype="f32", seed=22,
                     init_std=0.1))
    # tensor-core kernels on the scratch the CUDA-core calls left: four streams of
    # 64 chunks (the within-call sequence split runs), then a ragged tail chunk
    _run_pair(custom(B=1, T=4096, H=4, K=128, V=128, chunk=64, dtype="bf16", seed=23,
                     init_std=0.1))
    _run_pair(custom(B=2, T=2000, H=3, K=128, V=128, chunk=64, dtype="bf16", seed=24,
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
