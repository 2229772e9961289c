"""GPU parity of the within-call sequence split (two-level scan) of the
tensor-core path.  Over a run of chunks the state map is affine ("Sparse Delta
Memory: layer and kernels", What the layer computes: Phase 2), so a stream's
chunks can be cut into pieces that run side by side and be linked afterwards;
the results must match the float64 oracle with the usual bf16 tolerances
(2e-2 outputs and states, 3e-2 gradients) and the unsplit scan up to rounding."""
import numpy as np
import pytest
import torch

from gated_delta_rule_19_gb300 import gdn
from gated_delta_rule_19_gb300.inputs import custom, make_inputs, make_varlen_inputs
from gdn_testutil import compare, gpu_run, oracle_run, rel_l2, sample_gpu, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_19_gb300 import _build

    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.fixture(autouse=True)
def _policy():
    gdn.gdn_set_sequence_split(0)
    yield
    gdn.gdn_set_sequence_split(0)


def _run_profiled(w, inp, **kw):
    gdn.gdn_profiler_start(256)
    out = gpu_run(w, inp, True, **kw)
    gdn.gdn_profiler_stop()
    return out, gdn.gdn_profiler_summary()


# alpha_lo = 0.97: gates in (0.97, 1), so a piece's transition is far from zero
# and the chain between pieces decides the result (with the default gates a
# chunk's decay is below float32 resolution and every piece forgets its start).
@pytest.mark.parametrize("alpha_lo", [0.0, 0.97])
@pytest.mark.parametrize("B,T,H", [(1, 2048, 2), (2, 1024, 2), (1, 1000, 3)])
def test_automatic_split_matches_oracle(oracle_mod, B, T, H, alpha_lo):
    """Few streams: the automatic policy splits (B = 1, or T a multiple of the
    chunk); forward and backward against the oracle on every stream."""
    w = custom(B=B, T=T, H=H, K=128, V=128, chunk=64, dtype="bf16", seed=500 + T + H, init_std=0.2,
               dfinal_std=0.02, alpha_lo=alpha_lo)
    inp = make_inputs(w)
    got, prof = _run_profiled(w, inp)
    assert "scan_fwd_tc(split pass 1)" in prof and "scan_bwd_tc(split pass 1)" in prof, prof
    compare(got, oracle_run(oracle_mod, inp, True), "bf16")


@pytest.mark.parametrize("pieces", [2, 3, 7, 40])
def test_forced_split_matches_unsplit_and_oracle(oracle_mod, pieces):
    """Any number of pieces, including more pieces than chunks (empty pieces pass
    their state through), against the unsplit scan and the oracle; slow decay, so
    every piece's start state matters."""
    w = custom(B=1, T=1024, H=2, K=128, V=128, chunk=64, dtype="bf16", seed=510, init_std=0.2, dfinal_std=0.02,
               alpha_lo=0.97)
    inp = make_inputs(w)
    gdn.gdn_set_sequence_split(1)
    plain, prof0 = _run_profiled(w, inp)
    assert "scan_fwd_tc(split pass 1)" not in prof0
    gdn.gdn_set_sequence_split(pieces)
    split, prof1 = _run_profiled(w, inp)
    assert "scan_fwd_tc(split pass 1)" in prof1
    compare(split, oracle_run(oracle_mod, inp, True), "bf16")
    for n in plain:  # the same bf16 operands; only the chain's fp32 rounding differs
        assert rel_l2(split[n], plain[n]) < 1e-2, (n, rel_l2(split[n], plain[n]))


def test_split_backward_recompute_equals_saved():
    """Without `saved` the backward recomputes the chunk-start states with the
    same split: bit-identical gradients."""
    w = custom(B=1, T=2048, H=2, K=128, V=128, chunk=64, dtype="bf16", seed=520, init_std=0.2, dfinal_std=0.02,
               alpha_lo=0.97)
    inp = make_inputs(w)
    a = gpu_run(w, inp, True, saved_mode="saved")
    b = gpu_run(w, inp, True, saved_mode="recompute")
    for n in a:
        np.testing.assert_array_equal(a[n], b[n], err_msg=n)


def test_split_in_place_state_and_error_word():
    """final_state may be initial_state itself; the bounded waits never give up."""
    w = custom(B=1, T=1024, H=2, K=128, V=128, chunk=64, dtype="bf16", seed=530, init_std=0.2)
    d = {n: (t.cuda() if t is not None else None) for n, t in make_inputs(w).items()}
    args = (d["q"], d["k"], d["v"], d["alpha"], d["beta"])
    p = gdn.make_problem(w.B, w.T, w.H, w.K, w.V, w.chunk, torch.bfloat16)
    ws = torch.full((gdn.gdn_fwd_workspace_bytes(p),), 0x5A, dtype=torch.uint8, device="cuda")
    o1, s1, _ = gdn.gdn_fwd(*args, d["initial_state"], workspace=ws)
    state = d["initial_state"].clone()
    o2, _, _ = gdn.gdn_fwd(*args, state, final_state=state)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    assert torch.equal(o1, o2) and torch.equal(s1, state)


def test_split_varlen_matches_oracle(oracle_mod):
    """Packed sequences with every sequence cut into 3 pieces (short sequences
    get empty pieces)."""
    lengths = [1, 63, 64, 65, 700, 0, 130, 1200]
    inp = make_varlen_inputs(lengths, 2, 128, 128, "bf16", seed=540, init_std=0.3, dfinal_std=0.05, alpha_lo=0.97)
    d = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in inp.items()}
    gdn.gdn_set_sequence_split(3)
    gdn.gdn_profiler_start(256)
    o, sT, saved = gdn.gdn_varlen_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["cu_seqlens"], None,
                                      d["initial_state"], saved=True, check=True)
    g = gdn.gdn_varlen_bwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["cu_seqlens"], None,
                           d["initial_state"], d["d_o"], d["d_final_state"], saved=saved, check=True)
    gdn.gdn_profiler_stop()
    torch.cuda.synchronize()
    assert "scan_fwd_tc(split pass 1)" in gdn.gdn_profiler_summary()
    names = ("dq", "dk", "dv", "dalpha", "dbeta", "d_initial_state")
    got = dict(o=o, final_state=sT, **dict(zip(names, g)))
    cu = inp["cu_seqlens"].tolist()
    ref = {n: [] for n in ("o", "dq", "dk", "dv", "dalpha", "dbeta")}
    ref_sT, ref_ds0 = [], []
    for s in range(len(lengths)):
        a, e = cu[s], cu[s + 1]
        seq = {n: to_np(inp[n][a:e])[None] for n in ("q", "k", "v", "alpha", "beta", "d_o")}
        s0 = to_np(inp["initial_state"][s:s + 1])
        dsT = to_np(inp["d_final_state"][s:s + 1])
        o_r, sT_r = oracle_mod.gated_delta_fwd(seq["q"], seq["k"], seq["v"], seq["alpha"], seq["beta"], s0)
        gr = oracle_mod.gated_delta_bwd(seq["q"], seq["k"], seq["v"], seq["alpha"], seq["beta"], s0, seq["d_o"],
                                        dsT)
        ref["o"].append(o_r[0])
        for n in ("dq", "dk", "dv", "dalpha", "dbeta"):
            ref[n].append(gr[n][0])
        ref_sT.append(sT_r[0])
        ref_ds0.append(gr["d_initial_state"][0])
    want = {n: np.concatenate(x, 0) for n, x in ref.items()}
    want["final_state"] = np.stack(ref_sT)
    want["d_initial_state"] = np.stack(ref_ds0)
    compare({n: to_np(x) for n, x in got.items()}, want, "bf16")


def test_long_context_workload_sampled(oracle_mod):
    """The long context the bench times (B=1, T=65536, H=4, K=V=128 bf16: 1024
    chunks per stream), split automatically as the bench runs it; two of its four
    streams against the oracle over the whole sequence, forward and backward."""
    w = custom(B=1, T=65536, H=4, K=128, V=128, chunk=64, dtype="bf16", seed=7, init_std=0.1)
    inp = make_inputs(w)
    got, prof = _run_profiled(w, inp)
    assert "scan_fwd_tc(split pass 1)" in prof and "scan_bwd_tc(split pass 1)" in prof, prof
    streams = [(0, 0), (0, 3)]
    compare(sample_gpu(got, streams), oracle_run(oracle_mod, inp, True, streams=streams), "bf16")
