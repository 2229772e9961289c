"""GPU parity: the CUDA path (called through the C ABI binding) against the
float64 oracle on the same seeded inputs, element by element (relative L2 per
output tensor; 1e-5 for fp32 inputs, 2e-2 outputs / 3e-2 gradients for bf16).

Small and medium workloads are compared in full; the large training shape and
the long stream are compared on sampled (b, h) streams, which the oracle
computes on their own (streams are independent)."""
import numpy as np
import pytest
import torch

from gated_delta_rule_19_gb300 import gdn
from gated_delta_rule_19_gb300.inputs import WORKLOADS, custom, make_inputs
from gdn_testutil import (compare, gpu_run, oracle_run, rel_l2, sample_gpu, select_states,
                          select_streams, to_np)

pytestmark = pytest.mark.gpu

W = WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_19_gb300 import _build

    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _check_workload(oracle_mod, w, streams=None):
    inp = make_inputs(w)
    got = gpu_run(w, inp, backward=w.backward)
    ref = oracle_run(oracle_mod, inp, backward=w.backward, streams=streams)
    if streams is not None:
        got = sample_gpu(got, streams)
    return compare(got, ref, w.dtype, chunk=w.chunk)


def test_tiny_fp32_fwd_bwd(oracle_mod):
    errs = _check_workload(oracle_mod, W["tiny_f32_B1_T64_H2_K16_V16"])
    assert set(errs) >= {"o", "final_state", "dq", "dk", "dv", "dalpha", "dbeta"}


def test_fwd_bf16_B2_T1024_H4_K64(oracle_mod):
    _check_workload(oracle_mod, W["fwd_bf16_B2_T1024_H4_K64_V64"])


def test_train_bf16_B4_T2048_H6_K128(oracle_mod):
    errs = _check_workload(oracle_mod, W["train_bf16_B4_T2048_H6_K128_V128"])
    assert "dalpha" in errs


def test_train_bf16_B8_T4096_H6_K128_sampled(oracle_mod):
    """Full-size training shape; the oracle checks 4 of the 48 streams."""
    _check_workload(oracle_mod, W["train_bf16_B8_T4096_H6_K128_V128"],
                    streams=[(0, 0), (3, 5), (5, 2), (7, 4)])


def test_stream_bf16_four_calls_equal_one_call(oracle_mod):
    """Long context in 4 calls of T/4 passing final_state forward: equals one
    call bit for bit (boundaries align with chunks) and matches the oracle on
    sampled heads."""
    w = W["stream_bf16_B1_T32768_H16_K128_V128_4calls"]
    inp = make_inputs(w)
    d = {n: (t.cuda() if t is not None else None) for n, t in inp.items()}
    o1, s1, _ = gdn.gdn_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["initial_state"],
                            chunk=w.chunk)
    L = w.T // w.calls
    state = d["initial_state"].clone()
    outs = []
    for i in range(w.calls):
        sl = slice(i * L, (i + 1) * L)
        o, state, _ = gdn.gdn_fwd(*(d[n][:, sl].contiguous() for n in ("q", "k", "v", "alpha",
                                                                       "beta")),
                                  state, chunk=w.chunk, final_state=state)  # in place
        outs.append(o)
    o4 = torch.cat(outs, 1)
    torch.cuda.synchronize()
    assert torch.equal(o4, o1)
    assert torch.equal(state, s1)
    streams = [(0, 0), (0, 9), (0, 15)]
    ref = oracle_run(oracle_mod, inp, backward=False, streams=streams)
    got = sample_gpu(dict(o=to_np(o4), final_state=to_np(state)), streams)
    compare(got, ref, "bf16")


@pytest.mark.parametrize("C", [16, 32, 64])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chunk_sizes(oracle_mod, C, dtype):
    w = custom(B=2, T=192, H=2, K=32, V=64, chunk=C, dtype=dtype, seed=10 + C, init_std=0.1,
               dfinal_std=0.01)
    inp = make_inputs(w)
    compare(gpu_run(w, inp, True), oracle_run(oracle_mod, inp, True), dtype, chunk=w.chunk)


@pytest.mark.parametrize("T", [1, 5, 63, 64, 65, 130])
def test_ragged_lengths_fp32(oracle_mod, T):
    w = custom(B=1, T=T, H=3, K=16, V=32, chunk=64, dtype="f32", seed=T, init_std=0.1,
               dfinal_std=0.1)
    inp = make_inputs(w)
    compare(gpu_run(w, inp, True), oracle_run(oracle_mod, inp, True), "f32", chunk=w.chunk)


# all run the tensor-core kernels: TMA fills the columns past K or V with zeros
# on every load and clips them on every store
@pytest.mark.parametrize("K,V", [(64, 128), (128, 64), (128, 32), (16, 128), (128, 16), (32, 32),
                                 (16, 64)])
def test_key_value_dims_differ_bf16(oracle_mod, K, V):
    w = custom(B=1, T=200, H=2, K=K, V=V, chunk=64, dtype="bf16", seed=K + V, init_std=0.1,
               dfinal_std=0.01)
    inp = make_inputs(w)
    compare(gpu_run(w, inp, True), oracle_run(oracle_mod, inp, True), "bf16", chunk=w.chunk)


@pytest.mark.parametrize("seed", [100, 101, 102])
def test_seeds_fp32_full_heads(oracle_mod, seed):
    w = custom(B=2, T=96, H=2, K=128, V=128, chunk=32, dtype="f32", seed=seed, init_std=0.1,
               dfinal_std=0.1)
    inp = make_inputs(w)
    compare(gpu_run(w, inp, True), oracle_run(oracle_mod, inp, True), "f32", chunk=w.chunk)


def test_backward_recompute_equals_saved():
    """gdn_bwd without the saved boundary states recomputes them with the same
    kernels: identical gradients."""
    w = custom(B=2, T=256, H=2, K=64, V=64, chunk=64, dtype="bf16", seed=7, init_std=0.1,
               dfinal_std=0.01)
    inp = make_inputs(w)
    a = gpu_run(w, inp, True, saved_mode="saved")
    b = gpu_run(w, inp, True, saved_mode="recompute")
    for n in a:
        np.testing.assert_array_equal(a[n], b[n], err_msg=n)


def test_empty_and_degenerate():
    # T = 0: final state is the initial state; d_initial_state is d_final_state
    dev = "cuda"
    q = torch.zeros(2, 0, 3, 16, device=dev)
    v = torch.zeros(2, 0, 3, 32, device=dev)
    g = torch.zeros(2, 0, 3, device=dev)
    s0 = torch.randn(2, 3, 32, 16, device=dev)
    o, sT, _ = gdn.gdn_fwd(q, q, v, g, g, s0, chunk=16)
    assert o.shape == (2, 0, 3, 32) and torch.equal(sT, s0)
    o, sT, _ = gdn.gdn_fwd(q, q, v, g, g, None, chunk=16)
    assert torch.count_nonzero(sT) == 0
    dsT = torch.randn_like(s0)
    *_, ds0 = gdn.gdn_bwd(q, q, v, g, g, s0, v, dsT, chunk=16)
    assert torch.equal(ds0, dsT)
    # B = 0
    z = torch.zeros(0, 8, 2, 16, device=dev)
    o, sT, _ = gdn.gdn_fwd(z, z, z, torch.zeros(0, 8, 2, device=dev),
                           torch.zeros(0, 8, 2, device=dev), chunk=16)
    assert o.shape == (0, 8, 2, 16)


def test_null_update_and_exact_write_on_gpu():
    """Closed forms on the GPU path too: beta=0, alpha=1 keeps the state;
    unit keys with beta=1 and q=k read back v."""
    w = custom(B=1, T=100, H=2, K=64, V=64, chunk=64, dtype="f32", seed=3, init_std=1.0)
    inp = make_inputs(w)
    d = {n: (t.cuda() if t is not None else None) for n, t in inp.items()}
    ones = torch.ones_like(d["alpha"])
    o, sT, _ = gdn.gdn_fwd(d["q"], d["k"], d["v"], ones, torch.zeros_like(ones),
                           d["initial_state"], chunk=64)
    ref = torch.einsum("bhvk,bthk->bthv", d["initial_state"], d["q"])
    assert rel_l2(to_np(o), to_np(ref)) < 1e-6
    assert rel_l2(to_np(sT), to_np(d["initial_state"])) < 1e-6
    o, _, _ = gdn.gdn_fwd(d["k"], d["k"], d["v"], d["alpha"], ones, d["initial_state"], chunk=64)
    assert rel_l2(to_np(o), to_np(d["v"])) < 1e-5


# ------------------------------------------------ tensor-core path (bf16, K=V=128, C=64)

@pytest.mark.parametrize("T", [1, 63, 65, 200])
def test_tc_path_ragged_lengths(oracle_mod, T):
    w = custom(B=2, T=T, H=3, K=128, V=128, chunk=64, dtype="bf16", seed=300 + T, init_std=0.1,
               dfinal_std=0.01)
    inp = make_inputs(w)
    compare(gpu_run(w, inp, True), oracle_run(oracle_mod, inp, True), "bf16", chunk=w.chunk)


def test_tc_path_many_streams_multiple_waves(oracle_mod):
    """B*H above the SM count: the scans run in several waves of CTAs."""
    w = custom(B=4, T=128, H=40, K=128, V=128, chunk=64, dtype="bf16", seed=77, init_std=0.1,
               dfinal_std=0.01)
    inp = make_inputs(w)
    got = gpu_run(w, inp, True)
    streams = [(0, 0), (1, 17), (2, 33), (3, 39)]
    ref = oracle_run(oracle_mod, inp, True, streams=streams)
    compare(sample_gpu(got, streams), ref, "bf16")


def test_tc_backward_recompute_equals_saved():
    w = custom(B=2, T=300, H=2, K=128, V=128, chunk=64, dtype="bf16", seed=8, init_std=0.1,
               dfinal_std=0.01)
    inp = make_inputs(w)
    a = gpu_run(w, inp, True, saved_mode="saved")
    b = gpu_run(w, inp, True, saved_mode="recompute")
    for n in a:
        np.testing.assert_array_equal(a[n], b[n], err_msg=n)


@pytest.mark.parametrize("dtype,K,V,C", [("bf16", 128, 128, 64), ("f32", 32, 64, 32), ("bf16", 64, 64, 64),
                                         ("bf16", 64, 128, 64), ("bf16", 128, 64, 64)])
def test_slow_decay_long_range(oracle_mod, dtype, K, V, C):
    """Gates in (0.97, 1): the state carries across many chunks (about 40% of it
    survives a 64-token chunk), so cross-chunk propagation, the initial state and
    the final-state gradient all reach far; forward and backward against the
    oracle on every stream."""
    w = custom(B=2, T=1000, H=2, K=K, V=V, chunk=C, dtype=dtype, seed=600 + K + C, init_std=0.3, dfinal_std=0.05,
               alpha_lo=0.97)
    inp = make_inputs(w)
    compare(gpu_run(w, inp, True), oracle_run(oracle_mod, inp, True), dtype, chunk=w.chunk)


@pytest.mark.parametrize("B,H", [(7, 6), (5, 9)])
def test_tc_scan_48_column_slices(oracle_mod, B, H):
    """39 to 50 streams run the scans in 48-column V-slices (three per stream,
    the third reaching past V = 128 into zero columns): forward and backward
    against the oracle on every stream, slow decay so the states carry."""
    w = custom(B=B, T=200, H=H, K=128, V=128, chunk=64, dtype="bf16", seed=650 + B * H, init_std=0.3,
               dfinal_std=0.05, alpha_lo=0.97)
    inp = make_inputs(w)
    compare(gpu_run(w, inp, True), oracle_run(oracle_mod, inp, True), "bf16", chunk=w.chunk)


@pytest.mark.parametrize("B,H", [(7, 6), (3, 20)])
def test_tc_k64_slices_and_tail(oracle_mod, B, H):
    """K = V = 64 on the tensor-core kernels with more streams than one wave of
    48-column slices (the second slice of each stream reaches past V = 64 into
    the zero columns) and a ragged tail chunk: forward and backward against the
    oracle on every stream, slow decay so the states carry."""
    w = custom(B=B, T=230, H=H, K=64, V=64, chunk=64, dtype="bf16", seed=660 + B * H, init_std=0.3,
               dfinal_std=0.05, alpha_lo=0.97)
    inp = make_inputs(w)
    compare(gpu_run(w, inp, True), oracle_run(oracle_mod, inp, True), "bf16", chunk=w.chunk)


def test_tc_error_flag_stays_clear():
    """The tensor-core kernels' bounded waits never give up in a normal run: the
    error word at the start of the caller's workspace stays 0."""
    w = custom(B=2, T=256, H=2, K=128, V=128, chunk=64, dtype="bf16", seed=9, init_std=0.1,
               dfinal_std=0.01)
    inp = make_inputs(w)
    d = {n: (t.cuda() if t is not None else None) for n, t in inp.items()}
    args = (d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["initial_state"])
    p = gdn.make_problem(w.B, w.T, w.H, w.K, w.V, w.chunk, torch.bfloat16)
    wsf = torch.full((gdn.gdn_fwd_workspace_bytes(p),), 0x5A, dtype=torch.uint8, device="cuda")
    wsb = torch.full((gdn.gdn_bwd_workspace_bytes(p),), 0x5A, dtype=torch.uint8, device="cuda")
    _, _, saved = gdn.gdn_fwd(*args, chunk=w.chunk, saved=True, workspace=wsf)
    gdn.gdn_bwd(*args, d["d_o"], d["d_final_state"], saved=saved, chunk=w.chunk, workspace=wsb)
    torch.cuda.synchronize()
    assert int(wsf[:4].view(torch.int32).item()) == 0
    assert int(wsb[:4].view(torch.int32).item()) == 0


def test_tc_dirty_workspace_and_repeated_calls_bitwise():
    """grad_qk and grad_wy hand out chunks from counters kept in the workspace's
    error-flag area, reset by each call.  With 1536 chunks (far more than the
    persistent grids' CTAs), results from workspaces full of 0x7F bytes, used for
    two calls in a row, equal those from fresh workspaces bit for bit."""
    w = custom(B=4, T=4096, H=6, K=128, V=128, chunk=64, dtype="bf16", seed=31, init_std=0.1,
               dfinal_std=0.01)
    inp = make_inputs(w)
    d = {n: (t.cuda() if t is not None else None) for n, t in inp.items()}
    args = (d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["initial_state"])
    p = gdn.make_problem(w.B, w.T, w.H, w.K, w.V, w.chunk, torch.bfloat16)

    def run(wsf=None, wsb=None):
        o, s_t, saved = gdn.gdn_fwd(*args, chunk=w.chunk, saved=True, workspace=wsf)
        g = gdn.gdn_bwd(*args, d["d_o"], d["d_final_state"], saved=saved, chunk=w.chunk, workspace=wsb)
        torch.cuda.synchronize()
        return [o, s_t] + [x for x in g if x is not None]

    ref = run()
    wsf = torch.full((gdn.gdn_fwd_workspace_bytes(p),), 0x7F, dtype=torch.uint8, device="cuda")
    wsb = torch.full((gdn.gdn_bwd_workspace_bytes(p),), 0x7F, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        got = run(wsf, wsb)
        assert len(got) == len(ref)
        for i, (a, b) in enumerate(zip(ref, got)):
            assert torch.equal(a, b), f"output {i} differs"
