"""GPU parity of the packed variable-length calls (gdn_varlen_fwd / gdn_varlen_bwd).

Each sequence of a packed batch is an independent stream with its own initial
state, so its outputs and gradients must equal the float64 oracle run on that
sequence alone ("OpenGDN", Scope: ragged batches; "Sparse Delta Memory: layer and
kernels", What the layer computes: tokens past the end of a stream are masked).
Tolerances as for gdn_fwd / gdn_bwd: relative L2 1e-5 for fp32 inputs; 2e-2 for
bf16 outputs and states, 3e-2 for bf16 gradients."""
import numpy as np
import pytest
import torch

from gated_delta_rule_19_gb300 import gdn
from gated_delta_rule_19_gb300.inputs import custom, make_inputs, make_varlen_inputs
from gdn_testutil import TOL, local_failure, poisoned, rel_l2, to_np

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "dalpha", "dbeta")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_19_gb300 import _build

    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _cuda(inp):
    return {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in inp.items()}


def _run_varlen(d, chunk, max_len=None, backward=True):
    """Both calls on NaN-filled outputs: a row the kernels skip (or a ragged chunk's
    copy that misses one) shows up in the comparison."""
    S = d["cu_seqlens"].numel() - 1
    _, H, K = d["q"].shape
    V = d["v"].shape[-1]
    st_shape = (S, H, V, K)
    o, sT, saved = gdn.gdn_varlen_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["cu_seqlens"], max_len,
                                      d["initial_state"], chunk=chunk, saved=backward, check=True,
                                      o=poisoned(d["v"]), final_state=poisoned(d["v"], st_shape, torch.float32))
    out = dict(o=o, final_state=sT)
    if backward:
        grads = tuple(poisoned(d[n]) for n in ("q", "k", "v", "alpha", "beta"))
        g = gdn.gdn_varlen_bwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["cu_seqlens"], max_len,
                               d["initial_state"], d["d_o"], d["d_final_state"], saved=saved, chunk=chunk,
                               check=True, grads=grads,
                               d_initial_state=poisoned(d["v"], st_shape, torch.float32))
        out.update(zip(GRADS + ("d_initial_state",), g))
    torch.cuda.synchronize()
    return out


def _oracle_seq(oracle_mod, inp, s):
    """The oracle on sequence s alone (B = 1, T = its length)."""
    a, e = int(inp["cu_seqlens"][s]), int(inp["cu_seqlens"][s + 1])
    seq = {n: to_np(inp[n][a:e])[None] for n in ("q", "k", "v", "alpha", "beta", "d_o")}
    s0 = None if inp["initial_state"] is None else to_np(inp["initial_state"][s:s + 1])
    dsT = None if inp["d_final_state"] is None else to_np(inp["d_final_state"][s:s + 1])
    o, sT = oracle_mod.gated_delta_fwd(seq["q"], seq["k"], seq["v"], seq["alpha"], seq["beta"], s0)
    g = oracle_mod.gated_delta_bwd(seq["q"], seq["k"], seq["v"], seq["alpha"], seq["beta"], s0, seq["d_o"], dsT)
    return dict(o=o[0], final_state=sT[0], d_initial_state=g["d_initial_state"][0],
                **{n: g[n][0] for n in GRADS})


# bf16 with chunk 64 runs the tensor-core kernels on the flat chunk layout (each
# sequence starts a new chunk); other shapes pad to max_len.
CASES = [
    # lengths (one empty, ragged tails, exact chunks, several tiles), H, K, V, chunk, dtype
    ([1, 63, 64, 65, 200, 0, 130], 2, 64, 64, 64, "bf16"),
    ([65, 0, 1, 128, 70], 2, 32, 16, 64, "bf16"),
    ([64, 1, 128, 191], 2, 128, 128, 64, "bf16"),
    ([1, 63, 64, 65, 200, 0, 130, 0], 2, 128, 128, 64, "bf16"),
    # 40 sequences x 4 heads: more (sequence, head) streams than one wave of SMs
    ([(37 * i) % 150 + 1 for i in range(40)], 4, 128, 128, 64, "bf16"),
    ([5, 17, 33, 0, 48], 3, 32, 32, 16, "f32"),
    ([70, 9, 100], 1, 16, 64, 32, "f32"),
    ([129, 2], 2, 128, 128, 64, "f32"),
    # the longest sequence last and equal chunk counts: the scans run the
    # sequences longest first, through a permutation of the grid rows
    ([64, 300, 1, 700, 128, 128, 0, 1500], 3, 128, 128, 64, "bf16"),
    # one long sequence among short ones: the slice width follows the longest
    # chain (16-column slices)
    ([3000, 10, 10], 2, 128, 128, 64, "bf16"),
]


# alpha_lo = 0.97: slow decay, each sequence's initial state and the state
# carried across its chunks reach far (with the default gates a chunk forgets).
@pytest.mark.parametrize("alpha_lo", [0.0, 0.97])
@pytest.mark.parametrize("lengths,H,K,V,chunk,dtype", CASES)
def test_varlen_matches_oracle_per_sequence(oracle_mod, lengths, H, K, V, chunk, dtype, alpha_lo):
    inp = make_varlen_inputs(lengths, H, K, V, dtype, seed=700 + len(lengths) + K, init_std=0.3,
                             dfinal_std=0.05, alpha_lo=alpha_lo)
    got = _run_varlen(_cuda(inp), chunk)
    tol = TOL[dtype]
    cu = inp["cu_seqlens"].tolist()
    bad = []
    ref_all = {n: [] for n in ("o",) + GRADS}
    for s in range(len(lengths)):
        ref = _oracle_seq(oracle_mod, inp, s)
        a, e = cu[s], cu[s + 1]
        for n in ("final_state", "d_initial_state"):
            err = rel_l2(to_np(got[n][s]), ref[n])
            if err > tol["out" if n == "final_state" else "grad"]:
                bad.append(f"seq {s} {n}: {err:.2e}")
        for n in ("o",) + GRADS:
            ref_all[n].append(ref[n])
            # per sequence where the sequence has enough elements for a relative
            # norm to mean something; the packed tensors are compared as a whole
            if e - a >= 16:
                lim = tol["out" if n == "o" else "grad"]
                err = rel_l2(to_np(got[n][a:e]), ref[n])
                if err > lim:
                    bad.append(f"seq {s} {n}: {err:.2e}")
                msg = local_failure(to_np(got[n][a:e]), ref[n], n, lim, chunk, packed=True)
                if msg:
                    bad.append(f"seq {s} {msg}")
    for n in ("o",) + GRADS:
        err = rel_l2(to_np(got[n]), np.concatenate(ref_all[n], 0))
        if err > tol["out" if n == "o" else "grad"]:
            bad.append(f"packed {n}: {err:.2e}")
    assert not bad, "; ".join(bad)


@pytest.mark.parametrize("dtype,K", [("f32", 64), ("bf16", 128)])
def test_varlen_short_sequences_equal_their_own_dense_runs(dtype, K):
    """Each sequence of a packed batch, run alone through gdn_fwd / gdn_bwd (B = 1,
    T = its length), gives the same outputs and gradients: the varlen calls only
    move rows, so short sequences whose gradients are too small for a relative
    norm are checked against the dense path here.  Both layouts pad a sequence's
    last chunk exactly as the dense kernels pad a ragged tail, so the results are
    bit-identical."""
    lengths = [1, 2, 3, 7, 15, 64, 65]
    inp = make_varlen_inputs(lengths, 2, K, K, dtype, seed=41, init_std=0.3, dfinal_std=0.05)
    d = _cuda(inp)
    got = _run_varlen(d, 64)
    cu = inp["cu_seqlens"].tolist()
    for s in range(len(lengths)):
        a, e = cu[s], cu[s + 1]
        seq = {n: d[n][a:e].unsqueeze(0).clone() for n in ("q", "k", "v", "alpha", "beta", "d_o")}
        s0 = d["initial_state"][s:s + 1].clone()
        dsT = d["d_final_state"][s:s + 1].clone()
        o, sT, saved = gdn.gdn_fwd(seq["q"], seq["k"], seq["v"], seq["alpha"], seq["beta"], s0, saved=True)
        g = gdn.gdn_bwd(seq["q"], seq["k"], seq["v"], seq["alpha"], seq["beta"], s0, seq["d_o"], dsT,
                        saved=saved)
        torch.cuda.synchronize()
        pairs = [(got["o"][a:e], o[0]), (got["final_state"][s], sT[0]),
                 (got["d_initial_state"][s], g[5][0])]
        pairs += [(got[n][a:e], g[i][0]) for i, n in enumerate(GRADS)]
        for x, y in pairs:
            assert torch.equal(x, y), (s, float((x.float() - y.float()).abs().max()))


@pytest.mark.parametrize("dtype,K", [("bf16", 64), ("f32", 64), ("bf16", 128)])
def test_varlen_equal_lengths_bitwise_equal_to_dense(dtype, K):
    """S sequences of one length T are the dense [S, T] batch: both layouts then
    put the chunk boundaries where the dense batch has them, so every result is
    bit-identical."""
    S, T, H, V = 3, 130, 2, K
    w = custom(B=S, T=T, H=H, K=K, V=V, chunk=64, dtype=dtype, seed=42, init_std=0.2, dfinal_std=0.05)
    dense = {n: (t.cuda() if t is not None else None) for n, t in make_inputs(w).items()}
    o, sT, saved = gdn.gdn_fwd(dense["q"], dense["k"], dense["v"], dense["alpha"], dense["beta"],
                               dense["initial_state"], saved=True)
    g = gdn.gdn_bwd(dense["q"], dense["k"], dense["v"], dense["alpha"], dense["beta"], dense["initial_state"],
                    dense["d_o"], dense["d_final_state"], saved=saved)
    packed = {n: dense[n].reshape(S * T, *dense[n].shape[2:]) for n in ("q", "k", "v", "alpha", "beta", "d_o")}
    packed.update(initial_state=dense["initial_state"], d_final_state=dense["d_final_state"],
                  cu_seqlens=torch.arange(0, S * T + 1, T, dtype=torch.int32, device="cuda"))
    got = _run_varlen(packed, 64, max_len=T)
    assert torch.equal(got["o"], o.reshape(S * T, H, V))
    assert torch.equal(got["final_state"], sT)
    assert torch.equal(got["d_initial_state"], g[5])
    for i, n in enumerate(GRADS):
        assert torch.equal(got[n], g[i].reshape(got[n].shape)), n


def test_varlen_empty_batch_and_empty_sequences():
    """No tokens at all (and an empty sequence among others): outputs are empty,
    final state = initial state, and d_initial_state = d_final_state."""
    H, K, V = 2, 32, 32
    inp = make_varlen_inputs([0, 0], H, K, V, "f32", seed=43, init_std=0.5, dfinal_std=0.5)
    got = _run_varlen(_cuda(inp), 64, max_len=0)
    assert got["o"].shape == (0, H, V)
    assert torch.equal(got["final_state"].cpu(), inp["initial_state"])
    assert torch.equal(got["d_initial_state"].cpu(), inp["d_final_state"])
    # the tensor-core layout, with one empty sequence between two short ones
    H, K, V = 2, 128, 128
    inp = make_varlen_inputs([3, 0, 5], H, K, V, "bf16", seed=45, init_std=0.5, dfinal_std=0.5)
    got = _run_varlen(_cuda(inp), 64)
    assert torch.equal(got["final_state"][1].cpu(), inp["initial_state"][1])
    assert torch.equal(got["d_initial_state"][1].cpu(), inp["d_final_state"][1])
    inp = make_varlen_inputs([0, 0], H, K, V, "bf16", seed=46, init_std=0.5, dfinal_std=0.5)
    got = _run_varlen(_cuda(inp), 64, max_len=0)
    assert got["o"].shape == (0, H, V)
    assert torch.equal(got["final_state"].cpu(), inp["initial_state"])
    assert torch.equal(got["d_initial_state"].cpu(), inp["d_final_state"])


@pytest.mark.parametrize("cu,total,max_len", [
    ([0, 50, 40, 100], 100, 64),   # decreasing offsets
    ([0, 50, 100], 120, 64),       # the offsets do not reach total
    ([0, 10, 100], 100, 64),       # a sequence longer than max_len
    ([3, 50, 100], 100, 64),       # does not start at row 0
])
@pytest.mark.parametrize("dtype,K", [("f32", 32), ("bf16", 128)])
def test_varlen_invalid_offsets_are_flagged(cu, total, max_len, dtype, K):
    """An invalid cu_seqlens (read only on the device) sets the error bit; the
    kernels stay inside the buffers and the binding raises with check=True."""
    H, V = 2, K
    inp = make_varlen_inputs([total], H, K, V, dtype, seed=44)
    d = _cuda(inp)
    d["cu_seqlens"] = torch.tensor(cu, dtype=torch.int32, device="cuda")
    with pytest.raises(gdn.GdnError, match="cu_seqlens"):
        gdn.gdn_varlen_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["cu_seqlens"], max_len,
                           None, check=True)
    with pytest.raises(gdn.GdnError, match="cu_seqlens"):
        gdn.gdn_varlen_bwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["cu_seqlens"], max_len, None,
                           d["d_o"], None, check=True)
    # the context is still usable: a valid call afterwards succeeds
    d["cu_seqlens"] = torch.tensor([0, total], dtype=torch.int32, device="cuda")
    gdn.gdn_varlen_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["cu_seqlens"], None, None, check=True)
    torch.cuda.synchronize()


@pytest.mark.parametrize("dtype,K,chunk", [("bf16", 128, 64), ("f32", 32, 16)])
def test_reset_mask_matches_oracle(oracle_mod, dtype, K, chunk):
    """Streams with reset positions (the state is cleared just before a reset
    token; a reset at t = 0 discards the initial state) against the segment-wise
    float64 oracle.  Resets: adjacent, at t = 0, at a chunk boundary, at T - 1."""
    from oracle import resets
    from gdn_testutil import compare

    B, T, H = 3, 150, 2
    # slow decay: without a reset the state would carry across the reset points
    w = custom(B=B, T=T, H=H, K=K, V=K, chunk=chunk, dtype=dtype, seed=47, init_std=0.3, dfinal_std=0.05,
               alpha_lo=0.97)
    inp = make_inputs(w)
    reset = torch.zeros(B, T, dtype=torch.bool)
    for b, t in [(0, 1), (0, 2), (0, 64), (1, 0), (1, 100), (2, 70), (2, 149)]:
        reset[b, t] = True
    d = {n: (t.cuda() if t is not None else None) for n, t in inp.items()}
    ins = [d[n] for n in ("q", "k", "v", "alpha", "beta")]
    o, sT, saved, nseg = gdn.gdn_reset_fwd(*ins, reset.cuda(), d["initial_state"], chunk=chunk, saved=True,
                                           check=True)
    g = gdn.gdn_reset_bwd(*ins, reset.cuda(), d["initial_state"], d["d_o"], d["d_final_state"], chunk=chunk,
                          max_segments=nseg, saved=saved, check=True)
    torch.cuda.synchronize()
    assert nseg == B + 6
    got = dict(o=to_np(o), final_state=to_np(sT), **{n: to_np(x) for n, x in zip(GRADS + ("d_initial_state",), g)})
    npi = {n: to_np(inp[n]) for n in ("q", "k", "v", "alpha", "beta", "initial_state", "d_o", "d_final_state")}
    args = [npi[n] for n in ("q", "k", "v", "alpha", "beta")]
    ref_o, ref_sT = resets.fwd_resets(*args, reset.numpy(), npi["initial_state"])
    ref = dict(o=ref_o, final_state=ref_sT)
    ref.update(resets.bwd_resets(*args, reset.numpy(), npi["initial_state"], npi["d_o"], npi["d_final_state"]))
    compare(got, ref, dtype)
    assert np.all(got["d_initial_state"][1] == 0.0)  # row 1 was reset at t = 0


def _reset_case(dtype="bf16", K=128):
    B, T, H = 3, 150, 2
    w = custom(B=B, T=T, H=H, K=K, V=K, chunk=64, dtype=dtype, seed=48, init_std=0.3, dfinal_std=0.05,
               alpha_lo=0.97)
    d = {n: (t.cuda() if t is not None else None) for n, t in make_inputs(w).items()}
    reset = torch.zeros(B, T, dtype=torch.bool)
    for b, t in [(0, 5), (1, 0), (1, 64), (2, 149)]:
        reset[b, t] = True
    return d, reset.cuda()


def test_reset_loose_bound_gives_the_same_bits():
    """A bound above the true segment count (the mask has 3 + 3 segments) only
    adds empty segments: identical outputs and gradients, no host read."""
    d, reset = _reset_case()
    ins = [d[n] for n in ("q", "k", "v", "alpha", "beta")]
    out = []
    for bound in (6, 40):
        o, sT, sv, _ = gdn.gdn_reset_fwd(*ins, reset, d["initial_state"], max_segments=bound, saved=True,
                                         check=True)
        g = gdn.gdn_reset_bwd(*ins, reset, d["initial_state"], d["d_o"], d["d_final_state"], max_segments=bound,
                              saved=sv, check=True)
        out.append((o, sT) + tuple(g))
    torch.cuda.synchronize()
    for a, b in zip(*out):
        assert torch.equal(a, b)


def test_reset_too_small_bound_is_reported():
    """Fewer segments allowed than the mask has: the kernels flag it in the error
    word (and stay within the buffers); check=True raises, and the context stays
    usable."""
    d, reset = _reset_case()
    ins = [d[n] for n in ("q", "k", "v", "alpha", "beta")]
    with pytest.raises(gdn.GdnError, match="more segments than max_segments"):
        gdn.gdn_reset_fwd(*ins, reset, d["initial_state"], max_segments=4, check=True)
    gdn.gdn_reset_fwd(*ins, reset, d["initial_state"], max_segments=6, check=True)
    torch.cuda.synchronize()


def test_varlen_bench_workload_sampled(oracle_mod):
    """The packed batch the bench times (32768 tokens in 17 sequences of
    log-uniform lengths in [128, 8192], H=6, K=V=128, bf16), run whole in the
    bench's launch configuration; its longest, shortest and median sequences
    against the oracle."""
    from gated_delta_rule_19_gb300.inputs import VARLEN_WORKLOADS, varlen_lengths

    spec = VARLEN_WORKLOADS["varlen_bf16_T32768_H6_K128_V128"]
    lengths = varlen_lengths(spec["total"], spec["lo"], spec["hi"], spec["seed"])
    inp = make_varlen_inputs(lengths, spec["H"], spec["K"], spec["V"], spec["dtype"], seed=spec["seed"])
    got = _run_varlen(_cuda(inp), 64)
    tol = TOL["bf16"]
    cu = inp["cu_seqlens"].tolist()
    by_len = sorted(range(len(lengths)), key=lambda s: lengths[s])
    bad = []
    for s in (by_len[-1], by_len[0], by_len[len(by_len) // 2]):
        ref = _oracle_seq(oracle_mod, inp, s)
        a, e = cu[s], cu[s + 1]
        for n in ("o",) + GRADS:
            lim = tol["out" if n == "o" else "grad"]
            err = rel_l2(to_np(got[n][a:e]), ref[n])
            if err > lim:
                bad.append(f"seq {s} (len {e - a}) {n}: {err:.2e}")
            msg = local_failure(to_np(got[n][a:e]), ref[n], n, lim, 64, packed=True)
            if msg:
                bad.append(f"seq {s} {msg}")
        for n in ("final_state", "d_initial_state"):
            if got.get(n) is None:
                continue
            err = rel_l2(to_np(got[n][s]), ref[n])
            if err > tol["out" if n == "final_state" else "grad"]:
                bad.append(f"seq {s} {n}: {err:.2e}")
    assert not bad, "; ".join(bad)
