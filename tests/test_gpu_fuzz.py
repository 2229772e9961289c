"""Seeded random shapes against the float64 oracle: dense forward + backward,
packed variable-length batches, and the calls with the prologue folded in
(against the prologue oracle chained with the recurrence's).  Batch, heads,
length, K, V, chunk size, dtype, gate decay and the presence of initial /
final-state gradients are drawn from fixed generators, so that combinations the
hand-picked cases miss (a ragged tail with K != V, one head, a one-token stream,
slow decay with an initial state) are covered too; the cases are the same on
every run.  Tolerances and the per-block check are those of the other parity
tests."""
import numpy as np
import pytest
import torch

from gated_delta_rule_19_gb300.inputs import custom, make_inputs, make_varlen_inputs
from gdn_testutil import TOL, compare, gpu_run, local_failure, oracle_run, rel_l2, to_np
from test_gpu_raw import _gpu as _run_raw, _inputs as _raw_inputs, _oracle as _raw_oracle
from test_gpu_varlen import GRADS, _cuda, _oracle_seq, _run_varlen

pytestmark = pytest.mark.gpu

DIMS = (16, 32, 64, 128)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_19_gb300 import _build

    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _dense_cases(n=60, seed=2024):
    rng = np.random.RandomState(seed)
    cases = []
    for i in range(n):
        dtype = "bf16" if rng.rand() < 0.7 else "f32"
        chunk = 64 if (dtype == "bf16" and rng.rand() < 0.7) else int(rng.choice([16, 32, 64]))
        cases.append(dict(B=int(rng.randint(1, 4)), T=int(rng.choice([1, 2, 63, 64, 65]) if rng.rand() < 0.3
                                                           else rng.randint(1, 300)),
                          H=int(rng.randint(1, 5)), K=int(rng.choice(DIMS)), V=int(rng.choice(DIMS)),
                          chunk=chunk, dtype=dtype, seed=3000 + i,
                          init_std=float(rng.choice([0.0, 0.1])), dfinal_std=float(rng.choice([0.0, 0.01])),
                          alpha_lo=float(rng.choice([0.0, 0.97]))))
    return cases


def _large_cases(seed=31337):
    """Long streams with slow decay (the state carried across up to 47 chunks), and
    batches of up to 320 streams (more scan CTAs than one wave of SMs)."""
    rng = np.random.RandomState(seed)
    cases = []
    for i in range(12):
        dtype = "bf16" if rng.rand() < 0.8 else "f32"
        chunk = 64 if (dtype == "bf16" and rng.rand() < 0.8) else int(rng.choice([16, 32, 64]))
        cases.append(dict(B=int(rng.randint(1, 3)), T=int(rng.randint(700, 3000)), H=int(rng.randint(1, 3)),
                          K=int(rng.choice(DIMS)), V=int(rng.choice(DIMS)), chunk=chunk, dtype=dtype,
                          seed=110000 + i, init_std=float(rng.choice([0.0, 0.3])),
                          dfinal_std=float(rng.choice([0.0, 0.05])),
                          alpha_lo=float(rng.choice([0.0, 0.99, 0.999, 0.9999]))))
    for i in range(10):
        dtype = "bf16" if rng.rand() < 0.8 else "f32"
        chunk = 64 if (dtype == "bf16" and rng.rand() < 0.8) else int(rng.choice([16, 32, 64]))
        cases.append(dict(B=int(rng.randint(8, 20)), T=int(rng.randint(1, 200)), H=int(rng.randint(8, 17)),
                          K=int(rng.choice(DIMS)), V=int(rng.choice(DIMS)), chunk=chunk, dtype=dtype,
                          seed=120000 + i, init_std=float(rng.choice([0.0, 0.3])),
                          dfinal_std=float(rng.choice([0.0, 0.05])), alpha_lo=float(rng.choice([0.0, 0.97]))))
    return cases


def _varlen_cases(n=20, seed=4048):
    rng = np.random.RandomState(seed)
    cases = []
    for i in range(n):
        dtype = "bf16" if rng.rand() < 0.75 else "f32"
        chunk = 64 if dtype == "bf16" else int(rng.choice([16, 32, 64]))
        S = int(rng.randint(1, 7))
        lengths = [int(x) for x in rng.choice([0, 1, 63, 64, 65, 130, 200], S)] if rng.rand() < 0.4 \
            else [int(x) for x in rng.randint(0, 260, S)]
        cases.append(dict(lengths=lengths, H=int(rng.randint(1, 4)), K=int(rng.choice(DIMS)),
                          V=int(rng.choice(DIMS)), chunk=chunk, dtype=dtype, seed=5000 + i,
                          alpha_lo=float(rng.choice([0.0, 0.97]))))
    return cases


def _raw_cases(n=12, seed=6072):
    rng = np.random.RandomState(seed)
    cases = []
    for i in range(n):
        dtype = "bf16" if rng.rand() < 0.75 else "f32"
        chunk = 64 if (dtype == "bf16" and rng.rand() < 0.75) else int(rng.choice([16, 32, 64]))
        cases.append(dict(B=int(rng.randint(1, 3)), T=int(rng.randint(1, 300)), H=int(rng.randint(1, 4)),
                          K=int(rng.choice(DIMS)), V=int(rng.choice(DIMS)), C=chunk, dtype=dtype,
                          seed=7000 + 10 * i, slow=bool(rng.rand() < 0.5)))
    return cases


@pytest.fixture(scope="module")
def pro():
    from oracle import prologue

    return prologue


@pytest.mark.parametrize("case", _dense_cases() + _large_cases(), ids=lambda c: "B{B}_T{T}_H{H}_K{K}_V{V}_C{chunk}_{dtype}".format(**c))
def test_dense_random_shapes(oracle_mod, case):
    w = custom(**case)
    inp = make_inputs(w)
    got = gpu_run(w, inp, backward=True)
    ref = oracle_run(oracle_mod, inp, backward=True)
    compare(got, ref, w.dtype, chunk=w.chunk)


@pytest.mark.parametrize("case", _varlen_cases(), ids=lambda c: "S{}_H{H}_K{K}_V{V}_C{chunk}_{dtype}".format(
    len(c["lengths"]), **c))
def test_varlen_random_batches(oracle_mod, case):
    lengths, dtype, chunk = case["lengths"], case["dtype"], case["chunk"]
    inp = make_varlen_inputs(lengths, case["H"], case["K"], case["V"], dtype, seed=case["seed"], init_std=0.3,
                             dfinal_std=0.05, alpha_lo=case["alpha_lo"])
    got = _run_varlen(_cuda(inp), chunk)
    tol = TOL[dtype]
    cu = inp["cu_seqlens"].tolist()
    bad = []
    for s in range(len(lengths)):
        ref = _oracle_seq(oracle_mod, inp, s)
        a, e = cu[s], cu[s + 1]
        for n in ("final_state", "d_initial_state"):
            err = rel_l2(to_np(got[n][s]), ref[n])
            if err > tol["out" if n == "final_state" else "grad"]:
                bad.append(f"seq {s} {n}: {err:.2e}")
        if e - a >= 16:
            for n in ("o",) + GRADS:
                lim = tol["out" if n == "o" else "grad"]
                err = rel_l2(to_np(got[n][a:e]), ref[n])
                if err > lim:
                    bad.append(f"seq {s} {n}: {err:.2e}")
                msg = local_failure(to_np(got[n][a:e]), ref[n], n, lim, chunk, packed=True)
                if msg:
                    bad.append(f"seq {s} {msg}")
        elif e > a:  # too few elements for a relative norm: compare with an absolute bound
            for n in ("o",) + GRADS:
                diff = np.abs(to_np(got[n][a:e]) - ref[n]).max()
                scale = max(1.0, np.abs(ref[n]).max())
                if not diff <= 5 * tol["grad"] * scale:
                    bad.append(f"seq {s} {n}: max abs diff {diff:.2e}")
    assert not bad, "; ".join(bad)


@pytest.mark.parametrize("case", _raw_cases(), ids=lambda c: "B{B}_T{T}_H{H}_K{K}_V{V}_C{C}_{dtype}".format(**c))
def test_raw_random_shapes(oracle_mod, pro, case):
    c = dict(case)
    x, r = _raw_inputs(c["B"], c["T"], c["H"], c["K"], c["V"], c["C"], c["dtype"], seed=c["seed"], slow=c["slow"])
    got = {n: to_np(t) for n, t in _run_raw(x, r, c["C"]).items()}
    compare(got, _raw_oracle(oracle_mod, pro, x, r), c["dtype"], chunk=c["C"])
