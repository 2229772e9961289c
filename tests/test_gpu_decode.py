"""GPU parity of the recurrent decode step (gdn_decode) against the float64
oracle, which is the token recurrence itself ("OpenGDN", Core operator
reference: a stream continued through state=).  Tolerances as for gdn_fwd:
relative L2 1e-5 for fp32 inputs, 2e-2 for bf16 outputs and states."""
import numpy as np
import pytest
import torch

from gated_delta_rule_19_gb300 import gdn
from gated_delta_rule_19_gb300.inputs import DECODE_WORKLOADS, custom, make_inputs
from gdn_testutil import compare, oracle_run, sample_gpu, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_19_gb300 import _build

    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _decode(inp, calls=1):
    """Runs gdn_decode over the inputs' T tokens in `calls` equal calls."""
    d = {n: (t.cuda() if t is not None else None) for n, t in inp.items()}
    B, T, H, K = d["q"].shape
    V = d["v"].shape[-1]
    state = (d["initial_state"].clone() if d["initial_state"] is not None
             else torch.zeros(B, H, V, K, device="cuda"))
    L = T // calls
    outs = []
    for i in range(calls):
        sl = slice(i * L, (i + 1) * L)
        o, state = gdn.gdn_decode(*(d[n][:, sl].contiguous() for n in ("q", "k", "v", "alpha", "beta")),
                                  state)
        outs.append(o)
    torch.cuda.synchronize()
    return torch.cat(outs, 1), state


@pytest.mark.parametrize("B,T,H,K,V,dtype", [
    (2, 1, 3, 128, 128, "bf16"),
    (3, 5, 2, 64, 32, "f32"),
    (1, 3, 4, 16, 16, "f32"),
    (2, 16, 2, 32, 128, "bf16"),
    (1, 7, 1, 128, 64, "f32"),
    # more 8-row units (64 * 8 * 16 = 8192) than the persistent grid has warps
    (64, 2, 8, 128, 128, "bf16"),
    (40, 3, 9, 64, 64, "f32"),
])
def test_decode_matches_oracle(oracle_mod, B, T, H, K, V, dtype):
    w = custom(B=B, T=T, H=H, K=K, V=V, chunk=64, dtype=dtype, seed=900 + T + K, init_std=0.5)
    inp = make_inputs(w)
    o, state = _decode(inp)
    ref = oracle_run(oracle_mod, inp, backward=False)
    compare(dict(o=to_np(o), final_state=to_np(state)), ref, dtype)


def test_decode_token_calls_equal_one_call():
    """T calls of one token continue the stream exactly: bit-identical outputs
    and state to one call of T tokens (the state is kept in fp32 between calls)."""
    w = custom(B=2, T=12, H=3, K=128, V=128, chunk=64, dtype="bf16", seed=31, init_std=0.3)
    inp = make_inputs(w)
    o1, s1 = _decode(inp, calls=1)
    o12, s12 = _decode(inp, calls=12)
    assert torch.equal(o1, o12)
    assert torch.equal(s1, s12)


def test_decode_agrees_with_chunked_forward():
    """The decode step and the chunked forward compute the same recurrence."""
    w = custom(B=1, T=64, H=2, K=64, V=64, chunk=64, dtype="f32", seed=32, init_std=0.2)
    inp = make_inputs(w)
    o_dec, s_dec = _decode(inp)
    d = {n: (t.cuda() if t is not None else None) for n, t in inp.items()}
    o_fwd, s_fwd, _ = gdn.gdn_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["initial_state"],
                                  chunk=64)
    torch.cuda.synchronize()
    rel = lambda a, b: float((a - b).norm() / b.norm())
    assert rel(o_dec, o_fwd) < 1e-5
    assert rel(s_dec, s_fwd) < 1e-5


def test_decode_serving_batch_sampled(oracle_mod):
    """The decode workload (B=256 sequences, 16 heads, one token) on sampled heads."""
    w = DECODE_WORKLOADS["decode_bf16_B256_T1_H16_K128_V128"]
    inp = make_inputs(w)
    o, state = _decode(inp)
    streams = [(0, 0), (117, 5), (255, 15)]
    ref = oracle_run(oracle_mod, inp, backward=False, streams=streams)
    got = sample_gpu(dict(o=to_np(o), final_state=to_np(state)), streams)
    compare(got, ref, "bf16")


def test_decode_zero_tokens_keeps_state():
    q = torch.zeros(2, 0, 3, 32, device="cuda", dtype=torch.bfloat16)
    v = torch.zeros(2, 0, 3, 16, device="cuda", dtype=torch.bfloat16)
    g = torch.zeros(2, 0, 3, device="cuda", dtype=torch.bfloat16)
    s = torch.randn(2, 3, 16, 32, device="cuda")
    s_ref = s.clone()
    o, s2 = gdn.gdn_decode(q, q, v, g, g, s)
    torch.cuda.synchronize()
    assert o.shape == (2, 0, 3, 16) and torch.equal(s2, s_ref)
