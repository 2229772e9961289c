"""GPU tests of failure detection.  gdn_count_nonfinite: the count equals torch's
on tensors with NaN and +-inf planted at known places (fp32 and bf16, sizes with
ragged tails), calls accumulate, n = 0 leaves the count alone, and a NaN in one
head's input to gdn_fwd shows up in that head's outputs only (the (b, h) streams
are independent).  Bounded waits: with the wait limit cut to a few nanoseconds
every tensor-core kernel of a forward and a backward call takes its error path,
the calls report it in their error words, and the next calls, at the default
limit, give the same bits as before (the context and the device stay usable)."""
import pytest
import torch

from gated_delta_rule_19_gb300 import gdn
from gated_delta_rule_19_gb300.inputs import custom, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_19_gb300 import _build

    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _count(t):
    c = gdn.gdn_count_nonfinite(t.contiguous())
    torch.cuda.synchronize()
    return int(c.item())


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("n", [1, 7, 8, 1000, 1 << 20, (1 << 20) + 3])
def test_counts_match_torch(dtype, n):
    g = torch.Generator().manual_seed(n)
    x = torch.randn(n, generator=g).to(dtype)
    idx = torch.randperm(n, generator=g)[: max(1, n // 97)]
    vals = torch.tensor([float("nan"), float("inf"), -float("inf")])
    x[idx] = vals[torch.arange(len(idx)) % 3].to(dtype)
    x = x.cuda()
    want = int((~torch.isfinite(x)).sum().item())
    assert want == len(idx)
    c = gdn.gdn_count_nonfinite(x)
    gdn.gdn_count_nonfinite(x, c)  # a second call adds to the same count
    torch.cuda.synchronize()
    assert int(c.item()) == 2 * want


def test_empty_tensor_leaves_the_count():
    c = torch.full((1,), 5, dtype=torch.int64, device="cuda")
    gdn.gdn_count_nonfinite(torch.empty(0, device="cuda"), c)
    torch.cuda.synchronize()
    assert int(c.item()) == 5


def test_nan_input_reaches_only_its_stream():
    w = custom(B=1, T=128, H=2, K=128, V=128, chunk=64, dtype="bf16", seed=3, init_std=0.1)
    d = {n: (t.cuda() if t is not None else None) for n, t in make_inputs(w).items()}

    def run():
        o, sT, _ = gdn.gdn_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["initial_state"],
                               chunk=w.chunk)
        return o, sT

    o, sT = run()
    assert _count(o) == 0 and _count(sT) == 0
    d["v"][0, 10, 1, 5] = float("nan")  # head 1, token 10
    o, sT = run()
    assert _count(o[:, :, 1]) > 0 and _count(sT[:, 1]) > 0
    assert _count(o[:, :, 0]) == 0 and _count(sT[:, 0]) == 0


def _step(w, d, wsf, wsb):
    args = (d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["initial_state"])
    o, s_t, saved = gdn.gdn_fwd(*args, chunk=w.chunk, saved=True, workspace=wsf)
    g = gdn.gdn_bwd(*args, d["d_o"], d["d_final_state"], saved=saved, chunk=w.chunk, workspace=wsb)
    torch.cuda.synchronize()
    words = [int(ws[:4].view(torch.int32).item()) for ws in (wsf, wsb)]
    return [o, s_t] + [x for x in g if x is not None], words


def test_bounded_waits_give_up_and_the_context_stays_usable():
    # 2 x 6 streams of 16 chunks: the scans, prep and both gradient kernels run
    w = custom(B=2, T=1000, H=6, K=128, V=128, chunk=64, dtype="bf16", seed=51, init_std=0.1,
               dfinal_std=0.01)
    d = {n: (t.cuda() if t is not None else None) for n, t in make_inputs(w).items()}
    p = gdn.make_problem(w.B, w.T, w.H, w.K, w.V, w.chunk, torch.bfloat16)
    wsf = torch.zeros(gdn.gdn_fwd_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    wsb = torch.zeros(gdn.gdn_bwd_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    ref, words = _step(w, d, wsf, wsb)
    assert words == [0, 0]
    try:
        gdn.gdn_test_set_wait_limit(2)  # 2 ns: the first wait that does not succeed at once gives up
        _, words = _step(w, d, wsf, wsb)
    finally:
        gdn.gdn_test_set_wait_limit(0)
    assert words[0] != 0 and words[1] != 0, words
    for _ in range(2):
        got, words = _step(w, d, wsf, wsb)
        assert words == [0, 0]
        for i, (a, b) in enumerate(zip(ref, got)):
            assert torch.equal(a, b), f"output {i} differs after the error path ran"
