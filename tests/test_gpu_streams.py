"""Calls in flight at once on separate CUDA streams, each with its own workspace,
saved buffer and outputs, give the same bits as the same calls made one after
another: the library keeps no state between calls outside the caller's buffers
(the persistent kernels' work counters and the error word live in each call's
workspace).  Covers the tensor-core path (dense, K = V = 128 with a ragged tail;
K = V = 64) and the CUDA-core path side by side, forward and backward."""
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


CASES = [
    custom(B=2, T=1000, H=3, K=128, V=128, chunk=64, dtype="bf16", seed=41, init_std=0.1, dfinal_std=0.01),
    custom(B=1, T=2048, H=4, K=64, V=64, chunk=64, dtype="bf16", seed=42, init_std=0.1, dfinal_std=0.01),
    custom(B=1, T=300, H=2, K=64, V=32, chunk=32, dtype="f32", seed=43, init_std=0.1, dfinal_std=0.01),
]


class _Call:
    """One forward + backward with every buffer allocated up front."""

    def __init__(self, w):
        d = {n: (t.cuda() if t is not None else None) for n, t in make_inputs(w).items()}
        self.d = d
        self.w = w
        # the tensor-core path keeps an error word at the start of its workspaces
        self.tc = w.dtype == "bf16" and w.chunk == 64
        dt = d["q"].dtype
        p = gdn.make_problem(w.B, w.T, w.H, w.K, w.V, w.chunk, dt)
        dev = d["q"].device
        self.args = (d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["initial_state"])
        self.o = torch.empty_like(d["v"])
        self.s_t = torch.empty((w.B, w.H, w.V, w.K), dtype=torch.float32, device=dev)
        self.saved = torch.empty(max(gdn.gdn_saved_bytes(p), 1), dtype=torch.uint8, device=dev)
        self.wsf = torch.empty(max(gdn.gdn_fwd_workspace_bytes(p), 1), dtype=torch.uint8, device=dev)
        self.wsb = torch.empty(max(gdn.gdn_bwd_workspace_bytes(p), 1), dtype=torch.uint8, device=dev)
        self.grads = tuple(torch.empty_like(d[n]) for n in ("q", "k", "v", "alpha", "beta"))
        self.ds0 = torch.empty_like(self.s_t)

    def launch(self, stream):
        w, d = self.w, self.d
        gdn.gdn_fwd(*self.args, chunk=w.chunk, o=self.o, final_state=self.s_t, saved=self.saved,
                    workspace=self.wsf, stream=stream)
        gdn.gdn_bwd(*self.args, d["d_o"], d["d_final_state"], saved=self.saved, chunk=w.chunk,
                    grads=self.grads, d_initial_state=self.ds0, workspace=self.wsb, stream=stream)

    def results(self):
        return [x.clone() for x in (self.o, self.s_t) + self.grads + (self.ds0,)]

    def error_words(self):
        if not self.tc:
            return [0, 0]
        return [int(ws[:4].view(torch.int32).item()) for ws in (self.wsf, self.wsb)]


def test_concurrent_streams_bitwise():
    calls = [_Call(w) for w in CASES]
    cur = torch.cuda.current_stream()
    refs = []
    for c in calls:  # one after another on the current stream
        c.launch(cur)
        torch.cuda.synchronize()
        refs.append(c.results())
        assert c.error_words() == [0, 0]
    streams = [torch.cuda.Stream() for _ in calls]
    for rep in range(3):
        for c in calls:  # outputs and workspaces dirtied between repetitions
            for t in (c.o, c.s_t, c.ds0) + c.grads:
                t.fill_(float("nan"))
            c.wsf.fill_(0x5A)
            c.wsb.fill_(0xA5)
        torch.cuda.synchronize()
        for c, s in zip(calls, streams):  # all in flight together
            c.launch(s)
        torch.cuda.synchronize()
        for i, (c, ref) in enumerate(zip(calls, refs)):
            got = c.results()
            for j, (a, b) in enumerate(zip(ref, got)):
                assert torch.equal(a, b), f"repetition {rep}, case {i}: output {j} differs"
            assert c.error_words() == [0, 0]
