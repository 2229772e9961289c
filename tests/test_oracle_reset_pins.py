"""Pins of the reset-position oracle (oracle/resets.py).

The reading: a reset at (b, t) clears the state just before token t.  In the
recurrence S_t = alpha_t S_{t-1}(I - beta_t k_t k_t^T) + beta_t v_t k_t^T that is
the same as alpha_t = 0 at t (the old state is multiplied by zero), so the
segment-wise oracle is checked against one plain token-recurrence run with
alpha_t set to 0 at every reset: outputs, final states and every gradient except
d alpha at the reset positions must agree (there the segment-wise run gives the
gradient of an alpha that multiplies a zero state, i.e. 0).  Central finite
differences pin the backward independently."""
import numpy as np
import pytest

from oracle import resets


def _case(B, T, H, K, V, seed, reset_at):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    alpha = rng.uniform(0.4, 1.0, (B, T, H))
    beta = rng.uniform(0.1, 1.0, (B, T, H))
    s0 = rng.standard_normal((B, H, V, K))
    do = rng.standard_normal((B, T, H, V))
    dsT = rng.standard_normal((B, H, V, K))
    reset = np.zeros((B, T), dtype=bool)
    for b, t in reset_at:
        reset[b, t] = True
    return q, k, v, alpha, beta, reset, s0, do, dsT


RESETS = [(0, 3), (0, 4), (1, 0), (1, 7), (2, 8)]  # adjacent resets, one at t = 0, one at T - 1


def test_reset_equals_zero_gate(oracle_mod):
    q, k, v, alpha, beta, reset, s0, do, dsT = _case(3, 9, 2, 4, 3, 11, RESETS)
    o, sT = resets.fwd_resets(q, k, v, alpha, beta, reset, s0)
    a0 = alpha.copy()
    a0[reset] = 0.0
    o_ref, sT_ref = oracle_mod.gated_delta_fwd(q, k, v, a0, beta, s0)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sT, sT_ref, rtol=1e-12, atol=1e-12)
    g = resets.bwd_resets(q, k, v, alpha, beta, reset, s0, do, dsT)
    g_ref = oracle_mod.gated_delta_bwd(q, k, v, a0, beta, s0, do, dsT)
    for n in ("dq", "dk", "dv", "dbeta", "d_initial_state"):
        np.testing.assert_allclose(g[n], g_ref[n], rtol=1e-11, atol=1e-11, err_msg=n)
    keep = ~reset
    np.testing.assert_allclose(g["dalpha"][keep], g_ref["dalpha"][keep], rtol=1e-11, atol=1e-11)
    assert np.all(g["dalpha"][reset] == 0.0)
    # a reset at t = 0 cuts the row off its initial state
    assert np.all(g["d_initial_state"][1] == 0.0)


def test_no_resets_is_the_plain_recurrence(oracle_mod):
    q, k, v, alpha, beta, reset, s0, do, dsT = _case(2, 6, 1, 3, 2, 12, [])
    o, sT = resets.fwd_resets(q, k, v, alpha, beta, reset, s0)
    o_ref, sT_ref = oracle_mod.gated_delta_fwd(q, k, v, alpha, beta, s0)
    np.testing.assert_array_equal(o, o_ref)
    np.testing.assert_array_equal(sT, sT_ref)


def test_segments():
    assert resets.segments(np.array([0, 0, 1, 1, 0, 1], dtype=bool)) == [(0, 2), (2, 3), (3, 5), (5, 6)]
    assert resets.segments(np.array([1, 0], dtype=bool)) == [(0, 2)]
    assert resets.segments(np.zeros(0, dtype=bool)) == []


@pytest.mark.parametrize("name", ["q", "k", "v", "alpha", "beta", "s0"])
def test_reset_gradients_match_central_differences(oracle_mod, name):
    q, k, v, alpha, beta, reset, s0, do, dsT = _case(2, 6, 1, 3, 2, 13, [(0, 2), (1, 0), (1, 5)])
    inputs = dict(q=q, k=k, v=v, alpha=alpha, beta=beta, s0=s0)
    g = resets.bwd_resets(q, k, v, alpha, beta, reset, s0, do, dsT)
    gname = dict(q="dq", k="dk", v="dv", alpha="dalpha", beta="dbeta", s0="d_initial_state")[name]

    def loss(args):
        o, sT = resets.fwd_resets(args["q"], args["k"], args["v"], args["alpha"], args["beta"], reset, args["s0"])
        return float((o * do).sum() + (sT * dsT).sum())

    arr = inputs[name]
    fd = np.zeros_like(arr)
    h = 1e-6
    for idx in np.ndindex(arr.shape):
        args = {n: a.copy() for n, a in inputs.items()}
        args[name][idx] += h
        lp = loss(args)
        args[name][idx] -= 2 * h
        lm = loss(args)
        fd[idx] = (lp - lm) / (2 * h)
    err = np.abs(g[gname] - fd).max() / max(np.abs(fd).max(), 1e-30)
    assert err < 1e-7, err
