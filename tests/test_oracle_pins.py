"""Pins of the float64 oracle against what the pages and the mathematics fix.

None of these compare the oracle with itself: each checks a closed form, an
invariant, a hand-worked value, finite differences, or an independent chunkwise
restatement (numpy, tests/chunkwise_ref.py).  A plausible mistake in the oracle
(dropped term, wrong sign or index, transposed operand, decay applied after the
write, read before the write) fails at least one of them.
"""
import numpy as np
import pytest

import chunkwise_ref as cw

RNG = np.random.default_rng(1234)


def _rand_case(B=1, T=7, H=2, K=4, V=5, rng=None, unit_k=True, s0=True):
    rng = rng or np.random.default_rng(7)
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    alpha = rng.uniform(0.3, 1.0, (B, T, H))
    beta = rng.uniform(0.05, 1.0, (B, T, H))
    S0 = rng.standard_normal((B, H, V, K)) if s0 else None
    return q, k, v, alpha, beta, S0


# ---------------------------------------------------------------- closed forms

def test_null_update_keeps_state(oracle_mod):
    """beta=0, alpha=1 leaves the state unchanged: o_t = S0 q_t, final = S0."""
    q, k, v, alpha, beta, S0 = _rand_case(T=9)
    alpha[:] = 1.0
    beta[:] = 0.0
    o, sT = oracle_mod.gated_delta_fwd(q, k, v, alpha, beta, S0)
    np.testing.assert_allclose(sT, S0, rtol=0, atol=1e-14)
    exp = np.einsum("bhvk,bthk->bthv", S0, q)
    np.testing.assert_allclose(o, exp, rtol=1e-13, atol=1e-13)


def test_pure_decay(oracle_mod):
    """beta=0: S_t = (prod_{i<=t} alpha_i) S0, so o_t = (prod alpha) S0 q_t."""
    q, k, v, alpha, beta, S0 = _rand_case(T=11)
    beta[:] = 0.0
    o, sT = oracle_mod.gated_delta_fwd(q, k, v, alpha, beta, S0)
    cp = np.cumprod(alpha, axis=1)  # [B,T,H]
    exp_o = cp[..., None] * np.einsum("bhvk,bthk->bthv", S0, q)
    np.testing.assert_allclose(o, exp_o, rtol=1e-12, atol=1e-13)
    exp_s = cp[:, -1][..., None, None] * S0
    np.testing.assert_allclose(sT, exp_s, rtol=1e-12, atol=1e-13)


def test_exact_write_any_alpha(oracle_mod):
    """Unit k_t and beta_t=1 write v_t exactly along k_t for any alpha_t and any
    previous state: S_t k_t = v_t.  Reading with q_t = k_t returns v_t (read after
    the write; the decay is applied before the write)."""
    q, k, v, alpha, beta, S0 = _rand_case(T=13, K=6, V=3)
    beta[:] = 1.0
    o, _ = oracle_mod.gated_delta_fwd(k, k, v, alpha, beta, S0)
    np.testing.assert_allclose(o, v, rtol=1e-12, atol=1e-12)


def test_orthonormal_keys_store_every_value(oracle_mod):
    """alpha=1, beta=1 with orthonormal keys (T <= K): the final state maps every
    key to its value, S_T k_j = v_j for all j."""
    K, V, T = 16, 16, 16  # the tiny workload's head dims
    rng = np.random.default_rng(3)
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    k = Qm.T[:T][None, :, None, :]  # rows are orthonormal keys, [1,T,1,K]
    v = rng.standard_normal((1, T, 1, V))
    S0 = rng.standard_normal((1, 1, V, K))
    alpha = np.ones((1, T, 1))
    beta = np.ones((1, T, 1))
    _, sT = oracle_mod.gated_delta_fwd(k, k, v, alpha, beta, S0)
    got = np.einsum("vk,tk->tv", sT[0, 0], k[0, :, 0])
    np.testing.assert_allclose(got, v[0, :, 0], rtol=1e-12, atol=1e-12)


def test_householder_isometry(oracle_mod):
    """alpha=1, beta=2, unit k, v=0: each step is S <- S (I - 2 k k^T), an
    orthogonal reflection, so the Frobenius norm is preserved."""
    q, k, v, alpha, beta, S0 = _rand_case(T=10, K=5, V=4)
    alpha[:] = 1.0
    beta[:] = 2.0
    v[:] = 0.0
    for T in (1, 4, 10):
        _, sT = oracle_mod.gated_delta_fwd(q[:, :T], k[:, :T], v[:, :T], alpha[:, :T],
                                           beta[:, :T], S0)
        np.testing.assert_allclose(np.linalg.norm(sT, axis=(2, 3)),
                                   np.linalg.norm(S0, axis=(2, 3)), rtol=1e-13)
        # and it is not the identity map
        assert np.abs(sT - S0).max() > 1e-3


def test_linearity(oracle_mod):
    """o is linear in q; (o, S_T) is jointly linear in (v, S0)."""
    q, k, v, alpha, beta, S0 = _rand_case(T=8)
    q2 = RNG.standard_normal(q.shape)
    o1, _ = oracle_mod.gated_delta_fwd(q, k, v, alpha, beta, S0)
    o2, _ = oracle_mod.gated_delta_fwd(q2, k, v, alpha, beta, S0)
    o3, _ = oracle_mod.gated_delta_fwd(q + 2.5 * q2, k, v, alpha, beta, S0)
    np.testing.assert_allclose(o3, o1 + 2.5 * o2, rtol=1e-12, atol=1e-12)
    v2 = RNG.standard_normal(v.shape)
    S02 = RNG.standard_normal(S0.shape)
    oa, sa = oracle_mod.gated_delta_fwd(q, k, v, alpha, beta, S0)
    ob, sb = oracle_mod.gated_delta_fwd(q, k, v2, alpha, beta, S02)
    oc, sc = oracle_mod.gated_delta_fwd(q, k, 2 * v - 3 * v2, alpha, beta, 2 * S0 - 3 * S02)
    np.testing.assert_allclose(oc, 2 * oa - 3 * ob, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(sc, 2 * sa - 3 * sb, rtol=1e-11, atol=1e-11)


def test_zero_state_zero_values_gives_zero(oracle_mod):
    q, k, v, alpha, beta, _ = _rand_case(T=6, s0=False)
    o, sT = oracle_mod.gated_delta_fwd(q, k, 0 * v, alpha, beta, None)
    assert np.abs(o).max() == 0 and np.abs(sT).max() == 0


def test_empty_sequence(oracle_mod):
    q, k, v, alpha, beta, S0 = _rand_case(T=0)
    o, sT = oracle_mod.gated_delta_fwd(q, k, v, alpha, beta, S0)
    assert o.shape == (1, 0, 2, 5)
    np.testing.assert_array_equal(sT, S0)


# ------------------------------------------------------------ hand-worked value

def test_hand_worked_two_tokens(oracle_mod):
    """K=V=2, two tokens, worked by hand from the definition.

    S0 = [[1,0],[0,2]].
    t=1: k=[1,0], v=[3,4], q=[0,1], alpha=1/2, beta=1/2.
         S0 (I - k k^T/2) = [[1/2,0],[0,2]]; times alpha -> [[1/4,0],[0,1]];
         beta v k^T = [[3/2,0],[2,0]];  S1 = [[7/4,0],[2,1]];  o1 = S1 q = [0,1].
    t=2: k=[0.6,0.8], v=[1,-1], q=[1,1], alpha=1, beta=1.
         S1 k = [1.05, 2.0]; v - S1 k = [-0.05, -3];
         S2 = S1 + (v - S1 k) k^T = [[1.72,-0.04],[0.2,-1.4]];  o2 = S2 q = [1.68,-1.2].
    """
    S0 = np.array([[[[1.0, 0.0], [0.0, 2.0]]]])
    k = np.array([[[[1.0, 0.0]], [[0.6, 0.8]]]])
    v = np.array([[[[3.0, 4.0]], [[1.0, -1.0]]]])
    q = np.array([[[[0.0, 1.0]], [[1.0, 1.0]]]])
    alpha = np.array([[[0.5], [1.0]]])
    beta = np.array([[[0.5], [1.0]]])
    o, sT = oracle_mod.gated_delta_fwd(q, k, v, alpha, beta, S0)
    np.testing.assert_allclose(o[0, :, 0], [[0.0, 1.0], [1.68, -1.2]], atol=1e-14)
    np.testing.assert_allclose(sT[0, 0], [[1.72, -0.04], [0.2, -1.4]], atol=1e-14)


def test_hand_worked_gradients_one_token(oracle_mod):
    """One token, K=V=2, L = <do, o>, worked by hand from the chain rule.

    S0 = [[1,0],[0,2]], k=[1,0], v=[3,4], q=[1,1], alpha=1/2, beta=1/2, do=[1,2].
    S1 = [[7/4,0],[2,1]], o = [7/4, 3]; dS = do q^T = [[1,1],[2,2]].
    dq = S1^T do = [23/4, 2];  dv = beta dS k = [1/2, 1];
    dbeta = (dS k).(v - alpha S0 k) = [1,2].[5/2,4] = 21/2;
    dalpha = <dS, S0 (I - beta k k^T)> = <[[1,1],[2,2]], [[1/2,0],[0,2]]> = 9/2;
    dk = beta dS^T v - alpha beta (S0^T dS k + dS^T S0 k)
       = [11/2, 11/2] - 1/4 ([1,4] + [1,1]) = [5, 17/4];
    dS0 = alpha dS (I - beta k k^T) = [[1/4,1/2],[1/2,1]].
    """
    S0 = np.array([[[[1.0, 0.0], [0.0, 2.0]]]])
    k = np.array([[[[1.0, 0.0]]]])
    v = np.array([[[[3.0, 4.0]]]])
    q = np.array([[[[1.0, 1.0]]]])
    alpha = np.array([[[0.5]]])
    beta = np.array([[[0.5]]])
    do = np.array([[[[1.0, 2.0]]]])
    o, _ = oracle_mod.gated_delta_fwd(q, k, v, alpha, beta, S0)
    np.testing.assert_allclose(o[0, 0, 0], [1.75, 3.0], atol=1e-14)
    g = oracle_mod.gated_delta_bwd(q, k, v, alpha, beta, S0, do)
    np.testing.assert_allclose(g["dq"][0, 0, 0], [23 / 4, 2], atol=1e-14)
    np.testing.assert_allclose(g["dv"][0, 0, 0], [0.5, 1.0], atol=1e-14)
    np.testing.assert_allclose(g["dbeta"][0, 0, 0], 21 / 2, atol=1e-14)
    np.testing.assert_allclose(g["dalpha"][0, 0, 0], 9 / 2, atol=1e-14)
    np.testing.assert_allclose(g["dk"][0, 0, 0], [5.0, 17 / 4], atol=1e-14)
    np.testing.assert_allclose(g["d_initial_state"][0, 0], [[0.25, 0.5], [0.5, 1.0]],
                               atol=1e-14)


# ------------------------------------------------------------- streaming split

@pytest.mark.parametrize("split", [1, 17, 32, 45])
def test_streaming_split_equals_single_call(oracle_mod, split):
    """Passing final_state of one call as the next call's state equals one call
    ("OpenGDN", "Core operator reference": exact streaming continuation)."""
    q, k, v, alpha, beta, S0 = _rand_case(B=2, T=48, H=3, K=6, V=4)
    o, sT = oracle_mod.gated_delta_fwd(q, k, v, alpha, beta, S0)
    o1, s1 = oracle_mod.gated_delta_fwd(q[:, :split], k[:, :split], v[:, :split],
                                        alpha[:, :split], beta[:, :split], S0)
    o2, s2 = oracle_mod.gated_delta_fwd(q[:, split:], k[:, split:], v[:, split:],
                                        alpha[:, split:], beta[:, split:], s1)
    np.testing.assert_allclose(np.concatenate([o1, o2], 1), o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(s2, sT, rtol=0, atol=1e-13)


# ------------------------------------------- independent chunkwise restatement

@pytest.mark.parametrize("C", [16, 32, 64])
@pytest.mark.parametrize("T", [64, 100])
def test_chunkwise_forward_matches_token_oracle(oracle_mod, C, T):
    """Chunk size changes the result only by rounding ("Sparse Delta Memory",
    "What the layer computes": the chunked form equals the token loop)."""
    q, k, v, alpha, beta, S0 = _rand_case(B=2, T=T, H=2, K=16, V=8)
    o, sT = oracle_mod.gated_delta_fwd(q, k, v, alpha, beta, S0)
    oc, sc = cw.chunk_fwd(q, k, v, alpha, beta, S0, C=C)
    np.testing.assert_allclose(oc, o, rtol=0, atol=1e-11)
    np.testing.assert_allclose(sc, sT, rtol=0, atol=1e-11)


@pytest.mark.parametrize("C", [16, 32, 64])
@pytest.mark.parametrize("T", [64, 77])
def test_chunkwise_backward_matches_token_oracle(oracle_mod, C, T):
    q, k, v, alpha, beta, S0 = _rand_case(B=1, T=T, H=2, K=8, V=12)
    rng = np.random.default_rng(11)
    do = rng.standard_normal(v.shape)
    dsT = rng.standard_normal(S0.shape)
    g = oracle_mod.gated_delta_bwd(q, k, v, alpha, beta, S0, do, dsT, seg=13)
    gc = cw.chunk_bwd(q, k, v, alpha, beta, S0, do, dsT, C=C)
    for name in g:
        ref = g[name]
        err = np.abs(gc[name] - ref).max() / max(np.abs(ref).max(), 1e-30)
        assert err < 1e-10, (name, err)


# ------------------------------------------------------- finite differences

def _loss(oracle_mod, q, k, v, alpha, beta, S0, do, dsT):
    o, sT = oracle_mod.gated_delta_fwd(q, k, v, alpha, beta, S0)
    return float((o * do).sum() + (sT * dsT).sum())


@pytest.mark.parametrize("seg", [2, 64])
def test_gradients_match_central_differences(oracle_mod, seg):
    """Every gradient of the reverse recurrence against central finite
    differences of the forward, element by element, in float64."""
    q, k, v, alpha, beta, S0 = _rand_case(B=1, T=5, H=2, K=3, V=4, unit_k=False)
    rng = np.random.default_rng(5)
    do = rng.standard_normal(v.shape)
    dsT = rng.standard_normal(S0.shape)
    g = oracle_mod.gated_delta_bwd(q, k, v, alpha, beta, S0, do, dsT, seg=seg)
    inputs = dict(q=q, k=k, v=v, alpha=alpha, beta=beta, S0=S0)
    names = dict(q="dq", k="dk", v="dv", alpha="dalpha", beta="dbeta", S0="d_initial_state")
    h = 1e-6
    for name, arr in inputs.items():
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            args = {n: a.copy() for n, a in inputs.items()}
            args[name][idx] += h
            lp = _loss(oracle_mod, args["q"], args["k"], args["v"], args["alpha"],
                       args["beta"], args["S0"], do, dsT)
            args[name][idx] -= 2 * h
            lm = _loss(oracle_mod, args["q"], args["k"], args["v"], args["alpha"],
                       args["beta"], args["S0"], do, dsT)
            fd[idx] = (lp - lm) / (2 * h)
        got = g[names[name]]
        err = np.abs(got - fd).max() / max(np.abs(fd).max(), 1e-30)
        assert err < 1e-7, (name, err)


def test_backward_without_final_grad_and_state(oracle_mod):
    """NULL initial state and NULL d_final_state act as zeros."""
    q, k, v, alpha, beta, _ = _rand_case(T=9, s0=False)
    do = np.random.default_rng(2).standard_normal(v.shape)
    g1 = oracle_mod.gated_delta_bwd(q, k, v, alpha, beta, None, do, None)
    z = np.zeros((1, 2, 5, 4))
    g2 = oracle_mod.gated_delta_bwd(q, k, v, alpha, beta, z, do, z)
    for n in g1:
        np.testing.assert_array_equal(g1[n], g2[n])


# ------------------------------------------------------------ golden regression

def test_golden_regression(oracle_mod):
    """The oracle still reproduces the stored float64 values of two small seeded
    cases (tests/golden/oracle_small_cases.json, written by make_golden.py)."""
    import json
    import os

    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_small_cases.json")
    with open(path) as f:
        cases = json.load(f)["cases"]
    for name, c in cases.items():
        a = {n: np.array(d["data"]).reshape(d["shape"]) for n, d in c.items()}
        o, sT = oracle_mod.gated_delta_fwd(a["q"], a["k"], a["v"], a["alpha"], a["beta"],
                                           a["initial_state"])
        np.testing.assert_allclose(o, a["o"], rtol=1e-12, atol=1e-14, err_msg=name)
        np.testing.assert_allclose(sT, a["final_state"], rtol=1e-12, atol=1e-14)
        g = oracle_mod.gated_delta_bwd(a["q"], a["k"], a["v"], a["alpha"], a["beta"],
                                       a["initial_state"], a["d_o"], a["d_final_state"])
        for n in g:
            np.testing.assert_allclose(g[n], a[n], rtol=1e-12, atol=1e-13, err_msg=n)
