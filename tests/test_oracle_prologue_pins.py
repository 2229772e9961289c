"""Pins of the prologue oracle (oracle/prologue.py) against facts that do not
come from its own formulas: closed forms of the normalised length, the direction
it keeps, an independent logistic routine, exact values at zero, the identity
exp(-softplus(x)) + sigmoid(x) = 1, the normalisation's insensitivity to radial
changes, and central finite differences for every gradient."""
import numpy as np
import pytest
from scipy.special import expit

from oracle import prologue as pro


def _raw(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return rng.standard_normal(shape) * scale


def test_normalised_length_closed_form_and_direction():
    x = _raw((2, 5, 3, 16), 0, scale=0.7)
    q, k, _, _ = pro.prologue_fwd(x, 2 * x, np.zeros((2, 5, 3)), np.zeros((2, 5, 3)))
    s = (x * x).sum(-1)
    np.testing.assert_allclose((q * q).sum(-1), s / (s + pro.EPS), rtol=1e-13)
    # q keeps the direction of x: cosine 1
    cos = (q * x).sum(-1) / np.sqrt((q * q).sum(-1) * s)
    np.testing.assert_allclose(cos, 1.0, rtol=1e-13)
    # k_raw = 2 x: the same unit direction, the eps effect scaled down
    np.testing.assert_allclose(k, q, atol=2e-6)


def test_gates_match_an_independent_logistic():
    a = np.linspace(-40.0, 40.0, 801).reshape(1, 801, 1)
    _, _, alpha, beta = pro.prologue_fwd(np.ones((1, 801, 1, 4)), np.ones((1, 801, 1, 4)), a, a)
    np.testing.assert_allclose(alpha, expit(-a), rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(beta, expit(a), rtol=1e-12, atol=1e-300)
    # exp(-softplus(x)) + sigmoid(x) = 1
    np.testing.assert_allclose(alpha + beta, 1.0, rtol=1e-14)


def test_gates_exact_and_extreme_values():
    z = np.zeros((1, 1, 1))
    _, _, alpha, beta = pro.prologue_fwd(np.ones((1, 1, 1, 4)), np.ones((1, 1, 1, 4)), z, z)
    assert alpha.item() == 0.5 and beta.item() == 0.5
    big = np.array([[[800.0, -800.0]]])
    _, _, alpha, beta = pro.prologue_fwd(np.ones((1, 1, 2, 4)), np.ones((1, 1, 2, 4)), big, big)
    assert np.isfinite(alpha).all() and np.isfinite(beta).all()
    assert alpha[0, 0, 0] == 0.0 and alpha[0, 0, 1] == 1.0
    assert beta[0, 0, 0] == 1.0 and beta[0, 0, 1] == 0.0


def test_radial_gradient_vanishes():
    """An upstream gradient along q itself only changes the length, which the
    normalisation removes (up to the eps term)."""
    x = _raw((1, 3, 2, 32), 1, scale=3.0)
    q, _, _, _ = pro.prologue_fwd(x, x, np.zeros((1, 3, 2)), np.zeros((1, 3, 2)))
    dq_raw, _, _, _ = pro.prologue_bwd(x, x, np.zeros((1, 3, 2)), np.zeros((1, 3, 2)), q, np.zeros_like(q),
                                       np.zeros((1, 3, 2)), np.zeros((1, 3, 2)))
    assert np.abs(dq_raw).max() < 1e-6


@pytest.mark.parametrize("K", [4, 16])
def test_gradients_match_central_differences(K):
    shape = (2, 3, 2, K)
    qr, kr = _raw(shape, 2), _raw(shape, 3, scale=0.3)
    a, b = _raw(shape[:3], 4, 2.0), _raw(shape[:3], 5, 2.0)
    wq, wk = _raw(shape, 6), _raw(shape, 7)
    wa, wb = _raw(shape[:3], 8), _raw(shape[:3], 9)

    def loss(qr_, kr_, a_, b_):
        q, k, al, be = pro.prologue_fwd(qr_, kr_, a_, b_)
        return (q * wq).sum() + (k * wk).sum() + (al * wa).sum() + (be * wb).sum()

    got = pro.prologue_bwd(qr, kr, a, b, wq, wk, wa, wb)
    h = 1e-6
    for idx, x in enumerate((qr, kr, a, b)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            m = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[m] += h
            xm[m] -= h
            args_p = [qr, kr, a, b]
            args_m = [qr, kr, a, b]
            args_p[idx], args_m[idx] = xp, xm
            fd[m] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(got[idx], fd, rtol=1e-6, atol=1e-8)
