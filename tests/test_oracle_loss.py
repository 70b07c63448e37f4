"""Pins of the joint-loss oracle (DeepSpec walkthrough section 7.2): central
finite differences of the loss against its gradient, closed forms, the
identity 1/2 ||p_d - p_t||_1 = 1 - sum min(p_d, p_t), invariances."""
import numpy as np
import pytest

from oracle import loss as L


def _rows(R=3, V=37, seed=0):
    rng = np.random.default_rng(seed)
    d = rng.normal(0, 1.5, (R, V))
    t = d + rng.normal(0, 1.0, (R, V))
    target = rng.integers(0, V, R)
    s = rng.normal(0, 1.0, R)
    omega = rng.uniform(0.2, 1.0, R)
    return d, t, target, s, omega


def test_position_weights():
    w = L.position_weights(np.array([1, 2, 5, 16]))
    assert w[0] == 1.0
    assert np.isclose(w[2], np.exp(-1.0))
    assert np.isclose(w[1] / w[0], np.exp(-0.25)) and np.isclose(w[3], np.exp(-15 / 4))


def test_grad_d_matches_central_differences():
    # the confidence term's c* is a target (no gradient through it): difference
    # the CE + L1 part only
    d, t, target, s, omega = _rows()
    kw = dict(alpha_ce=0.3, alpha_l1=0.7, alpha_conf=0.0)
    g, _ = L.dspark_loss_grad(d, t, target, s, omega, **kw)
    h = 1e-6
    num = np.zeros_like(d)
    for r in range(d.shape[0]):
        for v in range(d.shape[1]):
            dp, dm = d.copy(), d.copy()
            dp[r, v] += h
            dm[r, v] -= h
            num[r, v] = (L.dspark_loss(dp, t, target, s, omega, **kw)["loss"]
                         - L.dspark_loss(dm, t, target, s, omega, **kw)["loss"]) / (2 * h)
    assert np.max(np.abs(num - g)) < 1e-7


def test_grad_s_matches_central_differences():
    d, t, target, s, omega = _rows(seed=1)
    _, gs = L.dspark_loss_grad(d, t, target, s, omega)
    h = 1e-6
    for r in range(len(s)):
        sp, sm = s.copy(), s.copy()
        sp[r] += h
        sm[r] -= h
        num = (L.dspark_loss(d, t, target, sp, omega)["loss"] - L.dspark_loss(d, t, target, sm, omega)["loss"]) / (2 * h)
        assert abs(num - gs[r]) < 1e-8


def test_closed_forms():
    V = 50
    d = np.zeros((2, V))
    t = np.zeros((2, V))
    t[1, 3] = np.log(V + 1.0)                      # p_t(3) = (V+1)/(2V), the others 1/(2V)
    out = L.dspark_loss(d, t, np.array([0, 0]), np.zeros(2), np.ones(2))
    assert np.isclose(out["ce"][0], np.log(V))    # uniform logits
    assert out["c_star"][0] == 1.0 and out["l1"][0] == 0.0
    # p_d uniform 1/V, p_t: token 3 has (V+1)/(2V), the others 1/(2V)
    assert np.isclose(out["c_star"][1], 1.0 / V + (V - 1) / (2 * V))
    assert np.allclose(out["bce"], np.log(2.0))   # s = 0: softplus(0) - c* 0
    g, gs = L.dspark_loss_grad(d, t, np.array([0, 0]), np.zeros(2), np.ones(2))
    assert np.allclose(gs, L.ALPHA_CONF * (0.5 - out["c_star"]))


def test_l1_equals_one_minus_c_star_and_shift_invariance():
    d, t, target, s, omega = _rows(R=4, V=91, seed=2)
    out = L.dspark_loss(d, t, target, s, omega)
    assert np.allclose(out["l1"], 1.0 - out["c_star"], atol=1e-13)
    g, _ = L.dspark_loss_grad(d, t, target, s, omega)
    assert np.allclose(g.sum(axis=1), 0.0, atol=1e-15 * d.shape[1] + 1e-14)   # softmax gradients sum to 0
    out2 = L.dspark_loss(d + 3.0, t - 1.0, target, s, omega)
    assert np.allclose(out2["row"], out["row"], atol=1e-12)


def test_identical_rows_have_no_l1_gradient():
    d, _, target, s, omega = _rows(R=2, V=20, seed=3)
    g, _ = L.dspark_loss_grad(d, d.copy(), target, s, omega, alpha_ce=0.0, alpha_l1=1.0, alpha_conf=0.0)
    assert np.all(g == 0.0)
