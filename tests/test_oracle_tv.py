"""Pins for oracle.tv.accept_rate_tv (c* = 1 - 1/2 ||p_d - p_t||_1): values the
definition fixes, a two-point closed form, the min-sum identity by brute force,
and torch's own float64 softmax as an independent library routine."""
import numpy as np
import torch

from oracle import tv


def test_identical_rows_give_one():
    rng = np.random.default_rng(0)
    d = rng.normal(0, 2, (5, 300))
    assert np.allclose(tv.accept_rate_tv(d, d), 1.0, atol=1e-14)


def test_shift_invariance():
    rng = np.random.default_rng(1)
    d = rng.normal(0, 2, (5, 300))
    assert np.allclose(tv.accept_rate_tv(d, d + 3.7), 1.0, atol=1e-13)


def test_disjoint_supports_give_zero():
    V = 64
    d = np.full((1, V), -1e30)
    t = np.full((1, V), -1e30)
    d[0, : V // 2] = 0.0
    t[0, V // 2:] = 0.0
    assert tv.accept_rate_tv(d, t)[0] == 0.0


def test_symmetric_and_in_unit_interval():
    rng = np.random.default_rng(2)
    d = rng.normal(0, 3, (20, 50))
    t = rng.normal(0, 3, (20, 50))
    a, b = tv.accept_rate_tv(d, t), tv.accept_rate_tv(t, d)
    assert np.allclose(a, b, atol=1e-15)
    assert np.all((a >= 0) & (a <= 1))


def test_two_point_closed_form():
    rng = np.random.default_rng(3)
    d = rng.normal(0, 2, (100, 2))
    t = rng.normal(0, 2, (100, 2))
    sig = lambda x: 1.0 / (1.0 + np.exp(-x))
    expect = 1.0 - np.abs(sig(d[:, 1] - d[:, 0]) - sig(t[:, 1] - t[:, 0]))
    assert np.allclose(tv.accept_rate_tv(d, t), expect, atol=1e-14)


def test_min_sum_identity_brute_force():
    # sum_v min(p_v, q_v) = 1 - 1/2 sum |p - q|, with p, q built by explicit loops
    rng = np.random.default_rng(4)
    for V in (1, 3, 16):
        d = rng.normal(0, 2, V)
        t = rng.normal(0, 2, V)
        ed = [np.exp(x) for x in d]
        et = [np.exp(x) for x in t]
        p = [e / sum(ed) for e in ed]
        q = [e / sum(et) for e in et]
        expect = sum(min(pi, qi) for pi, qi in zip(p, q))
        assert abs(tv.accept_rate_tv(d[None], t[None])[0] - expect) < 1e-14


def test_against_torch_softmax_float64():
    rng = np.random.default_rng(5)
    d = rng.normal(0, 2, (8, 1000))
    t = d + rng.normal(0, 1, (8, 1000))
    pd = torch.softmax(torch.from_numpy(d), dim=-1)
    pt = torch.softmax(torch.from_numpy(t), dim=-1)
    expect = (1.0 - 0.5 * (pd - pt).abs().sum(-1)).numpy()
    assert np.allclose(tv.accept_rate_tv(d, t), expect, atol=1e-13)
