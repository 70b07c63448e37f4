"""Pins for oracle.schedule.schedule_prefix (Algorithm 1): brute force over
every allocation on tiny instances, the mediant closed form, extreme
confidences, and a non-concave SPS table where the literal early stop and the
global optimum differ."""
import itertools
from fractions import Fraction

import numpy as np

from oracle import schedule


def _sps(B, gamma, alpha=20.0, beta=0.05):
    N = np.arange(B * (gamma + 1) + 1, dtype=np.float64)
    return N / (alpha + beta * N)


def _survival(c):
    return np.cumprod(np.asarray(c, np.float32), axis=1, dtype=np.float32)


def test_greedy_stop_is_global_optimum_for_rational_sps():
    # For SPS(N) = N / (alpha + beta N), Theta = E / (alpha + beta N): the mediant of
    # Theta and a / beta, so Theta rises then falls along the sorted scan and the first
    # drop is the best allocation over all (gamma + 1)^B choices of prefix lengths.
    rng = np.random.default_rng(0)
    checked = 0
    for trial in range(3000):
        B = int(rng.integers(1, 4))
        G = int(rng.integers(1, 4))
        alpha = float(rng.choice([0.5, 2.0, 20.0]))
        beta = float(rng.choice([0.05, 0.3, 1.0]))
        c = rng.uniform(0.05, 1.0, (B, G))
        a = _survival(c)
        sps = _sps(B, G, alpha, beta)
        ell, n, theta = schedule.schedule_prefix(a, sps)
        best, best_alloc, second = -1.0, None, -1.0
        for alloc in itertools.product(range(G + 1), repeat=B):
            E = B + sum(float(a[b, :alloc[b]].astype(np.float64).sum()) for b in range(B))
            N = B + sum(alloc)
            th = E / N * sps[N]
            if th > best:
                best, best_alloc, second = th, alloc, best
            elif th > second:
                second = th
        assert abs(theta - best) <= 1e-12 * best
        assert n == B + int(ell.sum())
        if best - second > 1e-9 * best:
            assert tuple(ell) == best_alloc
            checked += 1
    assert checked > 2500


def test_mediant_rule_closed_form():
    # accept the next sorted pair iff a > beta * Theta_current (exact rationals)
    rng = np.random.default_rng(1)
    alpha, beta = 20.0, 0.05
    for trial in range(200):
        B, G = int(rng.integers(1, 40)), int(rng.integers(1, 17))
        q = rng.uniform(0.3, 0.999, B)
        a = _survival(np.repeat(q[:, None], G, axis=1))
        sps = _sps(B, G, alpha, beta)
        ell, n, _ = schedule.schedule_prefix(a, sps)
        vals = sorted(((-float(a[b, j]), b, j) for b in range(B) for j in range(G)))
        E, N, taken = Fraction(B), B, np.zeros(B, int)
        for negv, b, j in vals:
            v = Fraction(-negv)
            if v * (Fraction(alpha) + Fraction(beta) * N) > Fraction(beta) * E:
                E += v
                N += 1
                taken[b] += 1
            else:
                break
        assert np.array_equal(ell, taken)


def test_extremes():
    B, G = 5, 7
    sps = _sps(B, G)
    ell, n, theta = schedule.schedule_prefix(np.ones((B, G), np.float32), sps)
    assert np.all(ell == G) and n == B * (G + 1)
    ell, n, theta = schedule.schedule_prefix(_survival(np.full((B, G), 1e-6)), sps)
    assert np.all(ell == 0) and n == B and theta == sps[B]


def test_literal_break_on_non_concave_sps():
    # Theta dips at N = B + 1 and rises after: Algorithm 1 stops at the first drop
    B, G = 2, 2
    a = np.full((B, G), 0.9, np.float32)
    sps = np.array([0.0, 1.0, 1.0, 0.5, 5.0, 5.0, 5.0])
    ell, n, theta = schedule.schedule_prefix(a, sps)
    assert list(ell) == [0, 0] and n == 2 and theta == 1.0
    # the best allocation is elsewhere
    E4 = 2 + 2 * float(np.float32(0.9))
    assert E4 / 4 * sps[4] > theta


def test_tie_break_lower_request_then_position():
    B, G = 3, 2
    a = np.array([[0.5, 0.5], [0.5, 0.5], [0.5, 0.5]], np.float32)
    # with beta tuned so exactly three pairs fit, the first three in (b, j) order win
    sps = np.zeros(B * (G + 1) + 1)
    sps[3:] = [1.0, 1.2, 1.4, 1.6, 1.0, 0.5, 0.5]
    ell, n, _ = schedule.schedule_prefix(a, sps)
    assert list(ell) == [2, 1, 0] and n == 6


def test_equal_theta_stops_the_scan():
    # "Theta > Theta_best" is strict: an exactly equal Theta ends the scan
    a = np.array([[1.0, 1.0]], np.float32)
    ell, n, theta = schedule.schedule_prefix(a, np.array([0.0, 1.0, 1.0, 2.0]))
    assert list(ell) == [0] and n == 1 and theta == 1.0
    ell, n, theta = schedule.schedule_prefix(a, np.array([0.0, 1.0, 1.0 + 2 ** -40, 2.0]))
    assert list(ell) == [2] and n == 3 and theta == 2.0
