"""Pins for oracle.verify: losslessness (the emitted tokens follow the target
distribution) by chi-square over independent requests, the link between the
empirical acceptance rate and c* = sum_v min(p_d, p_t), and the degenerate
cases p_d = p_t and greedy agreement."""
import numpy as np
from scipy import stats

from oracle import draft, verify, tv


def _chi2_p(samples, probs):
    counts = np.bincount(samples, minlength=len(probs)).astype(float)
    expect = probs * counts.sum()
    keep = expect >= 5
    obs, exp = counts[keep], expect[keep]
    rest_o, rest_e = counts[~keep].sum(), expect[~keep].sum()
    if rest_e >= 5:
        obs, exp = np.append(obs, rest_o), np.append(exp, rest_e)
    else:
        obs[-1] += rest_o
        exp[-1] += rest_e
    return stats.chisquare(obs, exp).pvalue


def _softmax(x):
    e = np.exp(x - x.max())
    return e / e.sum()


def _round(R, V, G, r, T, seed, ell, t_noise=1.0, rng_seed=0):
    rng = np.random.default_rng(rng_seed)
    U1 = rng.normal(0, 1.5, (G, V))
    t1 = np.concatenate([U1, rng.normal(0, 1.5, (1, V))]) + rng.normal(0, t_noise, (G + 1, V))
    W1 = rng.normal(0, 0.5, (V, r))
    W2 = rng.normal(0, 0.5, (V, r))
    H = 2
    x0 = np.full(R, 3)
    U = np.broadcast_to(U1, (R, G, V))
    t = np.broadcast_to(t1, (R, G + 1, V))
    d = draft.draft_block(U, np.zeros((R, G, H)), W1, W2, np.zeros(H + r), 0.0, x0, T, seed)
    ell = np.full(R, ell)
    out = verify.verify(t, U, W1, W2, x0, d["x"], d["lse_d"], d["logp_d"], ell, T, seed)
    return U1, t1, W1, W2, d, out


def test_first_emitted_token_follows_target():
    R, V, G, r, T = 60000, 70, 3, 8, 1.0
    U1, t1, W1, W2, d, out = _round(R, V, G, r, T, seed=11, ell=G)
    first = np.where(out["n_accept"] >= 1, d["x"][:, 0], out["next_token"])
    pt1 = _softmax(t1[0] / T)
    assert _chi2_p(first, pt1) > 1e-3
    # the draft distribution alone is rejected by the same test
    z1 = U1[0] + W2 @ W1[3]
    assert _chi2_p(d["x"][:, 0], pt1) < 1e-6
    # acceptance rate at position 1 equals c*(z_1 / T, t_1 / T) = sum min(p_d, p_t)
    cstar = tv.accept_rate_tv((z1 / T)[None], (t1[0] / T)[None])[0]
    acc = np.mean(out["n_accept"] >= 1)
    assert abs(acc - cstar) < 4.5 * np.sqrt(cstar * (1 - cstar) / R)


def test_token_after_a_rejection_follows_the_residual():
    """Given a rejection at position 1, the emitted token follows the residual
    law norm(max(0, p_t - p_d)) of the rejection sampler, in closed form here."""
    R, V, G, r, T = 60000, 70, 3, 8, 1.0
    U1, t1, W1, W2, d, out = _round(R, V, G, r, T, seed=11, ell=G)
    rej = out["n_accept"] == 0
    p_t = _softmax(t1[0] / T)
    p_d = _softmax((U1[0] + W2 @ W1[3]) / T)
    q = np.maximum(0.0, p_t - p_d)
    assert rej.sum() > 5000
    assert _chi2_p(out["next_token"][rej], q / q.sum()) > 1e-3
    # the sample has the power to tell the residual from p_t itself
    assert _chi2_p(out["next_token"][rej], p_t) < 1e-6


def test_second_token_follows_target_given_first_accepted():
    R, V, G, r, T = 80000, 40, 3, 8, 0.9
    U1, t1, W1, W2, d, out = _round(R, V, G, r, T, seed=5, ell=G, rng_seed=1)
    acc1 = out["n_accept"] >= 1
    second = np.where(out["n_accept"] >= 2, d["x"][:, 1], out["next_token"])
    assert _chi2_p(second[acc1], _softmax(t1[1] / T)) > 1e-3


def test_bonus_token_when_nothing_is_scheduled():
    R, V, G, r, T = 50000, 50, 3, 8, 1.3
    U1, t1, W1, W2, d, out = _round(R, V, G, r, T, seed=9, ell=0, rng_seed=2)
    assert np.all(out["n_accept"] == 0)
    assert _chi2_p(out["next_token"], _softmax(t1[0] / T)) > 1e-3


def test_bonus_after_full_acceptance_is_from_row_after_prefix():
    R, V, G, r, T = 50000, 30, 2, 4, 1.0
    U1, t1, W1, W2, d, out = _round(R, V, G, r, T, seed=21, ell=1, rng_seed=3, t_noise=0.3)
    full = out["n_accept"] == 1
    assert np.all(out["n_accept"] <= 1)
    assert _chi2_p(out["next_token"][full], _softmax(t1[1] / T)) > 1e-3


def test_identical_distributions_accept_everything():
    rng = np.random.default_rng(4)
    R, V, G, r, H, T = 200, 90, 4, 8, 2, 0.7
    U = rng.normal(0, 2, (R, G, V))
    W1 = rng.normal(0, 0.5, (V, r))
    W2 = rng.normal(0, 0.5, (V, r))
    x0 = rng.integers(0, V, R)
    d = draft.draft_block(U, np.zeros((R, G, H)), W1, W2, np.zeros(H + r), 0.0, x0, T, seed=3)
    prev = np.concatenate([x0[:, None], d["x"][:, :-1]], axis=1)
    t = np.zeros((R, G + 1, V))
    for k in range(G):
        t[:, k] = U[:, k] + (W1[prev[:, k]] @ W2.T)
    t[:, G] = rng.normal(0, 1, (R, V))
    out = verify.verify(t, U, W1, W2, x0, d["x"], d["lse_d"], d["logp_d"], np.full(R, G), T, seed=3)
    assert np.all(out["n_accept"] == G)


def test_greedy_agreement_and_first_disagreement():
    rng = np.random.default_rng(5)
    R, V, G, r, H = 100, 60, 5, 4, 2
    U = rng.normal(0, 2, (R, G, V))
    W1 = rng.normal(0, 0.5, (V, r))
    W2 = rng.normal(0, 0.5, (V, r))
    x0 = rng.integers(0, V, R)
    d = draft.draft_block(U, np.zeros((R, G, H)), W1, W2, np.zeros(H + r), 0.0, x0, 0.0, seed=1)
    t = rng.normal(0, 1, (R, G + 1, V))
    cut = rng.integers(0, G + 1, R)        # rows before `cut` agree with the draft
    for b in range(R):
        for k in range(cut[b]):
            t[b, k, d["x"][b, k]] = 100.0
        if cut[b] < G:
            t[b, cut[b], d["x"][b, cut[b]]] = -100.0
    ell = rng.integers(0, G + 1, R)
    out = verify.verify(t, U, W1, W2, x0, d["x"], d["lse_d"], d["logp_d"], ell, 0.0, seed=1)
    assert np.array_equal(out["n_accept"], np.minimum(cut, ell))
    stop = np.minimum(cut, ell)
    assert np.array_equal(out["next_token"], np.argmax(t[np.arange(R), stop], axis=-1))


def test_rejection_with_an_empty_residual_draws_from_the_target():
    """Reading 7: a residual with no mass falls back to a draw from p_t.  With the
    target row equal to the draft logits (p_t = p_d) and the caller's logp_d
    raised by 1, every test accepts with probability 1/e, and each rejected row's
    residual max(0, p_t - p_d) is zero everywhere."""
    rng = np.random.default_rng(8)
    R, V, G, r, H, T = 40000, 24, 1, 4, 2, 1.0
    U1 = rng.normal(0, 1.0, (G, V))
    W1 = rng.normal(0, 0.5, (V, r))
    W2 = rng.normal(0, 0.5, (V, r))
    x0 = np.full(R, 5)
    U = np.broadcast_to(U1, (R, G, V))
    d = draft.draft_block(U, np.zeros((R, G, H)), W1, W2, np.zeros(H + r), 0.0, x0, T, seed=13)
    # the target row is the draft's own logits, rebuilt as verification rebuilds them,
    # so p_t and p_d agree bit for bit and the residual is exactly empty
    z1 = verify.draft_logits(U, W1, W2, x0, d["x"], np.arange(1), np.ones(1, int))[0]
    from oracle.sampling import logsumexp
    p_d = np.exp(z1 / T - d["lse_d"][0, 0])
    p_t = np.exp(z1 / T - logsumexp((z1 / T)[None], axis=-1)[0])   # as verification forms p_t
    assert np.all(np.maximum(0.0, p_t - p_d) == 0.0)
    t = np.empty((R, G + 1, V))
    t[:, 0] = z1
    t[:, 1] = rng.normal(0, 1.0, V)
    out = verify.verify(t, U, W1, W2, x0, d["x"], d["lse_d"], d["logp_d"] + 1.0, np.full(R, G), T, seed=13)
    rej = out["n_accept"] == 0
    assert abs(1.0 - rej.mean() - np.exp(-1.0)) < 4.5 * np.sqrt(np.exp(-1.0) * (1 - np.exp(-1.0)) / R)
    assert _chi2_p(out["next_token"][rej], _softmax(z1 / T)) > 1e-3
