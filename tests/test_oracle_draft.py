"""Pins for oracle.sampling and oracle.draft: distribution tests of the
Gumbel-max sampler and a brute-force restatement of it, closed forms of the Markov bias / confidence head /
survival product built from structured weights, and a deterministic chain that
shows the bias of step k uses x_{k-1}."""
import numpy as np
from scipy import stats

from oracle import sampling, draft, philox


def _chi2_p(samples, probs):
    counts = np.bincount(samples, minlength=len(probs)).astype(float)
    n = counts.sum()
    expect = probs * n
    keep = expect >= 5
    obs, exp = counts[keep], expect[keep]
    # pool the sparse bins into one bin (or into the last kept bin if still sparse)
    rest_o, rest_e = counts[~keep].sum(), expect[~keep].sum()
    if rest_e >= 5:
        obs, exp = np.append(obs, rest_o), np.append(exp, rest_e)
    else:
        obs[-1] += rest_o
        exp[-1] += rest_e
    return stats.chisquare(obs, exp).pvalue


def test_gumbel_max_matches_softmax():
    # a ragged vocabulary (not a multiple of the 4 words of a Philox block) with
    # zero-weight entries
    rng = np.random.default_rng(10)
    V = 150
    logw = rng.normal(0, 1.5, V)
    logw[[3, 70, 149]] = -np.inf
    R = 100000
    tok, _ = sampling.gumbel_max(np.broadcast_to(logw, (R, V)), 123, np.arange(R), 1, philox.STREAM_DRAFT_TOKEN)
    p = np.exp(logw - logw[np.isfinite(logw)].max())
    p /= p.sum()
    assert np.all(np.isfinite(logw[tok]))
    assert _chi2_p(tok, p) > 1e-3


def test_gumbel_max_detects_a_wrong_law():
    # sanity of the test itself: the same draws do not fit a tempered law
    rng = np.random.default_rng(11)
    V = 150
    logw = rng.normal(0, 1.5, V)
    R = 100000
    tok, _ = sampling.gumbel_max(np.broadcast_to(logw, (R, V)), 5, np.arange(R), 2, philox.STREAM_DRAFT_TOKEN)
    p_wrong = np.exp(0.8 * (logw - logw.max()))
    p_wrong /= p_wrong.sum()
    assert _chi2_p(tok, p_wrong) < 1e-6


def test_gumbel_max_single_finite_entry_and_dead_row():
    V = 200
    logw = np.full((2, V), -np.inf)
    logw[0, 131] = 0.0
    tok, _ = sampling.gumbel_max(logw, 1, np.arange(2), 1, philox.STREAM_VERIFY_TOKEN)
    assert tok[0] == 131 and tok[1] == -1


def test_gumbel_max_is_the_literal_definition():
    """Brute force, one scalar at a time with Python's own math.log: for every
    index v, the word (v & 3) of Philox(seed; (v >> 2, k, b, stream)), the uniform
    ((w >> 9) + 1/2) 2^-23, the Gumbel -ln(-ln u), then the first maximum of
    lw_v + G.  The vectorised sampler must give the same tokens and margins."""
    import math
    rng = np.random.default_rng(12)
    seed, k, stream = 0xDEADBEEF12345678, 3, philox.STREAM_DRAFT_TOKEN
    R, V = 6, 37
    logw = rng.normal(0, 2.0, (R, V))
    logw[2, :] = 0.0                      # only the noise decides
    logw[4, 5] = -np.inf
    b = np.array([0, 1, 7, 1000, 65535, 3])
    tok, mar = sampling.gumbel_max(logw, seed, b, k, stream)
    for i in range(R):
        best, second, arg = -math.inf, -math.inf, -1
        for v in range(V):
            words = philox.philox4x32_10(v >> 2, k, int(b[i]), stream, seed & 0xFFFFFFFF, seed >> 32)
            w = int(words[v & 3])
            u = ((w >> 9) + 0.5) * 2.0 ** -23
            score = float(logw[i, v]) - math.log(-math.log(u))
            if score > best:
                best, second, arg = score, best, v
            elif score > second:
                second = score
        assert tok[i] == arg
        assert abs(mar[i] - (best - second)) < 1e-12


def test_gumbel_max_noise_is_keyed_by_index_request_position_stream():
    """Changing any of seed, request, position or stream changes the draw for a
    flat log-weight row (where only the noise decides) in most cases, and the
    same key always gives the same draw."""
    V, R = 64, 400
    flat = np.zeros((R, V))
    base, _ = sampling.gumbel_max(flat, 9, np.arange(R), 2, 0)
    again, _ = sampling.gumbel_max(flat, 9, np.arange(R), 2, 0)
    assert np.array_equal(base, again)
    for other in (sampling.gumbel_max(flat, 10, np.arange(R), 2, 0)[0],
                  sampling.gumbel_max(flat, 9, np.arange(R) + 1, 2, 0)[0],
                  sampling.gumbel_max(flat, 9, np.arange(R), 3, 0)[0],
                  sampling.gumbel_max(flat, 9, np.arange(R), 2, 1)[0]):
        assert np.mean(other == base) < 0.1


def test_greedy_lowest_index_on_ties():
    tok, gap = sampling.greedy(np.array([[1.0, 3.0, 3.0, 2.0], [0.0, -1.0, 5.0, 4.5]]))
    assert list(tok) == [1, 2]
    assert gap[0] == 0.0 and gap[1] == 0.5


def _structured(V, r, H, boost=30.0):
    """W1[p] = e_(p mod r); W2[v, j] = boost iff v = g(j) = (7 j + 3) mod V."""
    W1 = np.zeros((V, r))
    W1[np.arange(V), np.arange(V) % r] = 1.0
    W2 = np.zeros((V, r))
    g = (7 * np.arange(r) + 3) % V
    W2[g, np.arange(r)] = boost
    return W1, W2, g


def test_markov_bias_orientation():
    V, r = 40, 6
    W1, W2, g = _structured(V, r, 1)
    prev = np.array([0, 5, 13, 39])
    Bk = draft.markov_bias(W1, W2, prev)
    for i, p in enumerate(prev):
        expect = np.zeros(V)
        expect[g[p % r]] = 30.0
        assert np.array_equal(Bk[i], expect)


def test_chain_uses_previous_token():
    # with U = 0 the bias forces x_k = g(x_{k-1} mod r): any use of x_0 or x_k
    # in place of x_{k-1} breaks the chain
    V, r, H, B, G = 97, 11, 4, 6, 5
    W1, W2, g = _structured(V, r, H)
    U = np.zeros((B, G, V))
    x0 = np.array([1, 2, 50, 60, 95, 96])
    out = draft.draft_block(U, np.zeros((B, G, H)), W1, W2, np.zeros(H + r), 0.0, x0, 1.0, seed=3)
    prev = x0.copy()
    for k in range(G):
        prev = g[prev % r]
        assert np.array_equal(out["x"][:, k], prev)
    greedy_out = draft.draft_block(U, np.zeros((B, G, H)), W1, W2, np.zeros(H + r), 0.0, x0, 0.0, seed=3)
    assert np.array_equal(greedy_out["x"], out["x"])


def test_confidence_markov_part_reads_previous_token():
    V, r, H, B, G = 97, 11, 4, 6, 5
    W1, W2, g = _structured(V, r, H)
    j, s = 2, 1.7
    w = np.zeros(H + r)
    w[H + j] = s
    x0 = np.array([2, 13, 24, 3, 4, 5])          # x0 mod 11 == 2 for the first three
    out = draft.draft_block(np.zeros((B, G, V)), np.zeros((B, G, H)), W1, W2, w, 0.0, x0, 1.0, seed=1)
    prev = np.concatenate([x0[:, None], out["x"][:, :-1]], axis=1)
    expect = np.where(prev % r == j, 1.0 / (1.0 + np.exp(-s)), 0.5)
    assert np.allclose(out["c"], expect, atol=1e-15)


def test_confidence_hidden_part_and_survival():
    rng = np.random.default_rng(4)
    V, r, H, B, G = 50, 4, 8, 3, 4
    h = rng.normal(0, 1, (B, G, H))
    w = np.zeros(H + r)
    w[5] = 1.0
    out = draft.draft_block(rng.normal(0, 1, (B, G, V)), h, rng.normal(0, 1, (V, r)),
                            rng.normal(0, 1, (V, r)), w, 0.25, rng.integers(0, V, B), 1.0, seed=2)
    expect_c = 1.0 / (1.0 + np.exp(-(h[:, :, 5] + 0.25)))
    assert np.allclose(out["c"], expect_c, atol=1e-15)
    assert np.allclose(out["a"], np.cumprod(expect_c, axis=1), atol=1e-15)
    assert np.all(np.diff(out["a"], axis=1) <= 0)


def test_zero_head_gives_halving_survival():
    rng = np.random.default_rng(5)
    V, r, H, B, G = 30, 4, 8, 2, 7
    out = draft.draft_block(rng.normal(0, 1, (B, G, V)), rng.normal(0, 1, (B, G, H)),
                            rng.normal(0, 1, (V, r)), rng.normal(0, 1, (V, r)), np.zeros(H + r), 0.0,
                            rng.integers(0, V, B), 0.9, seed=9)
    assert np.all(out["c"] == 0.5)
    assert np.all(out["a"] == 2.0 ** -np.arange(1, G + 1)[None, :])


def test_draft_sample_distribution_with_strong_bias():
    # x_1 ~ softmax((U_1 + B(x_0)) / T) and x_2 | x_1 ~ softmax((U_2 + B(x_1)) / T);
    # weights N(0, 0.5^2) at r = 16 make the bias O(1), so using the wrong
    # previous token or dropping the bias is visible
    rng = np.random.default_rng(6)
    V, r, H, G, T = 130, 16, 4, 2, 0.8
    R = 60000
    U1 = rng.normal(0, 1, (G, V))
    W1 = rng.normal(0, 0.5, (V, r))
    W2 = rng.normal(0, 0.5, (V, r))
    x0 = 17
    out = draft.draft_block(np.broadcast_to(U1, (R, G, V)), np.zeros((R, G, H)), W1, W2,
                            np.zeros(H + r), 0.0, np.full(R, x0), T, seed=77)
    z1 = U1[0] + W2 @ W1[x0]
    p1 = np.exp((z1 - z1.max()) / T)
    p1 /= p1.sum()
    assert _chi2_p(out["x"][:, 0], p1) > 1e-3
    p1_nobias = np.exp((U1[0] - U1[0].max()) / T)
    p1_nobias /= p1_nobias.sum()
    assert _chi2_p(out["x"][:, 0], p1_nobias) < 1e-6
    top = np.bincount(out["x"][:, 0]).argmax()
    sel = out["x"][:, 0] == top
    z2 = U1[1] + W2 @ W1[top]
    p2 = np.exp((z2 - z2.max()) / T)
    p2 /= p2.sum()
    assert _chi2_p(out["x"][sel, 1], p2) > 1e-3
    # lse_d and logp_d are the normaliser and the log-probability of x_1
    L1 = np.log(np.sum(np.exp(z1 / T - (z1 / T).max()))) + (z1 / T).max()
    assert np.allclose(out["lse_d"][:, 0], L1, atol=1e-12)
    assert np.allclose(out["logp_d"][:, 0], z1[out["x"][:, 0]] / T - L1, atol=1e-12)
