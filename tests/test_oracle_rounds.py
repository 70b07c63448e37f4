"""Pins of the multi-round oracle (DeepSpec walkthrough sections 8.1 / 8.3):
the anchor carried from round to round, the emitted tokens when the target
agrees with the draft, per-round keys, and E[tau] against the scheduler's own
Theta."""
import numpy as np

from oracle import rounds as R
from oracle import schedule


def _pool(n, B, G, V, H, rng, agree=True):
    out = []
    for _ in range(n):
        U = rng.normal(0, 2.0, (B, G, V))
        t = np.concatenate([U, rng.normal(0, 2.0, (B, 1, V))], axis=1) if agree else \
            np.concatenate([U, rng.normal(0, 2.0, (B, 1, V))], axis=1) + rng.normal(0, 1.0, (B, G + 1, V))
        out.append(dict(U=U, h=rng.normal(0, 1.0, (B, G, H)), t=t))
    return out


def _sps(B, G):
    N = np.arange(B * (G + 1) + 1, dtype=np.float64)
    return N / (20.0 + 0.05 * N)


def test_anchor_is_the_last_emitted_token():
    """W1[v, 0] = v / V and a head that reads only that coordinate: c_1 of each
    round reveals the anchor it used, which must be the previous round's last
    emitted token."""
    rng = np.random.default_rng(0)
    B, G, V, H, r = 5, 4, 64, 3, 2
    pool = _pool(3, B, G, V, H, rng, agree=False)
    W1 = np.zeros((V, r))
    W1[:, 0] = np.arange(V) / V
    W2 = rng.normal(0, 0.3, (V, r))
    w = np.zeros(H + r)
    w[H] = 4.0
    x0 = rng.integers(0, V, B)
    out, final = R.decode_rounds(pool, W1, W2, w, 0.0, _sps(B, G), x0, 1.0, 7, rounds=5)
    prev_last = x0
    for o in out:
        used = np.log(o["c"][:, 0] / (1.0 - o["c"][:, 0])) / 4.0 * V
        assert np.allclose(used, prev_last, atol=1e-6)
        last = o["tokens"][np.arange(B), o["n_emitted"] - 1]
        assert np.array_equal(last, o["next_token"])
        prev_last = last
    assert np.array_equal(final, prev_last)


def test_agreeing_target_accepts_every_scheduled_token():
    """t = U and no Markov bias: p_t = p_d, so every scheduled draft token is
    accepted and a round emits l_b + 1 tokens, the last from row l_b + 1."""
    rng = np.random.default_rng(1)
    B, G, V, H, r = 6, 5, 40, 4, 2
    pool = _pool(2, B, G, V, H, rng, agree=True)
    W1 = rng.normal(0, 0.3, (V, r))
    W2 = np.zeros((V, r))
    w = rng.normal(0, 0.5, H + r)
    for T in (1.0, 0.0):
        out, _ = R.decode_rounds(pool, W1, W2, w, 0.5, _sps(B, G), rng.integers(0, V, B), T, 3, rounds=4)
        for i, o in enumerate(out):
            assert np.array_equal(o["n_accept"], o["ell"])
            assert np.array_equal(o["n_emitted"], o["ell"] + 1)
            assert o["tau"] == np.mean(o["ell"] + 1)
            for b in range(B):
                L = o["ell"][b]
                assert np.array_equal(o["tokens"][b, :L], o["x"][b, :L])
                assert np.all(o["tokens"][b, L + 1:] == -1)
                if T == 0.0:
                    assert o["tokens"][b, L] == np.argmax(pool[i % 2]["t"][b, L])


def test_rounds_draw_with_their_own_keys():
    """With the anchor made irrelevant (no bias, a head blind to W1), rounds 0
    and 1 on a one-slot pool see identical inputs; their draws must differ."""
    rng = np.random.default_rng(2)
    B, G, V, H, r = 8, 6, 300, 2, 2
    pool = _pool(1, B, G, V, H, rng, agree=True)
    W1 = rng.normal(0, 1.0, (V, r))
    W2 = np.zeros((V, r))
    w = np.concatenate([rng.normal(0, 0.5, H), np.zeros(r)])
    out, _ = R.decode_rounds(pool, W1, W2, w, 0.0, _sps(B, G), rng.integers(0, V, B), 1.0, 11, rounds=2)
    assert np.array_equal(out[0]["a"], out[1]["a"])
    assert not np.array_equal(out[0]["x"], out[1]["x"])
    assert R.round_seed((1 << 64) - 1, 1) == 0


def test_expected_tau_matches_the_schedulers_theta():
    """E = Theta_best * N / SPS(N) from the scheduler's own scan."""
    rng = np.random.default_rng(3)
    B, G = 7, 6
    c = rng.uniform(0.3, 1.0, (B, G)).astype(np.float32)
    a = np.cumprod(c, axis=1, dtype=np.float32)
    sps = _sps(B, G)
    ell, N, theta = schedule.schedule_prefix(a, sps)
    E = R.expected_tau(a, ell) * B
    assert abs(E - theta * N / sps[N]) <= 1e-12 * E
    assert R.expected_tau(a, np.zeros(B, int)) == 1.0
