"""Pins of the gated and recurrent heads (DeepSpec walkthrough section 3.2,
markov_head.py): closed forms where the gate is 0, 1/2 or saturated, the
unrolled recurrence, position alignment of h_k, and bf16 rounding."""
import numpy as np

from oracle import draft, heads


def _setup(B=4, G=5, V=48, H=3, r=4, seed=0):
    rng = np.random.default_rng(seed)
    U = rng.normal(0, 2.0, (B, G, V))
    h = rng.normal(0, 1.0, (B, G, H))
    W1 = rng.normal(0, 0.7, (V, r))
    W2 = rng.normal(0, 0.7, (V, r))
    w = rng.normal(0, 0.3, H + r)
    x0 = rng.integers(0, V, B)
    return U, h, W1, W2, w, x0, rng


def _same(a, b):
    for k in ("x", "lse_d", "logp_d", "c", "a"):
        assert np.array_equal(a[k], b[k]), k


def test_round_bf16():
    assert heads.round_bf16(1.0) == 1.0
    assert heads.round_bf16(1.0 + 2 ** -8) == 1.0                  # tie -> even
    assert heads.round_bf16(1.0 + 3 * 2 ** -8) == 1.0 + 2 ** -6     # tie -> even (upwards)
    assert heads.round_bf16(1.0 + 2 ** -8 + 2 ** -20) == 1.0 + 2 ** -7
    assert heads.round_bf16(-3.0) == -3.0
    assert heads.round_bf16(0.1) == 0.10009765625


def test_gated_zero_gate_halves_the_markov_bias():
    U, h, W1, W2, w, x0, _ = _setup()
    H, r = h.shape[-1], W1.shape[-1]
    g = heads.Head(heads.GATED, Wg=np.zeros((r, H + r)))
    for T in (0.9, 0.0):
        a = draft.draft_block(U, h, W1, W2, w, 0.1, x0, T, 3, head=g)
        b = draft.draft_block(U, h, W1, 0.5 * W2, w, 0.1, x0, T, 3)
        _same(a, b)
        assert np.array_equal(a["E"], 0.5 * b["E"])


def test_saturated_gates_reduce_to_closed_forms():
    """sigmoid(80) is 1 in float64: the gated head becomes the Markov head, and the
    RNN keeps its zero state (no bias at all)."""
    U, h, W1, W2, w, x0, _ = _setup(seed=1)
    H, r = h.shape[-1], W1.shape[-1]
    h = h.copy()
    h[:, :, 0] = 1.0
    Wg = np.zeros((r, H + r))
    Wg[:, 0] = 80.0
    a = draft.draft_block(U, h, W1, W2, w, 0.0, x0, 1.0, 5, head=heads.Head(heads.GATED, Wg=Wg))
    b = draft.draft_block(U, h, W1, W2, w, 0.0, x0, 1.0, 5)
    _same(a, b)
    Wg = np.zeros((r, 2 * r + H))
    Wg[:, 2 * r] = 80.0
    rng = np.random.default_rng(2)
    Wc = rng.normal(0, 1.0, (r, 2 * r + H))
    a = draft.draft_block(U, h, W1, W2, w, 0.0, x0, 1.0, 5, head=heads.Head(heads.RNN, Wg=Wg, Wc=Wc))
    b = draft.draft_block(U, h, W1, np.zeros_like(W2), w, 0.0, x0, 1.0, 5)
    _same(a, b)
    assert np.all(a["E"] == 0.0)


def test_rnn_half_gate_is_the_unrolled_sum():
    """g = 1/2 and a candidate that ignores the state: s_k = sum_{i<=k} 2^-(k-i+1) tanh(c_i),
    c_i = Wc_x W1[x_{i-1}] + Wc_h h_i."""
    U, h, W1, W2, w, x0, rng = _setup(seed=3)
    B, G, _ = U.shape
    H, r = h.shape[-1], W1.shape[-1]
    Wc = rng.normal(0, 1.0, (r, 2 * r + H))
    Wc[:, :r] = 0.0
    out = draft.draft_block(U, h, W1, W2, w, 0.0, x0, 0.8, 9,
                            head=heads.Head(heads.RNN, Wg=np.zeros((r, 2 * r + H)), Wc=Wc))
    prev = np.concatenate([x0[:, None], out["x"][:, :-1]], axis=1)    # x_{k-1}
    for k in range(1, G + 1):
        s = np.zeros((B, r))
        for i in range(1, k + 1):
            c = W1[prev[:, i - 1]] @ Wc[:, r:2 * r].T + h[:, i - 1, :] @ Wc[:, 2 * r:].T
            s += 0.5 ** (k - i + 1) * np.tanh(c)
        assert np.allclose(out["E"][:, k - 1, :], s, atol=1e-14)


def test_gate_reads_h_of_its_own_position():
    U, h, W1, W2, w, x0, _ = _setup(seed=4)
    B, G, _ = U.shape
    H, r = h.shape[-1], W1.shape[-1]
    W1 = np.ones_like(W1)
    Wg = np.zeros((r, H + r))
    Wg[:, 0] = 1.0
    out = draft.draft_block(U, h, W1, W2, w, 0.0, x0, 1.0, 2, head=heads.Head(heads.GATED, Wg=Wg))
    for k in range(1, G + 1):
        assert np.allclose(out["E"][:, k - 1, :], (1.0 / (1.0 + np.exp(-h[:, k - 1, 0])))[:, None], atol=1e-15)


def test_bf16_rounding_of_e():
    U, h, W1, W2, w, x0, rng = _setup(seed=5)
    H, r = h.shape[-1], W1.shape[-1]
    Wg = rng.normal(0, 1.0, (r, H + r))
    a = draft.draft_block(U, h, W1, W2, w, 0.0, x0, 1.0, 2, head=heads.Head(heads.GATED, Wg=Wg, bf16=True))
    assert np.array_equal(a["E"], heads.round_bf16(a["E"]))
    b = draft.draft_block(U, h, W1, W2, w, 0.0, x0, 1.0, 2, head=heads.Head(heads.GATED, Wg=Wg))
    assert not np.array_equal(a["E"], b["E"])
