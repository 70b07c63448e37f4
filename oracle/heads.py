"""Gated and recurrent sequential heads (test infrastructure only; see
oracle/__init__.py).

DeepSpec walkthrough, section 3.2, the three heads of markov_head.py.  Every
head adds B_k(v) = W2[v] . e_k to the parallel logits U_k; the heads differ in
the rank-r vector e_k:

  Markov (eq. 5)  e_k = W1[x_{k-1}]
  Gated           e_k = sigmoid(Wg [h_k ; W1[x_{k-1}]]) * W1[x_{k-1}]
  RNN (eq. 6)     s_k = g * s_{k-1} + (1 - g) * tanh(Wc z_k),
                  g = sigmoid(Wg z_k),  z_k = [s_{k-1} ; W1[x_{k-1}] ; h_k],  e_k = s_k

Readings of what the page's figure leaves open (its text is garbled there):
  * the gated head's figure shows no output projection; the plainest reading
    that yields a vocabulary bias keeps the Markov head's W2, and reads the
    product as element-wise (the only shape-consistent one), so Wg is
    [r, H + r];
  * the RNN head's "(1-sigma)(Wg z_k)" reads as 1 - sigmoid(Wg z_k); the state
    has r entries, s_0 = 0, Wg and Wc are [r, 2r + H] over [s; W1 row; h], and
    the bias projects the state with W2;
  * with bf16 weights e_k is rounded to bf16 (round to nearest even) before the
    projection, as the W1 rows of the Markov head are bf16 values; the RNN
    state itself is carried unrounded.
"""
import numpy as np

MARKOV, GATED, RNN = 0, 1, 2


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-np.asarray(x, np.float64)))


def round_bf16(x):
    """Round to the nearest bf16 value (ties to even), via float32."""
    f = np.asarray(x, np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


class Head:
    """A sequential head: kind, Wg, Wc (float64 copies of the weights) and
    whether e_k is rounded to bf16."""

    def __init__(self, kind, Wg=None, Wc=None, bf16=False):
        self.kind = kind
        self.Wg = None if Wg is None else np.asarray(Wg, np.float64)
        self.Wc = None if Wc is None else np.asarray(Wc, np.float64)
        self.bf16 = bf16

    def start(self, B, r):
        """The recurrent state before position 1."""
        return np.zeros((B, r))

    def step(self, W1_prev, h_k, state):
        """(e_k [B, r], next state) from W1[x_{k-1}] [B, r], h_k [B, H] and the state."""
        W1_prev = np.asarray(W1_prev, np.float64)
        h_k = np.asarray(h_k, np.float64)
        if self.kind == MARKOV:
            e = W1_prev
        elif self.kind == GATED:
            g = sigmoid(np.concatenate([h_k, W1_prev], axis=1) @ self.Wg.T)
            e = g * W1_prev
        else:
            z = np.concatenate([state, W1_prev, h_k], axis=1)
            g = sigmoid(z @ self.Wg.T)
            state = g * state + (1.0 - g) * np.tanh(z @ self.Wc.T)
            e = state
        if self.bf16 and self.kind != MARKOV:
            e = round_bf16(e)
        return e, state
