"""Semi-autoregressive draft block, confidence head and survival product
(test infrastructure only; see oracle/__init__.py).

Follows the DeepSpec walkthrough (wangjunjian.com, "DSpark" post):
  * section 3.2, stage two: p_k(v) = softmax(U_k(v) + B_k(x_0, x_<k, v)) and the
    per-position loop of `sample_block_tokens` -- the bias of step k is built
    from the token sampled at step k-1 (the anchor x_0 for k = 1);
  * section 3.2, VanillaMarkovHead figure (paper eq. 5): B(x_{k-1}, .) =
    W2 . W1[x_{k-1}], rank r;
  * section 3.3, confidence head figure: c_k = sigmoid(linear([h_k; W1[x_{k-1}]]))
    (the model card's AcceptRatePredictor is one nn.Linear(input_dim, 1) that
    returns a logit; the sigmoid is applied at use);
  * section 3.3, Algorithm 1 figure: a_{r,j} = prod_{i<=j} c_{r,i}.

Temperature T divides the whole logit U + B; T = 0 means greedy argmax.
Everything is float64; inputs arrive as exact float64 copies of bf16/fp32.
"""
import numpy as np

from . import philox
from .sampling import gumbel_max, greedy, logsumexp


def markov_bias(W1, W2, prev):
    """B[b, v] = sum_j W2[v, j] * W1[prev[b], j]  for every request b."""
    W1 = np.asarray(W1, dtype=np.float64)
    W2 = np.asarray(W2, dtype=np.float64)
    E = W1[np.asarray(prev, dtype=np.int64)]          # [B, r]: the rows W1[x_{k-1}]
    return E @ W2.T                                   # [B, V]


def confidence(w, bias, h_k, W1_prev):
    """c = sigmoid(w . [h_k ; W1[x_{k-1}]] + bias) per request."""
    w = np.asarray(w, dtype=np.float64)
    H = h_k.shape[-1]
    logit = np.asarray(h_k, np.float64) @ w[:H] + np.asarray(W1_prev, np.float64) @ w[H:] + float(bias)
    return 1.0 / (1.0 + np.exp(-logit))


def draft_block(U, h, W1, W2, w, bias, x0, temperature, seed, forced_tokens=None, requests=None, head=None):
    """One draft block for B requests.

    U[B, gamma, V], h[B, gamma, H], W1/W2[V, r], w[H + r], x0[B].
    forced_tokens[B, gamma] (optional): use these as x_k when building step k+1
    (teacher forcing), so each position can be checked on its own.
    requests[B] (optional): the request index b that keys each row's random
    draws (default 0..B-1), so a sample of rows can be checked on its own.
    head (optional): an oracle.heads.Head (gated or recurrent) whose e_k replaces
    W1[x_{k-1}] in the bias B_k = W2 . e_k (section 3.2's other two heads).
    Returns a dict of x, lse_d, logp_d, c, a [B, gamma], margin [B, gamma] and
    E [B, gamma, r] (the e_k of every position).
    """
    U = np.asarray(U, dtype=np.float64)
    B, gamma, V = U.shape
    x = np.zeros((B, gamma), np.int64)
    lse_d = np.zeros((B, gamma))
    logp_d = np.zeros((B, gamma))
    c = np.zeros((B, gamma))
    a = np.zeros((B, gamma))
    margin = np.zeros((B, gamma))
    prev = np.asarray(x0, dtype=np.int64).copy()
    surv = np.ones(B)
    req = np.arange(B)
    keys = req if requests is None else np.asarray(requests, dtype=np.int64)
    T = float(temperature)
    W1f = np.asarray(W1, np.float64)
    E = np.zeros((B, gamma, W1f.shape[1]))
    state = None if head is None else head.start(B, W1f.shape[1])
    for k in range(1, gamma + 1):
        if head is None:
            E[:, k - 1, :] = W1f[prev]
            z = U[:, k - 1, :] + markov_bias(W1, W2, prev)
        else:
            E[:, k - 1, :], state = head.step(W1f[prev], np.asarray(h, np.float64)[:, k - 1, :], state)
            z = U[:, k - 1, :] + E[:, k - 1, :] @ np.asarray(W2, np.float64).T
        if T > 0.0:
            l = z / T
            L = logsumexp(l, axis=-1)
            tok, mar = gumbel_max(l, seed, keys, k, philox.STREAM_DRAFT_TOKEN)
            lse_d[:, k - 1] = L
            logp_d[:, k - 1] = l[req, tok] - L
        else:
            tok, mar = greedy(z)
        x[:, k - 1] = tok
        margin[:, k - 1] = mar
        c[:, k - 1] = confidence(w, bias, h[:, k - 1, :], np.asarray(W1, np.float64)[prev])
        surv = surv * c[:, k - 1]
        a[:, k - 1] = surv
        prev = tok if forced_tokens is None else np.asarray(forced_tokens, np.int64)[:, k - 1]
    return dict(x=x, lse_d=lse_d, logp_d=logp_d, c=c, a=a, margin=margin, E=E)


def draft_logits(U, W1, W2, x0, tokens, b, k, E=None):
    """z = U_k + B_k for request rows b at (1-based) position k, given the tokens
    x[b, 1..gamma] (x_{k-1} is x0 for k = 1), or given E [B, gamma, r], the e_k a
    gated or recurrent head used.  Used by the residual of verify."""
    U = np.asarray(U, dtype=np.float64)
    b = np.asarray(b, dtype=np.int64)
    k = np.asarray(k, dtype=np.int64)
    if E is not None:
        return U[b, k - 1, :] + np.asarray(E, np.float64)[b, k - 1, :] @ np.asarray(W2, np.float64).T
    tokens = np.asarray(tokens, dtype=np.int64)
    x0 = np.asarray(x0, dtype=np.int64)
    prev = np.where(k == 1, x0[b], tokens[b, np.maximum(k - 2, 0)])
    return U[b, k - 1, :] + markov_bias(W1, W2, prev)
