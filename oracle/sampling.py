"""Exact sampling from a softmax by Gumbel-max over the whole vocabulary (test
infrastructure only; see oracle/__init__.py).

The pages sample each draft position from p_k = softmax(U_k + B_k) (DeepSpec
walkthrough, section 3.2, the p_k formula and `sample_block_tokens`), sample
the residual norm(max(0, p_t - p_d)) on a rejection and a bonus token from p_t
(section 8.2) -- but fix no sampler.  The reading used throughout this library
is the textbook Gumbel-max draw with the noise keyed by vocabulary index:

    token = argmax_v ( lw_v + G(u_v) )          (lowest v on ties)
    u_v   = U01(Philox word of (seed; counter (v >> 2, k, b, stream), word v & 3))
    G(u)  = -ln(-ln u)                           (a standard Gumbel variate)

where lw are the log-weights (logits / T, or ln q for the residual) and
entries with lw_v = -inf (no mass) never win.  Because every G(u_v) is an
independent standard Gumbel variate, token v is drawn with probability
exp(lw_v) / sum_w exp(lw_w) (the Gumbel-max property).

The decision margin of a draw is the gap between the largest and the second
largest perturbed score lw_v + G(u_v): a draw closer than that may flip under
the rounding of another implementation.
"""
import numpy as np

from . import philox

_CHUNK_ELEMS = 1 << 21      # noise is drawn for about this many (row, index) pairs at a time


def logsumexp(x, axis=-1):
    """log(sum(exp(x))) in float64; -inf where every entry is -inf."""
    x = np.asarray(x, dtype=np.float64)
    m = np.max(x, axis=axis, keepdims=True)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    with np.errstate(divide="ignore"):
        s = np.log(np.sum(np.exp(x - m_safe), axis=axis, keepdims=True)) + m_safe
    s = np.where(finite, s, -np.inf)
    return np.squeeze(s, axis=axis)


def _top2_gap(scores):
    """Gap between the largest and second-largest entry of each row (inf if < 2 finite)."""
    s = np.partition(scores, scores.shape[-1] - 2, axis=-1) if scores.shape[-1] > 1 else scores
    top = s[..., -1]
    second = s[..., -2] if s.shape[-1] > 1 else np.full(s.shape[:-1], -np.inf)
    with np.errstate(invalid="ignore"):
        gap = top - second
    return np.where(np.isfinite(second), gap, np.inf)


def gumbel_noise(seed, b, k, stream, V):
    """G(u_v) for v = 0 .. V-1 of every request b[R] at position k: [R, V] float64."""
    words = philox.row_words(seed, b, k, stream, V)
    return philox.gumbel(philox.uniform_open(words))


def gumbel_max(logw, seed, b, k, stream):
    """Draw one index per row of logw[R, V] with probability softmax(logw).

    b[R] are the request indices that key each row's noise, k the position,
    `stream` the draw's Philox stream.  Returns (tokens[R] int64, margin[R]
    float64), margin the top-2 gap of the perturbed scores.  Rows whose
    log-weights are all -inf return token -1.
    """
    logw = np.atleast_2d(np.asarray(logw, dtype=np.float64))
    R, V = logw.shape
    b = np.broadcast_to(np.asarray(b, dtype=np.int64), (R,))
    tokens = np.zeros(R, np.int64)
    margin = np.zeros(R)
    rc = max(1, _CHUNK_ELEMS // max(V, 1))       # rows per chunk: bounds the float64 temporaries
    for r0 in range(0, R, rc):
        lw = logw[r0:r0 + rc]
        g = gumbel_noise(seed, b[r0:r0 + rc], k, stream, V)
        score = np.where(np.isfinite(lw), lw + g, -np.inf)
        tokens[r0:r0 + rc] = np.argmax(score, axis=-1)          # first maximum
        margin[r0:r0 + rc] = _top2_gap(score)
    dead = ~np.isfinite(np.max(logw, axis=-1))
    tokens = np.where(dead, -1, tokens)
    return tokens.astype(np.int64), margin


def greedy(logits):
    """argmax per row (lowest index on ties) and the top-2 gap as its margin."""
    logits = np.atleast_2d(np.asarray(logits, dtype=np.float64))
    return np.argmax(logits, axis=-1).astype(np.int64), _top2_gap(logits)
