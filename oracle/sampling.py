"""Exact sampling from a softmax by two-level Gumbel-max (test infrastructure
only; see oracle/__init__.py).

The pages sample each draft position from p_k = softmax(U_k + B_k) (DeepSpec
walkthrough, section 3.2, the p_k formula and `sample_block_tokens`), sample
the residual norm(max(0, p_t - p_d)) on a rejection and a bonus token from p_t
(section 8.2) -- but fix no sampler.  The reading used throughout this library:

  * split the vocabulary into blocks of SAMPLE_BLOCK consecutive indices;
  * block key  K_j = logsumexp_{v in block j}(lw_v) + G(u_j)   (block stream)
  * j*         = argmax_j K_j                                   (lowest j on ties)
  * token      = argmax_{v in j*, lw_v > -inf} (lw_v + G(u_v))  (token stream)

where lw are the log-weights (logits / T, or ln q for the residual) and G is a
standard Gumbel variate.  The block maximum of lw_v + G(u_v) is itself
Gumbel-distributed around the block's logsumexp and independent of where in
the block it falls, so the two levels together draw token v with probability
exp(lw_v) / sum exp(lw): the same law as one Gumbel-max over the whole
vocabulary.  Ties go to the lowest index at both levels.
"""
import numpy as np

from . import philox

SAMPLE_BLOCK = 64


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
    s = np.sort(scores, axis=-1)
    top, second = s[..., -1], s[..., -2] if s.shape[-1] > 1 else np.full(s.shape[:-1], -np.inf)
    with np.errstate(invalid="ignore"):
        gap = top - second
    return np.where(np.isfinite(second), gap, np.inf)


def two_level_gumbel(logw, seed, b, k, block_stream, token_stream):
    """Draw one index per row of logw[R, V] with probability softmax(logw).

    b[R] are the request indices that key each row's noise, k the position.
    Returns (tokens[R] int64, margin[R] float64): margin is the smaller of the
    top-2 gaps among block keys and among perturbed scores inside the chosen
    block -- a decision closer than that may legitimately flip under rounding.
    Rows whose log-weights are all -inf return token -1.
    """
    logw = np.atleast_2d(np.asarray(logw, dtype=np.float64))
    R, V = logw.shape
    b = np.broadcast_to(np.asarray(b, dtype=np.int64), (R,))
    nblk = -(-V // SAMPLE_BLOCK)
    padded = np.full((R, nblk * SAMPLE_BLOCK), -np.inf)
    padded[:, :V] = logw
    blocks = padded.reshape(R, nblk, SAMPLE_BLOCK)

    block_lse = logsumexp(blocks, axis=-1)                                    # [R, nblk]
    blk_idx = np.arange(nblk, dtype=np.uint64)[None, :]
    u_blk = philox.uniform_open(philox.draw_words(seed, b[:, None], k, block_stream, blk_idx))
    block_key = block_lse + philox.gumbel(u_blk)                              # -inf stays -inf
    best_blk = np.argmax(block_key, axis=-1)                                  # first max
    block_margin = _top2_gap(block_key)

    tok_idx = best_blk[:, None] * SAMPLE_BLOCK + np.arange(SAMPLE_BLOCK)[None, :]   # [R, 64]
    lw = np.take_along_axis(padded, tok_idx, axis=-1)
    u_tok = philox.uniform_open(philox.draw_words(seed, b[:, None], k, token_stream,
                                                  tok_idx.astype(np.uint64)))
    score = np.where(np.isfinite(lw), lw + philox.gumbel(u_tok), -np.inf)
    inner = np.argmax(score, axis=-1)
    tokens = best_blk * SAMPLE_BLOCK + inner
    margin = np.minimum(block_margin, _top2_gap(score))

    dead = ~np.isfinite(np.max(logw, axis=-1))
    tokens = np.where(dead, -1, tokens)
    return tokens.astype(np.int64), margin


def greedy(logits):
    """argmax per row (lowest index on ties) and the top-2 gap as its margin."""
    logits = np.atleast_2d(np.asarray(logits, dtype=np.float64))
    return np.argmax(logits, axis=-1).astype(np.int64), _top2_gap(logits)
