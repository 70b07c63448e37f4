"""Target verification by rejection sampling (test infrastructure only; see
oracle/__init__.py).

DeepSpec walkthrough, section 8.2 "verify_draft_tokens": for each draft
position k, accept x_k if u < min(1, p_t(x_k) / p_d(x_k)); at the first
rejection drop x_k and everything after it and draw the next token from the
residual max(0, p_t - p_d) renormalised; section 2.1 diagram: a round that
accepts every proposed token adds one bonus token from the target.  Only the
scheduled prefix l*_b is verified (section 3.3, Algorithm 1 flowchart), so
the bonus row of request b is row l*_b + 1.

Readings: p_t = softmax(t_k / T) and p_d = softmax((U_k + B_k) / T), with the
draft's own log-normaliser lse_d and log p_d(x_k) passed in from the draft
step; the residual is drawn by the Gumbel-max of oracle.sampling over ln q;
if q has no mass (p_t <= p_d everywhere) the token is drawn from p_t at that
row.  Every token the verifier emits (residual, bonus, or that fallback) takes
its noise from one stream (STREAM_VERIFY_TOKEN) at (b, row of the draw): a
request draws exactly one such token per round, and the stream is separate
from the draft's noise and from the acceptance uniforms, so the draw is
independent of every event that led to it.  T = 0 is greedy: accept iff x_k = argmax t_k, and the next
token is argmax t at the stop row.  Ties go to the lowest index.
"""
import numpy as np

from . import philox
from .sampling import gumbel_max, greedy, logsumexp
from .draft import draft_logits


def verify(t_logits, U, W1, W2, x0, x, lse_d, logp_d, ell, temperature, seed, requests=None, E=None):
    """Return dict(n_accept[B], next_token[B], margin[B]).

    t_logits[B, gamma+1, V], U[B, gamma, V], W1/W2[V, r], x0[B], x[B, gamma],
    lse_d/logp_d[B, gamma], ell[B] in 0..gamma.  margin[b] is the smallest
    decision margin of request b: |u - ratio| of each acceptance test taken
    and the margin of the final draw (greedy: top-2 logit gaps).
    requests[B] (optional): the request index b that keys each row's random
    draws (default 0..B-1).
    """
    t_logits = np.asarray(t_logits, dtype=np.float64)
    B, gp1, V = t_logits.shape
    gamma = gp1 - 1
    x = np.asarray(x, dtype=np.int64)
    ell = np.asarray(ell, dtype=np.int64)
    lse_d = np.asarray(lse_d, dtype=np.float64)
    logp_d = np.asarray(logp_d, dtype=np.float64)
    req = np.arange(B)
    keys = req if requests is None else np.asarray(requests, dtype=np.int64)
    T = float(temperature)
    n_accept = np.zeros(B, np.int64)
    next_token = np.full(B, -1, np.int64)
    margin = np.full(B, np.inf)
    alive = np.ones(B, bool)                       # still accepting

    for k in range(1, gamma + 1):
        test = alive & (ell >= k)
        if not np.any(test):
            break
        rows = req[test]
        trow = t_logits[rows, k - 1, :]
        if T > 0.0:
            Lt = logsumexp(trow / T, axis=-1)
            log_pt = trow[np.arange(len(rows)), x[rows, k - 1]] / T - Lt
            ratio = np.exp(log_pt - logp_d[rows, k - 1])
            u = philox.uniform_accept(philox.draw_words(seed, keys[rows], k, philox.STREAM_ACCEPT, 0))
            ok = u < ratio
            margin[rows] = np.minimum(margin[rows], np.abs(u - ratio))
        else:
            arg, gap = greedy(trow)
            ok = arg == x[rows, k - 1]
            margin[rows] = np.minimum(margin[rows], gap)
        n_accept[rows[ok]] += 1
        alive[rows[~ok]] = False

    stop = n_accept + 1                             # 1-based row of the final draw
    rejected = n_accept < ell
    for k in range(1, gamma + 2):
        at_k = stop == k
        if not np.any(at_k):
            continue
        if T == 0.0:
            rows = req[at_k]
            tok, gap = greedy(t_logits[rows, k - 1, :])
            next_token[rows] = tok
            margin[rows] = np.minimum(margin[rows], gap)
            continue
        bonus_rows = req[at_k & ~rejected]
        res_rows = req[at_k & rejected]
        fallback = np.zeros(0, np.int64)
        if len(res_rows):
            trow = t_logits[res_rows, k - 1, :] / T
            p_t = np.exp(trow - logsumexp(trow, axis=-1)[:, None])
            z = draft_logits(U, W1, W2, x0, x, res_rows, np.full(len(res_rows), k), E=E)
            p_d = np.exp(z / T - lse_d[res_rows, k - 1][:, None])
            q = np.maximum(0.0, p_t - p_d)
            has_mass = np.sum(q, axis=-1) > 0.0
            with np.errstate(divide="ignore"):
                logq = np.where(q > 0.0, np.log(q), -np.inf)
            if np.any(has_mass):
                r = res_rows[has_mass]
                tok, mar = gumbel_max(logq[has_mass], seed, keys[r], k, philox.STREAM_VERIFY_TOKEN)
                next_token[r] = tok
                margin[r] = np.minimum(margin[r], mar)
            fallback = res_rows[~has_mass]
        from_target = np.concatenate([bonus_rows, fallback])
        if len(from_target):
            tok, mar = gumbel_max(t_logits[from_target, k - 1, :] / T, seed, keys[from_target], k,
                                  philox.STREAM_VERIFY_TOKEN)
            next_token[from_target] = tok
            margin[from_target] = np.minimum(margin[from_target], mar)
    return dict(n_accept=n_accept, next_token=next_token, margin=margin)
