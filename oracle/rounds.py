"""Several speculative-decoding rounds in a row (test infrastructure only; see
oracle/__init__.py).

DeepSpec walkthrough, section 8.1 / 8.3 (`generate_decoding_sample`): each
round proposes a draft block from the current context, verifies it against
the target, emits the accepted draft tokens followed by the one token the
verifier draws (residual or bonus), and continues from the new context.  With
synthetic inputs the context carried from round to round is the anchor: the
next round's x_0 is the last token emitted.  Readings:

  * round i takes its logits U, h and t from a pool of synthetic rounds, slot
    i mod pool (the target model that would produce them is out of scope);
  * round i keys its random draws with seed + i (64-bit wrap-around), so no two
    rounds share a Philox key;
  * the scheduler sees the survivals a as float32, as the draft writes them;
  * expected emitted tokens per request, E[tau] = sum_b (1 + sum_{j <= l_b}
    a_{b,j}) / B (the quantity the scheduler maximises, section 3.3), and the
    realised value sum_b (n_accept_b + 1) / B.
"""
import numpy as np

from .draft import draft_block
from .schedule import schedule_prefix
from .verify import verify

MASK64 = (1 << 64) - 1


def round_seed(seed, i):
    return (int(seed) + int(i)) & MASK64


def emitted_tokens(x, n_accept, next_token):
    """[B, gamma+1]: the accepted draft tokens, then the verifier's token, then -1."""
    x = np.asarray(x, np.int64)
    B, gamma = x.shape
    out = np.full((B, gamma + 1), -1, np.int64)
    for b in range(B):
        n = int(n_accept[b])
        out[b, :n] = x[b, :n]
        out[b, n] = next_token[b]
    return out


def expected_tau(a, ell):
    """E[tau] = sum_b (1 + sum_{j <= l_b} a_{b,j}) / B, summed exactly."""
    from fractions import Fraction
    a = np.asarray(a, np.float32)
    B = a.shape[0]
    E = Fraction(B)
    for b in range(B):
        for j in range(int(ell[b])):
            E += Fraction(float(a[b, j]))
    return float(E / B)


def decode_rounds(pool, W1, W2, w, bias, sps, x0, temperature, seed, rounds, forced=None):
    """Run `rounds` rounds.  pool: list of dicts with U [B, gamma, V], h [B, gamma, H]
    and t [B, gamma+1, V] (float64).  forced (optional): per round a dict with the
    anchor, x and a of another implementation (teacher forcing: round i then starts
    from forced[i]['anchor'], builds each draft position on forced x, and schedules
    forced a), so each round can be checked on its own.  Returns a list of per-round
    dicts (anchor, x, lse_d, logp_d, c, a, draft margin, ell, n_sched, n_accept,
    next_token, verify margin, tokens, n_emitted, E_tau, tau) and the final anchor."""
    anchor = np.asarray(x0, np.int64).copy()
    out = []
    for i in range(rounds):
        slot = pool[i % len(pool)]
        s = round_seed(seed, i)
        f = None if forced is None else forced[i]
        if f is not None:
            anchor = np.asarray(f["anchor"], np.int64).copy()
        d = draft_block(slot["U"], slot["h"], W1, W2, w, bias, anchor, temperature, s,
                        forced_tokens=None if f is None else f["x"])
        x = d["x"] if f is None else np.asarray(f["x"], np.int64)
        a32 = (d["a"] if f is None else np.asarray(f["a"])).astype(np.float32)
        lse_d = d["lse_d"] if f is None else np.asarray(f["lse_d"], np.float64)
        logp_d = d["logp_d"] if f is None else np.asarray(f["logp_d"], np.float64)
        ell, n_sched, _ = schedule_prefix(a32, sps)
        v = verify(slot["t"], slot["U"], W1, W2, anchor, x, lse_d, logp_d, ell, temperature, s)
        tokens = emitted_tokens(x, v["n_accept"], v["next_token"])
        out.append(dict(anchor=anchor.copy(), x=d["x"], lse_d=d["lse_d"], logp_d=d["logp_d"], c=d["c"], a=d["a"],
                        draft_margin=d["margin"], ell=ell, n_sched=n_sched, n_accept=v["n_accept"],
                        next_token=v["next_token"], verify_margin=v["margin"], tokens=tokens,
                        n_emitted=np.asarray(v["n_accept"], np.int64) + 1,
                        E_tau=expected_tau(a32, ell), tau=float(np.mean(np.asarray(v["n_accept"]) + 1))))
        anchor = np.asarray(v["next_token"], np.int64).copy()
    return out, anchor
