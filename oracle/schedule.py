"""Hardware-aware prefix scheduler, Algorithm 1 (test infrastructure only;
see oracle/__init__.py).

DeepSpec walkthrough, section 3.3, "Hardware-aware prefix scheduler
(Algorithm 1)" flowchart: take every request's confidence sequence, form the
survival a_{r,j} = prod_{i<=j} c_{r,i}, sort all (r, j) pairs by a descending,
scan them greedily, accept a pair while Theta > Theta_best (updating l*_r),
and stop at the first pair that does not raise Theta -- the early stop keeps
the schedule non-anticipating.  Theta = tau * SPS(B) there.

Reading of the symbols (the page leaves them implicit):
  * N = sum_r (l_r + 1) verified rows per round: each request always verifies
    its bonus row (the serving verify width counts the bonus token), so the
    scan starts from l_r = 0, N = B;
  * E = sum_r (1 + sum_{j<=l_r} a_{r,j}) expected emitted tokens;
  * tau = E / N expected emitted tokens per verified row, and SPS(N) the
    verification rate at N rows (a caller-supplied table), so
    Theta(N) = (E / N) * SPS(N);
  * "Theta > Theta_best" is strict; sort ties go to the lower request index,
    then the lower position.
E is the exact sum of the float32 a values, rounded once to float64; Theta is
then one IEEE double division and one multiplication.
"""
from fractions import Fraction

import numpy as np


def schedule_prefix(a, sps):
    """Return (ell[B] int64, n_sched, theta_best) for survival a[B, gamma]
    (float32 values in [0, 1]) and the table sps[N] for N = 0..B*(gamma+1)."""
    a = np.asarray(a, dtype=np.float32)
    B, gamma = a.shape
    sps = [float(s) for s in np.asarray(sps, dtype=np.float64)]
    pairs = sorted(((b, j) for b in range(B) for j in range(1, gamma + 1)),
                   key=lambda p: (-float(a[p[0], p[1] - 1]), p[0], p[1]))
    ell = np.zeros(B, np.int64)
    E = Fraction(B)
    N = B
    theta_best = (float(E) / N) * sps[N]
    for b, j in pairs:
        E_new = E + Fraction(float(a[b, j - 1]))   # exact: float32 -> dyadic rational
        N_new = N + 1
        theta = (float(E_new) / N_new) * sps[N_new]
        if theta > theta_best:
            ell[b] += 1
            E, N, theta_best = E_new, N_new, theta
        else:
            break
    return ell, N, theta_best

