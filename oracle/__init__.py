"""Oracle: a plain, slow, float64 CPU statement of the DSpark draft / schedule /
verify / accept-rate path.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline leg (and its `--impl reference` arm) may import or run anything
here; the library under serving_draft_verify_gb300/ never does, and the two
share no code.  Every function names the passage of the DeepSpec walkthrough
(wangjunjian.com, "DSpark" post) or the model card (dpshk.com) it follows.

Modules
  philox    Philox4x32-10 (Salmon et al., SC'11) and the uniforms / Gumbel draws
  sampling  Gumbel-max over the vocabulary, noise keyed by vocabulary index
  draft     Markov bias, draft sampling, confidence head, survival product
  schedule  Algorithm 1, literal, with an exact sum of survivals
  verify    rejection-sampling verification, residual and bonus tokens
  tv        c* = 1 - 1/2 ||softmax(d) - softmax(t)||_1
  loss      the joint training loss (CE + L1 + BCE, position weights) and its gradient
  rounds    several draft -> schedule -> verify rounds with the anchor carried
  heads     the gated and recurrent sequential heads (the rank-r row behind the bias)

Parity status: every function is pinned by tests/test_oracle_*.py against
closed forms, brute force, the generator's published vectors or distribution
tests; none is "parity unpinned".
"""
from . import philox, sampling, draft, schedule, verify, tv, loss, rounds, heads  # noqa: F401
from .draft import draft_block, markov_bias, confidence, draft_logits  # noqa: F401
from .schedule import schedule_prefix  # noqa: F401
from .verify import verify as verify_round  # noqa: F401
from .tv import accept_rate_tv  # noqa: F401
from .sampling import gumbel_max  # noqa: F401
