"""The joint DSpark training loss and its gradient (test infrastructure only;
see oracle/__init__.py).

DeepSpec walkthrough, section 7.2 "joint loss" (`compute_dspark_loss`):

    L = alpha_ce L_ce + alpha_l1 L_l1 + alpha_conf L_conf

  L_ce    cross entropy of the draft logits against the target token,
  L_l1    1/2 ||p_d - p_t||_1 = 1 - c*, dense distribution matching,
  L_conf  BCE(confidence prediction, c*), calibrating the confidence head,

with the default weights 0.1 / 0.9 / 1.0 of that section's table, and
position weights exp(-(k-1) / 4) for block position k (`_build_loss_weight_mask`,
loss_decay_gamma = 4).  Readings of what the page leaves open:

  * each term is a weighted sum over rows with per-row weights omega_r; the
    caller normalises (omega_r = w_k / sum of w over the batch gives the
    weighted mean);
  * the confidence prediction is the head's logit s and the BCE is taken with
    logits: softplus(s) - c* s;
  * c* is the BCE's target: no gradient flows into the logits through it (the
    distribution-matching gradient comes from L_l1);
  * where p_d(v) = p_t(v) exactly the L1 subgradient takes sign(0) = 0.

Written out literally in float64 per row.
"""
import numpy as np

from .tv import softmax

ALPHA_CE, ALPHA_L1, ALPHA_CONF = 0.1, 0.9, 1.0
DECAY_GAMMA = 4.0


def position_weights(k, decay=DECAY_GAMMA):
    """exp(-(k-1)/decay) for block positions k = 1, 2, ..."""
    return np.exp(-(np.asarray(k, dtype=np.float64) - 1.0) / decay)


def logsumexp_rows(x):
    x = np.asarray(x, dtype=np.float64)
    m = np.max(x, axis=-1, keepdims=True)
    return np.squeeze(m, -1) + np.log(np.sum(np.exp(x - m), axis=-1))


def softplus(s):
    s = np.asarray(s, dtype=np.float64)
    return np.maximum(s, 0.0) + np.log1p(np.exp(-np.abs(s)))


def dspark_loss(d, t, target, conf_logit, omega, alpha_ce=ALPHA_CE, alpha_l1=ALPHA_L1, alpha_conf=ALPHA_CONF):
    """Per-row terms and the total.

    d, t [R, V] draft / target logits; target [R] target token ids; conf_logit
    [R] the confidence head's logit s; omega [R] row weights.  Returns a dict
    with ce, c_star, l1, bce (each [R]), row (the weighted row total [R]) and
    loss (their sum).
    """
    d = np.asarray(d, dtype=np.float64)
    t = np.asarray(t, dtype=np.float64)
    R = d.shape[0]
    target = np.asarray(target, dtype=np.int64)
    s = np.asarray(conf_logit, dtype=np.float64)
    omega = np.asarray(omega, dtype=np.float64)
    ce = logsumexp_rows(d) - d[np.arange(R), target]
    c_star = np.sum(np.minimum(softmax(d), softmax(t)), axis=-1)
    l1 = 0.5 * np.sum(np.abs(softmax(d) - softmax(t)), axis=-1)
    bce = softplus(s) - c_star * s
    row = omega * (alpha_ce * ce + alpha_l1 * l1 + alpha_conf * bce)
    return dict(ce=ce, c_star=c_star, l1=l1, bce=bce, row=row, loss=float(np.sum(row)))


def dspark_loss_grad(d, t, target, conf_logit, omega, alpha_ce=ALPHA_CE, alpha_l1=ALPHA_L1, alpha_conf=ALPHA_CONF):
    """Gradients of the total loss: dL/dd [R, V] and dL/ds [R].

      d(CE)/dd_v = p_d(v) - [v = target]
      d(L1)/dd_v = 1/2 sum_u sign(p_d(u) - p_t(u)) dp_d(u)/dd_v
                 = 1/2 p_d(v) (sign_v - sum_u p_d(u) sign_u)
      d(BCE)/ds  = sigmoid(s) - c*           (c* held fixed, see above)
    """
    d = np.asarray(d, dtype=np.float64)
    t = np.asarray(t, dtype=np.float64)
    R = d.shape[0]
    p_d, p_t = softmax(d), softmax(t)
    target = np.asarray(target, dtype=np.int64)
    s = np.asarray(conf_logit, dtype=np.float64)
    omega = np.asarray(omega, dtype=np.float64)[:, None]
    onehot = np.zeros_like(d)
    onehot[np.arange(R), target] = 1.0
    sgn = np.sign(p_d - p_t)
    g_ce = p_d - onehot
    g_l1 = 0.5 * p_d * (sgn - np.sum(p_d * sgn, axis=-1, keepdims=True))
    grad_d = omega * (alpha_ce * g_ce + alpha_l1 * g_l1)
    c_star = np.sum(np.minimum(p_d, p_t), axis=-1)
    grad_s = omega[:, 0] * alpha_conf * (1.0 / (1.0 + np.exp(-s)) - c_star)
    return grad_d, grad_s
