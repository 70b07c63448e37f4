"""Analytic accept rate c* = 1 - 1/2 ||softmax(d) - softmax(t)||_1 (test
infrastructure only; see oracle/__init__.py).

DeepSpec walkthrough, section 3.3 "Confidence head design", paper eq. 8 and the
`_compute_accept_rate_3d` snippet: both logit rows go through a softmax over the
full vocabulary (no temperature), the absolute difference is summed, and half
of it is subtracted from 1.  Written out literally in float64.
"""
import numpy as np


def softmax(x):
    """Row softmax in float64 (max-shifted; exact up to rounding)."""
    x = np.asarray(x, dtype=np.float64)
    m = np.max(x, axis=-1, keepdims=True)
    e = np.exp(x - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def accept_rate_tv(d, t):
    """c*[row] for draft logits d[rows, V] and target logits t[rows, V]."""
    p_d = softmax(d)
    p_t = softmax(t)
    return 1.0 - 0.5 * np.sum(np.abs(p_d - p_t), axis=-1)
