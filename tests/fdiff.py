"""Central finite differences in float64 (test machinery).

The convention (loss = sum of cotangent * output, gradients by central
differences) is itself pinned by the causal-conv worked example in
``test_oracle_pins.py``.
"""
import numpy as np


def central_grad(loss, x, idx=None, h=1e-6):
    """d loss / d x at the flat indices ``idx`` (all if None); ``x`` is modified and restored."""
    flat = x.reshape(-1)
    if idx is None:
        idx = np.arange(flat.size)
    g = np.zeros(len(idx))
    for n, i in enumerate(idx):
        old = flat[i]
        flat[i] = old + h
        lp = loss()
        flat[i] = old - h
        lm = loss()
        flat[i] = old
        g[n] = (lp - lm) / (2 * h)
    return g


def causal_conv1d(x, w, bias):
    """y_t = bias + sum_k w_k x_{t-K+1+k}, zero left padding, no activation."""
    K = len(w)
    xp = np.concatenate([np.zeros(K - 1), x])
    return np.array([bias + sum(w[k] * xp[t + k] for k in range(K)) for t in range(len(x))])
