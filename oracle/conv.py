"""Causal depthwise conv1d (+ SiLU) and its backward, float64 (TEST INFRASTRUCTURE ONLY).

Only the tests, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg use this
module; it shares no code with the CUDA path.

It writes out the definitions of "第三章 反向传播的完整推导" (starbuckoverflow.cn, the
causal-convolution series, chapter 3), per channel c with K taps and zero state before
each sequence's first token:

* forward:  z_t = bias_c + sum_k w_{c,k} x~_{t-K+1+k}  (x~ = x, zero before the sequence
  start), y = SiLU(z) = z sigmoid(z) or y = z without the activation;
* the upstream gradient g = dL/dy becomes delta = dL/dz = g sigmoid(z) (1 + z (1 - sigmoid(z)))
  with SiLU (taken at the pre-activation z), delta = g without it;
* dbias_c = sum_t delta_t;  dw_{c,k} = sum_t delta_t x~_{t-K+1+k};
  dx_s = sum_k w_{c,k} delta_{s+K-1-k}, delta zero past the sequence end;
* packed sequences ("分段数据的公式扩展"): every sum stays inside one sequence.
"""
import numpy as np


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def conv1d_fwd(x, w, bias, cu_seqlens, silu):
    """x [T, C], w [C, K], bias [C] or None -> y [T, C] (and z)."""
    x, w, bias = _f64(x), _f64(w), _f64(bias)
    T, C = x.shape
    K = w.shape[1]
    z = np.zeros((T, C))
    for b, e in zip(cu_seqlens[:-1], cu_seqlens[1:]):
        xp = np.concatenate([np.zeros((K - 1, C)), x[b:e]])  # zero state before the sequence
        for k in range(K):
            z[b:e] += w[:, k][None, :] * xp[k:k + e - b]
        if bias is not None:
            z[b:e] += bias[None, :]
    y = z * _sigmoid(z) if silu else z
    return y, z


def conv1d_bwd(x, w, bias, dy, cu_seqlens, silu):
    """Returns dict(dx [T, C], dw [C, K], dbias [C] or None)."""
    x, w, dy = _f64(x), _f64(w), _f64(dy)
    T, C = x.shape
    K = w.shape[1]
    _, z = conv1d_fwd(x, w, bias, cu_seqlens, silu)
    if silu:
        s = _sigmoid(z)
        delta = dy * s * (1.0 + z * (1.0 - s))
    else:
        delta = dy
    dx = np.zeros((T, C))
    dw = np.zeros((C, K))
    for b, e in zip(cu_seqlens[:-1], cu_seqlens[1:]):
        L = e - b
        xp = np.concatenate([np.zeros((K - 1, C)), x[b:e]])
        dp = np.concatenate([delta[b:e], np.zeros((K - 1, C))])  # delta past the end is zero
        for k in range(K):
            dw[:, k] += (delta[b:e] * xp[k:k + L]).sum(axis=0)
            dx[b:e] += w[:, k][None, :] * dp[K - 1 - k:K - 1 - k + L]
    dbias = None if bias is None else delta.sum(axis=0)
    return {"dx": dx, "dw": dw, "dbias": dbias}
