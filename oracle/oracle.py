"""Float64 CPU oracle for the chunked gated delta-rule backward (GDN and KDA).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` call it.  It shares no code with the CUDA path.

The token-by-token recurrence and its hand-derived reverse mode are in
``gdr_oracle.c`` (see that file's header for every formula and its source).
This module adds the two gate front ends:

* GDN: one natural-log gate per (token, head).  It is broadcast over the
  channels and its gradient is the channel sum of the per-channel gradient.
* KDA: ``g = -exp(A_log[h]) * softplus(g_raw + dt_bias[h, d])`` per channel (the
  gate function of the KDA benchmark workload).  Its chain
  rule follows the pattern of "FlashKDA之backward（K1）", §5.2 (chain through
  the gate function per element, parameter gradients summed over tokens, the
  A_log gradient picking up one factor from the exp):
      dg_raw[t,h,d]  = dg[t,h,d] * (-exp(A_log[h]) * sigmoid(g_raw + dt_bias))
      ddt_bias[h,d]  = sum_t dg_raw[t,h,d]
      dA_log[h]      = sum_{t,d} dg[t,h,d] * g[t,h,d]

Layout everywhere: token-major ``[T_total, H, D]``; ``cu_seqlens`` (int64,
``[N+1]``) gives the sequence boundaries on the token axis; states are
``[N, H, D, D]`` with the key channel as the row index.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        lib.oracle_gdr.restype = ctypes.c_int
        lib.oracle_gdr.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int64), ctypes.c_int,
                                   ctypes.c_int, ctypes.c_double] + [dp] * 16 + [ctypes.c_int]
        lib.oracle_max_threads.restype = ctypes.c_int
        _LIB = lib
    return _LIB


def max_threads() -> int:
    return int(_lib().oracle_max_threads())


def _f64(x):
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x):
    if x is None:
        return ctypes.POINTER(ctypes.c_double)()
    return x.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def gated_delta(q, k, v, glog, beta_logit, scale, cu_seqlens, h0=None, dO=None, dht=None,
                nthreads=0):
    """Per-channel log-gate recurrence, forward and (if ``dO`` is given) backward.

    Returns a dict with ``o`` [T,H,D], ``ht`` [N,H,D,D] and, with ``dO``,
    ``dq, dk, dv, dglog`` [T,H,D], ``dbeta`` [T,H] (logit space), ``dh0`` [N,H,D,D].

    Grouped heads (GQA: q, k with Hk heads, v and everything else with H = r Hk heads):
    value head h reads q / k head h // r, i.e. each q / k head is shared by r consecutive
    value heads (the grouped-query layout of the FlashQLA page's GQA tests); the shared
    q / k is the same as r copies of it, so dq and dk are the sums over each group.
    """
    q, k = _f64(q), _f64(k)
    if q.shape[1] != np.shape(v)[1]:
        Hk, H = q.shape[1], np.shape(v)[1]
        assert H % Hk == 0 and k.shape == q.shape
        r = H // Hk
        out = gated_delta(np.repeat(q, r, axis=1), np.repeat(k, r, axis=1), v, glog, beta_logit, scale,
                          cu_seqlens, h0, dO, dht, nthreads)
        for name in ("dq", "dk"):
            if name in out:
                T, _, D = out[name].shape
                out[name] = out[name].reshape(T, Hk, r, D).sum(axis=2)
        return out
    q, k, v, glog, beta_logit = map(_f64, (q, k, v, glog, beta_logit))
    h0, dO, dht = _f64(h0), _f64(dO), _f64(dht)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    T, H, D = q.shape
    N = cu.shape[0] - 1
    assert cu[0] == 0 and cu[-1] == T and np.all(np.diff(cu) >= 0)
    for x in (k, v, glog):
        assert x.shape == (T, H, D)
    assert beta_logit.shape == (T, H)
    for x in (h0, dht):
        assert x is None or x.shape == (N, H, D, D)
    out = {"o": np.zeros((T, H, D)), "ht": np.zeros((N, H, D, D))}
    if dO is not None:
        assert dO.shape == (T, H, D)
        out.update(dq=np.zeros((T, H, D)), dk=np.zeros((T, H, D)), dv=np.zeros((T, H, D)),
                   dglog=np.zeros((T, H, D)), dbeta=np.zeros((T, H)),
                   dh0=np.zeros((N, H, D, D)))
    g = out.get
    rc = _lib().oracle_gdr(N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), H, D,
                           float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(glog), _ptr(beta_logit),
                           _ptr(h0), _ptr(dO), _ptr(dht), _ptr(g("o")), _ptr(g("ht")),
                           _ptr(g("dq")), _ptr(g("dk")), _ptr(g("dv")), _ptr(g("dglog")),
                           _ptr(g("dbeta")), _ptr(g("dh0")), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gdr rejected its arguments")
    return out


def gdn(q, k, v, g, beta_logit, scale, cu_seqlens, h0=None, dO=None, dht=None, nthreads=0):
    """GDN: scalar natural-log gate ``g`` [T,H].  Backward returns ``dg`` [T,H]."""
    g = _f64(g)
    T, H, D = np.shape(v)
    assert g.shape == (T, H)
    glog = np.ascontiguousarray(np.broadcast_to(g[:, :, None], (T, H, D)))
    out = gated_delta(q, k, v, glog, beta_logit, scale, cu_seqlens, h0, dO, dht, nthreads)
    if "dglog" in out:
        out["dg"] = out.pop("dglog").sum(axis=2)
    return out


def softplus(x):
    return np.logaddexp(0.0, x)


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def kda_gate(g_raw, A_log, dt_bias):
    """Per-channel log gate of KDA: -exp(A_log[h]) * softplus(g_raw + dt_bias[h, d])."""
    g_raw, A_log, dt_bias = map(_f64, (g_raw, A_log, dt_bias))
    return -np.exp(A_log)[None, :, None] * softplus(g_raw + dt_bias[None, :, :])


LN2 = np.log(2.0)


def kda_sigmoid_gate(g_raw, A_log, dt_bias, gate_scale):
    """Sigmoid-bounded per-channel log gate of the FlashKDA kernels ("FlashKDA之backward（K1）",
    §5.2: the base-2 log gate is gate_scale * sigmoid(e^{A_log[h]} (g_raw + dt_bias[h, d]))),
    written as a natural-log gate: ln 2 * gate_scale * sigmoid(e^{A_log} (g_raw + dt_bias))."""
    g_raw, A_log, dt_bias = map(_f64, (g_raw, A_log, dt_bias))
    z = np.exp(A_log)[None, :, None] * (g_raw + dt_bias[None, :, :])
    return LN2 * float(gate_scale) * sigmoid(z)


def kda(q, k, v, g_raw, A_log, dt_bias, beta_logit, scale, cu_seqlens, h0=None, dO=None,
        dht=None, nthreads=0, gate="softplus", gate_scale=None):
    """KDA: per-channel gate from ``g_raw`` [T,H,D], ``A_log`` [H], ``dt_bias`` [H,D].

    ``gate="softplus"``: g = -e^{A_log} softplus(g_raw + dt_bias); ``gate="sigmoid"``: the
    sigmoid-bounded gate of ``kda_sigmoid_gate`` with ``gate_scale``.  Backward returns
    ``dg_raw`` [T,H,D], ``dA_log`` [H] and ``ddt_bias`` [H,D] in place of ``dg``.
    """
    g_raw, A_log, dt_bias = map(_f64, (g_raw, A_log, dt_bias))
    if gate == "softplus":
        glog = kda_gate(g_raw, A_log, dt_bias)
    elif gate == "sigmoid":
        glog = kda_sigmoid_gate(g_raw, A_log, dt_bias, gate_scale)
    else:
        raise ValueError("gate must be 'softplus' or 'sigmoid'")
    out = gated_delta(q, k, v, glog, beta_logit, scale, cu_seqlens, h0, dO, dht, nthreads)
    if "dglog" in out:
        dglog = out.pop("dglog")
        a = np.exp(A_log)[None, :, None]
        x = g_raw + dt_bias[None, :, :]
        if gate == "softplus":
            # g = -a softplus(x): dg/dx = -a sigmoid(x), dg/dA_log = g
            dg_raw = dglog * (-a * sigmoid(x))
            dA = dglog * glog
        else:
            # g = ln2 gs sigmoid(z), z = a x: dg/dz = ln2 gs s (1 - s); dz/dx = a, dz/dA_log = a x
            s = sigmoid(a * x)
            dz = dglog * LN2 * float(gate_scale) * s * (1.0 - s)
            dg_raw = dz * a
            dA = dz * a * x
        out["dg_raw"] = dg_raw
        out["ddt_bias"] = dg_raw.sum(axis=0)
        out["dA_log"] = dA.sum(axis=(0, 2))
        out["dA_terms"] = dA  # per-element terms of dA_log (their magnitudes condition short sums)
    return out
