"""Float64 chunk-form reference of the gated delta rule (forward and backward).

TEST INFRASTRUCTURE ONLY (diagnostics for small cases); it shares no code with
the CUDA path and nothing on the product path imports it.

It restates, chunk by chunk, the algebra the pages describe for the chunked
method, in numpy float64 and without any range tricks:

* per chunk of C tokens: the inclusive gate cumsum gc and its last row gT, and
  the derived tiles kd = kn*e^{gc}, ki = kn*e^{-gc}, kr = kn*e^{gT-gc},
  qd = scale*qn*e^{gc} ("FlashKDA之backward（K1）", the forward workspace in the
  kernel signature and §3.2(a));
* the intra-chunk UT/WY form: A = strict_lower(diag(beta) kd ki^T),
  T = (I + A)^-1, u = T diag(beta) (V - kd S0), O = qd S0 + lower(qd ki^T) u,
  S_C = diag(e^{gT}) S0 + kr^T u;
* the state-gradient recurrence of the FlashQLA dh kernel
  ("FlashQLA ... GDN 反向", §三): dS0 = e^{gT} dS_C + R^T dO - X^T (kr dS_C)
  with X = W = T diag(beta) kd and R = qd - lower(P) X;
* the FlashKDA K1_bwd assembly of the input gradients from the gradients of
  the derived tiles ("FlashKDA之backward（K1）", §3.2-§3.3 and §5): the
  numerically stable dgc, the L2-norm backward, and the reverse cumsum of dgc
  plus the per-chunk constant dgT.

It is pinned against the token-level oracle (``oracle.py``): the two are
independent derivations of the same gradients.
"""
import numpy as np

CHUNK = 64


def reverse_cumsum(x, axis=0):
    """Suffix sums along ``axis`` (the adjoint of a prefix sum), as in
    "FlashKDA之backward（K1）", §5.0."""
    x = np.asarray(x)
    return np.flip(np.cumsum(np.flip(x, axis=axis), axis=axis), axis=axis)


def _l2n(x):
    n = np.sqrt((x * x).sum(axis=-1, keepdims=True) + 1e-6)
    return x / n, n


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _chunk_consts(qn, kn, glog, beta, scale):
    gc = np.cumsum(glog, axis=0)
    gT = gc[-1]
    Kd = kn * np.exp(gc)
    Ki = kn * np.exp(-gc)
    Kr = kn * np.exp(gT[None, :] - gc)
    Qd = scale * qn * np.exp(gc)
    n = qn.shape[0]
    Araw = Kd @ Ki.T
    A = np.tril(beta[:, None] * Araw, -1)
    T = np.linalg.inv(np.eye(n) + A)
    P = np.tril(Qd @ Ki.T)
    W = T @ (beta[:, None] * Kd)
    return dict(gc=gc, gT=gT, Kd=Kd, Ki=Ki, Kr=Kr, Qd=Qd, Araw=Araw, A=A, T=T, P=P, W=W)


def pair(q, k, v, glog, blogit, h0, dO, dht, scale, C=CHUNK, keep=False):
    """One (sequence, head): q, k, v, glog, dO are [L, D]; blogit [L]; h0, dht [D, D].

    Returns the forward outputs, the gradients and (``keep=True``) a list of
    per-chunk intermediates (S0, dSC, W, U, Kr, R, T).
    """
    L, D = q.shape
    qn, nq = _l2n(q)
    kn, nk = _l2n(k)
    beta = _sigmoid(blogit)
    S = np.zeros((D, D)) if h0 is None else h0.copy()
    o = np.zeros((L, D))
    chunks = []
    for r0 in range(0, L, C):
        r1 = min(r0 + C, L)
        cst = _chunk_consts(qn[r0:r1], kn[r0:r1], glog[r0:r1], beta[r0:r1], scale)
        E = v[r0:r1] - cst["Kd"] @ S
        u = cst["T"] @ (beta[r0:r1, None] * E)
        o[r0:r1] = cst["Qd"] @ S + cst["P"] @ u
        U = cst["T"] @ (beta[r0:r1, None] * v[r0:r1])
        R = cst["Qd"] - cst["P"] @ cst["W"]
        chunks.append(dict(r0=r0, r1=r1, S0=S.copy(), u=u, E=E, U=U, R=R, **cst))
        S = np.exp(cst["gT"])[:, None] * S + cst["Kr"].T @ u
    out = dict(o=o, ht=S)
    if dO is None:
        return out
    dq = np.zeros((L, D)); dk = np.zeros((L, D)); dv = np.zeros((L, D))
    dglog = np.zeros((L, D)); dblogit = np.zeros(L)
    dS = np.zeros((D, D)) if dht is None else dht.copy()
    for ch in reversed(chunks):
        r0, r1 = ch["r0"], ch["r1"]
        S0, u, E, T, P = ch["S0"], ch["u"], ch["E"], ch["T"], ch["P"]
        Kd, Ki, Kr, Qd, Araw = ch["Kd"], ch["Ki"], ch["Kr"], ch["Qd"], ch["Araw"]
        gc, gT = ch["gc"], ch["gT"]
        b = beta[r0:r1]
        do = dO[r0:r1]
        ch["dSC"] = dS.copy()
        # O = Qd S0 + lower(Qd Ki^T) u
        dP = np.tril(do @ u.T)
        dQd = do @ S0.T + dP @ Ki
        dKi = dP.T @ Qd
        # S_C = diag(e^gT) S0 + Kr^T u
        du = P.T @ do + Kr @ dS
        dKr = u @ dS.T
        # u = T Y, Y = diag(beta) E, T = (I + A)^-1
        dY = T.T @ du
        dA = -np.tril(dY @ u.T, -1)
        dbeta = (dY * E).sum(axis=1) + (dA * Araw).sum(axis=1)
        dKd = (b[:, None] * dA) @ Ki
        dKi = dKi + (b[:, None] * dA).T @ Kd
        dE = b[:, None] * dY
        dv[r0:r1] = dE
        dKd = dKd - dE @ S0.T
        dS0 = np.exp(gT)[:, None] * dS + Qd.T @ do - Kd.T @ dE
        # gate: stable dgc, per-chunk constant dgT, reverse cumsum
        eg, emg, egr = np.exp(gc), np.exp(-gc), np.exp(gT[None, :] - gc)
        knc, qnc = kn[r0:r1], qn[r0:r1]
        dgc = knc * (dKd * eg - dKi * emg - dKr * egr) + qnc * scale * dQd * eg
        dgT = np.exp(gT) * (dS * S0).sum(axis=1) + (dKr * Kr).sum(axis=0)
        dglog[r0:r1] = reverse_cumsum(dgc, axis=0) + dgT[None, :]
        dkn = dKd * eg + dKi * emg + dKr * egr
        dqn = scale * dQd * eg
        dq[r0:r1] = (dqn - qnc * (dqn * qnc).sum(axis=1, keepdims=True)) / nq[r0:r1]
        dk[r0:r1] = (dkn - knc * (dkn * knc).sum(axis=1, keepdims=True)) / nk[r0:r1]
        dblogit[r0:r1] = dbeta * b * (1.0 - b)
        dS = dS0
    out.update(dq=dq, dk=dk, dv=dv, dglog=dglog, dbeta=dblogit, dh0=dS)
    if keep:
        out["chunks"] = chunks
    return out


def gated_delta(q, k, v, glog, beta_logit, scale, cu_seqlens, h0=None, dO=None, dht=None,
                keep=False):
    """Same arguments and layout as ``oracle.gated_delta``; float64 numpy arrays.

    With ``keep=True`` also returns ``chunks[(global_chunk, head)]``; global chunk
    indices enumerate the chunks of sequence 0, then sequence 1, and so on.
    """
    q, k, v, glog, beta_logit = (np.asarray(x, dtype=np.float64) for x in (q, k, v, glog, beta_logit))
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T, H, D = q.shape
    N = len(cu) - 1
    res = {"o": np.zeros((T, H, D)), "ht": np.zeros((N, H, D, D))}
    if dO is not None:
        dO = np.asarray(dO, dtype=np.float64)
        for name in ("dq", "dk", "dv", "dglog"):
            res[name] = np.zeros((T, H, D))
        res["dbeta"] = np.zeros((T, H))
        res["dh0"] = np.zeros((N, H, D, D))
    chunks = {}
    cbase = 0
    for s in range(N):
        a, e = int(cu[s]), int(cu[s + 1])
        for h in range(H):
            r = pair(q[a:e, h], k[a:e, h], v[a:e, h], glog[a:e, h], beta_logit[a:e, h],
                     None if h0 is None else np.asarray(h0, np.float64)[s, h],
                     None if dO is None else dO[a:e, h],
                     None if dht is None else np.asarray(dht, np.float64)[s, h], scale, keep=keep)
            res["o"][a:e, h] = r["o"]
            res["ht"][s, h] = r["ht"]
            if dO is not None:
                for name in ("dq", "dk", "dv", "dglog", "dbeta"):
                    res[name][a:e, h] = r[name]
                res["dh0"][s, h] = r["dh0"]
            if keep:
                for i, ch in enumerate(r["chunks"]):
                    chunks[(cbase + i, h)] = ch
        cbase += (e - a + CHUNK - 1) // CHUNK
    if keep:
        res["chunks"] = chunks
    return res
