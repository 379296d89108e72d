"""Rounding-site replay of the chunk-parallel backward, float64 (one sequence, one head).

TEST INFRASTRUCTURE ONLY: a diagnostic for the precision design of the CUDA kernels.
Nothing on the product path imports it, and it shares no code with the CUDA path.

It replays the chunk algebra the main backward kernels use (the tiles referenced to the
middle of each chunk's gate range, the products G1..G11 and the element-wise assembly of
"FlashKDA之backward（K1）" §3.2-§3.3 and §5) in float64, and rounds to bf16 exactly the
operand sites named in ``sites``; everything else stays float64.  With no site rounded it
reproduces the oracle's gradients (a test checks this).  Sites:

    S      the chunk-start state S0 as a product operand      dS   the state gradient dS_C
    derX   kd of X = kd S0                                     derR kr of du and dkr
    derA   kd', ki', qd' of [A; P] = [kd'; qd'] ki'^T           derG ki', qd', kd' of G10 / G11
    A, P   the in-chunk matrices as operands                   T    the inverse T
    uF     beta E = beta (V - X)                               uG   u
    du     du (and dY)                                         dP   dP and beta dA
    chain  the state recurrences run as the state kernel runs them, i.e. all three of
           chainW  the chunk tiles W, kr (and U) in bf16
           chainS  the state (or state gradient) as the first product's operand in bf16
           chainY  the second product's operand (U - X, or Y = kr dS) in bf16

The per-channel (KDA) kernel keeps uF, uG, dP, derG and P as bf16 pairs, which this replay
treats as exact ("precise mode"); the scalar-gate kernel rounds every site once.
``python -m oracle.precision_sites`` prints the error of dg and of the per-head dA_log sum
over 16 heads for both models and with each remaining site made exact.  ``replay`` also returns
dh0 and ht, which only the chain sites touch.
"""
import numpy as np

from . import chunk_form, oracle

ALL_SITES = frozenset({"S", "dS", "derX", "derR", "derA", "derG", "A", "P", "T", "uF", "uG", "du", "dP", "chain"})
PRECISE_MODE = ALL_SITES - {"uF", "uG", "dP", "derG", "P"}


def bf16(x):
    """Round-to-nearest-even to bf16, returned as float64."""
    x = np.asarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def replay(q, k, v, glog, blogit, dO, scale, sites, C=64, h0=None, dht=None):
    """q, k, v, glog, dO: [L, D]; blogit [L] (bf16-representable inputs); h0, dht [D, D] or
    None (zero).  Returns the gradients dq, dk, dv and dglog (the per-channel log-gate
    gradient), dh0 and the forward's final state ht of one sequence, computed with the named
    sites rounded to bf16."""
    R = lambda name, x: bf16(x) if name in sites else x
    cW, cS, cY = (("chain" in sites) or (n in sites) for n in ("chainW", "chainS", "chainY"))
    rW = lambda x: bf16(x) if cW else x
    rS = lambda x: bf16(x) if cS else x
    rY = lambda x: bf16(x) if cY else x
    L, D = q.shape
    qn, nq = chunk_form._l2n(q)
    kn, nk = chunk_form._l2n(k)
    beta = chunk_form._sigmoid(blogit)
    spans = [(r0, min(r0 + C, L)) for r0 in range(0, L, C)]
    # forward state chain (S_C = e^{gT} S0 + kr^T (U - W S0)): the chunk-start states
    S = np.zeros((D, D)) if h0 is None else np.array(h0, dtype=np.float64)
    starts = []
    for r0, r1 in spans:
        c = chunk_form._chunk_consts(qn[r0:r1], kn[r0:r1], glog[r0:r1], beta[r0:r1], scale)
        starts.append(S.copy())
        U = c["T"] @ (beta[r0:r1, None] * v[r0:r1])
        S = np.exp(c["gT"])[:, None] * S + rW(c["Kr"]).T @ rY(rW(U) - rW(c["W"]) @ rS(S))
    ht = S.copy()  # the final state
    # backward state-gradient chain (dS0 = e^{gT} dS_C + R^T dO - W^T (kr dS_C), R = qd - P W
    # carried exactly, as the kernel's bf16 pair): dS at each chunk's end
    dS = np.zeros((D, D)) if dht is None else np.array(dht, dtype=np.float64)
    ends = [None] * len(spans)
    for i in range(len(spans) - 1, -1, -1):
        r0, r1 = spans[i]
        c = chunk_form._chunk_consts(qn[r0:r1], kn[r0:r1], glog[r0:r1], beta[r0:r1], scale)
        ends[i] = dS.copy()
        Rm = c["Qd"] - c["P"] @ c["W"]
        dS = np.exp(c["gT"])[:, None] * dS + Rm.T @ dO[r0:r1] - rW(c["W"]).T @ rY(rW(c["Kr"]) @ rS(dS))
    dg = np.zeros((L, D))
    dqn = np.zeros((L, D))
    dkn = np.zeros((L, D))
    dv = np.zeros((L, D))
    for (r0, r1), S0, dSc in zip(spans, starts, ends):
        sl = slice(r0, r1)
        bt = beta[sl]
        gc = np.cumsum(glog[sl], axis=0)
        gT = gc[-1]
        ref = 0.5 * (gc.max(axis=0) + gc.min(axis=0))
        eg, egp, egi, egr = np.exp(gc), np.exp(gc - ref), np.exp(ref - gc), np.exp(gT - gc)
        S0r, dSr = R("S", S0), R("dS", dSc)
        Kd, Kr = R("derX", kn[sl] * eg), R("derR", kn[sl] * egr)
        Kdp, Kip, Qdp = R("derA", kn[sl] * egp), R("derA", kn[sl] * egi), R("derA", scale * qn[sl] * egp)
        KdpG, KipG, QdpG = R("derG", kn[sl] * egp), R("derG", kn[sl] * egi), R("derG", scale * qn[sl] * egp)
        A = np.tril(bt[:, None] * (Kdp @ Kip.T), -1)
        P = R("P", np.tril(Qdp @ Kip.T))
        T = R("T", np.linalg.inv(np.eye(r1 - r0) + A))
        bE = R("uF", bt[:, None] * (v[sl] - Kd @ S0r))
        u = R("uG", T @ bE)
        dQd = dO[sl] @ S0r.T                       # state part of dqd
        du = R("du", P.T @ dO[sl] + Kr @ dSr)
        dY = R("du", T.T @ du)
        Z = dY @ S0r.T                             # dkd from E: -beta Z
        dKr = u @ dSr.T
        dP = R("dP", np.tril(dO[sl] @ u.T))
        bdA = R("dP", bt[:, None] * -np.tril(dY @ u.T, -1))
        dQdp, dKdp = dP @ KipG, bdA @ KipG
        dKip = dP.T @ QdpG + bdA.T @ KdpG
        dgc = (qn[sl] * scale * eg) * dQd + QdpG * dQdp + (kn[sl] * eg) * (-bt[:, None] * Z) \
            + KdpG * dKdp - KipG * dKip - (kn[sl] * egr) * dKr
        dgT = np.exp(gT) * (dSc * S0).sum(axis=1) + ((kn[sl] * egr) * dKr).sum(axis=0)
        dg[sl] = chunk_form.reverse_cumsum(dgc, 0) + dgT[None]
        dv[sl] = bt[:, None] * dY
        dqn[sl] = scale * eg * dQd + scale * egp * dQdp
        dkn[sl] = eg * (-bt[:, None] * Z) + egp * dKdp + egi * dKip + egr * dKr
    dq = (dqn - qn * (dqn * qn).sum(axis=1, keepdims=True)) / nq
    dk = (dkn - kn * (dkn * kn).sum(axis=1, keepdims=True)) / nk
    return dict(dq=dq, dk=dk, dv=dv, dglog=dg, dh0=dS, ht=ht)


def kda_head(seed, L=512, D=128):
    """One head of the KDA workload's distributions (bf16 inputs, softplus gate)."""
    rng = np.random.default_rng(seed)
    q, k, v, dO = (bf16(rng.standard_normal((L, D))) for _ in range(4))
    b = bf16(rng.standard_normal(L))
    raw = bf16(rng.standard_normal((L, D)))
    A_log = rng.uniform(-1.0, 0.0)
    dt = 0.1 * rng.standard_normal(D)
    glog = -np.exp(A_log) * oracle.softplus(raw + dt)
    return q, k, v, glog, b, dO, D ** -0.5


def errors(sites, heads=16, L=512):
    """Relative L2 error of dglog over all heads, and of the per-head dA_log sums
    (sum over tokens and channels of dglog * glog) as one vector over the heads."""
    num = den = 0.0
    da, da_ref = [], []
    for h in range(heads):
        q, k, v, glog, b, dO, scale = kda_head(h, L)
        ref = replay(q, k, v, glog, b, dO, scale, frozenset())
        got = replay(q, k, v, glog, b, dO, scale, sites)
        num += np.sum((got["dglog"] - ref["dglog"]) ** 2)
        den += np.sum(ref["dglog"] ** 2)
        da.append(np.sum(got["dglog"] * glog))
        da_ref.append(np.sum(ref["dglog"] * glog))
    da, da_ref = np.array(da), np.array(da_ref)
    return float(np.sqrt(num / den)), float(np.linalg.norm(da - da_ref) / np.linalg.norm(da_ref))


if __name__ == "__main__":
    for name, s in (("every site once in bf16 (scalar-gate kernel)", ALL_SITES),
                    ("precise mode (per-channel kernel)", PRECISE_MODE)):
        print("%-48s dg %.2e  dA_log %.2e" % ((name,) + errors(s)), flush=True)
    for site in sorted(PRECISE_MODE):
        print("precise mode, %-6s exact                       dg %.2e  dA_log %.2e"
              % ((site,) + errors(PRECISE_MODE - {site})), flush=True)
