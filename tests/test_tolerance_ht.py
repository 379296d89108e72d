"""Where the forward final-state tolerance (TOL_HT in tests/helpers.py) comes from.

The final state ht is returned in fp32, but the kernels build it from bf16 chunk
tiles: per chunk  S_C = e^{gT} S0 + kr^T (U - W S0),  with W, U and kr stored as
bf16 tiles, S0 rounded to bf16 as the operand of W S0, and U - W S0 rounded to bf16
as the operand of the update product (fp32 accumulation everywhere).  This test
replays that chain in float64 on the oracle's chunk algebra, rounding exactly those
sites to bf16, and checks that the error it predicts for ht sits in the class the
tolerance assumes: each of the roundings of U, kr and U - W S0 costs about 1.6e-3
relative (2^-9 unit roundoff, averaged over a tile), ~2.3e-3 together, at any
length, because the workloads' gates forget a chunk's start state within the chunk.
TOL_HT = 5e-3 is about twice that.  (The backward's dh0 is built from R = qd - P W
carried as a bf16 pair, which is why it meets 1e-3.)
"""
import numpy as np
import pytest
import torch

from chunked_gated_delta_bwd_gb300 import inputs
from oracle import chunk_form, oracle
from tests import helpers as H


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).to(torch.float64).numpy()


def _chain(q, k, v, glog, blogit, h0, scale, sites):
    """Chunk-form forward state chain of one (sequence, head), rounding `sites` to bf16."""
    L = q.shape[0]
    qn, _ = chunk_form._l2n(q)
    kn, _ = chunk_form._l2n(k)
    beta = chunk_form._sigmoid(blogit)
    S = h0.copy()
    for r0 in range(0, L, 64):
        r1 = min(r0 + 64, L)
        c = chunk_form._chunk_consts(qn[r0:r1], kn[r0:r1], glog[r0:r1], beta[r0:r1], scale)
        W, Kr = c["W"], c["Kr"]
        U = c["T"] @ (beta[r0:r1, None] * v[r0:r1])
        if "W" in sites:
            W = _bf16(W)
        if "U" in sites:
            U = _bf16(U)
        if "Kr" in sites:
            Kr = _bf16(Kr)
        Y = U - W @ (_bf16(S) if "S" in sites else S)
        if "Y" in sites:
            Y = _bf16(Y)
        S = np.exp(c["gT"])[:, None] * S + Kr.T @ Y
    return S


@pytest.mark.parametrize("mode", ["gdn", "kda"])
def test_ht_tolerance_covers_the_kernels_rounding_sites(mode):
    x = inputs.custom(mode, [640], heads=1, dim=128, seed=5, with_h0=True)
    f = lambda n: x[n].to(torch.float64).numpy()
    q, k, v = f("q")[:, 0], f("k")[:, 0], f("v")[:, 0]
    D = q.shape[1]
    if mode == "gdn":
        glog = np.repeat(f("g")[:, 0:1], D, axis=1)
    else:
        glog = oracle.kda_gate(f("g_raw"), f("A_log"), f("dt_bias"))[:, 0]
    b, h0 = f("beta_logit")[:, 0], f("h0")[0, 0]
    exact = _chain(q, k, v, glog, b, h0, x["scale"], set())
    # the exact chain is the oracle's final state (the token recurrence)
    ref = oracle.gated_delta(q[:, None], k[:, None], v[:, None], glog[:, None], b[:, None], x["scale"],
                             np.array([0, q.shape[0]]), h0=h0[None, None])["ht"][0, 0]
    assert H.rel_l2(exact, ref) < 1e-10
    err = {s: H.rel_l2(_chain(q, k, v, glog, b, h0, x["scale"], {s}), exact) for s in ("U", "Kr", "Y")}
    for s, e in err.items():
        assert 1e-3 < e < 2.5e-3, (s, e)  # one bf16 rounding of a tile: the 2^-9 class
    every = H.rel_l2(_chain(q, k, v, glog, b, h0, x["scale"], {"W", "U", "Kr", "S", "Y"}), exact)
    assert 1.5e-3 < every < 3.5e-3, every
    assert H.TOL_HT >= 1.4 * every
