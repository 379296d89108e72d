"""The rounding-site replay behind the kernels' precision design (oracle/precision_sites.py):
with nothing rounded it is the oracle's backward, and rounding the kernels' sites gives the
error classes the GPU parity tests measure: every site once in bf16 (the scalar-gate kernel)
leaves the log-gate gradient at the 2^-9 class (~3-4e-3), while the per-channel kernel's
precise mode (bf16 pairs at beta E, u, dP / beta dA and the tiles of the gradient products)
brings it several times lower, the class the per-head dA_log / ddt_bias sums need."""
import numpy as np

from oracle import oracle, precision_sites as ps
from tests import helpers as H


def test_unrounded_replay_is_the_oracle_backward():
    q, k, v, glog, b, dO, scale = ps.kda_head(7, L=200, D=16)
    rng = np.random.default_rng(8)
    h0, dht = 0.1 * rng.standard_normal((16, 16)), 0.1 * rng.standard_normal((16, 16))
    got = ps.replay(q, k, v, glog, b, dO, scale, frozenset(), h0=h0, dht=dht)
    ref = oracle.gated_delta(q[:, None], k[:, None], v[:, None], glog[:, None], b[:, None], scale,
                             np.array([0, 200]), h0=h0[None, None], dO=dO[:, None], dht=dht[None, None])
    for name in ("dq", "dk", "dv", "dglog"):
        assert H.rel_l2(got[name], ref[name][:, 0]) < 1e-9, name
    assert H.rel_l2(got["dh0"], ref["dh0"][0, 0]) < 1e-9


def test_precise_mode_lowers_the_gate_gradient_error():
    plain, _ = ps.errors(ps.ALL_SITES, heads=2, L=256)
    precise, _ = ps.errors(ps.PRECISE_MODE, heads=2, L=256)
    assert 1.5e-3 < plain < 8e-3, plain
    assert precise < plain / 4, (precise, plain)


def _scalar_gate_head(seed, L, D, decay):
    """One head of the scalar-gate workload's distributions (bf16 inputs), its log gate
    -softplus(a), a ~ N(0, 1), on every channel; or, without decay, a log gate of 0."""
    rng = np.random.default_rng(seed)
    q, k, v, dO = (ps.bf16(rng.standard_normal((L, D))) for _ in range(4))
    b = ps.bf16(rng.standard_normal(L))
    g = -oracle.softplus(rng.standard_normal(L)) if decay else np.zeros(L)
    h0, dht = 0.1 * rng.standard_normal((D, D)), 0.1 * rng.standard_normal((D, D))
    return q, k, v, np.repeat(g[:, None], D, axis=1), b, dO, D ** -0.5, h0, dht


def test_dh0_error_without_decay():
    """dh0 depends only on the state-gradient chain.  Without decay every bf16 operand of that
    chain -- the tiles W and kr, the state gradient in the first product, Y = kr dS_C in the
    second -- leaves more than 1e-3 on dh0 by itself, ~2e-3 together (the bound of the
    no-decay GPU case is twice that); with the workloads' decay the same roundings stay far
    below 1e-3, because each chunk's contribution to dh0 fades."""
    def err(sites, decay):
        q, k, v, glog, b, dO, scale, h0, dht = _scalar_gate_head(11, 1024, 128, decay)
        exact = ps.replay(q, k, v, glog, b, dO, scale, frozenset(), h0=h0, dht=dht)["dh0"]
        got = ps.replay(q, k, v, glog, b, dO, scale, frozenset(sites), h0=h0, dht=dht)["dh0"]
        return H.rel_l2(got, exact)
    for site in ("chainW", "chainS", "chainY"):
        e = err({site}, decay=False)
        assert 8e-4 < e < 2.5e-3, (site, e)
    together = err({"chain"}, decay=False)
    assert 1.5e-3 < together < H.TOL_DH0_NO_DECAY / 2, together
    assert err({"chain"}, decay=True) < H.TOL_FP32 / 2


def test_ht_error_without_decay():
    """The forward's final state without decay: the chain's bf16 operands leave ~3.9e-3 on
    ht together (the bound of the no-decay GPU case is twice that), against ~2.3e-3 with the
    workloads' decay (within TOL_HT)."""
    def err(decay):
        q, k, v, glog, b, dO, scale, h0, dht = _scalar_gate_head(12, 1024, 128, decay)
        exact = ps.replay(q, k, v, glog, b, dO, scale, frozenset(), h0=h0, dht=dht)["ht"]
        got = ps.replay(q, k, v, glog, b, dO, scale, frozenset({"chain"}), h0=h0, dht=dht)["ht"]
        return H.rel_l2(got, exact)
    e = err(False)
    assert 3e-3 < e <= H.TOL_HT_NO_DECAY / 2, e
    assert err(True) < H.TOL_HT, "the decayed workloads' bound"
