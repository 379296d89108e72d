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
    got = ps.replay(q, k, v, glog, b, dO, scale, frozenset())
    ref = oracle.gated_delta(q[:, None], k[:, None], v[:, None], glog[:, None], b[:, None], scale,
                             np.array([0, 200]), dO=dO[:, None])
    for name in ("dq", "dk", "dv", "dglog"):
        assert H.rel_l2(got[name], ref[name][:, 0]) < 1e-9, name


def test_precise_mode_lowers_the_gate_gradient_error():
    plain, _ = ps.errors(ps.ALL_SITES, heads=2, L=256)
    precise, _ = ps.errors(ps.PRECISE_MODE, heads=2, L=256)
    assert 1.5e-3 < plain < 8e-3, plain
    assert precise < plain / 4, (precise, plain)
