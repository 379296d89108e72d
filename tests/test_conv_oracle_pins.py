"""Pins of the float64 causal conv1d backward (oracle/conv.py) against things other than
itself: the worked example of "第三章 反向传播的完整推导" (tests/golden), central differences
of its forward (with and without SiLU, two packed sequences, K from 1 to 4), the SiLU slope
1/2 at z = 0 the page points out, and packed sequences equal separate runs."""
import json
import os

import numpy as np
import pytest

from oracle import conv
from tests.fdiff import central_grad

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_worked_example():
    ex = json.load(open(os.path.join(GOLDEN, "causal_conv_backward_example.json")))
    x = np.array(ex["x"], dtype=np.float64)[:, None]
    w = np.array(ex["w"], dtype=np.float64)[None, :]
    b = np.array([ex["bias"]], dtype=np.float64)
    g = np.array(ex["g"], dtype=np.float64)[:, None]
    cu = np.array([0, len(ex["x"])])
    y, _ = conv.conv1d_fwd(x, w, b, cu, silu=False)
    assert (g * y).sum() == ex["L"]
    r = conv.conv1d_bwd(x, w, b, g, cu, silu=False)
    assert r["dx"][:, 0].tolist() == ex["dx"]
    assert r["dw"][0].tolist() == ex["dw"]
    assert r["dbias"].tolist() == [ex["dbias"]]


@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("silu", [False, True])
def test_backward_matches_fd(K, silu):
    rng = np.random.default_rng(30 + K)
    cu = np.array([0, 5, 7])  # two packed sequences of 5 and 2 tokens
    C = 3
    x = rng.standard_normal((7, C))
    w = rng.standard_normal((C, K))
    b = rng.standard_normal(C)
    dy = rng.standard_normal((7, C))
    an = conv.conv1d_bwd(x, w, b, dy, cu, silu)

    def loss():
        return (dy * conv.conv1d_fwd(x, w, b, cu, silu)[0]).sum()
    for name, arr, key in (("x", x, "dx"), ("w", w, "dw"), ("bias", b, "dbias")):
        fd = central_grad(loss, arr)
        ref = an[key].reshape(-1)
        assert np.abs(fd - ref).max() <= 1e-7 + 1e-6 * np.abs(ref).max(), name


def test_silu_slope_at_zero_is_half():
    # at z = 0 the SiLU derivative is 1/2 (not the 1 of the identity): x = 0 and no bias
    # give z = 0 everywhere, so delta = dy / 2
    rng = np.random.default_rng(41)
    cu = np.array([0, 6])
    dy = rng.standard_normal((6, 2))
    r = conv.conv1d_bwd(np.zeros((6, 2)), rng.standard_normal((2, 3)), np.zeros(2), dy, cu, silu=True)
    np.testing.assert_allclose(r["dbias"], dy.sum(axis=0) / 2, rtol=0, atol=1e-15)


def test_packed_sequences_equal_separate_runs():
    rng = np.random.default_rng(42)
    x = rng.standard_normal((9, 4))
    dy = rng.standard_normal((9, 4))
    w = rng.standard_normal((4, 4))
    b = rng.standard_normal(4)
    packed = conv.conv1d_bwd(x, w, b, dy, np.array([0, 2, 2, 9]), silu=True)
    a = conv.conv1d_bwd(x[:2], w, b, dy[:2], np.array([0, 2]), silu=True)
    c = conv.conv1d_bwd(x[2:], w, b, dy[2:], np.array([0, 7]), silu=True)
    np.testing.assert_allclose(packed["dx"], np.concatenate([a["dx"], c["dx"]]), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(packed["dw"], a["dw"] + c["dw"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(packed["dbias"], a["dbias"] + c["dbias"], rtol=1e-13, atol=1e-13)
