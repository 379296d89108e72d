"""GPU parity of the causal conv1d (+ SiLU) backward (gdr_conv1d_bwd) against the float64
oracle (oracle/conv.py) on the same seeded inputs.  Tolerances: relative L2 <= 2e-2 for dx
(bf16 output, like the other bf16 gradients) and <= 1e-3 for dweight / dbias (fp32 sums
over tokens)."""
import numpy as np
import pytest
import torch

from chunked_gated_delta_bwd_gb300 import inputs
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from chunked_gated_delta_bwd_gb300 import build
    build.build()


def _run(c, dense=None):
    import chunked_gated_delta_bwd_gb300 as gdr
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in c.items()}
    if dense:
        B, T = dense
        out = gdr.conv1d_bwd(d["x"].reshape(B, T, -1), d["weight"], d["bias"], d["dy"].reshape(B, T, -1),
                             silu=c["silu"])
        out["dx"] = out["dx"].reshape(B * T, -1)
    else:
        out = gdr.conv1d_bwd(d["x"], d["weight"], d["bias"], d["dy"], cu_seqlens=d["cu_seqlens"], silu=c["silu"])
    torch.cuda.synchronize()
    return {k: (None if v is None else v.cpu()) for k, v in out.items()}


def _check(c, gpu, channels=None, label=""):
    from oracle import conv
    sel = (lambda t: t) if channels is None else (lambda t: t[..., channels])
    x, dy = sel(H.f64(c["x"])), sel(H.f64(c["dy"]))
    w = H.f64(c["weight"])[channels] if channels is not None else H.f64(c["weight"])
    b = None if c["bias"] is None else (H.f64(c["bias"])[channels] if channels is not None else H.f64(c["bias"]))
    ref = conv.conv1d_bwd(x, w, b, dy, c["cu_seqlens"].numpy(), c["silu"])
    res = {"dx": (H.rel_l2(sel(H.f64(gpu["dx"])), ref["dx"]), H.TOL_BF16)}
    gw = H.f64(gpu["dweight"])
    res["dweight"] = (H.rel_l2(gw[channels] if channels is not None else gw, ref["dw"]), H.TOL_FP32)
    if b is not None:
        gb = H.f64(gpu["dbias"])
        res["dbias"] = (H.rel_l2(gb[channels] if channels is not None else gb, ref["dbias"]), H.TOL_FP32)
    print(label, H.assert_parity(res, label))


@pytest.mark.parametrize("width", [1, 2, 3, 4])
@pytest.mark.parametrize("silu", [False, True])
def test_varlen_ragged(width, silu):
    # empty and one-token sequences, tile boundaries inside and between sequences, a
    # channel count that leaves a partial block
    c = inputs.conv_case([1, 0, 127, 129, 5, 0, 260, 64], 516, width, seed=200 + width, silu=silu)
    _check(c, _run(c), label="conv_k%d_silu%d" % (width, silu))


def test_no_bias_dense_layout():
    c = inputs.conv_case([300, 300], 256, 4, seed=210, with_bias=False)
    gpu = _run(c, dense=(2, 300))
    assert gpu["dbias"] is None
    _check(c, gpu, label="conv_dense_nobias")


def test_worked_example_exactly():
    # the page's example (x = [1, 2, 3, 4], w = [2, 3, 5], bias 1, no activation, g = [1, 2, 3, 4]:
    # dx = [17, 27, 27, 20], dw = [11, 20, 30], dbias = 10) on four identical channels; every
    # value is an integer that bf16 holds exactly
    import json, os
    import chunked_gated_delta_bwd_gb300 as gdr
    ex = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "causal_conv_backward_example.json")))
    x = torch.tensor(ex["x"], dtype=torch.bfloat16)[:, None].repeat(1, 4).cuda()
    g = torch.tensor(ex["g"], dtype=torch.bfloat16)[:, None].repeat(1, 4).cuda()
    w = torch.tensor(ex["w"], dtype=torch.float32)[None].repeat(4, 1).cuda()
    b = torch.full((4,), float(ex["bias"]), dtype=torch.float32).cuda()
    out = gdr.conv1d_bwd(x, w, b, g, silu=False)
    assert out["dx"][:, 0].float().tolist() == ex["dx"]
    assert out["dweight"][0].tolist() == ex["dw"]
    assert out["dbias"].tolist() == [ex["dbias"]] * 4


def test_full_size_sampled_channels():
    # the q, k, v channels of the H16 D128 layer (C = 3 * 16 * 128) over 32768 tokens, K = 4,
    # SiLU, bias; 64 channels checked against the oracle (channels are independent)
    c = inputs.conv_case([32768], 3 * 16 * 128, 4, seed=220)
    gpu = _run(c)
    chans = list(np.linspace(0, 3 * 16 * 128 - 1, 64).astype(int))
    _check(c, gpu, channels=chans, label="conv_full")
