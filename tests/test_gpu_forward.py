"""GPU parity of the forward (gdr_fwd / kda_fwd: output o and final state ht) against
the float64 oracle's forward on the same seeded inputs.  Tolerances: relative L2
<= 2e-2 for o (a bf16 output, like the gradients) and <= 5e-3 for ht (fp32, built
from bf16 chunk tiles; the derivation is beside TOL_HT in tests/helpers.py)."""
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


def _check(x, heads=None, label="", tol_ht=H.TOL_HT):
    gpu = H.run_gpu_fwd(x)
    ref = H.run_oracle_fwd(x, heads)
    print(label, H.assert_parity(H.compare_fwd(gpu, ref, heads, x=x, tol_ht=tol_ht), label))
    return gpu


def test_gdn_tiny_config():
    _check(inputs.make(inputs.CASES["gdn_tiny"]), label="fwd_gdn_tiny")


@pytest.mark.parametrize("mode", ["gdn", "kda", "kda_sigmoid"])
@pytest.mark.parametrize("dim", [64, 128])
def test_varlen_ragged_with_h0(mode, dim):
    gate = "sigmoid" if mode == "kda_sigmoid" else "softplus"
    x = inputs.custom(mode.split("_")[0], [1, 63, 64, 65, 200, 130], heads=3, dim=dim, seed=111, with_h0=True,
                      kda_gate=gate, gate_scale=-2.0)
    _check(x, label="fwd_%s_ragged_d%d" % (mode, dim))


@pytest.mark.parametrize("dim", [64, 128])
def test_grouped_qk_heads(dim):
    x = inputs.custom("gdn", [1, 63, 200, 130], heads=4, dim=dim, seed=117, with_h0=True, k_heads=2)
    _check(x, label="fwd_gqa_d%d" % dim)


@pytest.mark.parametrize("dim", [64, 128])
def test_empty_and_single_token_sequences(dim):
    x = inputs.custom("kda", [0, 1, 0, 64, 1], heads=2, dim=dim, seed=112, with_h0=True)
    gpu = _check(x, label="fwd_empty_d%d" % dim)
    # an empty sequence leaves its initial state unchanged
    torch.testing.assert_close(gpu["ht"][0], x["h0"][0], rtol=0, atol=0)
    torch.testing.assert_close(gpu["ht"][2], x["h0"][2], rtol=0, atol=0)


@pytest.mark.parametrize("mode,lengths,dim", [("gdn", [200, 77], 128), ("kda", [200, 77], 128),
                                             ("gdn", [16000, 64], 128), ("kda", [16000, 64], 128),
                                             ("gdn", [200, 77], 64), ("kda", [200, 77], 64)])
def test_forward_states_feed_the_backward(mode, lengths, dim):
    # the chunk-start states kept by the forward equal gdr_fwd_states's, and a backward from
    # them equals the backward that recomputes them (the long case runs the state chains as
    # segments: forward-only, backward-only and both directions)
    import chunked_gated_delta_bwd_gb300 as gdr
    x = inputs.custom(mode, lengths, heads=2, dim=dim, seed=113, with_h0=True, with_dht=True)
    d = H.to_gpu(x)
    kw = dict(h0=d["h0"], cu_seqlens=d["cu_seqlens"], scale=d["scale"])
    if mode == "gdn":
        ref_states = gdr.gdr_fwd_states(d["q"], d["k"], d["v"], d["g"], d["beta_logit"], **kw)
    else:
        ref_states = gdr.gdr_fwd_states(d["q"], d["k"], d["v"], None, d["beta_logit"], gate="kda",
                                        g_raw=d["g_raw"], A_log=d["A_log"], dt_bias=d["dt_bias"], **kw)
    fwd = H.run_gpu_fwd(x, states=True)
    # chunks are numbered sequence after sequence; the buffer's tail past the last chunk
    # (its size is a bound for varlen) is not written; head_dim 64 keeps the states of the
    # channels zero-padded to 128
    used = 256 + sum((n + 63) // 64 for n in lengths) * 2 * 128 * 128 * 2  # header + the states
    assert torch.equal(fwd["states"][:used], ref_states.cpu()[:used])
    a = H.run_gpu(x, states=fwd["states"].cuda())
    b = H.run_gpu(x)
    for k in a:
        if k in ("dA_log", "ddt_bias"):
            torch.testing.assert_close(a[k], b[k], rtol=1e-5, atol=1e-6)
        else:
            assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("mode", ["gdn", "kda"])
def test_segmented_forward_varlen(mode):
    # few (sequence, head) pairs and a long sequence: the forward's state chains run as
    # time-parallel segments (3 here); the 64-token sequence leaves two segments empty
    x = inputs.custom(mode, [16000, 64], heads=2, dim=128, seed=115, with_h0=True)
    _check(x, label="fwd_segments_%s" % mode)


@pytest.mark.parametrize("mode", ["gdn", "kda"])
def test_forward_eight_segments(mode):
    # one sequence of 256 chunks over 2 heads: the forward's chains run as the most segments
    # (8), whose boundary composition takes 7 steps
    x = inputs.custom(mode, [16384], heads=2, dim=128, seed=132, with_h0=True)
    _check(x, label="fwd_eight_segments_%s" % mode)


def test_forward_without_decay():
    # degenerate gate: g = 0 everywhere (the ungated delta rule); nothing is forgotten, so
    # every bf16 operand of the forward chain counts in ht: held to the no-decay bound derived
    # beside TOL_HT_NO_DECAY (o keeps its usual bound)
    x = inputs.custom("gdn", [3072, 130], heads=2, dim=128, seed=133, with_h0=True)
    x["g"] = torch.zeros_like(x["g"])
    _check(x, label="fwd_no_decay", tol_ht=H.TOL_HT_NO_DECAY)


def test_forward_is_deterministic():
    x = inputs.custom("gdn", [500, 3], heads=4, dim=128, seed=114, with_h0=True)
    a, b = H.run_gpu_fwd(x), H.run_gpu_fwd(x)
    for k in a:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("name", ["gdn_b2_h16_t4k", "kda_b1_h16_t8k", "gdn_varlen_h32", "gdn_h16_t32k",
                                  "kda_h16_t32k"])
def test_full_size_all_heads(name):
    _check(inputs.make(inputs.CASES[name]), label="fwd_" + name)


@pytest.mark.parametrize("seed", range(12))
def test_random_shapes(seed):
    # the backward's seeded random shapes (tests/test_gpu_parity.py), through the forward:
    # gate kinds, head dims, head grouping, packed sequences of 0-1500 tokens, h0 or not
    from tests.test_gpu_parity import _random_case
    x, label = _random_case(seed)
    _check(x, label="fwd_" + label)
