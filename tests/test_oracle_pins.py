"""Pins of the float64 oracle against things other than itself.

* central finite differences of the oracle's own forward (every gradient, both
  gate modes, varlen with two sequences, h0 and dht present, a sequence longer
  than the oracle's 64-token checkpoint block);
* closed forms: beta = 0 (the output is the decayed h0 only) and g = 0 with
  beta = 0 (the state never moves), forward and backward;
* the retrieval invariant of the delta rule with beta = 1 (the state returns
  v for the key just written), which fixes the order of decay and update;
* tangency of the L2-norm backward ("FlashKDA之backward（K1）", §3.3.2);
* varlen equals separate per-sequence runs; linearity in (dO, dht);
* the KDA gate values at points where softplus and sigmoid have closed forms
  (ln 2, ln 4, ln(4/3); 1/2, 3/4, 1/4) and the identities softplus(x) - softplus(-x)
  = x and sigmoid(z) + sigmoid(-z) = 1, alone and through the whole KDA path;
* the worked examples of the pages (tests/golden/);
* torch float64 autograd through a token recurrence written out independently (both gate
  kinds, both per-channel gate functions, grouped q / k heads, sequences crossing the
  oracle's checkpoint blocks);
* the chunk form at chunk lengths 16, 32 and 64 equals the token recurrence.
"""
import json
import os

import numpy as np
import pytest

from oracle import chunk_form, oracle
from tests.fdiff import causal_conv1d, central_grad

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(rng, lens, H, D, gate="gdn", h0=True, dht=True):
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    N = len(lens)
    c = dict(cu=cu, q=rng.standard_normal((T, H, D)), k=rng.standard_normal((T, H, D)),
             v=rng.standard_normal((T, H, D)), b=rng.standard_normal((T, H)),
             dO=rng.standard_normal((T, H, D)),
             h0=0.3 * rng.standard_normal((N, H, D, D)) if h0 else None,
             dht=0.3 * rng.standard_normal((N, H, D, D)) if dht else None, scale=D ** -0.5)
    if gate == "gdn":
        c["g"] = -np.logaddexp(0, rng.standard_normal((T, H)))
    elif gate == "glog":
        c["glog"] = -0.5 * np.logaddexp(0, rng.standard_normal((T, H, D)))
    else:
        c["g_raw"] = rng.standard_normal((T, H, D))
        c["A_log"] = rng.uniform(-1, 0, H)
        c["dt_bias"] = 0.1 * rng.standard_normal((H, D))
    return c


def _loss_gdn(c):
    r = oracle.gdn(c["q"], c["k"], c["v"], c["g"], c["b"], c["scale"], c["cu"], h0=c["h0"])
    L = (r["o"] * c["dO"]).sum()
    if c["dht"] is not None:
        L += (r["ht"] * c["dht"]).sum()
    return L


def _loss_kda(c, gate="softplus", gate_scale=None):
    r = oracle.kda(c["q"], c["k"], c["v"], c["g_raw"], c["A_log"], c["dt_bias"], c["b"],
                   c["scale"], c["cu"], h0=c["h0"], gate=gate, gate_scale=gate_scale)
    L = (r["o"] * c["dO"]).sum()
    if c["dht"] is not None:
        L += (r["ht"] * c["dht"]).sum()
    return L


def _check(fd, an, name):
    err = np.abs(fd - an).max()
    tol = 1e-7 + 1e-6 * np.abs(an).max()
    assert err <= tol, f"{name}: max |fd - analytic| = {err:.3e} > {tol:.3e}"


# ----------------------------------------------------------------------------
# FD machinery convention, pinned by the conv worked example (page 2)
# ----------------------------------------------------------------------------
def test_fd_convention_on_conv_worked_example():
    ex = json.load(open(os.path.join(GOLDEN, "causal_conv_backward_example.json")))
    x = np.array(ex["x"], float)
    w = np.array(ex["w"], float)
    bias = np.array([float(ex["bias"])])
    g = np.array(ex["g"], float)
    loss = lambda: float((g * causal_conv1d(x, w, bias[0])).sum())
    assert loss() == pytest.approx(ex["L"], abs=1e-9)
    np.testing.assert_allclose(central_grad(loss, x), ex["dx"], atol=1e-6)
    np.testing.assert_allclose(central_grad(loss, w), ex["dw"], atol=1e-6)
    np.testing.assert_allclose(central_grad(loss, bias), [ex["dbias"]], atol=1e-6)


def test_reverse_cumsum_worked_example():
    ex = json.load(open(os.path.join(GOLDEN, "reverse_cumsum_example.json")))
    np.testing.assert_array_equal(chunk_form.reverse_cumsum(np.array(ex["dgc"])),
                                  ex["suffix_sums"])


# ----------------------------------------------------------------------------
# finite differences of the whole backward
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("lens,D,sample", [((3, 5), 4, None), ((70, 81), 3, 160)])
def test_gdn_backward_matches_fd(lens, D, sample):
    rng = np.random.default_rng(11)
    c = _rand_case(rng, lens, 2, D, "gdn")
    an = oracle.gdn(c["q"], c["k"], c["v"], c["g"], c["b"], c["scale"], c["cu"], h0=c["h0"],
                    dO=c["dO"], dht=c["dht"])
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("b", "dbeta"),
                      ("h0", "dh0")):
        x = c[name]
        idx = None if sample is None else rng.choice(x.size, min(sample, x.size), replace=False)
        fd = central_grad(lambda: _loss_gdn(c), x, idx)
        ref = an[key].reshape(-1) if idx is None else an[key].reshape(-1)[idx]
        _check(fd, ref, name)


@pytest.mark.parametrize("gate,gate_scale", [("softplus", None), ("sigmoid", -2.0)])
def test_kda_backward_matches_fd(gate, gate_scale):
    rng = np.random.default_rng(12)
    c = _rand_case(rng, (4, 3), 2, 4, "kda")
    an = oracle.kda(c["q"], c["k"], c["v"], c["g_raw"], c["A_log"], c["dt_bias"], c["b"],
                    c["scale"], c["cu"], h0=c["h0"], dO=c["dO"], dht=c["dht"], gate=gate, gate_scale=gate_scale)
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g_raw", "dg_raw"),
                      ("A_log", "dA_log"), ("dt_bias", "ddt_bias"), ("b", "dbeta"),
                      ("h0", "dh0")):
        fd = central_grad(lambda: _loss_kda(c, gate, gate_scale), c[name])
        _check(fd, an[key].reshape(-1), name)


def test_sigmoid_gate_value_at_vanishing_slope():
    # with e^{A_log} -> 0 the sigmoid-bounded gate is ln2 * gate_scale * sigmoid(0) = ln2 * gate_scale / 2
    # for every token and channel, so the KDA path equals the plain recurrence with that constant
    # log gate, and no gradient reaches g_raw
    rng = np.random.default_rng(21)
    c = _rand_case(rng, (9, 5), 2, 4, "kda")
    c["A_log"] = np.full(2, -60.0)
    gs = -3.0
    a = oracle.kda(c["q"], c["k"], c["v"], c["g_raw"], c["A_log"], c["dt_bias"], c["b"], c["scale"], c["cu"],
                   h0=c["h0"], dO=c["dO"], dht=c["dht"], gate="sigmoid", gate_scale=gs)
    glog = np.full(c["q"].shape, np.log(2.0) * gs / 2)
    b = oracle.gated_delta(c["q"], c["k"], c["v"], glog, c["b"], c["scale"], c["cu"], h0=c["h0"], dO=c["dO"],
                           dht=c["dht"])
    for key in ("o", "ht", "dq", "dk", "dv", "dbeta", "dh0"):
        np.testing.assert_allclose(a[key], b[key], rtol=1e-12, atol=1e-12, err_msg=key)
    assert np.abs(a["dg_raw"]).max() < 1e-20
    # and the gate parameters' gradients are the chain-rule sums of the per-element terms
    np.testing.assert_allclose(a["ddt_bias"], a["dg_raw"].sum(axis=0), rtol=1e-12, atol=0)


# ----------------------------------------------------------------------------
# KDA gate values where they have a closed form (the finite-difference pins fix
# only the chain rule of whatever gate the oracle computes, not its value)
# ----------------------------------------------------------------------------
LN2, LN3 = np.log(2.0), np.log(3.0)


def _gate_inputs(x, A_log, dt_bias):
    """g_raw [1, H, D] such that g_raw + dt_bias = x (x [D]), for every head."""
    A_log = np.asarray(A_log, float)
    dt_bias = np.asarray(dt_bias, float)
    g_raw = (np.asarray(x, float)[None, :] - dt_bias)[None]
    return g_raw, A_log, dt_bias


def test_softplus_gate_values_at_closed_form_points():
    # softplus(0) = ln 2, softplus(ln 3) = ln 4, softplus(-ln 3) = ln(4/3); the gate is
    # -e^{A_log[h]} softplus(g_raw + dt_bias[h, d]); two heads with e^{A_log} = 1 and 2, and
    # dt_bias different per head and channel, so that a dropped or subtracted dt_bias, a
    # missing factor e^{A_log} or a wrong sign changes the value
    x = np.array([0.0, LN3, -LN3])
    g_raw, A_log, dt_bias = _gate_inputs(x, [0.0, LN2], [[0.25, -0.5, 1.0], [-0.75, 0.3, 0.1]])
    g = oracle.kda_gate(g_raw, A_log, dt_bias)
    sp = np.array([LN2, 2 * LN2, 2 * LN2 - LN3])
    expect = -np.array([1.0, 2.0])[:, None] * sp[None, :]
    np.testing.assert_allclose(g[0], expect, rtol=1e-14, atol=0)
    # far from zero: softplus(x) -> x for large x and -> e^{x} for very negative x
    g_raw, A_log, dt_bias = _gate_inputs([40.0, -40.0], [LN2], [[0.5, -0.5]])
    g = oracle.kda_gate(g_raw, A_log, dt_bias)[0, 0]
    assert g[0] == pytest.approx(-80.0, rel=1e-15)
    assert g[1] < 0 and g[1] == pytest.approx(-2 * np.exp(-40.0), rel=1e-12)
    # softplus(x) - softplus(-x) = x, so g(x) - g(-x) = -e^{A_log} x at any x
    rng = np.random.default_rng(51)
    xs = 3 * rng.standard_normal(16)
    gp = oracle.kda_gate(*_gate_inputs(xs, [-0.4], np.zeros((1, 16))))[0, 0]
    gm = oracle.kda_gate(*_gate_inputs(-xs, [-0.4], np.zeros((1, 16))))[0, 0]
    np.testing.assert_allclose(gp - gm, -np.exp(-0.4) * xs, rtol=1e-12, atol=1e-14)


def test_sigmoid_gate_values_at_closed_form_points():
    # sigmoid(0) = 1/2, sigmoid(ln 3) = 3/4, sigmoid(-ln 3) = 1/4; the natural-log gate is
    # ln2 gate_scale sigmoid(e^{A_log} (g_raw + dt_bias)); with e^{A_log} = 2, x = ln(3)/2
    # reaches the argument ln 3
    gs = -2.5
    x = np.array([0.0, LN3 / 2, -LN3 / 2])
    g_raw, A_log, dt_bias = _gate_inputs(x, [LN2], [[0.2, -0.7, 0.4]])
    g = oracle.kda_sigmoid_gate(g_raw, A_log, dt_bias, gs)[0, 0]
    np.testing.assert_allclose(g, LN2 * gs * np.array([0.5, 0.75, 0.25]), rtol=1e-14, atol=0)
    # sigmoid(z) + sigmoid(-z) = 1, so g(x) + g(-x) = ln2 gate_scale at any x
    rng = np.random.default_rng(52)
    xs = 2 * rng.standard_normal(16)
    gp = oracle.kda_sigmoid_gate(*_gate_inputs(xs, [0.3], np.zeros((1, 16))), gs)[0, 0]
    gm = oracle.kda_sigmoid_gate(*_gate_inputs(-xs, [0.3], np.zeros((1, 16))), gs)[0, 0]
    np.testing.assert_allclose(gp + gm, LN2 * gs, rtol=1e-13, atol=0)


@pytest.mark.parametrize("gate", ["softplus", "sigmoid"])
def test_kda_path_at_a_closed_form_gate(gate):
    # g_raw + dt_bias = x0 for every token and channel puts the whole KDA path on a constant
    # log gate known in closed form, so it must equal the plain recurrence with that gate;
    # its gradients are then the chain rule with the closed-form slope:
    #   softplus, e^{A_log} = 1, x0 = ln 3:  g = -ln 4,          dg/dx = -3/4,     dg/dA_log = g
    #   sigmoid,  e^{A_log} = 2, x0 = ln(3)/2: g = (3/4) ln2 gs,   dg/dx = 2 ln2 gs (3/16),
    #                                         dg/dA_log = x0 dg/dx
    rng = np.random.default_rng(53)
    c = _rand_case(rng, (7, 5), 2, 4, "kda")
    gs = -2.0
    if gate == "softplus":
        a, x0 = 1.0, LN3
        glog0, slope = -2 * LN2, -0.75
        dA_fac = glog0
    else:
        a, x0 = 2.0, LN3 / 2
        glog0, slope = 0.75 * LN2 * gs, a * LN2 * gs * 3.0 / 16.0
        dA_fac = x0 * slope
    T = c["q"].shape[0]
    A_log = np.full(2, np.log(a))
    g_raw = np.broadcast_to(x0 - c["dt_bias"][None], (T, 2, 4)).copy()
    r = oracle.kda(c["q"], c["k"], c["v"], g_raw, A_log, c["dt_bias"], c["b"], c["scale"], c["cu"],
                   h0=c["h0"], dO=c["dO"], dht=c["dht"], gate=gate, gate_scale=gs)
    glog = np.full(c["q"].shape, glog0)
    b = oracle.gated_delta(c["q"], c["k"], c["v"], glog, c["b"], c["scale"], c["cu"], h0=c["h0"], dO=c["dO"],
                           dht=c["dht"])
    for key in ("o", "ht", "dq", "dk", "dv", "dbeta", "dh0"):
        np.testing.assert_allclose(r[key], b[key], rtol=1e-12, atol=1e-13, err_msg=key)
    np.testing.assert_allclose(r["dg_raw"], slope * b["dglog"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["ddt_bias"], slope * b["dglog"].sum(axis=0), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["dA_log"], dA_fac * b["dglog"].sum(axis=(0, 2)), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("mode", ["gdn", "kda"])
def test_grouped_heads_backward_matches_fd(mode):
    # GQA: 2 q / k heads shared by 4 value heads (value head h reads q / k head h // 2)
    rng = np.random.default_rng(14)
    c = _rand_case(rng, (5, 3), 4, 3, mode)
    c["q"], c["k"] = c["q"][:, :2].copy(), c["k"][:, :2].copy()
    if mode == "gdn":
        an = oracle.gdn(c["q"], c["k"], c["v"], c["g"], c["b"], c["scale"], c["cu"], h0=c["h0"], dO=c["dO"],
                        dht=c["dht"])
        loss = lambda: _loss_gdn(c)
    else:
        an = oracle.kda(c["q"], c["k"], c["v"], c["g_raw"], c["A_log"], c["dt_bias"], c["b"], c["scale"],
                        c["cu"], h0=c["h0"], dO=c["dO"], dht=c["dht"])
        loss = lambda: _loss_kda(c)
    assert an["dq"].shape == c["q"].shape and an["dv"].shape == c["v"].shape
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("b", "dbeta"), ("h0", "dh0")):
        fd = central_grad(loss, c[name])
        _check(fd, an[key].reshape(-1), name)
    # the group's value heads see the same q / k: the output equals the run on expanded q / k
    ex = oracle.gated_delta(np.repeat(c["q"], 2, axis=1), np.repeat(c["k"], 2, axis=1), c["v"],
                            oracle.kda_gate(c["g_raw"], c["A_log"], c["dt_bias"]) if mode == "kda"
                            else np.repeat(c["g"][:, :, None], 3, axis=2), c["b"], c["scale"], c["cu"], h0=c["h0"])
    np.testing.assert_allclose(an["o"], ex["o"], rtol=1e-13, atol=1e-13)


def test_dht_gradient_is_the_final_state():
    # d L / d dht = ht, so FD in dht is the forward's final state; and the
    # gradient w.r.t. dO is o.  This pins which output each cotangent pairs with.
    rng = np.random.default_rng(13)
    c = _rand_case(rng, (5,), 1, 3, "gdn")
    r = oracle.gdn(c["q"], c["k"], c["v"], c["g"], c["b"], c["scale"], c["cu"], h0=c["h0"])
    _check(central_grad(lambda: _loss_gdn(c), c["dht"]), r["ht"].reshape(-1), "dht")
    _check(central_grad(lambda: _loss_gdn(c), c["dO"]), r["o"].reshape(-1), "dO")


# ----------------------------------------------------------------------------
# closed forms
# ----------------------------------------------------------------------------
def _l2n(x):
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + 1e-6)


@pytest.mark.parametrize("zero_gate", [False, True])
def test_beta_zero_closed_form(zero_gate):
    """beta = 0: S_t = diag(exp(cumsum g)) h0, so o_t = scale (Gamma_t h0)^T qn_t and
    dv = dk = 0, dh0 = sum_t scale Gamma_t qn_t dO_t^T + Gamma_T dht,
    dg_t[d] = sum_{s>=t} scale qn_s[d] (Gamma_s h0 dO_s)[d] + (Gamma_T h0 . dht)[d, :].sum()."""
    rng = np.random.default_rng(21)
    L_, D = 9, 5
    c = _rand_case(rng, (L_,), 1, D, "glog")
    if zero_gate:
        c["glog"][:] = 0.0
    b = np.full((L_, 1), -np.inf)
    r = oracle.gated_delta(c["q"], c["k"], c["v"], c["glog"], b, c["scale"], c["cu"], h0=c["h0"],
                           dO=c["dO"], dht=c["dht"])
    h0, dht, s = c["h0"][0, 0], c["dht"][0, 0], c["scale"]
    qn = _l2n(c["q"][:, 0])
    gam = np.exp(np.cumsum(c["glog"][:, 0], axis=0))          # [L, D]
    o = np.stack([s * (gam[t][:, None] * h0).T @ qn[t] for t in range(L_)])
    np.testing.assert_allclose(r["o"][:, 0], o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["ht"][0, 0], gam[-1][:, None] * h0, rtol=1e-12, atol=1e-13)
    assert np.abs(r["dv"]).max() == 0.0 and np.abs(r["dk"]).max() == 0.0
    assert np.abs(r["dbeta"]).max() == 0.0
    dh0 = sum(s * np.outer(gam[t] * qn[t], c["dO"][t, 0]) for t in range(L_)) + gam[-1][:, None] * dht
    np.testing.assert_allclose(r["dh0"][0, 0], dh0, rtol=1e-11, atol=1e-12)
    per_tok = np.stack([s * qn[t] * gam[t] * (h0 @ c["dO"][t, 0]) for t in range(L_)])
    dg = np.flip(np.cumsum(np.flip(per_tok, 0), 0), 0) + (gam[-1][:, None] * h0 * dht).sum(1)[None]
    np.testing.assert_allclose(r["dglog"][:, 0], dg, rtol=1e-10, atol=1e-12)
    dqn = np.stack([s * (gam[t][:, None] * h0) @ c["dO"][t, 0] for t in range(L_)])
    nq = np.sqrt((c["q"][:, 0] ** 2).sum(-1, keepdims=True) + 1e-6)
    dq = (dqn - qn * (dqn * qn).sum(-1, keepdims=True)) / nq
    np.testing.assert_allclose(r["dq"][:, 0], dq, rtol=1e-11, atol=1e-12)


def test_retrieval_invariant_fixes_update_order():
    """With beta = 1 and |kn| = 1 the delta rule overwrites the value stored
    under the key just written: S_t^T kn_t = v_t.  With q = k the output is then
    scale * v_t.  Holds for per-channel gates only with the decay applied before
    the update."""
    rng = np.random.default_rng(22)
    c = _rand_case(rng, (12,), 2, 6, "glog")
    b = np.full((12, 2), np.inf)
    r = oracle.gated_delta(c["k"], c["k"], c["v"], c["glog"], b, 1.0, c["cu"], h0=c["h0"])
    # |kn|^2 = |k|^2 / (|k|^2 + 1e-6): the identity holds to ~1e-6 relative
    np.testing.assert_allclose(r["o"], c["v"], rtol=2e-5, atol=2e-5)


def test_single_token_from_zero_state():
    """T = 1, h0 = 0: S_1 = beta kn v^T, so o = scale * beta * <kn, qn> v."""
    rng = np.random.default_rng(23)
    c = _rand_case(rng, (1,), 3, 7, "glog", h0=False, dht=False)
    r = oracle.gated_delta(c["q"], c["k"], c["v"], c["glog"], c["b"], c["scale"], c["cu"])
    beta = 1 / (1 + np.exp(-c["b"][0]))
    dot = (_l2n(c["k"][0]) * _l2n(c["q"][0])).sum(-1)
    np.testing.assert_allclose(r["o"][0], (c["scale"] * beta * dot)[:, None] * c["v"][0],
                               rtol=1e-12, atol=1e-14)


# ----------------------------------------------------------------------------
# invariants and consistency
# ----------------------------------------------------------------------------
def test_l2_backward_tangency():
    rng = np.random.default_rng(31)
    c = _rand_case(rng, (20,), 2, 8, "gdn")
    r = oracle.gdn(c["q"], c["k"], c["v"], c["g"], c["b"], c["scale"], c["cu"], h0=c["h0"],
                   dO=c["dO"], dht=c["dht"])
    for x, dx in ((c["q"], r["dq"]), (c["k"], r["dk"])):
        dots = (x * dx).sum(-1)
        scale = np.linalg.norm(x, axis=-1) * np.linalg.norm(dx, axis=-1)
        assert np.all(np.abs(dots) <= 1e-6 * scale + 1e-14)


def test_varlen_equals_separate_runs():
    rng = np.random.default_rng(32)
    lens = (7, 1, 66, 0, 13)
    c = _rand_case(rng, lens, 2, 4, "gdn")
    r = oracle.gdn(c["q"], c["k"], c["v"], c["g"], c["b"], c["scale"], c["cu"], h0=c["h0"],
                   dO=c["dO"], dht=c["dht"])
    cu = c["cu"]
    for s in range(len(lens)):
        a, e = cu[s], cu[s + 1]
        rs = oracle.gdn(c["q"][a:e], c["k"][a:e], c["v"][a:e], c["g"][a:e], c["b"][a:e],
                        c["scale"], np.array([0, e - a]), h0=c["h0"][s:s + 1],
                        dO=c["dO"][a:e], dht=c["dht"][s:s + 1])
        for key in ("o", "dq", "dk", "dv", "dg", "dbeta"):
            np.testing.assert_array_equal(r[key][a:e], rs[key])
        for key in ("ht", "dh0"):
            np.testing.assert_array_equal(r[key][s], rs[key][0])
    # an empty sequence passes the state gradient straight through
    np.testing.assert_array_equal(r["dh0"][3], c["dht"][3])
    np.testing.assert_array_equal(r["ht"][3], c["h0"][3])


def test_backward_is_linear_in_cotangents():
    rng = np.random.default_rng(33)
    c = _rand_case(rng, (10, 6), 2, 4, "gdn")
    args = (c["q"], c["k"], c["v"], c["g"], c["b"], c["scale"], c["cu"])
    dO2 = rng.standard_normal(c["dO"].shape)
    dht2 = rng.standard_normal(c["dht"].shape)
    r1 = oracle.gdn(*args, h0=c["h0"], dO=c["dO"], dht=c["dht"])
    r2 = oracle.gdn(*args, h0=c["h0"], dO=dO2, dht=dht2)
    r3 = oracle.gdn(*args, h0=c["h0"], dO=2 * c["dO"] - 3 * dO2, dht=2 * c["dht"] - 3 * dht2)
    for key in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        np.testing.assert_allclose(r3[key], 2 * r1[key] - 3 * r2[key], rtol=1e-10, atol=1e-11)


def test_gdn_is_kda_path_with_channel_constant_gate():
    rng = np.random.default_rng(34)
    c = _rand_case(rng, (9,), 2, 5, "gdn")
    r = oracle.gdn(c["q"], c["k"], c["v"], c["g"], c["b"], c["scale"], c["cu"], h0=c["h0"],
                   dO=c["dO"], dht=c["dht"])
    glog = np.repeat(c["g"][:, :, None], 5, axis=2)
    rk = oracle.gated_delta(c["q"], c["k"], c["v"], glog, c["b"], c["scale"], c["cu"],
                            h0=c["h0"], dO=c["dO"], dht=c["dht"])
    np.testing.assert_allclose(r["dg"], rk["dglog"].sum(2), rtol=1e-13, atol=1e-14)


# ----------------------------------------------------------------------------
# the chunk-form restatement agrees with the token recurrence
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("gate", ["gdn", "glog"])
def test_chunk_form_matches_token_oracle(gate):
    rng = np.random.default_rng(41)
    c = _rand_case(rng, (150, 64, 1), 2, 8, gate)
    glog = np.repeat(c["g"][:, :, None], 8, 2) if gate == "gdn" else c["glog"]
    a = oracle.gated_delta(c["q"], c["k"], c["v"], glog, c["b"], c["scale"], c["cu"], h0=c["h0"],
                           dO=c["dO"], dht=c["dht"])
    b = chunk_form.gated_delta(c["q"], c["k"], c["v"], glog, c["b"], c["scale"], c["cu"],
                               h0=c["h0"], dO=c["dO"], dht=c["dht"])
    for key in ("o", "ht", "dq", "dk", "dv", "dglog", "dbeta", "dh0"):
        np.testing.assert_allclose(b[key], a[key], rtol=1e-8, atol=1e-9 * np.abs(a[key]).max(),
                                   err_msg=key)


# ----------------------------------------------------------------------------
# torch float64 autograd through an independently written token recurrence
# ----------------------------------------------------------------------------
def _autograd_case(c, mode, gate_scale, Hk):
    """The loss sum(o . dO) + sum(ht . dht) of the recurrence written out token by token in
    torch float64 (decay, then the delta update, then the read-out), differentiated by autograd.
    Returns the leaf gradients by input name."""
    import torch
    t = {n: torch.tensor(c[n], dtype=torch.float64, requires_grad=True)
         for n in ("q", "k", "v", "b", "h0") + (("g",) if mode == "gdn" else ("g_raw", "A_log", "dt_bias"))}
    if mode == "gdn":
        glog = t["g"][:, :, None].expand_as(t["v"])
    elif mode == "softplus":
        glog = -torch.exp(t["A_log"])[None, :, None] * torch.nn.functional.softplus(t["g_raw"] + t["dt_bias"][None])
    else:
        glog = np.log(2.0) * gate_scale * torch.sigmoid(torch.exp(t["A_log"])[None, :, None] *
                                                        (t["g_raw"] + t["dt_bias"][None]))
    dO, dht = torch.tensor(c["dO"]), torch.tensor(c["dht"])
    H = c["v"].shape[1]
    r = H // Hk
    loss = torch.zeros((), dtype=torch.float64)
    for s in range(len(c["cu"]) - 1):
        for h in range(H):
            S = t["h0"][s, h]
            for i in range(int(c["cu"][s]), int(c["cu"][s + 1])):
                qv, kv = t["q"][i, h // r], t["k"][i, h // r]
                qn = qv / torch.sqrt((qv * qv).sum() + 1e-6)
                kn = kv / torch.sqrt((kv * kv).sum() + 1e-6)
                beta = torch.sigmoid(t["b"][i, h])
                S = torch.exp(glog[i, h])[:, None] * S
                S = S - beta * torch.outer(kn, kn @ S) + beta * torch.outer(kn, t["v"][i, h])
                loss = loss + ((c["scale"] * (S.T @ qn)) * dO[i, h]).sum()
            loss = loss + (S * dht[s, h]).sum()
    loss.backward()
    return {n: x.grad.numpy() for n, x in t.items()}


@pytest.mark.parametrize("mode,Hk", [("gdn", 2), ("softplus", 2), ("sigmoid", 2), ("softplus", 1)])
def test_backward_matches_torch_autograd(mode, Hk):
    """Every gradient of the hand-derived reverse mode equals autograd's on 150 + 70 tokens
    (both sequences cross the oracle's 64-token checkpoint blocks), with h0 and dht, for
    the scalar gate, both per-channel gate functions, and two value heads sharing one q / k
    head."""
    rng = np.random.default_rng(61)
    c = _rand_case(rng, (150, 70), 2, 6, "gdn" if mode == "gdn" else "kda")
    if Hk < 2:
        c["q"], c["k"] = c["q"][:, :Hk].copy(), c["k"][:, :Hk].copy()
    gs = -2.0 if mode == "sigmoid" else None
    if mode == "gdn":
        an = oracle.gdn(c["q"], c["k"], c["v"], c["g"], c["b"], c["scale"], c["cu"], h0=c["h0"],
                        dO=c["dO"], dht=c["dht"])
        pairs = (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("b", "dbeta"), ("h0", "dh0"))
    else:
        an = oracle.kda(c["q"], c["k"], c["v"], c["g_raw"], c["A_log"], c["dt_bias"], c["b"], c["scale"],
                        c["cu"], h0=c["h0"], dO=c["dO"], dht=c["dht"], gate=mode, gate_scale=gs)
        pairs = (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g_raw", "dg_raw"), ("A_log", "dA_log"),
                 ("dt_bias", "ddt_bias"), ("b", "dbeta"), ("h0", "dh0"))
    ag = _autograd_case(c, mode, gs, Hk)
    for name, key in pairs:
        np.testing.assert_allclose(an[key], ag[name], rtol=1e-9, atol=1e-11 * np.abs(ag[name]).max(),
                                   err_msg=name)


# ----------------------------------------------------------------------------
# the chunk algebra does not depend on the chunk length
# ----------------------------------------------------------------------------
def test_chunk_form_is_independent_of_chunk_length():
    """The chunk form at C = 16, 32 and 64 (the kernels' length) gives the token recurrence's
    outputs and gradients on one sequence of 150 tokens: every C leaves a ragged last chunk
    and puts chunk boundaries in different places."""
    rng = np.random.default_rng(62)
    c = _rand_case(rng, (150,), 1, 8, "glog")
    ref = oracle.gated_delta(c["q"], c["k"], c["v"], c["glog"], c["b"], c["scale"], c["cu"], h0=c["h0"],
                             dO=c["dO"], dht=c["dht"])
    for C in (16, 32, 64):
        got = chunk_form.pair(c["q"][:, 0], c["k"][:, 0], c["v"][:, 0], c["glog"][:, 0], c["b"][:, 0],
                              c["h0"][0, 0], c["dO"][:, 0], c["dht"][0, 0], c["scale"], C=C)
        for key, want in (("o", ref["o"][:, 0]), ("ht", ref["ht"][0, 0]), ("dq", ref["dq"][:, 0]),
                          ("dk", ref["dk"][:, 0]), ("dv", ref["dv"][:, 0]), ("dglog", ref["dglog"][:, 0]),
                          ("dbeta", ref["dbeta"][:, 0]), ("dh0", ref["dh0"][0, 0])):
            np.testing.assert_allclose(got[key], want, rtol=1e-8, atol=1e-9 * np.abs(want).max(),
                                       err_msg="%s at C = %d" % (key, C))
