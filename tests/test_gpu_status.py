"""Device-side status reporting, on the GPU, with no fault: a states buffer written
for another variant or shape is refused by the backward, and a bounded wait that runs
out (the test hook holds one CTA on a barrier that nothing arrives on) leaves a
status bit and a usable context behind."""
import pytest
import torch

import chunked_gated_delta_bwd_gb300 as gdr
from chunked_gated_delta_bwd_gb300 import inputs
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from chunked_gated_delta_bwd_gb300 import build
    build.build()


def _states(mode, x, **kw):
    d = H.to_gpu(x)
    if mode == "gdn":
        return gdr.gdr_fwd_states(d["q"], d["k"], d["v"], d["g"], d["beta_logit"], h0=d["h0"],
                                  cu_seqlens=d["cu_seqlens"], scale=d["scale"], **kw)
    return gdr.gdr_fwd_states(d["q"], d["k"], d["v"], None, d["beta_logit"], h0=d["h0"],
                              cu_seqlens=d["cu_seqlens"], scale=d["scale"], gate="kda", g_raw=d["g_raw"],
                              A_log=d["A_log"], dt_bias=d["dt_bias"], **kw)


def _status_after(x, states):
    ws = H._workspace(H.to_gpu(x), x, None)
    d = H.to_gpu(x)
    N = d["cu_seqlens"].numel() - 1
    common = dict(h0=d["h0"], dht=d["dht"], cu_seqlens=d["cu_seqlens"], num_seqs=N, scale=d["scale"],
                  states=states, workspace=ws)
    if x["mode"] == "gdn":
        gdr.gdr_bwd(d["q"], d["k"], d["v"], d["g"], d["beta_logit"], d["dO"], **common)
    else:
        gdr.kda_bwd(d["q"], d["k"], d["v"], d["g_raw"], d["A_log"], d["dt_bias"], d["beta_logit"], d["dO"],
                    kda_gate=x["kda_gate"], gate_scale=x["gate_scale"], **common)
    torch.cuda.synchronize()
    return gdr.workspace_status(ws)


@pytest.mark.parametrize("dim", [64, 128])
def test_states_of_another_variant_or_shape_are_refused(dim):
    lens = [200, 77]
    xg = inputs.custom("gdn", lens, heads=2, dim=dim, seed=120, with_h0=True, with_dht=True)
    xk = inputs.custom("kda", lens, heads=2, dim=dim, seed=120, with_h0=True, with_dht=True)
    st_g, st_k = _states("gdn", xg), _states("kda", xk)
    # the matching buffers are accepted
    assert _status_after(xg, st_g) == 0
    assert _status_after(xk, st_k) == 0
    # a GDN buffer given to the KDA backward and the other way round
    assert _status_after(xk, st_g) & gdr.api.GDR_DEV_STATES_MISMATCH
    assert _status_after(xg, st_k) & gdr.api.GDR_DEV_STATES_MISMATCH
    # the sigmoid-bounded gate is another variant of KDA
    xs = dict(xk, kda_gate="sigmoid", gate_scale=-2.0)
    assert _status_after(xs, st_k) & gdr.api.GDR_DEV_STATES_MISMATCH
    # states computed without h0 for a call with h0
    st_noh0 = _states("gdn", dict(xg, h0=None))
    assert _status_after(xg, st_noh0) & gdr.api.GDR_DEV_STATES_MISMATCH
    # another shape (a larger buffer: the same lengths plus a third sequence)
    x3 = inputs.custom("gdn", lens + [64], heads=2, dim=dim, seed=121, with_h0=True, with_dht=True)
    assert _status_after(xg, _states("gdn", x3)) & gdr.api.GDR_DEV_STATES_MISMATCH


def test_timed_out_wait_sets_the_status_and_leaves_the_context_usable():
    x = inputs.custom("gdn", [700, 300, 64], heads=4, dim=128, seed=122, with_h0=True, with_dht=True)
    d = H.to_gpu(x)
    ws = H._workspace(d, x, None)
    gdr.api.test_stall_next_call(0)
    gdr.gdr_bwd(d["q"], d["k"], d["v"], d["g"], d["beta_logit"], d["dO"], h0=d["h0"], dht=d["dht"],
                cu_seqlens=d["cu_seqlens"], num_seqs=3, scale=d["scale"], workspace=ws)
    torch.cuda.synchronize()  # the call returned and its work completed
    assert gdr.workspace_status(ws) & gdr.api.GDR_DEV_TIMEOUT
    # the hook is one-shot: the next call on the same device runs in full and passes parity
    gpu = H.run_gpu(x, workspace=ws)
    assert gdr.workspace_status(ws) == 0
    print(H.assert_parity(H.compare(gpu, H.run_oracle(x), x), "after timeout"))


@pytest.mark.parametrize("mode", ["gdn", "kda"])
def test_backward_captures_into_a_cuda_graph(mode):
    # every step of a call is a kernel or memset on the caller's stream and nothing waits on
    # the host, so a call can be captured once and replayed: the replay equals an eager call
    x = inputs.custom(mode, [700, 300, 64], heads=4, dim=128, seed=123, with_h0=True, with_dht=True)
    d = H.to_gpu(x)
    ws = H._workspace(d, x, None)
    N = d["cu_seqlens"].numel() - 1
    common = dict(h0=d["h0"], dht=d["dht"], cu_seqlens=d["cu_seqlens"], num_seqs=N, scale=d["scale"], workspace=ws)
    T, Hh, D = d["v"].shape
    out = gdr.alloc_outputs(T, Hh, D, N, mode)

    def call():
        if mode == "gdn":
            gdr.gdr_bwd(d["q"], d["k"], d["v"], d["g"], d["beta_logit"], d["dO"], out=out, **common)
        else:
            gdr.kda_bwd(d["q"], d["k"], d["v"], d["g_raw"], d["A_log"], d["dt_bias"], d["beta_logit"], d["dO"],
                        out=out, **common)

    call()  # eager, also the warm-up before capture
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in out.items()}
    for v in out.values():
        v.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for v in out.values():
        v.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert gdr.workspace_status(ws) == 0
    for k, v in out.items():
        if k in ("dA_log", "ddt_bias"):  # fp32 atomics: the order of the additions may differ
            torch.testing.assert_close(v, eager[k], rtol=1e-5, atol=1e-6)
        else:
            assert torch.equal(v, eager[k]), k


def test_profile_counts_kernels_not_sections():
    """The instrumentation counts kernels: a dense backward with time-parallel state
    passing launches the prep, two chain phases and the boundary kernel, and the main
    kernel (five), recorded as three timed sections."""
    from chunked_gated_delta_bwd_gb300 import api
    x = inputs.make(inputs.Case("prof", "gdn", 1, 4096, 2, 128, seed=3, with_h0=True, with_dht=True))
    d = H.to_gpu(x)
    gdr.gdr_bwd(d["q"], d["k"], d["v"], d["g"], d["beta_logit"], d["dO"], h0=d["h0"], dht=d["dht"],
                num_seqs=1, scale=d["scale"])
    torch.cuda.synchronize()
    api.profile_begin(8)
    gdr.gdr_bwd(d["q"], d["k"], d["v"], d["g"], d["beta_logit"], d["dO"], h0=d["h0"], dht=d["dht"],
                num_seqs=1, scale=d["scale"])
    prof = api.profile_end()
    counts = {k: n for k, (ms, n) in prof.items() if n}
    # one sequence of 64 chunks over 2 heads: two segments per (sequence, head)
    assert counts == {"prep": 1, "states": 3, "main": 1}, counts
    assert all(prof[k][0] > 0 for k in counts)


def test_two_streams_overlap_with_own_workspaces():
    """Two backward calls with their own workspaces, enqueued on two streams so that their
    kernels can run at the same time (each grid is smaller than the GPU), give the same
    results as the same calls run one after the other: the library keeps no state between
    calls outside the workspace.  Everything but the atomically summed dA_log / ddt_bias is
    bitwise reproducible."""
    xa = inputs.custom("gdn", [700, 300], heads=4, dim=128, seed=141, with_h0=True, with_dht=True)
    xb = inputs.custom("kda", [600, 380], heads=4, dim=128, seed=142, with_h0=True, with_dht=True)

    def launch(x, d, ws):
        common = dict(h0=d["h0"], dht=d["dht"], cu_seqlens=d["cu_seqlens"], num_seqs=d["cu_seqlens"].numel() - 1,
                      scale=d["scale"], workspace=ws)
        if x["mode"] == "gdn":
            return gdr.gdr_bwd(d["q"], d["k"], d["v"], d["g"], d["beta_logit"], d["dO"], **common)
        return gdr.kda_bwd(d["q"], d["k"], d["v"], d["g_raw"], d["A_log"], d["dt_bias"], d["beta_logit"], d["dO"],
                           kda_gate=x["kda_gate"], gate_scale=x["gate_scale"], **common)

    da, db = H.to_gpu(xa), H.to_gpu(xb)
    wsa, wsb = H._workspace(da, xa, None), H._workspace(db, xb, None)
    ref_a = {k: v.clone() for k, v in launch(xa, da, wsa).items()}
    ref_b = {k: v.clone() for k, v in launch(xb, db, wsb).items()}
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s1):
        got_a = launch(xa, da, wsa)
    with torch.cuda.stream(s2):
        got_b = launch(xb, db, wsb)
    torch.cuda.synchronize()
    assert gdr.workspace_status(wsa) == 0 and gdr.workspace_status(wsb) == 0
    for ref, got in ((ref_a, got_a), (ref_b, got_b)):
        for k in ref:
            if k in ("dA_log", "ddt_bias"):
                torch.testing.assert_close(got[k], ref[k], rtol=1e-5, atol=1e-6)
            else:
                assert torch.equal(got[k], ref[k]), k
