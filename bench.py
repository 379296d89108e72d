"""Benchmark of the chunked gated delta-rule backward on GB300.

One step = one GDN backward and one KDA backward over the long-sequence
workload (B=1, H=16, T=32768, D=128, chunk 64), each computing every gradient
(dq, dk, dv, dg / dg_raw, dbeta, dh0, dA_log, ddt_bias) from the inputs alone
(the chunk states are recomputed inside the call).  Inputs are seeded,
synthetic, resident in HBM before timing, and larger than L2 (about 0.6 GB per
variant), so no L2 flush is needed between steps.

Prints one JSON line (rank 0).  Under torchrun each rank runs its own replica
on its own GPU (weak scaling, no data-path collective); the barrier and the
max over ranks are the only cross-rank operations.

``--impl reference`` times the float64 CPU oracle instead (a bounded sample of
the same workload on the host cores) on the same metric.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from chunked_gated_delta_bwd_gb300 import inputs  # noqa: E402

WORKLOAD = "gdn+kda bwd, B=1 H=16 T=32768 D=128 chunk=64"
METRIC = "GDN+KDA bwd Mtokens/s at H16 T32k D128"
UNIT = "Mtokens/s"
CASE_G, CASE_K = inputs.CASES["gdn_h16_t32k"], inputs.CASES["kda_h16_t32k"]
TOKENS_PER_STEP = CASE_G.seq_len * CASE_G.num_seqs + CASE_K.seq_len * CASE_K.num_seqs

# Algorithmic figures of the backward per token-head (D = 128, C = 64), the method's own:
#   flops: the 18 products of a chunk (7 of C*D*D, 11 of C*C*D) = 14 D^2 + 22 C D = 409 600;
#   bytes with the chunk-start states saved in bf16: q, k, v, dO (4 * 2D) + gate + beta +
#   S0 (2 D^2 / C) read, dq, dk, dv (3 * 2D) + dgate + dbeta written = 2316 (GDN: fp32 scalar gate
#   and gradient) or 2820 (KDA: bf16 per-channel raw gate and gradient, 2D each); plus 4 D^2 per
#   (sequence, head) for each of h0, dht and dh0.
D_, C_ = 128, 64
BWD_FLOP_PER_TH = 14 * D_ * D_ + 22 * C_ * D_
BWD_BYTES_PER_TH = {"gdn": 4 * 2 * D_ + 4 + 2 + 2 * D_ * D_ // C_ + 3 * 2 * D_ + 4 + 2,
                    "kda": 4 * 2 * D_ + 2 * D_ + 2 + 2 * D_ * D_ // C_ + 3 * 2 * D_ + 2 * D_ + 2}
assert BWD_FLOP_PER_TH == 409600 and BWD_BYTES_PER_TH == {"gdn": 2316, "kda": 2820}
# What this design's main kernel moves per token-head besides, for the design-byte figure
# reported beside: the dS_C and T tiles it reads from the state and prep kernels' output, and
# (KDA) A and the P pair from the prep kernel.
MAIN_DESIGN_EXTRA_PER_TH = {"gdn": 2 * D_ * D_ // C_ + 2 * C_, "kda": 2 * D_ * D_ // C_ + 2 * C_ + 3 * 2 * C_}
# Forward output kernel (o = R S0 + P U per chunk) per token-head: reads S0 (2 D^2 / C), R^T and
# U^T (2 D each), P (2 C); writes o (2 D).  Flops: 2 (D^2 + C D).
OUT_BYTES_PER_TH = 2 * D_ * D_ // C_ + 2 * D_ + 2 * D_ + 2 * C_ + 2 * D_
OUT_FLOP_PER_TH = 2 * (D_ * D_ + C_ * D_)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(x, world):
    """Max of a float over ranks (identity for a single process)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi (every 10 ms, time-stamped); the
    summary keeps the samples taken inside the timed region [t0, t1] (host wall-clock)."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "10"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self, t0=None, t1=None):
        import datetime
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[2]), float(f[3]), f[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 is not None and t0 - 0.005 <= r[0] <= t1 + 0.005]
        use = inside if inside else rows
        sm = [r[1] for r in use]
        reasons = {n for r in use for n, v in zip(names, r[3]) if v.lower() == "active"}
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max((r[2] for r in use), default=None),
                "reasons": sorted(reasons), "samples": len(sm),
                "window": "timed region" if inside else "whole sampler run"}


# ---------------------------------------------------------------------------
# oracle (CPU) timing: bounded sample of the same workload
# ---------------------------------------------------------------------------
def oracle_sample_seconds(tokens):
    """Times the float64 oracle on the first `tokens` tokens of both variants, all heads."""
    from oracle import oracle
    import numpy as np
    t0 = time.perf_counter()
    for case in (CASE_G, CASE_K):
        x = inputs.make(inputs.Case(case.name + "_sample", case.mode, 1, tokens, case.heads, case.dim,
                                    case.seed, with_h0=case.with_h0, with_dht=case.with_dht))
        f = lambda t: None if t is None else t.to(torch.float64).numpy()
        cu = np.array([0, tokens])
        if case.mode == "gdn":
            oracle.gdn(f(x["q"]), f(x["k"]), f(x["v"]), f(x["g"]), f(x["beta_logit"]), x["scale"], cu,
                       h0=f(x["h0"]), dO=f(x["dO"]), dht=f(x["dht"]))
        else:
            oracle.kda(f(x["q"]), f(x["k"]), f(x["v"]), f(x["g_raw"]), f(x["A_log"]), f(x["dt_bias"]),
                       f(x["beta_logit"]), x["scale"], cu, h0=f(x["h0"]), dO=f(x["dO"]), dht=f(x["dht"]))
    return time.perf_counter() - t0


def cpu_baseline(tokens):
    from oracle import build as obuild, oracle
    obuild.build()
    secs = oracle_sample_seconds(tokens)
    cores = min(oracle.max_threads(), CASE_G.heads)
    return {"value": 2 * tokens / secs / 1e6, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "float64 oracle, first %d tokens of the GDN and the KDA sequence, all %d heads "
                      "(forward + backward); %.2f s on %d host threads (host has %d cores)"
                      % (tokens, CASE_G.heads, secs, cores, os.cpu_count() or 0)}


def run_reference(args):
    rank, world, _ = dist_info()
    if world > 1 and rank != 0:
        return
    tokens = args.ref_tokens
    from oracle import build as obuild, oracle
    obuild.build()
    for _ in range(args.warmup):
        oracle_sample_seconds(tokens)
    secs = [oracle_sample_seconds(tokens) for _ in range(args.steps)]
    total = sum(secs)
    value = 2 * tokens * args.steps / total / 1e6
    cores = min(oracle.max_threads(), CASE_G.heads)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD + " (oracle: first %d tokens per variant per step)" % tokens},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "float64 oracle, first %d tokens of the GDN and the KDA sequence, "
                                       "all %d heads, per step" % (tokens, CASE_G.heads)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def main_gpu(args):
    import chunked_gated_delta_bwd_gb300 as gdr
    from chunked_gated_delta_bwd_gb300 import api, build
    rank, world, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    build.build()

    xg = inputs.make(CASE_G)
    xk = inputs.make(CASE_K)
    dev = lambda x: {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    G, K = dev(xg), dev(xk)
    T, Hh, D = G["q"].shape
    N = 1
    ws_g = torch.empty(gdr.workspace_bytes(gdr.make_shape(N, T, Hh, D)), dtype=torch.uint8, device="cuda")
    ws_k = torch.empty_like(ws_g)
    out_g = gdr.alloc_outputs(T, Hh, D, N, "gdn")
    out_k = gdr.alloc_outputs(T, Hh, D, N, "kda")

    def step_g(A=G, o=out_g):
        gdr.gdr_bwd(A["q"], A["k"], A["v"], A["g"], A["beta_logit"], A["dO"], h0=A["h0"], dht=A["dht"],
                    num_seqs=N, scale=A["scale"], workspace=ws_g, out=o)

    def step_k(A=K, o=out_k):
        gdr.kda_bwd(A["q"], A["k"], A["v"], A["g_raw"], A["A_log"], A["dt_bias"], A["beta_logit"], A["dO"],
                    h0=A["h0"], dht=A["dht"], num_seqs=N, scale=A["scale"], workspace=ws_k, out=o)

    def step():
        step_g()
        step_k()

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for w in (ws_g, ws_k):
        st = gdr.workspace_status(w)
        if st:
            raise RuntimeError("device status %d raised by the warm-up steps" % st)

    # ---- timed region (device-resident inputs) ----
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        # untimed steps while the sampler starts (about half a second), then the timed steps
        t_settle = time.time()
        while time.time() - t_settle < 0.5:
            step()
            torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        api.profile_begin(16 * args.steps)
        t_clk0 = time.time()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        t_clk1 = time.time()
    barrier(world)
    prof = api.profile_end()
    ms_local = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(ms_local, world)
    value = world * TOKENS_PER_STEP / (ms * 1e-3) / 1e6
    launches = sum(n for _, n in prof.values())

    # per-variant step times (informational, separate short loops)
    per_variant = {}

    def time_loop(name, fn, n=max(3, args.steps // 2)):
        torch.cuda.synchronize()
        api.profile_begin(8 * n)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        per_variant[name] = {k: round(v[0] / n, 4) for k, v in api.profile_end().items() if v[1]}
        return a.elapsed_time(b) / n
    ms_g, ms_k = time_loop("gdn", step_g), time_loop("kda", step_k)

    # ---- the forward (o, ht) on the same inputs: informational, one loop per variant ----
    fwd_kernels = {}

    def fwd_loop(name, fn, n=max(3, args.steps // 2)):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        api.profile_begin(8 * n)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        fwd_kernels[name] = {k: round(v[0] / n, 4) for k, v in api.profile_end().items() if v[1]}
        return a.elapsed_time(b) / n
    fms_g = fwd_loop("gdn", lambda A=G: gdr.gdr_fwd(A["q"], A["k"], A["v"], A["g"], A["beta_logit"], h0=A["h0"],
                                                   num_seqs=N, scale=A["scale"], workspace=ws_g))
    fms_k = fwd_loop("kda", lambda A=K: gdr.kda_fwd(A["q"], A["k"], A["v"], A["g_raw"], A["A_log"], A["dt_bias"],
                                                   A["beta_logit"], h0=A["h0"], num_seqs=N, scale=A["scale"],
                                                   workspace=ws_k))
    # the backward from saved chunk states (the forward kept them): no forward recurrence
    saved = {}
    st_g = gdr.gdr_fwd_states(G["q"], G["k"], G["v"], G["g"], G["beta_logit"], h0=G["h0"], num_seqs=N,
                              scale=G["scale"], workspace=ws_g)
    st_k = gdr.gdr_fwd_states(K["q"], K["k"], K["v"], None, K["beta_logit"], h0=K["h0"], num_seqs=N,
                              scale=K["scale"], workspace=ws_k, gate="kda", g_raw=K["g_raw"], A_log=K["A_log"],
                              dt_bias=K["dt_bias"])
    saved_kernels = {}

    def saved_loop(name, fn, n=max(3, args.steps // 2)):
        fn()
        torch.cuda.synchronize()
        api.profile_begin(8 * n)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        saved_kernels[name] = {k: round(v[0] / n, 4) for k, v in api.profile_end().items() if v[1]}
        saved[name] = a.elapsed_time(b) / n
    saved_loop("gdn", lambda A=G, o=out_g: gdr.gdr_bwd(A["q"], A["k"], A["v"], A["g"], A["beta_logit"], A["dO"],
                                                       h0=A["h0"], dht=A["dht"], num_seqs=N, scale=A["scale"],
                                                       states=st_g, workspace=ws_g, out=o))
    saved_loop("kda", lambda A=K, o=out_k: gdr.kda_bwd(A["q"], A["k"], A["v"], A["g_raw"], A["A_log"],
                                                       A["dt_bias"], A["beta_logit"], A["dO"], h0=A["h0"],
                                                       dht=A["dht"], num_seqs=N, scale=A["scale"], states=st_k,
                                                       workspace=ws_k, out=o))
    del st_g, st_k

    # the KDA backward and forward with the sigmoid-bounded gate (gate_scale -2), same inputs
    sig = {}

    def sig_loop(name, fn, n=max(3, args.steps // 2)):
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        sig[name] = a.elapsed_time(b) / n
    sig_loop("bwd_ms", lambda A=K, o=out_k: gdr.kda_bwd(A["q"], A["k"], A["v"], A["g_raw"], A["A_log"], A["dt_bias"],
                                                        A["beta_logit"], A["dO"], h0=A["h0"], dht=A["dht"],
                                                        num_seqs=N, scale=A["scale"], workspace=ws_k, out=o,
                                                        kda_gate="sigmoid", gate_scale=-2.0))
    sig_loop("fwd_ms", lambda A=K: gdr.kda_fwd(A["q"], A["k"], A["v"], A["g_raw"], A["A_log"], A["dt_bias"],
                                               A["beta_logit"], h0=A["h0"], num_seqs=N, scale=A["scale"],
                                               workspace=ws_k, kda_gate="sigmoid", gate_scale=-2.0))
    # GDN with grouped q / k heads: 16 q / k heads shared by 32 value heads, T = 32768
    gqa = None
    gq_case = inputs.Case("gqa", "gdn", 1, CASE_G.seq_len, 2 * CASE_G.heads, CASE_G.dim, seed=231, with_h0=True,
                          with_dht=True, k_heads=CASE_G.heads)
    gx = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inputs.make(gq_case).items()}
    ws_q = torch.empty(gdr.workspace_bytes(gdr.make_shape(N, T, 2 * Hh, D, k_heads=Hh)), dtype=torch.uint8,
                       device="cuda")
    gqa_fn = lambda A=gx: gdr.gdr_bwd(A["q"], A["k"], A["v"], A["g"], A["beta_logit"], A["dO"], h0=A["h0"],
                                      dht=A["dht"], num_seqs=N, scale=A["scale"], workspace=ws_q)
    gqa_fn()
    torch.cuda.synchronize()
    ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_gqa = max(3, args.steps // 2)
    ga.record(stream)
    for _ in range(n_gqa):
        gqa_fn()
    gb.record(stream)
    torch.cuda.synchronize()
    gqa = {"workload": "GDN bwd, 16 q/k heads, 32 v heads, T=32768 D=128", "ms": ga.elapsed_time(gb) / n_gqa}
    del gx, ws_q

    # the causal conv1d (+ SiLU) backward feeding q, k, v of this layer: C = 3 H D channels, K = 4
    conv = None
    cc = inputs.conv_case([CASE_G.seq_len], 3 * CASE_G.heads * CASE_G.dim, 4, seed=230)
    cx = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in cc.items()}
    conv_fn = lambda: gdr.conv1d_bwd(cx["x"], cx["weight"], cx["bias"], cx["dy"], silu=True)
    for _ in range(2):
        conv_fn()
    torch.cuda.synchronize()
    n_conv = max(3, args.steps // 2)
    api.profile_begin(2 * n_conv)
    for _ in range(n_conv):
        conv_fn()
    torch.cuda.synchronize()
    conv_prof = api.profile_end()
    if conv_prof["conv"][1]:
        conv_ms = conv_prof["conv"][0] / conv_prof["conv"][1]
        conv_bytes = CASE_G.seq_len * cc["x"].shape[1] * 6  # x, dy read, dx written (bf16)
        conv = {"kernel": "k_conv1d_bwd", "ms": conv_ms, "tokens": CASE_G.seq_len, "channels": cc["x"].shape[1],
                "width": 4, "bound": "hbm", "achieved": conv_bytes / (conv_ms * 1e-3) / 1e9, "unit": "GB/s"}
    del cx
    th_v = CASE_G.seq_len * CASE_G.heads
    out_ms = (fwd_kernels["gdn"].get("out", 0.0) + fwd_kernels["kda"].get("out", 0.0)) / 2
    forward = {
        "ms_per_variant": {"gdn": fms_g, "kda": fms_k},
        "mtokens_per_s": (CASE_G.seq_len + CASE_K.seq_len) / ((fms_g + fms_k) * 1e-3) / 1e6,
        "kernels_ms_per_variant": fwd_kernels,
        "out_roofline": ({"kernel": "k_out (forward output)", "bound": "hbm",
                          "achieved": th_v * OUT_BYTES_PER_TH / (out_ms * 1e-3) / 1e9, "unit": "GB/s",
                          "tensor_tflops": th_v * OUT_FLOP_PER_TH / (out_ms * 1e-3) / 1e12}
                         if out_ms > 0 else None),
    }

    # ---- end to end: pinned host inputs -> device -> backward -> host gradients ----
    # Pipelined as a training loop runs it: two device sets of inputs and gradients; step i's
    # inputs upload on one copy stream while step i - 1 computes, and step i's gradients
    # download on another while step i + 1 computes.  Every step still moves all of its
    # inputs in and all of its gradients out inside the timed region.
    def pinned(x):
        return {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    hg, hk = pinned(xg), pinned(xk)
    hout_g = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in out_g.items()}
    hout_k = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in out_k.items()}
    keys_g = [k for k, v in hg.items() if isinstance(v, torch.Tensor) and k != "cu_seqlens"]
    keys_k = [k for k, v in hk.items() if isinstance(v, torch.Tensor) and k != "cu_seqlens"]
    h2d = sum(hg[k].numel() * hg[k].element_size() for k in keys_g) + \
        sum(hk[k].numel() * hk[k].element_size() for k in keys_k)
    d2h = sum(v.numel() * v.element_size() for v in out_g.values()) + \
        sum(v.numel() * v.element_size() for v in out_k.values())
    sets = [(G, K, out_g, out_k),
            (dev(xg), dev(xk), gdr.alloc_outputs(T, Hh, D, N, "gdn"), gdr.alloc_outputs(T, Hh, D, N, "kda"))]
    up_s, down_s = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: [torch.cuda.Event(), torch.cuda.Event()]
    ev_up, ev_comp, ev_down = ev(), ev(), ev()

    def e2e_steps(n):
        # the first upload, then per step: compute (after its upload and the previous download
        # from the same set), the next upload (after the compute that last read that set) and
        # this step's download
        up_s.wait_stream(stream)
        down_s.wait_stream(stream)
        with torch.cuda.stream(up_s):
            for k in keys_g:
                sets[0][0][k].copy_(hg[k], non_blocking=True)
            for k in keys_k:
                sets[0][1][k].copy_(hk[k], non_blocking=True)
            ev_up[0].record(up_s)
        for i in range(n):
            b = i & 1
            Gb, Kb, og, ok = sets[b]
            stream.wait_event(ev_up[b])
            if i >= 2:
                stream.wait_event(ev_down[b])
            step_g(A=Gb, o=og)
            step_k(A=Kb, o=ok)
            ev_comp[b].record(stream)
            if i + 1 < n:
                nb = b ^ 1
                with torch.cuda.stream(up_s):
                    if i >= 1:
                        up_s.wait_event(ev_comp[nb])
                    for k in keys_g:
                        sets[nb][0][k].copy_(hg[k], non_blocking=True)
                    for k in keys_k:
                        sets[nb][1][k].copy_(hk[k], non_blocking=True)
                    ev_up[nb].record(up_s)
            with torch.cuda.stream(down_s):
                down_s.wait_event(ev_comp[b])
                for k, v in og.items():
                    hout_g[k].copy_(v, non_blocking=True)
                for k, v in ok.items():
                    hout_k[k].copy_(v, non_blocking=True)
                ev_down[b].record(down_s)
        stream.wait_stream(up_s)
        stream.wait_stream(down_s)

    e2e_steps(2)
    torch.cuda.synchronize()
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    e2e_steps(args.steps)
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b) / args.steps, world)
    e2e_value = world * TOKENS_PER_STEP / (e2e_ms * 1e-3) / 1e6

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    # ---- roofline of the dominant kernel ----
    hbm, tf_burst, tf_sus, src = peaks()
    if conv:
        conv.update(peak=hbm, frac=conv["achieved"] / hbm, peak_source=src + " (hbm_gbs)")
    if forward["out_roofline"]:
        fr = forward["out_roofline"]
        fr.update(peak=hbm, frac=fr["achieved"] / hbm, peak_source=src + " (hbm_gbs)")
    dom = max(prof, key=lambda k: prof[k][0])
    th = CASE_G.seq_len * CASE_G.heads  # token-heads per variant
    pair_bytes = 3 * 4 * D_ * D_ * CASE_G.num_seqs * CASE_G.heads  # h0, dht read, dh0 written
    alg_bytes = {m: th * BWD_BYTES_PER_TH[m] + pair_bytes for m in ("gdn", "kda")}
    alg_flop = th * BWD_FLOP_PER_TH
    roof = None
    if dom == "main" and prof["main"][1] > 0:
        # the dominant kernel: the method's algorithmic bytes and flops of one backward over its
        # launch time (the main kernel is the step that reads the inputs and writes the gradients)
        n_main = prof["main"][1]
        avg_s = prof["main"][0] / n_main * 1e-3
        bytes_avg = (alg_bytes["gdn"] + alg_bytes["kda"]) / 2
        ach = bytes_avg / avg_s / 1e9
        design = bytes_avg + th * (MAIN_DESIGN_EXTRA_PER_TH["gdn"] + MAIN_DESIGN_EXTRA_PER_TH["kda"]) / 2
        traffic = None
        tp = os.path.join(ROOT, "profiles", "main_traffic.json")
        if os.path.exists(tp):
            t = json.load(open(tp))
            if t.get("source_sha") == build_sha():
                traffic = t.get("bytes_per_launch")
        roof = {"kernel": "k_main (avg of the GDN and KDA launches)", "bound": "hbm", "achieved": ach,
                "peak": hbm, "unit": "GB/s", "frac": ach / hbm, "traffic": traffic,
                "peak_source": src + " (hbm_gbs)",
                "bytes_per_launch": bytes_avg, "bytes_basis": "the method's: 2316 / 2820 B per token-head",
                "design_bytes_per_launch": design,
                "design_achieved": design / avg_s / 1e9,
                "design_basis": "the builder's count: also the dS_C and T tiles (and, KDA, A and the P pair) this design reads",
                "tensor_tflops": alg_flop / avg_s / 1e12, "tensor_frac": alg_flop / avg_s / 1e12 / tf_burst,
                "tensor_peak": tf_burst, "tensor_peak_source": src + " (bf16_tflops, burst)"}
    else:
        k = dom
        roof = {"kernel": k, "bound": "hbm", "achieved": None, "peak": hbm, "unit": "GB/s", "frac": None,
                "traffic": None, "note": "dominant kernel has no algorithmic figure yet"}
    # the whole backward call (every kernel of gdr_bwd / kda_bwd), per variant
    whole = {"flop_per_token_head": BWD_FLOP_PER_TH, "bytes_per_token_head": BWD_BYTES_PER_TH,
             "hbm_peak_gbs": hbm, "tensor_peak_tflops": {"burst": tf_burst, "sustained": tf_sus},
             "peak_source": src}
    for m, ms_v in (("gdn", ms_g), ("kda", ms_k)):
        s_ = ms_v * 1e-3
        tfl = alg_flop / s_ / 1e12
        gbs = alg_bytes[m] / s_ / 1e9
        whole[m] = {"ms": ms_v, "mtokens_per_s": CASE_G.seq_len / s_ / 1e6, "tflops": tfl,
                    "tensor_frac_burst": tfl / tf_burst, "tensor_frac_sustained": tfl / tf_sus,
                    "gbs": gbs, "hbm_frac": gbs / hbm}

    csum = clk.summary(t_clk0, t_clk1)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "variants_ms": {"gdn": ms_g, "kda": ms_k},
                   "l2": "inputs larger than L2 (no flush)", "parallelism": "replicas" if world > 1 else "1 GPU"},
        "roofline": roof,
        "backward_roofline": whole,
        "kernels_ms_per_step": {k: v[0] / args.steps for k, v in prof.items()},
        "kernels_ms_per_variant": per_variant,
        "forward": forward,
        "bwd_from_saved_states": {"ms_per_variant": saved, "kernels_ms_per_variant": saved_kernels},
        "kda_sigmoid_gate": sig,
        "conv1d_bwd": conv,
        "gqa": gqa,
        "gpu_launches": launches,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms},
        "clocks": csum,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_tokens)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_profile_case(args):
    """Small case for ncu captures: a few GDN or KDA backwards (or, with the _fwd cases,
    forwards) at B=1 H=16 T=8192 D=128 (inputs ~150 MB, larger than L2), or (conv) conv1d
    backwards of the benchmark's layer (T=32768, 6144 channels, ~1.2 GB); no timing line."""
    import chunked_gated_delta_bwd_gb300 as gdr
    from chunked_gated_delta_bwd_gb300 import build
    build.build()
    if args.profile_case == "conv":
        cc = inputs.conv_case([CASE_G.seq_len], 3 * CASE_G.heads * CASE_G.dim, 4, seed=230)
        cx = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in cc.items()}
        for _ in range(args.steps):
            gdr.conv1d_bwd(cx["x"], cx["weight"], cx["bias"], cx["dy"], silu=True)
        torch.cuda.synchronize()
        print("profile case conv: %d calls done" % args.steps)
        return
    mode = args.profile_case.replace("_fwd", "")
    fwd = args.profile_case.endswith("_fwd")
    case = inputs.Case("profile_" + mode, mode, 1, 8192, 16, 128, seed=5, with_h0=True, with_dht=True)
    x = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inputs.make(case).items()}
    ws = torch.empty(gdr.workspace_bytes(gdr.make_shape(1, 8192, 16, 128)), dtype=torch.uint8, device="cuda")
    for _ in range(args.steps):
        if fwd and mode == "gdn":
            gdr.gdr_fwd(x["q"], x["k"], x["v"], x["g"], x["beta_logit"], h0=x["h0"], num_seqs=1,
                        scale=x["scale"], workspace=ws)
        elif fwd:
            gdr.kda_fwd(x["q"], x["k"], x["v"], x["g_raw"], x["A_log"], x["dt_bias"], x["beta_logit"],
                        h0=x["h0"], num_seqs=1, scale=x["scale"], workspace=ws)
        elif mode == "gdn":
            gdr.gdr_bwd(x["q"], x["k"], x["v"], x["g"], x["beta_logit"], x["dO"], h0=x["h0"], dht=x["dht"],
                        num_seqs=1, scale=x["scale"], workspace=ws)
        else:
            gdr.kda_bwd(x["q"], x["k"], x["v"], x["g_raw"], x["A_log"], x["dt_bias"], x["beta_logit"],
                        x["dO"], h0=x["h0"], dht=x["dht"], num_seqs=1, scale=x["scale"], workspace=ws)
    torch.cuda.synchronize()
    print("profile case %s: %d calls done" % (args.profile_case, args.steps))


# the sources that define the main kernel (its .cu file and the headers it includes)
MAIN_SOURCES = ("gdr_main_kda.cu", "gdr_main_gdn.cu", "gdr_chunk.cuh", "gdr_common.cuh", "gdr_tc.cuh", "gdr_tma.h", "gdr_internal.h")


def build_sha():
    """Hash of the main kernel's sources: the stored DRAM traffic is reported only while it matches."""
    import hashlib
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "chunked_gated_delta_bwd_gb300", "csrc")
    for f in MAIN_SOURCES:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:12]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-tokens", type=int, default=8192)
    ap.add_argument("--ref-tokens", type=int, default=1024)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", choices=["gdn", "kda", "gdn_fwd", "kda_fwd", "conv"], default=None,
                    help="run a small case (B=1 H=16 T=8192) for ncu captures instead of the benchmark")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.profile_case:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        main_gpu(args)


if __name__ == "__main__":
    main()
