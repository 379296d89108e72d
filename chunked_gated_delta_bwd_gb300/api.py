"""Python binding of the C ABI in include/gdr.h (argument marshalling only).

Every step of the computation runs in the CUDA kernels of libgdr.so; this
module checks dtypes and shapes, allocates outputs and workspace with torch
(device memory plumbing), and passes raw pointers and the current CUDA stream.
It raises if the library has not been built: there is no fallback.

Layouts: q, k, v, dO are bf16 ``[T_total, H, D]`` (token-major; a dense
``[B, T, H, D]`` is accepted and flattened), beta logits bf16 ``[T_total, H]``,
GDN gate g float32 ``[T_total, H]``, KDA g_raw bf16 ``[T_total, H, D]``,
A_log float32 ``[H]``, dt_bias float32 ``[H, D]``, h0 / dht float32 ``[N, H, D, D]``.
"""
import ctypes
import os

import torch

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

GDR_DEV_BAD_SEQLENS = 1
GDR_DEV_GATE_RANGE = 2
GDR_DEV_TIMEOUT = 4
GDR_DEV_STATES_MISMATCH = 8


class GdrShape(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int64),
                ("num_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("cu_seqlens", ctypes.c_void_p), ("scale", ctypes.c_float),
                ("kda_gate", ctypes.c_int32), ("gate_scale", ctypes.c_float),
                ("num_k_heads", ctypes.c_int32)]

KDA_GATES = {"softplus": 0, "sigmoid": 1}  # GDR_KDA_GATE_SOFTPLUS / GDR_KDA_GATE_SIGMOID


class GdrError(RuntimeError):
    pass


def lib():
    """Loads libgdr.so (built by ``build.build()``); raises if it is missing."""
    global _LIB
    if _LIB is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise GdrError("libgdr.so is not built (run chunked_gated_delta_bwd_gb300.build.build())")
        L = ctypes.CDLL(path)
        vp, sz, sp = ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(GdrShape)
        L.gdr_workspace_bytes.restype = sz
        L.gdr_workspace_bytes.argtypes = [sp]
        L.gdr_states_bytes.restype = sz
        L.gdr_states_bytes.argtypes = [sp]
        L.gdr_fwd_states.restype = ctypes.c_int
        L.gdr_fwd_states.argtypes = [sp] + [vp] * 7 + [sz, vp, sz, vp]
        L.kda_fwd_states.restype = ctypes.c_int
        L.kda_fwd_states.argtypes = [sp] + [vp] * 9 + [sz, vp, sz, vp]
        L.gdr_fwd.restype = ctypes.c_int
        L.gdr_fwd.argtypes = [sp] + [vp] * 9 + [sz, vp, sz, vp]
        L.kda_fwd.restype = ctypes.c_int
        L.kda_fwd.argtypes = [sp] + [vp] * 11 + [sz, vp, sz, vp]
        L.gdr_bwd.restype = ctypes.c_int
        L.gdr_bwd.argtypes = [sp] + [vp] * 10 + [sz] + [vp] * 7
        L.kda_bwd.restype = ctypes.c_int
        L.kda_bwd.argtypes = [sp] + [vp] * 12 + [sz] + [vp] * 9
        L.gdr_conv1d_bwd.restype = ctypes.c_int
        L.gdr_conv1d_bwd.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32] + [vp] * 5 + \
            [ctypes.c_int32] + [vp] * 4
        L.gdr_workspace_status.restype = ctypes.c_int
        L.gdr_workspace_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int)]
        L.gdr_last_error.restype = ctypes.c_char_p
        L.gdr_last_error.argtypes = []
        L.gdr_profile_begin.restype = ctypes.c_int
        L.gdr_profile_begin.argtypes = [ctypes.c_int]
        L.gdr_profile_end.restype = ctypes.c_int
        L.gdr_profile_end.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)]
        L.gdr_test_stall_next_call.restype = None
        L.gdr_test_stall_next_call.argtypes = [ctypes.c_int]
        _LIB = L
    return _LIB


def _check(rc, what):
    if rc != 0:
        raise GdrError("%s failed (status %d): %s" % (what, rc, lib().gdr_last_error().decode()))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def make_shape(num_seqs, total_tokens, heads, dim, cu_seqlens=None, scale=None, kda_gate="softplus",
               gate_scale=0.0, k_heads=None):
    """The problem shape.  ``kda_gate`` selects the KDA gate function ("softplus":
    g = -e^{A_log} softplus(g_raw + dt_bias); "sigmoid": g = ln2 gate_scale sigmoid(e^{A_log} (g_raw +
    dt_bias)) with gate_scale <= 0); the GDN calls ignore it."""
    sh = GdrShape()
    sh.num_seqs = int(num_seqs)
    sh.total_tokens = int(total_tokens)
    sh.num_heads = int(heads)
    sh.head_dim = int(dim)
    sh.cu_seqlens = None if cu_seqlens is None else cu_seqlens.data_ptr()
    sh.scale = float(dim ** -0.5 if scale is None else scale)
    if kda_gate not in KDA_GATES:
        raise ValueError("kda_gate must be one of %s" % sorted(KDA_GATES))
    sh.kda_gate = KDA_GATES[kda_gate]
    sh.gate_scale = float(0.0 if gate_scale is None else gate_scale)
    sh.num_k_heads = 0 if k_heads is None or int(k_heads) == int(heads) else int(k_heads)
    return sh


def workspace_bytes(shape: GdrShape) -> int:
    return int(lib().gdr_workspace_bytes(ctypes.byref(shape)))


def states_bytes(shape: GdrShape) -> int:
    return int(lib().gdr_states_bytes(ctypes.byref(shape)))


def _need(t, dtype, shape, name):
    if t is None:
        raise ValueError("%s is required" % name)
    if not t.is_cuda or t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA %s tensor of shape %s (got %s %s %s)"
                         % (name, dtype, tuple(shape), t.device, t.dtype, tuple(t.shape)))
    return t


def _opt(t, dtype, shape, name):
    return None if t is None else _need(t, dtype, shape, name)


class _Problem:
    """Shape of one call: value heads H from v, q / k heads Hk from q (GQA when Hk < H)."""

    def __init__(self, q, cu_seqlens, num_seqs, scale, kda_gate="softplus", gate_scale=0.0, v=None):
        v = q if v is None else v
        if q.dim() == 4:
            B, T, Hk, D = q.shape
            H = v.shape[2]
            self.dense_shape = (B, T)
            N, Tt = B, B * T
        else:
            Tt, Hk, D = q.shape
            H = v.shape[1]
            self.dense_shape = None
            N = num_seqs if cu_seqlens is None else cu_seqlens.numel() - 1
            if N is None:
                N = 1
        if cu_seqlens is not None:
            _need(cu_seqlens, torch.int64, (N + 1,), "cu_seqlens")
        self.N, self.T, self.H, self.D, self.Hk = int(N), int(Tt), int(H), int(D), int(Hk)
        self.cu = cu_seqlens
        self.shape = make_shape(N, Tt, H, D, cu_seqlens, scale, kda_gate, gate_scale, k_heads=Hk)

    def flat(self, t):
        if t is None or self.dense_shape is None:
            return t
        return t.reshape(self.T, *t.shape[2:])

    def unflat(self, t):
        if self.dense_shape is None:
            return t
        return t.reshape(*self.dense_shape, *t.shape[1:])

    def workspace(self, ws):
        need = workspace_bytes(self.shape)
        if ws is None:
            return torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
        if ws.numel() < need or ws.dtype != torch.uint8:
            raise ValueError("workspace must be a uint8 tensor of at least %d bytes" % need)
        return ws


def gdr_fwd_states(q, k, v, g, beta_logit, h0=None, cu_seqlens=None, num_seqs=None, scale=None,
                   workspace=None, gate="gdn", g_raw=None, A_log=None, dt_bias=None, kda_gate="softplus",
                   gate_scale=0.0):
    """Chunk-start states of every 64-token chunk (bf16), for gdr_bwd / kda_bwd."""
    P = _Problem(q, cu_seqlens, num_seqs, scale, kda_gate, gate_scale, v=v)
    T, H, D, N, Hk = P.T, P.H, P.D, P.N, P.Hk
    q, k = (_need(P.flat(x), torch.bfloat16, (T, Hk, D), n) for x, n in ((q, "q"), (k, "k")))
    v = _need(P.flat(v), torch.bfloat16, (T, H, D), "v")
    beta_logit = _need(P.flat(beta_logit), torch.bfloat16, (T, H), "beta_logit")
    h0 = _opt(h0, torch.float32, (N, H, D, D), "h0")
    states = torch.empty(max(states_bytes(P.shape), 16), dtype=torch.uint8, device="cuda")
    ws = P.workspace(workspace)
    if gate == "gdn":
        g = _need(P.flat(g), torch.float32, (T, H), "g")
        rc = lib().gdr_fwd_states(ctypes.byref(P.shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                  _ptr(beta_logit), _ptr(h0), _ptr(states), states.numel(), _ptr(ws),
                                  ws.numel(), _stream())
    else:
        g_raw = _need(P.flat(g_raw), torch.bfloat16, (T, H, D), "g_raw")
        A_log = _need(A_log, torch.float32, (H,), "A_log")
        dt_bias = _need(dt_bias, torch.float32, (H, D), "dt_bias")
        rc = lib().kda_fwd_states(ctypes.byref(P.shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw),
                                  _ptr(A_log), _ptr(dt_bias), _ptr(beta_logit), _ptr(h0),
                                  _ptr(states), states.numel(), _ptr(ws), ws.numel(), _stream())
    _check(rc, "gdr_fwd_states" if gate == "gdn" else "kda_fwd_states")
    return states


def _fwd(gate, q, k, v, beta_logit, h0, cu_seqlens, num_seqs, scale, states, workspace, want_ht,
         g=None, g_raw=None, A_log=None, dt_bias=None, kda_gate="softplus", gate_scale=0.0):
    P = _Problem(q, cu_seqlens, num_seqs, scale, kda_gate, gate_scale, v=v)
    T, H, D, N, Hk = P.T, P.H, P.D, P.N, P.Hk
    q, k = (_need(P.flat(x), torch.bfloat16, (T, Hk, D), n) for x, n in ((q, "q"), (k, "k")))
    v = _need(P.flat(v), torch.bfloat16, (T, H, D), "v")
    beta_logit = _need(P.flat(beta_logit), torch.bfloat16, (T, H), "beta_logit")
    h0 = _opt(h0, torch.float32, (N, H, D, D), "h0")
    ws = P.workspace(workspace)
    o = torch.empty(T, H, D, dtype=torch.bfloat16, device="cuda")
    ht = torch.empty(N, H, D, D, dtype=torch.float32, device="cuda") if want_ht else None
    if states is True:
        states = torch.empty(max(states_bytes(P.shape), 16), dtype=torch.uint8, device="cuda")
    nst = 0 if states is None else states.numel()
    if gate == "gdn":
        g = _need(P.flat(g), torch.float32, (T, H), "g")
        rc = lib().gdr_fwd(ctypes.byref(P.shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta_logit),
                           _ptr(h0), _ptr(o), _ptr(ht), _ptr(states), nst, _ptr(ws), ws.numel(), _stream())
    else:
        g_raw = _need(P.flat(g_raw), torch.bfloat16, (T, H, D), "g_raw")
        A_log = _need(A_log, torch.float32, (H,), "A_log")
        dt_bias = _need(dt_bias, torch.float32, (H, D), "dt_bias")
        rc = lib().kda_fwd(ctypes.byref(P.shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(A_log),
                           _ptr(dt_bias), _ptr(beta_logit), _ptr(h0), _ptr(o), _ptr(ht), _ptr(states), nst,
                           _ptr(ws), ws.numel(), _stream())
    _check(rc, "gdr_fwd" if gate == "gdn" else "kda_fwd")
    out = {"o": P.unflat(o), "ht": ht}
    if states is not None:
        out["states"] = states
    return out


def gdr_fwd(q, k, v, g, beta_logit, h0=None, cu_seqlens=None, num_seqs=None, scale=None, states=None,
            workspace=None, want_ht=True):
    """GDN forward.  Returns dict(o, ht[, states]); ``states=True`` allocates and returns the
    chunk-start states for a later gdr_bwd (or pass a uint8 buffer of states_bytes)."""
    return _fwd("gdn", q, k, v, beta_logit, h0, cu_seqlens, num_seqs, scale, states, workspace, want_ht, g=g)


def kda_fwd(q, k, v, g_raw, A_log, dt_bias, beta_logit, h0=None, cu_seqlens=None, num_seqs=None, scale=None,
            states=None, workspace=None, want_ht=True, kda_gate="softplus", gate_scale=0.0):
    """KDA forward.  Returns dict(o, ht[, states]) as gdr_fwd; ``kda_gate`` / ``gate_scale`` as make_shape."""
    return _fwd("kda", q, k, v, beta_logit, h0, cu_seqlens, num_seqs, scale, states, workspace, want_ht,
                g_raw=g_raw, A_log=A_log, dt_bias=dt_bias, kda_gate=kda_gate, gate_scale=gate_scale)


def gdr_bwd(q, k, v, g, beta_logit, dO, h0=None, dht=None, cu_seqlens=None, num_seqs=None,
            scale=None, states=None, workspace=None, out=None):
    """GDN backward.  Returns dict(dq, dk, dv, dg, dbeta, dh0)."""
    P = _Problem(q, cu_seqlens, num_seqs, scale, v=v)
    T, H, D, N, Hk = P.T, P.H, P.D, P.N, P.Hk
    q, k = (_need(P.flat(x), torch.bfloat16, (T, Hk, D), n) for x, n in ((q, "q"), (k, "k")))
    v, dO = (_need(P.flat(x), torch.bfloat16, (T, H, D), n) for x, n in ((v, "v"), (dO, "dO")))
    g = _need(P.flat(g), torch.float32, (T, H), "g")
    beta_logit = _need(P.flat(beta_logit), torch.bfloat16, (T, H), "beta_logit")
    h0 = _opt(h0, torch.float32, (N, H, D, D), "h0")
    dht = _opt(dht, torch.float32, (N, H, D, D), "dht")
    ws = P.workspace(workspace)
    o = out if out is not None else alloc_outputs(T, H, D, N, "gdn", k_heads=Hk)
    rc = lib().gdr_bwd(ctypes.byref(P.shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta_logit),
                       _ptr(h0), _ptr(dO), _ptr(dht), _ptr(states), _ptr(ws), ws.numel(),
                       _ptr(o["dq"]), _ptr(o["dk"]), _ptr(o["dv"]), _ptr(o["dg"]), _ptr(o["dbeta"]),
                       _ptr(o["dh0"]), _stream())
    _check(rc, "gdr_bwd")
    return {k_: (P.unflat(t) if k_ != "dh0" else t) for k_, t in o.items()}


def kda_bwd(q, k, v, g_raw, A_log, dt_bias, beta_logit, dO, h0=None, dht=None, cu_seqlens=None,
            num_seqs=None, scale=None, states=None, workspace=None, out=None, kda_gate="softplus", gate_scale=0.0):
    """KDA backward.  Returns dict(dq, dk, dv, dg_raw, dbeta, dh0, dA_log, ddt_bias); ``kda_gate`` /
    ``gate_scale`` as make_shape."""
    P = _Problem(q, cu_seqlens, num_seqs, scale, kda_gate, gate_scale, v=v)
    T, H, D, N, Hk = P.T, P.H, P.D, P.N, P.Hk
    q, k = (_need(P.flat(x), torch.bfloat16, (T, Hk, D), n) for x, n in ((q, "q"), (k, "k")))
    v, dO, g_raw = (_need(P.flat(x), torch.bfloat16, (T, H, D), n)
                    for x, n in ((v, "v"), (dO, "dO"), (g_raw, "g_raw")))
    A_log = _need(A_log, torch.float32, (H,), "A_log")
    dt_bias = _need(dt_bias, torch.float32, (H, D), "dt_bias")
    beta_logit = _need(P.flat(beta_logit), torch.bfloat16, (T, H), "beta_logit")
    h0 = _opt(h0, torch.float32, (N, H, D, D), "h0")
    dht = _opt(dht, torch.float32, (N, H, D, D), "dht")
    ws = P.workspace(workspace)
    o = out if out is not None else alloc_outputs(T, H, D, N, "kda", k_heads=Hk)
    rc = lib().kda_bwd(ctypes.byref(P.shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(A_log),
                       _ptr(dt_bias), _ptr(beta_logit), _ptr(h0), _ptr(dO), _ptr(dht), _ptr(states),
                       _ptr(ws), ws.numel(), _ptr(o["dq"]), _ptr(o["dk"]), _ptr(o["dv"]),
                       _ptr(o["dg_raw"]), _ptr(o["dbeta"]), _ptr(o["dh0"]), _ptr(o["dA_log"]),
                       _ptr(o["ddt_bias"]), _stream())
    _check(rc, "kda_bwd")
    return {k_: (P.unflat(t) if k_ not in ("dh0", "dA_log", "ddt_bias") else t) for k_, t in o.items()}


def conv1d_bwd(x, weight, bias, dy, cu_seqlens=None, num_seqs=None, silu=True):
    """Backward of the causal depthwise conv1d (+ SiLU): x, dy bf16 [T, C] (or [B, T, C]),
    weight float32 [C, K], bias float32 [C] or None.  Returns dict(dx, dweight, dbias)."""
    dense = None
    if x.dim() == 3:
        B, T, C = x.shape
        dense = (B, T)
        N, Tt = B, B * T
        x, dy = x.reshape(Tt, C), dy.reshape(Tt, C)
    else:
        Tt, C = x.shape
        N = num_seqs if cu_seqlens is None else cu_seqlens.numel() - 1
        N = 1 if N is None else N
    K = weight.shape[1] if weight.dim() == 2 else -1
    _need(x, torch.bfloat16, (Tt, C), "x")
    _need(dy, torch.bfloat16, (Tt, C), "dy")
    _need(weight, torch.float32, (C, K), "weight")
    _opt(bias, torch.float32, (C,), "bias")
    if cu_seqlens is not None:
        _need(cu_seqlens, torch.int64, (N + 1,), "cu_seqlens")
    dx = torch.empty(Tt, C, dtype=torch.bfloat16, device="cuda")
    dw = torch.empty(C, K, dtype=torch.float32, device="cuda")
    db = torch.empty(C, dtype=torch.float32, device="cuda") if bias is not None else None
    rc = lib().gdr_conv1d_bwd(int(N), int(Tt), int(C), int(K), _ptr(cu_seqlens), _ptr(x), _ptr(weight), _ptr(bias),
                              _ptr(dy), 1 if silu else 0, _ptr(dx), _ptr(dw), _ptr(db), _stream())
    _check(rc, "gdr_conv1d_bwd")
    return {"dx": dx if dense is None else dx.reshape(*dense, C), "dweight": dw, "dbias": db}


def alloc_outputs(T, H, D, N, gate, device="cuda", k_heads=None):
    bf = dict(dtype=torch.bfloat16, device=device)
    Hk = H if k_heads is None else k_heads
    o = {"dq": torch.empty(T, Hk, D, **bf), "dk": torch.empty(T, Hk, D, **bf),
         "dv": torch.empty(T, H, D, **bf), "dbeta": torch.empty(T, H, **bf),
         "dh0": torch.empty(N, H, D, D, dtype=torch.float32, device=device)}
    if gate == "gdn":
        o["dg"] = torch.empty(T, H, dtype=torch.float32, device=device)
    else:
        o["dg_raw"] = torch.empty(T, H, D, **bf)
        o["dA_log"] = torch.empty(H, dtype=torch.float32, device=device)
        o["ddt_bias"] = torch.empty(H, D, dtype=torch.float32, device=device)
    return o


def workspace_status(workspace) -> int:
    """Waits for the current stream and returns the device status bits of ``workspace``."""
    st = ctypes.c_int(0)
    _check(lib().gdr_workspace_status(_ptr(workspace), _stream(), ctypes.byref(st)), "gdr_workspace_status")
    return st.value


def test_stall_next_call(cta: int):
    """Test hook: hold CTA ``cta`` of the next GDN backward's main kernel (head_dim 128) on a
    barrier nothing arrives on, so that its bounded wait runs out (GDR_DEV_TIMEOUT)."""
    lib().gdr_test_stall_next_call(int(cta))


KERNEL_NAMES = ("chunk_table", "prep", "states", "main", "out", "conv")


def profile_begin(max_launches: int):
    """Time the next ``max_launches`` timed sections of the library (one kernel kind of one
    call) with CUDA events."""
    _check(lib().gdr_profile_begin(int(max_launches)), "gdr_profile_begin")


def profile_end():
    """Returns {kernel: (total_ms, kernels launched)} for the sections recorded since profile_begin."""
    n = len(KERNEL_NAMES)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int * n)()
    _check(lib().gdr_profile_end(ms, cnt), "gdr_profile_end")
    return {KERNEL_NAMES[i]: (ms[i], cnt[i]) for i in range(n)}
