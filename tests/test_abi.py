"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/gdr.h declares, sizes its buffers, and rejects bad arguments
on the host before touching the device."""
import ctypes
import os
import re

import pytest

import chunked_gated_delta_bwd_gb300 as gdr
from chunked_gated_delta_bwd_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdr.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return api.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdr_\w+|kda_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("gdr_fwd_states", "kda_fwd_states", "gdr_fwd", "kda_fwd", "gdr_bwd", "kda_bwd", "gdr_workspace_bytes",
              "gdr_states_bytes", "gdr_workspace_status", "gdr_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in declared_functions():
        assert hasattr(L, n), n


def test_workspace_sizes(L):
    sh = gdr.make_shape(1, 32768, 16, 128)
    chunks = 512
    HDR = 256  # GDR_STATES_HEADER_BYTES
    assert gdr.states_bytes(sh) == HDR + chunks * 16 * 128 * 128 * 2
    ws = gdr.workspace_bytes(sh)
    # per chunk-head: W, U, Kr, R_hi, R_lo; T; A, P hi, P lo (the KDA backward's); gT, e^{gT}; S0, dS
    tiles = chunks * 16 * (5 * 64 * 128 * 2 + 64 * 64 * 2 + 3 * 64 * 64 * 2 + 2 * 128 * 4 + 2 * 128 * 128 * 2)
    # time-parallel state passing: 4 segments per (sequence, head) when both directions run,
    # 6 when one does; the buffers hold the larger count
    segments = 5 * 16 * 6 * 128 * 128 * 4
    assert tiles + segments <= ws <= tiles + segments + 64 * 256
    # one sequence of 256 chunks over 2 heads: the most segments (8) in both directions
    sh8 = gdr.make_shape(1, 16384, 2, 128)
    tiles8 = 256 * 2 * (5 * 64 * 128 * 2 + 64 * 64 * 2 + 3 * 64 * 64 * 2 + 2 * 128 * 4 + 2 * 128 * 128 * 2)
    segments8 = 5 * 2 * 8 * 128 * 128 * 4
    assert tiles8 + segments8 <= gdr.workspace_bytes(sh8) <= tiles8 + segments8 + 64 * 256
    # varlen bound: sum ceil(len/64) <= (T + 63 N) / 64
    fake_cu = ctypes.c_void_p(256)
    sh2 = api.GdrShape(3, 130, 2, 64, fake_cu.value, 0.125)
    # head_dim 64 runs on channels zero-padded to 128: its states keep the padded layout, and
    # its workspace holds the padded inputs and outputs beyond the 128-channel layout
    assert gdr.states_bytes(sh2) == HDR + ((130 + 63 * 3) // 64) * 2 * 128 * 128 * 2
    sh3 = api.GdrShape(3, 130, 2, 128, fake_cu.value, 0.125)
    # (10 token-major bf16 tensors, 4 fp32 states-shaped ones, dt_bias and ddt_bias)
    pads = 10 * 130 * 2 * 128 * 2 + 4 * 3 * 2 * 128 * 128 * 4 + 2 * 2 * 128 * 4
    assert gdr.workspace_bytes(sh3) + pads <= gdr.workspace_bytes(sh2) <= gdr.workspace_bytes(sh3) + pads + 17 * 256


@pytest.mark.parametrize("mutate,code", [
    (dict(head_dim=96), 2),
    (dict(num_heads=0), 1),
    (dict(num_seqs=0), 1),
    (dict(total_tokens=-1), 1),
    (dict(total_tokens=100, num_seqs=3), 1),  # dense needs T % N == 0
    (dict(total_tokens=1 << 34, num_seqs=2), 1),  # beyond the 32-bit tile addressing of one call
])
def test_bad_shapes_rejected(L, mutate, code):
    sh = gdr.make_shape(2, 128, 2, 64)
    for k, v in mutate.items():
        setattr(sh, k, v)
    assert L.gdr_workspace_bytes(ctypes.byref(sh)) == 0
    A = ctypes.c_void_p(4096)
    rc = L.gdr_bwd(ctypes.byref(sh), *([A] * 6), A, None, None, A, 1 << 40, *([A] * 6), None)
    assert rc == code
    assert L.gdr_last_error()


def test_largest_problem_accepted_next_token_rejected(L):
    # the kernels address the per chunk-head tiles by 32-bit row, the largest block being the
    # KDA backward's A / P pair block of 192 rows per chunk-head: chunks x heads x 192 < 2^31.
    # With 16 heads that allows 699050 chunks (44.7 M tokens in one sequence); one token more
    # opens chunk 699051 and is refused before any device work
    limit = ((1 << 31) - 1) // (16 * 192)
    assert limit == 699050
    ok = gdr.make_shape(1, limit * 64, 16, 128)
    assert L.gdr_workspace_bytes(ctypes.byref(ok)) > 0
    assert L.gdr_states_bytes(ctypes.byref(ok)) > 0
    over = gdr.make_shape(1, limit * 64 + 1, 16, 128)
    assert L.gdr_workspace_bytes(ctypes.byref(over)) == 0
    A = ctypes.c_void_p(4096)
    rc = L.gdr_bwd(ctypes.byref(over), *([A] * 6), A, None, None, A, 1 << 40, *([A] * 6), None)
    assert rc == 1 and b"too large" in L.gdr_last_error()


def _bwd_args(A, ws_bytes):
    # q k v g beta h0 dO dht states ws ws_bytes dq dk dv dg dbeta dh0 stream
    return [A, A, A, A, A, None, A, None, None, A, ws_bytes, A, A, A, A, A, A, None]


def test_null_and_misaligned_pointers_rejected(L):
    sh = gdr.make_shape(2, 128, 2, 64)
    ws = gdr.workspace_bytes(sh)
    A = ctypes.c_void_p(4096)
    args = _bwd_args(A, ws)
    for i in (0, 1, 2, 3, 4, 6, 9, 11, 12, 13, 14, 15, 16):
        bad = list(args)
        bad[i] = None
        assert L.gdr_bwd(ctypes.byref(sh), *bad) == 1, i
        bad[i] = ctypes.c_void_p(4096 + 8)
        assert L.gdr_bwd(ctypes.byref(sh), *bad) == 1, i
        assert b"aligned" in L.gdr_last_error()


def test_small_workspace_rejected(L):
    sh = gdr.make_shape(2, 128, 2, 64)
    ws = gdr.workspace_bytes(sh)
    A = ctypes.c_void_p(4096)
    assert L.gdr_bwd(ctypes.byref(sh), *_bwd_args(A, ws - 1)) == 3
    # KDA: A_log / dt_bias / dg_raw / dA_log / ddt_bias are required
    kargs = [A] * 7 + [None, A, None, None, A, ws] + [A] * 8 + [None]
    for i in (3, 4, 5):
        bad = list(kargs)
        bad[i] = None
        assert L.kda_bwd(ctypes.byref(sh), *bad) == 1
    bad = list(kargs)
    bad[12] = ws - 1
    assert L.kda_bwd(ctypes.byref(sh), *bad) == 3


def test_states_buffer_too_small_rejected(L):
    sh = gdr.make_shape(2, 128, 2, 64)
    ws = gdr.workspace_bytes(sh)
    st = gdr.states_bytes(sh)
    A = ctypes.c_void_p(4096)
    rc = L.gdr_fwd_states(ctypes.byref(sh), A, A, A, A, A, None, A, st - 1, A, ws, None)
    assert rc == 3


def test_kda_gate_choice_checked(L):
    sh = gdr.make_shape(2, 128, 2, 64)
    ws = gdr.workspace_bytes(sh)
    assert ws > 0
    sh.kda_gate = 2
    assert gdr.workspace_bytes(sh) == 0
    sh.kda_gate = 1
    sh.gate_scale = 0.5  # a growing gate
    assert gdr.workspace_bytes(sh) == 0
    sh.gate_scale = -2.0
    assert gdr.workspace_bytes(sh) == ws
    with pytest.raises(ValueError):
        gdr.make_shape(2, 128, 2, 64, kda_gate="tanh")


def test_forward_arguments_rejected(L):
    # gdr_fwd(shape, q, k, v, g, beta, h0, o, ht, states, states_bytes, ws, ws_bytes, stream)
    sh = gdr.make_shape(2, 128, 2, 64)
    ws = gdr.workspace_bytes(sh)
    st = gdr.states_bytes(sh)
    A = ctypes.c_void_p(4096)
    args = [A, A, A, A, A, None, A, None, None, 0, A, ws, None]
    for i in (0, 1, 2, 3, 4, 6, 10):  # q, k, v, g, beta, o, workspace are required
        bad = list(args)
        bad[i] = None
        assert L.gdr_fwd(ctypes.byref(sh), *bad) == 1, i
        bad[i] = ctypes.c_void_p(4096 + 8)
        assert L.gdr_fwd(ctypes.byref(sh), *bad) == 1, i
    for i in (5, 7, 8):  # h0, ht, states are optional but must be aligned
        bad = list(args)
        bad[i] = ctypes.c_void_p(4096 + 8)
        if i == 8:
            bad[9] = st
        assert L.gdr_fwd(ctypes.byref(sh), *bad) == 1, i
    small = list(args)
    small[11] = ws - 1
    assert L.gdr_fwd(ctypes.byref(sh), *small) == 3
    small = list(args)
    small[8], small[9] = A, st - 1
    assert L.gdr_fwd(ctypes.byref(sh), *small) == 3
    # kda_fwd: g_raw, A_log, dt_bias are required
    kargs = [A, A, A, A, A, A, A, None, A, None, None, 0, A, ws, None]
    for i in (3, 4, 5):
        bad = list(kargs)
        bad[i] = None
        assert L.kda_fwd(ctypes.byref(sh), *bad) == 1, i
    sh_bad = gdr.make_shape(2, 128, 2, 96)
    assert L.kda_fwd(ctypes.byref(sh_bad), *kargs) == 2


def test_conv1d_arguments_rejected(L):
    A = ctypes.c_void_p(4096)
    ok = [2, 256, 8, 4, None, A, A, A, A, 1, A, A, A, None]
    def call(args):
        return L.gdr_conv1d_bwd(*args)
    # every call here must be rejected on the host (the pointers are not device memory)
    for i, v, code in ((3, 5, 2), (3, 0, 2), (2, 7, 1), (0, 0, 1), (1, 255, 1)):  # width, channels, N, dense T
        bad = list(ok)
        bad[i] = v
        assert call(bad) == code, (i, v)
    for i in (5, 6, 8, 10, 11):  # x, weight, dy, dx, dweight required
        bad = list(ok)
        bad[i] = None
        assert call(bad) == 1, i
    for i in (7, 12):  # bias, dbias optional but aligned
        bad = list(ok)
        bad[i] = ctypes.c_void_p(4096 + 4)
        assert call(bad) == 1, i


def test_product_path_fails_loudly_without_library(monkeypatch):
    monkeypatch.setattr(api, "_LIB", None)
    monkeypatch.setattr(build, "LIB", "/nonexistent/libgdr.so")
    with pytest.raises(api.GdrError):
        api.lib()
