"""The allocation-free backward (gdr_bwd_fixed) against gdr_bwd, through the C ABI.

gdr_bwd_fixed serves callers that cannot allocate device memory where they run
the backward (a plug-in whose host framework owns every allocation, or code
where a cudaMalloc may not run): its scratch is a static device array inside
the library.  This file is collected last so that a run stopping at the first
failure has run every other test first; it passes alone in a fresh process
(the first call resolves the array's address) and after the other tests.
"""
import ctypes

import pytest
import torch

from chunked_gated_delta_bwd_gb300 import inputs
from tests import helpers as H

pytestmark = pytest.mark.gpu

FIXED_BYTES = 64 << 20  # GDR_FIXED_WORKSPACE_BYTES in include/gdr.h


def _lib():
    from chunked_gated_delta_bwd_gb300 import api, build
    build.build()
    L = api.lib()
    vp = ctypes.c_void_p
    L.gdr_bwd_fixed.restype = ctypes.c_int
    L.gdr_bwd_fixed.argtypes = [ctypes.POINTER(api.GdrShape)] + [vp] * 16
    return L, api


def _call_fixed(L, api, x):
    d = H.to_gpu(x)
    T, Hh, D = d["q"].shape
    N = d["cu_seqlens"].numel() - 1
    shape = api.make_shape(N, T, Hh, D, d["cu_seqlens"], d["scale"])
    o = api.alloc_outputs(T, Hh, D, N, "gdn")
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    rc = L.gdr_bwd_fixed(ctypes.byref(shape), p(d["q"]), p(d["k"]), p(d["v"]), p(d["g"]),
                         p(d["beta_logit"]), p(d["h0"]), p(d["dO"]), p(d["dht"]), None,
                         p(o["dq"]), p(o["dk"]), p(o["dv"]), p(o["dg"]), p(o["dbeta"]), p(o["dh0"]),
                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return rc, {k: v.cpu() for k, v in o.items()}


def test_fixed_workspace_matches_gdr_bwd_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    L, api = _lib()
    # two calls in a row, different inputs and shapes: the second reuses the
    # array with the first call's contents still in it
    for seed, lens in ((201, [200, 77, 64]), (202, [130, 1, 300])):
        x = inputs.custom("gdn", lens, heads=3, dim=128, seed=seed, with_h0=True, with_dht=True)
        rc, fixed = _call_fixed(L, api, x)
        assert rc == 0, L.gdr_last_error().decode()
        ref = H.run_gpu(x)  # the existing entry point, caller workspace
        # the GDN backward has no atomics and sums in a fixed order, so the two entry points
        # must agree bit for bit: any of the first call's scratch that leaked into the
        # second call's results would show here
        for name, t in ref.items():
            assert torch.equal(fixed[name], t), (seed, name, H.rel_l2(H.f64(fixed[name]), H.f64(t)))
        # and both are right: the oracle on the same inputs
        print(H.assert_parity(H.compare(fixed, H.run_oracle(x), x), "fixed %d" % seed))


def test_fixed_workspace_rejects_problems_beyond_its_size():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    L, api = _lib()
    big = api.make_shape(1, 32768, 16, 128)
    assert api.workspace_bytes(big) > FIXED_BYTES
    A = ctypes.c_void_p(4096)  # never dereferenced: the size check comes first
    rc = L.gdr_bwd_fixed(ctypes.byref(big), *([A] * 9), *([A] * 6), None)
    assert rc == 3
    assert b"fixed workspace" in L.gdr_last_error()
