"""GB300 (sm_103a) chunked gated delta-rule backward: GDN and KDA.

The computation lives in libgdr.so (CUDA kernels behind the C ABI of
include/gdr.h); ``api`` is a thin ctypes binding.  ``inputs`` draws the seeded
synthetic workloads.  Importing the package does not load the library; the
first call does, and raises if it has not been built.
"""
from .api import (GdrError, alloc_outputs, conv1d_bwd, gdr_bwd, gdr_fwd, gdr_fwd_states, kda_bwd, kda_fwd,
                  make_shape, states_bytes, workspace_bytes, workspace_status)

__all__ = ["GdrError", "alloc_outputs", "conv1d_bwd", "gdr_bwd", "gdr_fwd", "gdr_fwd_states", "kda_bwd",
           "kda_fwd", "make_shape", "states_bytes", "workspace_bytes", "workspace_status"]
