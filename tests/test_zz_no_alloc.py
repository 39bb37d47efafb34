"""The workspace-free forward entry point (mesa_forward_chunked_noalloc) against the regular
one, through the C ABI.

It serves callers that cannot allocate device memory where they run the layer (a host that
owns all GPU memory, a plugin that only gets its input and output buffers, code recorded
into a CUDA graph); its scratch is a fixed 32 MiB array inside the library.  This file is
collected last so that a run stopping at the first failure has run every other test first;
it passes alone in a fresh process too.
"""
import numpy as np
import pytest

from mesa_layer_gb300 import synth
from helpers import TOL, torch_inputs, unit_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mesa_layer_gb300 import binding, build
    build.build()
    binding.load()


@pytest.mark.parametrize("name,overrides", [
    ("fwd_fp32_d64", {}),                                  # fp32 SIMT path, whole workload
    ("fwd_bf16_d128", {"B": 1, "H": 2, "T": 520}),         # tensor-core path, ragged tail
])
def test_noalloc_matches_regular_entry_point_twice(name, overrides):
    import torch

    from mesa_layer_gb300 import binding
    w = synth.workload(name, **overrides)
    t = torch_inputs(synth.forward_inputs(w, seed=21), w.dtype)
    need = binding.mesa_forward_workspace_size(w.B, w.H, w.T, w.dk, w.dv, w.chunk)
    assert need <= binding.NOALLOC_MAX_BYTES
    ref, ref_it = binding.mesa_forward_chunked(t["q"], t["k"], t["v"], t["gamma"], t["lam"],
                                               w.cg_iters, w.cg_tol, w.chunk)
    torch.cuda.synchronize()
    ref = ref.float().cpu().numpy()[None]
    ref_it = ref_it.cpu().numpy()
    for call in range(2):  # the second call reuses the scratch the first one left behind
        out, it = binding.mesa_forward_chunked_noalloc(t["q"], t["k"], t["v"], t["gamma"], t["lam"],
                                                       w.cg_iters, w.cg_tol, w.chunk)
        torch.cuda.synchronize()
        o = out.float().cpu().numpy()[None]
        assert np.array_equal(it.cpu().numpy(), ref_it), f"call {call}: iteration counts differ"
        err = unit_err(o.reshape(-1, w.T, w.dv), ref.reshape(-1, w.T, w.dv)).max()
        assert err <= TOL[w.dtype], f"call {call}: max rel err {err:.3e}"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import torch

    from mesa_layer_gb300 import binding
    lib = binding.load()
    w = synth.workload("fwd_bf16_d128", B=8, H=16, T=4096)
    assert binding.mesa_forward_workspace_size(w.B, w.H, w.T, w.dk, w.dv, w.chunk) > binding.NOALLOC_MAX_BYTES
    x = torch.zeros(16, device="cuda")
    p = lambda: __import__("ctypes").c_void_p(x.data_ptr())
    st = lib.mesa_forward_chunked_noalloc(w.B, w.H, w.T, w.dk, w.dv, 1, p(), p(), p(), p(), p(), 15, 0.0, 64,
                                          p(), None, None)
    assert st == 3  # MESA_ERR_WORKSPACE, nothing enqueued
