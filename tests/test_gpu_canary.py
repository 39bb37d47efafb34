"""Out-of-bounds writes (a sanitizer stand-in): every buffer a call writes -- workspace,
outputs, iteration counts, final states, decode states -- is carved out of a larger byte
buffer whose 4 KB before and after it hold a fixed pattern; after the call the pattern must
be intact.  The workspace is handed over at exactly the size the library asked for."""
import numpy as np
import pytest

from mesa_layer_gb300 import synth
from helpers import torch_inputs

pytestmark = pytest.mark.gpu
PAD = 4096
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mesa_layer_gb300 import binding, build
    build.build()
    binding.load()


class Guarded:
    """`shape` of `dtype` inside a pattern-filled byte buffer (PAD bytes on each side)."""

    def __init__(self, shape, dtype, init=None):
        import torch
        n = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
        self.buf = torch.full((PAD + n + PAD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.t = self.buf[PAD:PAD + n].view(dtype).view(shape)
        if init is not None:
            self.t.copy_(init)

    def intact(self):
        import torch
        torch.cuda.synchronize()
        return bool((self.buf[:PAD] == PATTERN).all() and (self.buf[-PAD:] == PATTERN).all())


def workspace(nbytes):
    import torch
    return Guarded((nbytes,), torch.uint8)


FWD = [
    # (dtype, d, T, iters, tol, chunk): the four compute paths, ragged tails
    ("bf16", 128, 300, 30, 1e-3, 64),   # tensor cores, bf16
    ("f32", 64, 300, 20, 1e-4, 64),     # tensor cores, fp32 d = 64
    ("f32", 32, 77, 12, 0.0, 32),       # CUDA cores, d <= 32
    ("f32", 128, 130, 10, 0.0, 64),     # CUDA cores, d = 128
]


@pytest.mark.parametrize("case", FWD, ids=lambda c: f"{c[0]}-d{c[1]}")
def test_forward_writes_stay_inside_their_buffers(case):
    import torch

    from mesa_layer_gb300 import binding
    dtype, d, T, iters, tol, chunk = case
    w = synth.workload("fwd_fp32_d64", dtype=dtype, B=2, H=2, T=T, dk=d, dv=d, chunk=chunk)
    t = torch_inputs(synth.forward_inputs(w, seed=31), dtype)
    td = t["q"].dtype
    ws = workspace(binding.mesa_forward_workspace_size(w.B, w.H, T, d, d, chunk))
    out = Guarded((w.B, w.H, T, d), td)
    it = Guarded((w.B, w.H, T), torch.int32)
    Hf = Guarded((w.B, w.H, d, d), torch.float32)
    Gf = Guarded((w.B, w.H, d, d), torch.float32)
    binding.mesa_forward_chunked(t["q"], t["k"], t["v"], t["gamma"], t["lam"], iters, tol, chunk, out=out.t,
                                 iters_used=it.t, H_final=Hf.t, G_final=Gf.t, workspace=ws.t)
    for name, g in (("workspace", ws), ("out", out), ("iters", it), ("H_final", Hf), ("G_final", Gf)):
        assert g.intact(), f"a write landed next to {name}"
    assert binding.mesa_forward_status(ws.t) == 0


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("warm", [False, True])
def test_decode_writes_stay_inside_their_buffers(d, warm):
    import torch

    from mesa_layer_gb300 import binding
    w = synth.workload("decode_bf16_d128", B=3, H=2, dk=d, dv=d)
    lam = torch.from_numpy(synth.lambdas(w)).cuda()
    Hs = Guarded((w.B, w.H, d, d), torch.float32, torch.zeros(w.B, w.H, d, d))
    Gs = Guarded((w.B, w.H, d, d), torch.float32, torch.zeros(w.B, w.H, d, d))
    Xs = Guarded((w.B, w.H, d), torch.float32, torch.zeros(w.B, w.H, d))
    out = Guarded((w.B, w.H, d), torch.bfloat16)
    it = Guarded((w.B, w.H), torch.int32)
    for s in range(-4, 3):
        x = synth.decode_inputs(w, s)
        x = {k: torch.from_numpy(x[k]).cuda().to(torch.bfloat16 if k != "gamma" else torch.float32)
             for k in ("q", "k", "v", "gamma")}
        n = w.cg_iters if s >= 0 else 0
        if warm:
            binding.mesa_decode_step_warm(Hs.t, Gs.t, Xs.t, x["q"], x["k"], x["v"], x["gamma"], lam, n, w.cg_tol,
                                          out=out.t, iters_used=it.t)
        else:
            binding.mesa_decode_step(Hs.t, Gs.t, x["q"], x["k"], x["v"], x["gamma"], lam, n, w.cg_tol,
                                     out=out.t, iters_used=it.t)
    for name, g in (("H", Hs), ("G", Gs), ("X", Xs), ("out", out), ("iters", it)):
        assert g.intact(), f"a write landed next to {name}"
    assert binding.mesa_decode_status()[0] == binding.MESA_OK


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_preprocess_writes_stay_inside_their_buffers(dtype):
    import torch

    from mesa_layer_gb300 import binding
    w = synth.workload("qkpre_bf16_d128", dtype=dtype, B=1, H=3, T=333, dk=128, dv=128)
    inp = synth.preprocess_inputs(w, taps=4, seed=32)
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    q = torch.from_numpy(inp["q_raw"]).cuda().to(td)
    k = torch.from_numpy(inp["k_raw"]).cuda().to(td)
    wq, wk = torch.from_numpy(inp["wq"]).cuda(), torch.from_numpy(inp["wk"]).cuda()
    qo, ko = Guarded(q.shape, td), Guarded(k.shape, td)
    binding.mesa_qk_preprocess(q, k, wq, wk, q_out=qo.t, k_out=ko.t)
    assert qo.intact() and ko.intact()


def test_backward_writes_stay_inside_their_buffers():
    import torch

    from mesa_layer_gb300 import binding
    w = synth.workload("bwd_bf16_d128", B=1, H=2, T=200, cg_iters=8)
    inp = synth.backward_inputs(w, seed=33)
    t = torch_inputs(inp, "bf16")
    dout = torch.from_numpy(inp["dout"]).cuda().to(torch.bfloat16)
    ws = workspace(binding.mesa_backward_workspace_size(w.B, w.H, w.T, 128, 128))
    g = {"dq": Guarded((w.B, w.H, w.T, 128), torch.bfloat16), "dk": Guarded((w.B, w.H, w.T, 128), torch.bfloat16),
         "dv": Guarded((w.B, w.H, w.T, 128), torch.bfloat16), "dgamma": Guarded((w.B, w.H, w.T), torch.float32),
         "dlambda": Guarded((w.H, 128), torch.float32), "iters_fwd": Guarded((w.B, w.H, w.T), torch.int32),
         "iters_bwd": Guarded((w.B, w.H, w.T), torch.int32)}
    binding.mesa_backward_chunked(t["q"], t["k"], t["v"], t["gamma"], t["lam"], dout, w.cg_iters, 0.0,
                                  workspace=ws.t, **{k: v.t for k, v in g.items()})
    assert ws.intact(), "a write landed next to the workspace"
    for name, b in g.items():
        assert b.intact(), f"a write landed next to {name}"
