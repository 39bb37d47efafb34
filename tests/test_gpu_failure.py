"""Failure paths on the GPU, in forms that fault and hang nothing.

* A bounded wait made to give up: the test hook mesa_debug_set_wait_limit(0) makes the
  tensor-core kernels' waits for their matrix multiplies give up at once on working code.
  The kernels set the status bit, wait (with the default limit) for the multiplies still in
  flight, release their tensor memory and return; mesa_forward_status reports
  MESA_ERR_TIMEOUT, and the next call with the default limit is clean and correct.
* Non-finite inputs (NaN, infinity) in q, k, v or gamma: every call ends, the status word
  reports MESA_ERR_NONFINITE, and the propagation is the one include/mesa.h states (q_t:
  o_t alone; k_t, v_t, gamma_t: nothing before the 128-token block holding t, nothing in
  another unit), checked bit for bit against a clean run.
"""
import numpy as np
import pytest

from mesa_layer_gb300 import synth
from helpers import forward_check, torch_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mesa_layer_gb300 import binding, build
    build.build()
    binding.load()


def _run(t, iters, tol, chunk, ws):
    import torch

    from mesa_layer_gb300 import binding
    out, it = binding.mesa_forward_chunked(t["q"], t["k"], t["v"], t["gamma"], t["lam"], iters, tol, chunk,
                                           workspace=ws)
    code, flags = binding.mesa_forward_status_code(ws)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), it.cpu().numpy(), code, flags


def _workspace(w):
    import torch

    from mesa_layer_gb300 import binding
    n = binding.mesa_forward_workspace_size(w.B, w.H, w.T, w.dk, w.dv, w.chunk)
    return torch.empty(n, dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_wait_give_up_reports_timeout_and_the_next_call_is_clean(dtype, d):
    from mesa_layer_gb300 import binding
    # (fp32: the fp32 workload's Lambda range; with the bf16 workload's, down to 0.05, a plain
    # fp32 restatement of these 12 un-converged iterations already lands at 1.03e-4)
    w = synth.workload("fwd_bf16_d128" if dtype == "bf16" else "fwd_fp32_d64", dtype=dtype, dk=d, dv=d, B=1, H=2,
                       T=300, cg_iters=12, cg_tol=0.0)
    inp = synth.forward_inputs(w, seed=21)
    t = torch_inputs(inp, dtype)
    ws = _workspace(w)
    binding.mesa_debug_set_wait_limit(0)
    try:
        _, _, code, flags = _run(t, w.cg_iters, 0.0, w.chunk, ws)
    finally:
        binding.mesa_debug_set_wait_limit(-1)
    assert code == binding.MESA_ERR_TIMEOUT and flags & 1, (code, flags)
    assert not flags & 4, "the drain of the in-flight multiplies expired"
    o, it, code, flags = _run(t, w.cg_iters, 0.0, w.chunk, ws)
    assert code == binding.MESA_OK and flags == 0
    r = forward_check(inp, o, it, dtype, w.cg_iters, 0.0, "after a give-up")
    print(f"after a give-up: {r}")


PATHS = {
    # name: (dtype, d, chunk)
    "tensor_core": ("bf16", 128, 64),
    "tensor_core_fp32_d64": ("f32", 64, 64),
    "rows_fp32_d32": ("f32", 32, 64),
    "simt_fp32_d128": ("f32", 128, 64),
}
T_BAD = 150  # token with the planted value (inside the 128-token block [128, 256))


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("where", ["q_nan", "q_inf", "k_inf", "v_nan", "gamma_nan"])
def test_nonfinite_inputs(path, where):
    from mesa_layer_gb300 import binding
    dtype, d, chunk = PATHS[path]
    w = synth.workload("fwd_fp32_d64", dtype=dtype, B=1, H=2, T=300, dk=d, dv=d, chunk=chunk,
                       cg_iters=30, cg_tol=1e-3)
    inp = synth.forward_inputs(w, seed=22)
    ws = _workspace(w)
    o0, it0, code, _ = _run(torch_inputs(inp, dtype), w.cg_iters, w.cg_tol, chunk, ws)
    assert code == binding.MESA_OK
    bad = {k: v.copy() for k, v in inp.items()}
    name, kind = where.split("_")
    val = np.float32(np.nan if kind == "nan" else np.inf)
    if name == "gamma":
        bad["gamma"][0, 0, T_BAD] = val
    else:
        bad[name][0, 0, T_BAD, 3] = val
    o1, it1, code, flags = _run(torch_inputs(bad, dtype), w.cg_iters, w.cg_tol, chunk, ws)
    # the other unit: bit for bit the clean run
    assert np.array_equal(o1[0, 1], o0[0, 1]) and np.array_equal(it1[0, 1], it0[0, 1])
    if where == "q_inf" and np.isfinite(o1[0, 0, T_BAD]).all():
        # an infinite query meets the dynamic stopping rule at once (inf <= tol * inf): o_t = 0
        assert it1[0, 0, T_BAD] == 0 and np.all(o1[0, 0, T_BAD] == 0)
        assert code == binding.MESA_OK and flags == 0
    else:
        assert not np.isfinite(o1[0, 0, T_BAD]).all()
        assert code == binding.MESA_ERR_NONFINITE and flags == 2, (code, flags)
    if name == "q":  # the query enters its own token's solve only
        keep = np.ones(w.T, dtype=bool)
        keep[T_BAD] = False
    else:            # keys, values and gates enter every later state
        keep = np.arange(w.T) < (T_BAD // 128) * 128
    assert np.array_equal(o1[0, 0, keep], o0[0, 0, keep])
    assert np.array_equal(it1[0, 0, keep], it0[0, 0, keep])
    # and the next clean call reports nothing
    _, _, code, flags = _run(torch_inputs(inp, dtype), w.cg_iters, w.cg_tol, chunk, ws)
    assert code == binding.MESA_OK and flags == 0


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("where", ["q", "k", "v", "gamma"])
def test_nonfinite_decode_inputs(d, where):
    import torch

    from mesa_layer_gb300 import binding
    w = synth.workload("decode_bf16_d128", B=3, H=2, dk=d, dv=d)
    lam = torch.from_numpy(synth.lambdas(w)).cuda()
    H1 = torch.zeros(w.B, w.H, d, d, device="cuda")
    G1 = torch.zeros_like(H1)

    def dev(x):
        return {k: torch.from_numpy(x[k]).cuda().to(torch.bfloat16 if k != "gamma" else torch.float32)
                for k in ("q", "k", "v", "gamma")}

    for s in range(-16, 0):
        x = dev(synth.decode_inputs(w, s))
        binding.mesa_decode_step(H1, G1, x["q"], x["k"], x["v"], x["gamma"], lam, 0, 0.0)
    assert binding.mesa_decode_status()[0] == binding.MESA_OK
    H2, G2 = H1.clone(), G1.clone()
    inp = synth.decode_inputs(w, 0)
    o1, i1 = binding.mesa_decode_step(H1, G1, **{k: v for k, v in dev(inp).items()}, lambda_diag=lam,
                                      cg_iters=w.cg_iters, cg_tol=w.cg_tol)
    assert binding.mesa_decode_status()[0] == binding.MESA_OK
    bad = {k: v.copy() for k, v in inp.items()}
    if where == "gamma":
        bad["gamma"][1, 0] = np.nan
    else:
        bad[where][1, 0, 5] = np.nan
    o2, i2 = binding.mesa_decode_step(H2, G2, **{k: v for k, v in dev(bad).items()}, lambda_diag=lam,
                                      cg_iters=w.cg_iters, cg_tol=w.cg_tol)
    code, flags = binding.mesa_decode_status()
    assert code == binding.MESA_ERR_NONFINITE and flags == 2, (code, flags)
    assert binding.mesa_decode_status() == (binding.MESA_OK, 0)  # the query cleared it
    other = np.ones((w.B, w.H), dtype=bool)
    other[1, 0] = False
    for a, b in ((o1, o2), (i1, i2), (H1, H2), (G1, G2)):
        a, b = a.float().cpu().numpy(), b.float().cpu().numpy()
        assert np.array_equal(a[other], b[other])
    assert not np.isfinite(o2[1, 0].float().cpu().numpy()).all()


def test_decode_wait_give_up_reports_timeout_and_leaves_the_state():
    """d = 128 decode: its bounded wait for the bulk copy of H made to give up at once; the
    step reports MESA_ERR_TIMEOUT through mesa_decode_status, leaves H and G as they were, and
    the next step with the default limit is clean and equals a step from the same state."""
    import torch

    from mesa_layer_gb300 import binding
    w = synth.workload("decode_bf16_d128", B=3, H=2)
    lam = torch.from_numpy(synth.lambdas(w)).cuda()
    H1 = torch.zeros(w.B, w.H, 128, 128, device="cuda")
    G1 = torch.zeros_like(H1)

    def dev(x):
        return {k: torch.from_numpy(x[k]).cuda().to(torch.bfloat16 if k != "gamma" else torch.float32)
                for k in ("q", "k", "v", "gamma")}

    for s in range(-16, 0):
        x = dev(synth.decode_inputs(w, s))
        binding.mesa_decode_step(H1, G1, x["q"], x["k"], x["v"], x["gamma"], lam, 0, 0.0)
    assert binding.mesa_decode_status()[0] == binding.MESA_OK
    H0, G0 = H1.clone(), G1.clone()
    x = dev(synth.decode_inputs(w, 0))
    binding.mesa_debug_set_wait_limit(0)
    try:
        binding.mesa_decode_step(H1, G1, **x, lambda_diag=lam, cg_iters=w.cg_iters, cg_tol=w.cg_tol)
    finally:
        binding.mesa_debug_set_wait_limit(-1)
    code, flags = binding.mesa_decode_status()
    assert code == binding.MESA_ERR_TIMEOUT and flags & 1 and not flags & 4, (code, flags)
    assert torch.equal(H1, H0) and torch.equal(G1, G0)
    o1, i1 = binding.mesa_decode_step(H1, G1, **x, lambda_diag=lam, cg_iters=w.cg_iters, cg_tol=w.cg_tol)
    assert binding.mesa_decode_status() == (binding.MESA_OK, 0)
    H2, G2 = H0.clone(), G0.clone()
    o2, i2 = binding.mesa_decode_step(H2, G2, **x, lambda_diag=lam, cg_iters=w.cg_iters, cg_tol=w.cg_tol)
    assert torch.equal(o1, o2) and torch.equal(i1, i2) and torch.equal(H1, H2) and torch.equal(G1, G2)


def test_backward_wait_give_up_reports_timeout_and_the_next_call_is_clean():
    """The backward's tensor-core kernels (bf16, d = 128: the solves, the state sweeps and the
    products of the rows with the chunk states) made to give up their waits at once: the
    status word reports MESA_ERR_TIMEOUT with no expired drain, and the next call with the
    default limit equals a call that never gave up, bit for bit."""
    import torch

    from mesa_layer_gb300 import binding
    w = synth.workload("fwd_bf16_d128", B=1, H=2, T=300, cg_iters=10, cg_tol=0.0)
    inp = synth.forward_inputs(w, seed=23)
    t = torch_inputs(inp, "bf16")
    g = torch.Generator().manual_seed(5)
    dout = torch.randn(t["q"].shape, generator=g).to(torch.bfloat16).cuda()
    ws = torch.empty(binding.mesa_backward_workspace_size(w.B, w.H, w.T, w.dk, w.dv), dtype=torch.uint8,
                     device="cuda")

    def call():
        r = binding.mesa_backward_chunked(t["q"], t["k"], t["v"], t["gamma"], t["lam"], dout, w.cg_iters, 0.0,
                                          workspace=ws)
        code, flags = binding.mesa_forward_status_code(ws)
        torch.cuda.synchronize()
        return [x.float().cpu() for x in r[:5]], code, flags

    clean, code, flags = call()
    assert code == binding.MESA_OK and flags == 0
    binding.mesa_debug_set_wait_limit(0)
    try:
        _, code, flags = call()
    finally:
        binding.mesa_debug_set_wait_limit(-1)
    assert code == binding.MESA_ERR_TIMEOUT and flags & 1, (code, flags)
    assert not flags & 4, "the drain of the in-flight multiplies expired"
    again, code, flags = call()
    assert code == binding.MESA_OK and flags == 0
    for a, b in zip(again, clean):
        assert torch.equal(a, b)
