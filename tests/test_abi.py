"""Host-side checks of the C ABI (no GPU needed): the library builds, loads, exports every
function include/mesa.h declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

from mesa_layer_gb300 import binding, build

HEADER_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


def declared_functions():
    names = []
    for fn in sorted(os.listdir(HEADER_DIR)):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(mesa_\w+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("mesa_forward_chunked", "mesa_decode_step", "mesa_forward_workspace_size"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_version_and_status_strings(lib):
    assert lib.mesa_version() >= 100
    assert lib.mesa_status_string(0) == b"ok"
    assert lib.mesa_status_string(3).startswith(b"workspace")
    assert b"wait" in lib.mesa_status_string(5) and b"non-finite" in lib.mesa_status_string(6)


def test_status_queries_and_wait_limit_hook_validate_on_the_host(lib):
    """The status queries reject a null flags pointer before touching a stream, and the
    wait-limit hook only records a host-side number (range-checked)."""
    assert lib.mesa_decode_status(None, None) == 1
    assert lib.mesa_forward_status(None, None, None) == 1
    assert lib.mesa_debug_set_wait_limit(1 << 33) == 1
    assert lib.mesa_debug_set_wait_limit(0) == 0
    assert lib.mesa_debug_set_wait_limit(-1) == 0


def test_workspace_size(lib):
    ws = lib.mesa_forward_workspace_size
    assert ws(1, 1, 256, 16, 16, 64) >= 4 * (256 + 2 * 4 * 16 * 16)
    assert ws(1, 1, 100, 16, 16, 32) <= ws(1, 1, 128, 16, 16, 32)   # ragged last chunk
    assert ws(1, 1, 256, 17, 17, 64) == 0     # unsupported d
    assert ws(1, 1, 256, 64, 32, 64) == 0     # dk != dv
    assert ws(1, 1, 256, 64, 64, 48) == 0     # unsupported chunk
    # state sections scale with the number of working chunks: ceil(T / chunk) for d = 128,
    # ceil(T / min(chunk, 32)) for d <= 64 (the fp32 CUDA-core path's chunk cap)
    assert ws(2, 4, 2048, 128, 128, 64) > ws(2, 4, 2048, 128, 128, 128)
    assert ws(2, 4, 2048, 64, 64, 16) > ws(2, 4, 2048, 64, 64, 32)
    assert ws(2, 4, 2048, 64, 64, 32) == ws(2, 4, 2048, 64, 64, 64) == ws(2, 4, 2048, 64, 64, 128)


def _fwd(lib, **kw):
    args = dict(B=1, H=1, T=64, dk=16, dv=16, dtype=0, q=8, k=8, v=8, gamma=8, lam=8, iters=4, tol=0.0,
                chunk=64, out=8, it=None, H0=None, G0=None, Hf=None, Gf=None, ws=256, wsb=1 << 20)
    args.update(kw)
    a = args
    return lib.mesa_forward_chunked(a["B"], a["H"], a["T"], a["dk"], a["dv"], a["dtype"], a["q"], a["k"],
                                    a["v"], a["gamma"], a["lam"], a["iters"], a["tol"], a["chunk"], a["out"],
                                    a["it"], a["H0"], a["G0"], a["Hf"], a["Gf"], a["ws"], a["wsb"], None)


def test_forward_rejects_bad_arguments_without_launching(lib):
    # every case below returns before any CUDA call, so it runs without a GPU
    assert _fwd(lib, dk=24, dv=24) == 2
    assert _fwd(lib, dk=64, dv=32) == 2
    assert _fwd(lib, chunk=48) == 2
    assert _fwd(lib, B=-1) == 1
    assert _fwd(lib, iters=-1) == 1
    assert _fwd(lib, iters=100000) == 1
    assert _fwd(lib, dtype=7) == 1
    assert _fwd(lib, tol=float("nan")) == 1
    assert _fwd(lib, H0=8) == 1               # H0 without G0
    assert _fwd(lib, Hf=8) == 1               # H_final without G_final
    assert _fwd(lib, q=None) == 1
    assert _fwd(lib, ws=None) == 3
    assert _fwd(lib, wsb=16) == 3
    assert _fwd(lib, ws=264) == 3             # misaligned workspace
    assert _fwd(lib, B=0) == 0                # empty batch: nothing to do
    assert _fwd(lib, T=0) == 0                # empty sequence: nothing to do


def test_decode_rejects_bad_arguments_without_launching(lib):
    f = lib.mesa_decode_step
    base = [1, 1, 16, 16, 0, 16, 16, 8, 8, 8, 8, 8, 4, 0.0, 8, None, None]
    def call(i, val):
        a = list(base)
        a[i] = val
        return f(*a)
    assert call(2, 20) == 2 and call(3, 32) == 2
    assert call(0, -1) == 1 and call(12, -2) == 1 and call(4, 3) == 1
    assert call(5, None) == 1 and call(14, None) == 1
    assert call(5, 20) == 1                   # H_state not 16-byte aligned
    assert call(0, 0) == 0                    # no sequences


def test_binding_raises_without_gpu_or_library():
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    q = torch.zeros(1, 1, 4, 16)
    with pytest.raises(Exception):
        binding.mesa_forward_chunked(q, q, q, torch.ones(1, 1, 4), torch.ones(1, 16), 2, 0.0, 16)


def test_qk_preprocess_validation(lib):
    f = lib.mesa_qk_preprocess
    p = ctypes.c_void_p(256)
    args = lambda **kw: [kw.get(k, v) for k, v in dict(B=1, H=2, T=8, d=64, W=4, dtype=0, q=p, k=p, wq=p, wk=p,
                                                     qo=ctypes.c_void_p(512), ko=ctypes.c_void_p(768), st=None).items()]
    assert f(*args(W=0)) == 1 and f(*args(W=9)) == 1          # window out of range
    assert f(*args(dtype=5)) == 1
    assert f(*args(d=48)) == 2                                  # unsupported channel count
    assert f(*args(B=70000)) == 2                               # B * H over the grid limit
    assert f(*args(q=None)) == 1 and f(*args(wk=None)) == 1
    assert f(*args(qo=p)) == 1                                  # output aliases the input
    assert f(*args(q=ctypes.c_void_p(264))) == 1                # misaligned activation
    assert f(*args(T=0)) == 0                                   # nothing to do, nothing enqueued


def test_qk_preprocess_step_validation(lib):
    f = lib.mesa_qk_preprocess_step
    p = ctypes.c_void_p(256)
    args = lambda **kw: [kw.get(k, v) for k, v in dict(N=2, H=2, d=32, W=3, dtype=1, q=p, k=p, wq=p, wk=p,
                                                     cs=p, qo=p, ko=p, st=None).items()]
    assert f(*args(W=0)) == 1 and f(*args(W=9)) == 1
    assert f(*args(d=24)) == 2
    assert f(*args(cs=None)) == 1                               # a window needs its state
    assert f(*args(cs=ctypes.c_void_p(264))) == 1               # misaligned state
    assert f(*args(N=0)) == 0


def test_decode_step_warm_validation(lib):
    f = lib.mesa_decode_step_warm  # argument types set by the binding
    p = ctypes.c_void_p(256)
    def call(**kw):
        a = dict(N=2, H=2, dk=64, dv=64, dt=1, Hs=p, Gs=p, Xs=p, q=p, k=p, v=p, g=p, lam=p, it=5, tol=0.0,
                 out=p, its=None, st=None)
        a.update(kw)
        return f(a["N"], a["H"], a["dk"], a["dv"], a["dt"], a["Hs"], a["Gs"], a["Xs"], a["q"], a["k"], a["v"],
                 a["g"], a["lam"], a["it"], a["tol"], a["out"], a["its"], a["st"])
    assert call(Xs=None) == 1                        # the start vectors are required
    assert call(Xs=ctypes.c_void_p(264)) == 1        # misaligned start vectors
    assert call(dk=48, dv=48) == 2
    assert call(it=-1) == 1
    assert call(N=0) == 0


def test_backward_workspace_and_validation(lib):
    ws = lib.mesa_backward_workspace_size
    assert ws(2, 3, 100, 48, 48) == 0          # unsupported d
    assert ws(2, 3, 100, 64, 32) == 0          # dk != dv
    small, big = ws(2, 3, 100, 64, 64), ws(2, 3, 1000, 64, 64)
    assert 0 < small < big
    # d = 128 also holds the 128-token states of the tensor-core solves, and the four fp32
    # products of each token's row with the chunk states (4 T d floats per unit) with one
    # Frobenius pair per 32-token chunk
    assert ws(1, 1, 256, 128, 128) > 2 * ws(1, 1, 256, 64, 64)
    assert ws(1, 1, 256, 128, 128) >= 4 * 4 * 256 * 128 + 4 * (256 // 32) + 2 * 4 * (256 // 32) * 128 * 128
    f = lib.mesa_backward_chunked  # argument types set by the binding
    p = ctypes.c_void_p(256)

    def call(**kw):
        a = dict(B=2, H=2, T=64, dk=64, dv=64, dt=1, q=p, k=p, v=p, g=p, lam=p, do=p, xs=None, it=5, tol=0.0,
                 dq=p, dk_=p, dv_=p, dg=p, dl=p, itf=None, itb=None, ws=p, wsz=1 << 40, st=None)
        a.update(kw)
        return f(a["B"], a["H"], a["T"], a["dk"], a["dv"], a["dt"], a["q"], a["k"], a["v"], a["g"], a["lam"],
                 a["do"], a["xs"], a["it"], a["tol"], a["dq"], a["dk_"], a["dv_"], a["dg"], a["dl"], a["itf"],
                 a["itb"], a["ws"], a["wsz"], a["st"])
    assert call(dk=48, dv=48) == 2
    assert call(dv=32) == 2
    assert call(it=-1) == 1
    assert call(dt=7) == 1
    assert call(do=None) == 1
    assert call(dl=None) == 1
    assert call(dg=None) == 1
    assert call(wsz=1000) == 3                 # workspace too small
    assert call(ws=ctypes.c_void_p(264)) == 3  # workspace not 256-byte aligned
    assert call(B=0, H=0) == 0                 # nothing to do, nothing launched
    assert call(q=ctypes.c_void_p(264)) == 1   # operands must be 16-byte aligned
    assert call(dv_=ctypes.c_void_p(264)) == 1
    assert call(xs=ctypes.c_void_p(264)) == 1   # saved iterates must be 16-byte aligned
    fs = lib.mesa_forward_chunked_save          # the saved iterates are required
    assert fs(1, 1, 64, 64, 64, 0, p, p, p, p, p, 4, 0.0, 64, p, None, None, p, 1 << 40, None) == 1


def test_fused_preprocessing_forward_validation(lib):
    """mesa_forward_chunked_pre: workspace sizes (fused: the forward's; otherwise two more
    activation buffers) and argument checks before anything is launched."""
    fw = lib.mesa_forward_workspace_size(2, 4, 300, 128, 128, 64)
    assert lib.mesa_forward_pre_workspace_size(2, 4, 300, 128, 128, 64, 1) == fw
    fw64 = lib.mesa_forward_workspace_size(2, 4, 300, 64, 64, 64)
    assert lib.mesa_forward_pre_workspace_size(2, 4, 300, 64, 64, 64, 0) >= fw64 + 2 * 2 * 4 * 300 * 64 * 4
    assert lib.mesa_forward_pre_workspace_size(2, 4, 300, 64, 64, 64, 7) == 0
    f = lib.mesa_forward_chunked_pre
    f.restype = ctypes.c_int
    vp = ctypes.c_void_p
    f.argtypes = [ctypes.c_int] * 6 + [vp, vp, vp, vp, ctypes.c_int, vp, vp, vp, ctypes.c_int, ctypes.c_float,
                                       ctypes.c_int, vp, vp, vp, ctypes.c_size_t, vp]
    p = vp(4096)  # never dereferenced: every call below fails validation first
    args = lambda W=4, dt=1, ws=p, nbytes=1 << 30, q=p: (1, 2, 300, 128, 128, dt, q, p, p, p, W, p, p, p, 8, 0.0,
                                                         64, p, None, ws, nbytes, None)
    assert f(*args(W=0)) == 1 and f(*args(W=9)) == 1
    assert f(*args(dt=3)) == 1
    assert f(*args(q=None)) == 1
    assert f(*args(q=vp(4098))) == 1          # misaligned activations
    assert f(*args(ws=None)) == 3 and f(*args(nbytes=16)) == 3
