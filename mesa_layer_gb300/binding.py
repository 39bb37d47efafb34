"""Thin ctypes binding of libmesa_gb300.so (include/mesa.h).

Argument marshalling only: torch tensors supply device pointers and the current CUDA
stream; every step of the computation runs in the library's kernels.  Output tensors and
the workspace are allocated with torch on the caller's side when not given.  There is no
CPU fallback: if the library is missing or no GPU is present, calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

MESA_F32, MESA_BF16 = 0, 1
MESA_OK, MESA_ERR_TIMEOUT, MESA_ERR_NONFINITE = 0, 5, 6
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported size or option",
           3: "workspace missing or too small", 4: "CUDA launch failed",
           5: "a bounded device wait gave up", 6: "a kernel wrote a non-finite value"}

_lib = None
_vp, _fp, _ip = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
_i, _f, _sz = ctypes.c_int, ctypes.c_float, ctypes.c_size_t


class MesaError(RuntimeError):
    pass


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load the shared library (building it first if it is missing and nvcc exists)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise MesaError(f"{path} is not built: call mesa_layer_gb300.build.build()")
        _build.build()
    lib = ctypes.CDLL(path)
    lib.mesa_version.restype = _i
    lib.mesa_status_string.restype = ctypes.c_char_p
    lib.mesa_status_string.argtypes = [_i]
    lib.mesa_forward_workspace_size.restype = _sz
    lib.mesa_forward_workspace_size.argtypes = [_i] * 6
    lib.mesa_forward_chunked.restype = _i
    lib.mesa_forward_chunked.argtypes = [_i] * 6 + [_vp] * 5 + [_i, _f, _i, _vp, _ip] + \
        [_fp] * 4 + [_vp, _sz, _vp]
    lib.mesa_forward_chunked_noalloc.restype = _i
    lib.mesa_forward_chunked_noalloc.argtypes = [_i] * 6 + [_vp] * 5 + [_i, _f, _i, _vp, _ip, _vp]
    lib.mesa_forward_pre_workspace_size.restype = _sz
    lib.mesa_forward_pre_workspace_size.argtypes = [_i] * 7
    lib.mesa_forward_chunked_pre.restype = _i
    lib.mesa_forward_chunked_pre.argtypes = [_i] * 6 + [_vp, _vp, _fp, _fp, _i, _vp, _fp, _fp, _i, _f, _i, _vp, _ip,
                                                        _vp, _sz, _vp]
    lib.mesa_forward_status.restype = _i
    lib.mesa_forward_status.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_uint)]
    lib.mesa_decode_status.restype = _i
    lib.mesa_decode_status.argtypes = [_vp, ctypes.POINTER(ctypes.c_uint)]
    lib.mesa_debug_set_wait_limit.restype = _i
    lib.mesa_debug_set_wait_limit.argtypes = [ctypes.c_longlong]
    lib.mesa_tc_selftest.restype = _i
    lib.mesa_tc_selftest.argtypes = [_vp] * 6 + [_vp]
    lib.mesa_decode_step.restype = _i
    lib.mesa_decode_step.argtypes = [_i] * 5 + [_fp, _fp, _vp, _vp, _vp, _fp, _fp, _i, _f, _vp, _ip, _vp]
    lib.mesa_decode_step_warm.restype = _i
    lib.mesa_decode_step_warm.argtypes = [_i] * 5 + [_fp, _fp, _fp, _vp, _vp, _vp, _fp, _fp, _i, _f, _vp, _ip, _vp]
    lib.mesa_qk_preprocess.restype = _i
    lib.mesa_qk_preprocess.argtypes = [_i] * 6 + [_vp, _vp, _fp, _fp, _vp, _vp, _vp]
    lib.mesa_qk_preprocess_step.restype = _i
    lib.mesa_qk_preprocess_step.argtypes = [_i] * 5 + [_vp, _vp, _fp, _fp, _fp, _vp, _vp, _vp]
    lib.mesa_backward_workspace_size.restype = _sz
    lib.mesa_backward_workspace_size.argtypes = [_i] * 5
    lib.mesa_backward_chunked.restype = _i
    lib.mesa_backward_chunked.argtypes = [_i] * 6 + [_vp] * 3 + [_fp, _fp, _vp, _fp, _i, _f] + [_vp] * 3 + [
        _fp, _fp, _ip, _ip, _vp, _sz, _vp]
    lib.mesa_forward_chunked_save.restype = _i
    lib.mesa_forward_chunked_save.argtypes = [_i] * 6 + [_vp] * 5 + [_i, _f, _i, _vp, _ip, _fp, _vp, _sz, _vp]
    _lib = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(status: int, what: str):
    if status != 0:
        raise MesaError(f"{what}: {_STATUS.get(status, status)}")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return MESA_F32
    if t.dtype == torch.bfloat16:
        return MESA_BF16
    raise MesaError(f"unsupported dtype {t.dtype}: use float32 or bfloat16")


def _require(t, name, dtype=None, device=None):
    if t is None:
        return
    if not t.is_cuda:
        raise MesaError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise MesaError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise MesaError(f"{name} must be {dtype}, got {t.dtype}")


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def mesa_forward_workspace_size(B, H, T, dk, dv, chunk) -> int:
    return int(load().mesa_forward_workspace_size(B, H, T, dk, dv, chunk))


def mesa_forward_chunked(q, k, v, gamma, lambda_diag, cg_iters, cg_tol, chunk, out=None,
                         iters_used=None, H0=None, G0=None, H_final=None, G_final=None,
                         workspace=None, stream=None):
    """Chunked Mesa layer forward.  q, k [B, H, T, dk], v [B, H, T, dv] (fp32 or bf16),
    gamma [B, H, T] fp32, lambda_diag [H, dk] fp32.  Returns (out, iters_used)."""
    lib = load()
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    code = _dtype_code(q)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _require(t, name, q.dtype)
    _require(gamma, "gamma", torch.float32)
    _require(lambda_diag, "lambda_diag", torch.float32)
    for name, t in (("H0", H0), ("G0", G0), ("H_final", H_final), ("G_final", G_final)):
        _require(t, name, torch.float32)
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=q.dtype, device=q.device)
    if iters_used is None:
        iters_used = torch.empty((B, H, T), dtype=torch.int32, device=q.device)
    _require(out, "out", q.dtype)
    _require(iters_used, "iters_used", torch.int32)
    need = mesa_forward_workspace_size(B, H, T, dk, dv, chunk)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _require(workspace, "workspace")
    st = lib.mesa_forward_chunked(B, H, T, dk, dv, code, _ptr(q), _ptr(k), _ptr(v), _ptr(gamma),
                                  _ptr(lambda_diag), int(cg_iters), float(cg_tol), int(chunk),
                                  _ptr(out), _ptr(iters_used), _ptr(H0), _ptr(G0), _ptr(H_final),
                                  _ptr(G_final), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "mesa_forward_chunked")
    return out, iters_used


def mesa_forward_pre_workspace_size(B, H, T, dk, dv, chunk, dtype_code) -> int:
    return int(load().mesa_forward_pre_workspace_size(B, H, T, dk, dv, chunk, dtype_code))


def mesa_forward_chunked_pre(q_raw, k_raw, wq, wk, v, gamma, lambda_diag, cg_iters, cg_tol, chunk, out=None,
                             iters_used=None, workspace=None, stream=None):
    """The query/key preprocessing (taps wq, wk [H, dk, W] fp32) and the chunked forward in one
    call (zero initial state).  q_raw, k_raw [B, H, T, dk], v [B, H, T, dv] (fp32 or bf16).
    Returns (out, iters_used)."""
    lib = load()
    B, H, T, dk = q_raw.shape
    dv = v.shape[-1]
    W = wq.shape[-1]
    code = _dtype_code(q_raw)
    for name, t in (("q_raw", q_raw), ("k_raw", k_raw), ("v", v)):
        _require(t, name, q_raw.dtype)
    for name, t in (("wq", wq), ("wk", wk), ("gamma", gamma), ("lambda_diag", lambda_diag)):
        _require(t, name, torch.float32)
    if tuple(wk.shape) != tuple(wq.shape):
        raise MesaError("wq and wk must have the same shape [H, dk, W]")
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=q_raw.dtype, device=q_raw.device)
    if iters_used is None:
        iters_used = torch.empty((B, H, T), dtype=torch.int32, device=q_raw.device)
    _require(out, "out", q_raw.dtype)
    _require(iters_used, "iters_used", torch.int32)
    need = mesa_forward_pre_workspace_size(B, H, T, dk, dv, chunk, code)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q_raw.device)
    _require(workspace, "workspace")
    st = lib.mesa_forward_chunked_pre(B, H, T, dk, dv, code, _ptr(q_raw), _ptr(k_raw), _ptr(wq), _ptr(wk), int(W),
                                      _ptr(v), _ptr(gamma), _ptr(lambda_diag), int(cg_iters), float(cg_tol),
                                      int(chunk), _ptr(out), _ptr(iters_used), _ptr(workspace), workspace.numel(),
                                      _stream(stream))
    _check(st, "mesa_forward_chunked_pre")
    return out, iters_used


def mesa_backward_workspace_size(B, H, T, dk, dv) -> int:
    return int(load().mesa_backward_workspace_size(B, H, T, dk, dv))


def mesa_forward_chunked_save(q, k, v, gamma, lambda_diag, cg_iters, cg_tol, chunk, out=None,
                              iters_used=None, x_saved=None, workspace=None, stream=None):
    """mesa_forward_chunked (zero initial state) that also returns its CG iterates x_saved
    [B, H, T, dk] fp32 for mesa_backward_chunked.  Returns (out, iters_used, x_saved)."""
    lib = load()
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    code = _dtype_code(q)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _require(t, name, q.dtype)
    _require(gamma, "gamma", torch.float32)
    _require(lambda_diag, "lambda_diag", torch.float32)
    out = torch.empty((B, H, T, dv), dtype=q.dtype, device=q.device) if out is None else out
    iters_used = torch.empty((B, H, T), dtype=torch.int32, device=q.device) if iters_used is None else iters_used
    x_saved = torch.empty((B, H, T, dk), dtype=torch.float32, device=q.device) if x_saved is None else x_saved
    _require(out, "out", q.dtype)
    _require(iters_used, "iters_used", torch.int32)
    _require(x_saved, "x_saved", torch.float32)
    need = mesa_forward_workspace_size(B, H, T, dk, dv, chunk)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _require(workspace, "workspace")
    st = lib.mesa_forward_chunked_save(B, H, T, dk, dv, code, _ptr(q), _ptr(k), _ptr(v), _ptr(gamma),
                                       _ptr(lambda_diag), int(cg_iters), float(cg_tol), int(chunk), _ptr(out),
                                       _ptr(iters_used), _ptr(x_saved), _ptr(workspace), workspace.numel(),
                                       _stream(stream))
    _check(st, "mesa_forward_chunked_save")
    return out, iters_used, x_saved


def mesa_backward_chunked(q, k, v, gamma, lambda_diag, dout, cg_iters, cg_tol, dq=None, dk=None, dv=None,
                          dgamma=None, dlambda=None, iters_fwd=None, iters_bwd=None, workspace=None,
                          stream=None, x_saved=None):
    """Backward pass of mesa_forward_chunked (zero initial states): gradients of a loss given
    dout = dL/dout [B, H, T, dv] (dtype of q).  x_saved: None (the forward's solves are
    recomputed) or the iterates from mesa_forward_chunked_save.  Returns (dq, dk, dv, dgamma,
    dlambda, iters_fwd, iters_bwd); dlambda [H, dk] is summed over the batch; iters_fwd is
    left unwritten when x_saved is given."""
    lib = load()
    B, H, T, dkk = q.shape
    dvv = v.shape[-1]
    code = _dtype_code(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("dout", dout)):
        _require(t, name, q.dtype)
    _require(gamma, "gamma", torch.float32)
    _require(lambda_diag, "lambda_diag", torch.float32)
    dev = q.device
    dq = torch.empty((B, H, T, dkk), dtype=q.dtype, device=dev) if dq is None else dq
    dk = torch.empty((B, H, T, dkk), dtype=q.dtype, device=dev) if dk is None else dk
    dv = torch.empty((B, H, T, dvv), dtype=q.dtype, device=dev) if dv is None else dv
    dgamma = torch.empty((B, H, T), dtype=torch.float32, device=dev) if dgamma is None else dgamma
    dlambda = torch.empty((H, dkk), dtype=torch.float32, device=dev) if dlambda is None else dlambda
    iters_fwd = torch.empty((B, H, T), dtype=torch.int32, device=dev) if iters_fwd is None else iters_fwd
    iters_bwd = torch.empty((B, H, T), dtype=torch.int32, device=dev) if iters_bwd is None else iters_bwd
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _require(t, name, q.dtype)
    for name, t in (("dgamma", dgamma), ("dlambda", dlambda)):
        _require(t, name, torch.float32)
    _require(iters_fwd, "iters_fwd", torch.int32)
    _require(iters_bwd, "iters_bwd", torch.int32)
    _require(x_saved, "x_saved", torch.float32)
    need = mesa_backward_workspace_size(B, H, T, dkk, dvv)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _require(workspace, "workspace")
    st = lib.mesa_backward_chunked(B, H, T, dkk, dvv, code, _ptr(q), _ptr(k), _ptr(v), _ptr(gamma),
                                   _ptr(lambda_diag), _ptr(dout), _ptr(x_saved), int(cg_iters), float(cg_tol), _ptr(dq),
                                   _ptr(dk), _ptr(dv), _ptr(dgamma), _ptr(dlambda), _ptr(iters_fwd),
                                   _ptr(iters_bwd), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "mesa_backward_chunked")
    return dq, dk, dv, dgamma, dlambda, iters_fwd, iters_bwd


def mesa_decode_step(H_state, G_state, q, k, v, gamma, lambda_diag, cg_iters, cg_tol, out=None,
                     iters_used=None, stream=None):
    """One decode step in place on H_state [N, H, dk, dk] and G_state [N, H, dv, dk] (fp32).
    q, k [N, H, dk], v [N, H, dv] (fp32 or bf16), gamma [N, H].  Returns (out, iters_used)."""
    lib = load()
    N, H, dk = q.shape
    dv = v.shape[-1]
    code = _dtype_code(q)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _require(t, name, q.dtype)
    _require(H_state, "H_state", torch.float32)
    _require(G_state, "G_state", torch.float32)
    _require(gamma, "gamma", torch.float32)
    _require(lambda_diag, "lambda_diag", torch.float32)
    if out is None:
        out = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    if iters_used is None:
        iters_used = torch.empty((N, H), dtype=torch.int32, device=q.device)
    st = lib.mesa_decode_step(N, H, dk, dv, code, _ptr(H_state), _ptr(G_state), _ptr(q), _ptr(k),
                              _ptr(v), _ptr(gamma), _ptr(lambda_diag), int(cg_iters), float(cg_tol),
                              _ptr(out), _ptr(iters_used), _stream(stream))
    _check(st, "mesa_decode_step")
    return out, iters_used


def mesa_qk_preprocess(q_raw, k_raw, wq, wk, q_out=None, k_out=None, stream=None):
    """Query/key preprocessing: causal depthwise convolution with W taps per (head, channel),
    then each token divided by its Euclidean norm.  q_raw, k_raw [B, H, T, d] (fp32 or bf16),
    wq, wk [H, d, W] fp32.  Returns (q_out, k_out) of the input dtype."""
    lib = load()
    B, H, T, d = q_raw.shape
    W = wq.shape[-1]
    code = _dtype_code(q_raw)
    _require(q_raw, "q_raw")
    _require(k_raw, "k_raw", q_raw.dtype)
    _require(wq, "wq", torch.float32)
    _require(wk, "wk", torch.float32)
    if q_out is None:
        q_out = torch.empty_like(q_raw)
    if k_out is None:
        k_out = torch.empty_like(k_raw)
    st = lib.mesa_qk_preprocess(B, H, T, d, W, code, _ptr(q_raw), _ptr(k_raw), _ptr(wq), _ptr(wk),
                                _ptr(q_out), _ptr(k_out), _stream(stream))
    _check(st, "mesa_qk_preprocess")
    return q_out, k_out


def mesa_qk_preprocess_step(q_raw, k_raw, wq, wk, conv_state, q_out=None, k_out=None, stream=None):
    """One decode step of the preprocessing.  q_raw, k_raw [N, H, d]; conv_state
    [N, H, 2, W-1, d] fp32, updated in place (None when W = 1).  Returns (q_out, k_out)."""
    lib = load()
    N, H, d = q_raw.shape
    W = wq.shape[-1]
    code = _dtype_code(q_raw)
    _require(q_raw, "q_raw")
    _require(k_raw, "k_raw", q_raw.dtype)
    _require(wq, "wq", torch.float32)
    _require(wk, "wk", torch.float32)
    _require(conv_state, "conv_state", torch.float32)
    if q_out is None:
        q_out = torch.empty_like(q_raw)
    if k_out is None:
        k_out = torch.empty_like(k_raw)
    st = lib.mesa_qk_preprocess_step(N, H, d, W, code, _ptr(q_raw), _ptr(k_raw), _ptr(wq), _ptr(wk),
                                     _ptr(conv_state), _ptr(q_out), _ptr(k_out), _stream(stream))
    _check(st, "mesa_qk_preprocess_step")
    return q_out, k_out


def mesa_decode_step_warm(H_state, G_state, X_state, q, k, v, gamma, lambda_diag, cg_iters, cg_tol,
                          out=None, iters_used=None, stream=None):
    """mesa_decode_step whose CG starts from X_state [N, H, dk] (fp32, in/out: replaced by this
    step's solution).  Returns (out, iters_used)."""
    lib = load()
    N, H, dk = q.shape
    dv = v.shape[-1]
    code = _dtype_code(q)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _require(t, name, q.dtype)
    for name, t in (("H_state", H_state), ("G_state", G_state), ("X_state", X_state), ("gamma", gamma),
                    ("lambda_diag", lambda_diag)):
        _require(t, name, torch.float32)
    if out is None:
        out = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    if iters_used is None:
        iters_used = torch.empty((N, H), dtype=torch.int32, device=q.device)
    st = lib.mesa_decode_step_warm(N, H, dk, dv, code, _ptr(H_state), _ptr(G_state), _ptr(X_state), _ptr(q),
                                   _ptr(k), _ptr(v), _ptr(gamma), _ptr(lambda_diag), int(cg_iters), float(cg_tol),
                                   _ptr(out), _ptr(iters_used), _stream(stream))
    _check(st, "mesa_decode_step_warm")
    return out, iters_used


def mesa_forward_status(workspace, stream=None) -> int:
    """Synchronise the stream and return the device status word of the last forward call
    that used ``workspace`` (0: every kernel completed with finite outputs; bit 0: a bounded
    wait gave up; bit 1: a non-finite output; bit 2: the drain after a give-up expired)."""
    return mesa_forward_status_code(workspace, stream)[1]


def mesa_forward_status_code(workspace, stream=None):
    """(status code, flags) of mesa_forward_status: MESA_OK, MESA_ERR_TIMEOUT or
    MESA_ERR_NONFINITE, and the raw word."""
    lib = load()
    flags = ctypes.c_uint(0)
    rc = lib.mesa_forward_status(_ptr(workspace), _stream(stream), ctypes.byref(flags))
    if rc not in (MESA_OK, MESA_ERR_TIMEOUT, MESA_ERR_NONFINITE):
        _check(rc, "mesa_forward_status")
    return int(rc), int(flags.value)


def mesa_decode_status(stream=None):
    """(status code, flags) of the decode steps on the current device since the last query
    (the word is cleared): MESA_OK, MESA_ERR_TIMEOUT (bits 0 / 2 of flags) or
    MESA_ERR_NONFINITE (bit 1)."""
    lib = load()
    flags = ctypes.c_uint(0)
    rc = lib.mesa_decode_status(_stream(stream), ctypes.byref(flags))
    if rc not in (MESA_OK, MESA_ERR_TIMEOUT, MESA_ERR_NONFINITE):
        _check(rc, "mesa_decode_status")
    return int(rc), int(flags.value)


def mesa_debug_set_wait_limit(polls: int):
    """Test hook: polls after which the tensor-core kernels' (and the d = 128 decode step's)
    bounded waits give up (< 0: default)."""
    _check(load().mesa_debug_set_wait_limit(int(polls)), "mesa_debug_set_wait_limit")


def mesa_tc_selftest(A, B, stream=None):
    """Tensor-core building-block check: returns (C1 = A B^T, C2 = A B, C3 = A^T B, status)
    computed by tcgen05.mma on fp16-rounded [128, 128] inputs."""
    lib = load()
    _require(A, "A", torch.float32)
    _require(B, "B", torch.float32)
    C1 = torch.empty(128, 128, device=A.device)
    C2 = torch.empty(128, 128, device=A.device)
    C3 = torch.empty(128, 128, device=A.device)
    status = torch.zeros(1, dtype=torch.int32, device=A.device)
    _check(lib.mesa_tc_selftest(_ptr(A), _ptr(B), _ptr(C1), _ptr(C2), _ptr(C3), _ptr(status),
                                _stream(stream)), "mesa_tc_selftest")
    return C1, C2, C3, status


NOALLOC_MAX_BYTES = 32 << 20


def mesa_forward_chunked_noalloc(q, k, v, gamma, lambda_diag, cg_iters, cg_tol, chunk, out=None,
                                 iters_used=None, stream=None):
    """mesa_forward_chunked with the library's fixed device scratch instead of a workspace
    (no device allocation inside the call; calls must not overlap on the GPU)."""
    lib = load()
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    code = _dtype_code(q)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _require(t, name, q.dtype)
    _require(gamma, "gamma", torch.float32)
    _require(lambda_diag, "lambda_diag", torch.float32)
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=q.dtype, device=q.device)
    if iters_used is None:
        iters_used = torch.empty((B, H, T), dtype=torch.int32, device=q.device)
    st = lib.mesa_forward_chunked_noalloc(B, H, T, dk, dv, code, _ptr(q), _ptr(k), _ptr(v), _ptr(gamma),
                                          _ptr(lambda_diag), int(cg_iters), float(cg_tol), int(chunk),
                                          _ptr(out), _ptr(iters_used), _stream(stream))
    _check(st, "mesa_forward_chunked_noalloc")
    return out, iters_used
