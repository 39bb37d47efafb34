"""fp64 CPU oracle for the Mesa layer forward and backward passes (ctypes wrapper over mesa_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py``.  The product path (``mesa_layer_gb300``)
never imports it.  It shares no code with the CUDA path.

What it computes follows the MesaNet technical summary (gist.science/pt/paper/2506.05233),
section "A Camada Mesa": the Mesa objective, the query solve q*_t = (H_t + Lambda)^-1 q_t
by conjugate gradient, the state variables G_t and H_t, and the per-token stopping
criterion.  The readings taken where the page is silent are listed in mesa_oracle.c.

All arrays are converted to contiguous float64 before the call; callers round inputs to
the tested dtype first (the oracle sees exactly what the kernels see, upcast to fp64).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mesa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmesa_oracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int32)


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle with gcc (OpenMP if available).  No -march flags, no fused
    multiply-add contraction, so x86 and Arm builds round the same way."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off"]
    tail = [src, "-o", out, "-lm", *extra_flags]
    try:
        subprocess.run(base + ["-fopenmp"] + tail, check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + tail, check=True, capture_output=True)
    return out


def _needs_build() -> bool:
    return (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)


def _bind(lib):
    lib.oracle_cg.restype = ctypes.c_int
    lib.oracle_cg.argtypes = [ctypes.c_int, _D, _D, _D, ctypes.c_int, ctypes.c_double, _D, _D]
    lib.oracle_forward.restype = ctypes.c_int
    lib.oracle_forward.argtypes = [ctypes.c_int] * 5 + [_D] * 5 + [
        ctypes.c_int, ctypes.c_double, _I, _D, _D, _D, _I, _D, _D, _D, ctypes.c_int]
    lib.oracle_decode_step.restype = ctypes.c_int
    lib.oracle_decode_step.argtypes = [ctypes.c_int] * 4 + [_D] * 7 + [
        ctypes.c_int, ctypes.c_double, _D, _I, _D, ctypes.c_int]
    lib.oracle_state_trace.restype = None
    lib.oracle_state_trace.argtypes = [ctypes.c_int] * 3 + [_D] * 5
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    lib.oracle_cg_from.restype = ctypes.c_int
    lib.oracle_cg_from.argtypes = [ctypes.c_int, _D, _D, _D, _D, ctypes.c_int, ctypes.c_double, _D, _D]
    lib.oracle_decode_step_from.restype = ctypes.c_int
    lib.oracle_decode_step_from.argtypes = [ctypes.c_int] * 4 + [_D] * 7 + [
        ctypes.c_int, ctypes.c_double, _D, _D, _I, _D, ctypes.c_int]
    lib.oracle_qk_preprocess.restype = None
    lib.oracle_qk_preprocess.argtypes = [ctypes.c_int] * 5 + [_D] * 3
    lib.oracle_qk_preprocess_step.restype = None
    lib.oracle_qk_preprocess_step.argtypes = [ctypes.c_int] * 4 + [_D] * 4
    lib.oracle_backward.restype = ctypes.c_int
    lib.oracle_backward.argtypes = [ctypes.c_int] * 5 + [_D] * 6 + [ctypes.c_int, ctypes.c_double] + [_D] * 5 + [
        _I, _I, ctypes.c_int]
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library.  ``path`` selects another build of
    the same source (used by the planted-mistake tests)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _needs_build():
                compile_oracle()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a, t=_D):
    return None if a is None else a.ctypes.data_as(t)


def _scale_buf(a, shape):
    """The caller's readout-magnitude array, checked (None stays None)."""
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags.c_contiguous and a.shape == tuple(shape), \
        f"scale_out must be float64 C-contiguous {tuple(shape)}"
    return a


def max_threads(lib=None) -> int:
    return (lib or load()).oracle_max_threads()


def cg(Hm, lam, q, maxit, tol=0.0, x0=None, lib=None):
    """Textbook CG on (Hm + diag(lam)) x = q from x0 (None: 0; the stopping rule stays
    relative to ||q||).  Returns (x, iterations)."""
    lib = lib or load()
    Hm, lam, q = _f64(Hm), _f64(lam), _f64(q)
    n = q.shape[0]
    x = np.zeros(n)
    work = np.zeros(3 * n)
    if x0 is None:
        it = lib.oracle_cg(n, _ptr(Hm), _ptr(lam), _ptr(q), int(maxit), float(tol), _ptr(x), _ptr(work))
    else:
        x0 = _f64(x0)
        it = lib.oracle_cg_from(n, _ptr(Hm), _ptr(lam), _ptr(q), _ptr(x0), int(maxit), float(tol), _ptr(x),
                                _ptr(work))
    return x, it


def forward(q, k, v, gamma, lam, cg_iters, cg_tol=0.0, replay=None, H0=None, G0=None,
            want_final=False, nthreads=None, lib=None, scale_out=None):
    """Mesa layer forward.  q, k: [B, heads, T, dk]; v: [B, heads, T, dv];
    gamma: [B, heads, T]; lam: [heads, dk].  Returns (out [B, heads, T, dv] fp64,
    iters [B, heads, T] int32[, H_final [B, heads, dk, dk], G_final [B, heads, dv, dk]]).
    ``replay`` (int32 [B, heads, T]) runs each token for exactly that many iterations.
    ``scale_out``: None, or a float64 C-contiguous [B, heads, T] array that receives each
    token's readout magnitude || |G_t| |x_t| ||_2 (>= ||out_t||)."""
    lib = lib or load()
    q, k, v, gamma, lam = _f64(q), _f64(k), _f64(v), _f64(gamma), _f64(lam)
    B, heads, T, dk = q.shape
    dv = v.shape[-1]
    U = B * heads
    out = np.zeros((B, heads, T, dv))
    iters = np.zeros((B, heads, T), dtype=np.int32)
    rep = None if replay is None else np.ascontiguousarray(replay, dtype=np.int32)
    H0 = None if H0 is None else _f64(H0)
    G0 = None if G0 is None else _f64(G0)
    Hf = np.zeros((B, heads, dk, dk)) if want_final else None
    Gf = np.zeros((B, heads, dv, dk)) if want_final else None
    nt = nthreads if nthreads is not None else (os.cpu_count() or 1)
    lib.oracle_forward(U, heads, T, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(gamma), _ptr(lam),
                       int(cg_iters), float(cg_tol), _ptr(rep, _I), _ptr(H0), _ptr(G0),
                       _ptr(out), _ptr(iters, _I), _ptr(Hf), _ptr(Gf), _ptr(_scale_buf(scale_out, (B, heads, T))),
                       int(nt))
    if want_final:
        return out, iters, Hf, Gf
    return out, iters


def backward(q, k, v, gamma, lam, dout, cg_iters, cg_tol=0.0, nthreads=None, lib=None):
    """Gradients of a loss through the Mesa layer forward, given dout = dL/do
    [B, heads, T, dv]: implicit differentiation through each token's solve (one more CG per
    token, on (H_t + Lambda) y = G_t^T g_t, with the forward's CG rule), then the state
    recurrence differentiated backwards in time.  Zero initial states.  Returns a dict with
    dq, dk [B, heads, T, dk], dv [B, heads, T, dv], dgamma [B, heads, T], dlam [heads, dk]
    (summed over the batch), iters_fwd and iters_bwd [B, heads, T] int32."""
    lib = lib or load()
    q, k, v, gamma, lam, dout = _f64(q), _f64(k), _f64(v), _f64(gamma), _f64(lam), _f64(dout)
    B, heads, T, dk = q.shape
    dv = v.shape[-1]
    r = {"dq": np.zeros((B, heads, T, dk)), "dk": np.zeros((B, heads, T, dk)), "dv": np.zeros((B, heads, T, dv)),
         "dgamma": np.zeros((B, heads, T)), "dlam": np.zeros((heads, dk)),
         "iters_fwd": np.zeros((B, heads, T), dtype=np.int32), "iters_bwd": np.zeros((B, heads, T), dtype=np.int32)}
    nt = nthreads if nthreads is not None else (os.cpu_count() or 1)
    lib.oracle_backward(B * heads, heads, T, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(gamma), _ptr(lam), _ptr(dout),
                        int(cg_iters), float(cg_tol), _ptr(r["dq"]), _ptr(r["dk"]), _ptr(r["dv"]), _ptr(r["dgamma"]),
                        _ptr(r["dlam"]), _ptr(r["iters_fwd"], _I), _ptr(r["iters_bwd"], _I), int(nt))
    return r


def decode_step(Hs, Gs, q, k, v, gamma, lam, cg_iters, cg_tol=0.0, nthreads=None, X=None, lib=None,
                scale_out=None):
    """One decode step, in place on the fp64 states Hs [N, heads, dk, dk] and
    Gs [N, heads, dv, dk] (must be float64 C-contiguous).  q, k: [N, heads, dk];
    v: [N, heads, dv]; gamma: [N, heads].  X: None, or [N, heads, dk] float64 C-contiguous,
    the start of each unit's CG (warm start), replaced in place by this step's solution.
    scale_out: None, or float64 C-contiguous [N, heads], each unit's || |G| |x| ||_2.
    Returns (out [N, heads, dv], iters [N, heads])."""
    lib = lib or load()
    assert Hs.dtype == np.float64 and Hs.flags.c_contiguous
    assert Gs.dtype == np.float64 and Gs.flags.c_contiguous
    q, k, v, gamma, lam = _f64(q), _f64(k), _f64(v), _f64(gamma), _f64(lam)
    N, heads, dk = q.shape
    dv = v.shape[-1]
    out = np.zeros((N, heads, dv))
    iters = np.zeros((N, heads), dtype=np.int32)
    nt = nthreads if nthreads is not None else (os.cpu_count() or 1)
    if X is None:
        lib.oracle_decode_step(N * heads, heads, dk, dv, _ptr(Hs), _ptr(Gs), _ptr(q), _ptr(k), _ptr(v),
                               _ptr(gamma), _ptr(lam), int(cg_iters), float(cg_tol), _ptr(out),
                               _ptr(iters, _I), _ptr(_scale_buf(scale_out, (N, heads))), int(nt))
    else:
        assert X.dtype == np.float64 and X.flags.c_contiguous
        lib.oracle_decode_step_from(N * heads, heads, dk, dv, _ptr(Hs), _ptr(Gs), _ptr(q), _ptr(k), _ptr(v),
                                    _ptr(gamma), _ptr(lam), int(cg_iters), float(cg_tol), _ptr(X), _ptr(out),
                                    _ptr(iters, _I), _ptr(_scale_buf(scale_out, (N, heads))), int(nt))
    return out, iters


def state_trace(k, v, gamma, lib=None):
    """States after every token for one unit: k [T, dk], v [T, dv], gamma [T] ->
    (H_all [T, dk, dk], G_all [T, dv, dk]) from the recurrence."""
    lib = lib or load()
    k, v, gamma = _f64(k), _f64(v), _f64(gamma)
    T, dk = k.shape
    dv = v.shape[1]
    Ha = np.zeros((T, dk, dk))
    Ga = np.zeros((T, dv, dk))
    lib.oracle_state_trace(T, dk, dv, _ptr(k), _ptr(v), _ptr(gamma), _ptr(Ha), _ptr(Ga))
    return Ha, Ga


def qk_preprocess(x, w, lib=None):
    """Query/key preprocessing ("Arquitetura (MesaNet)", "Pre-processamento"): causal
    depthwise convolution over time with W taps per (head, channel), then each token divided
    by its Euclidean norm.  x: [B, heads, T, d]; w: [heads, d, W] (tap s multiplies the input
    s tokens back).  Returns [B, heads, T, d] fp64."""
    lib = lib or load()
    x, w = _f64(x), _f64(w)
    B, heads, T, d = x.shape
    W = w.shape[-1]
    out = np.zeros_like(x)
    lib.oracle_qk_preprocess(B * heads, heads, T, d, W, _ptr(x), _ptr(w), _ptr(out))
    return out


def qk_preprocess_step(x, w, hist, lib=None):
    """One decode step of qk_preprocess.  x: [N, heads, d]; w: [heads, d, W]; hist:
    [N, heads, W-1, d] float64 C-contiguous, the previous raw inputs (hist[..., s, :] is the
    input s+1 tokens back), updated in place.  Returns [N, heads, d] fp64."""
    lib = lib or load()
    assert hist.dtype == np.float64 and hist.flags.c_contiguous
    x, w = _f64(x), _f64(w)
    N, heads, d = x.shape
    W = w.shape[-1]
    out = np.zeros_like(x)
    lib.oracle_qk_preprocess_step(N * heads, heads, d, W, _ptr(x), _ptr(w), _ptr(hist), _ptr(out))
    return out
