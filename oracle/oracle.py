"""Python face of the float64 CPU oracle (``opam_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test-suite, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  Nothing here is shared
with the CUDA library.  Inputs are converted to float64 numpy arrays (exact
for float32 and bf16 values) and handed to the C recurrences unchanged.

Every function's meaning is documented in ``opam_oracle.c`` next to the
passage of the pages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "opam_oracle.c")
_LIB = os.path.join(_HERE, "libopam_oracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.POINTER(ctypes.c_int64)
_I32 = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP) into libopam_oracle.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i, d = ctypes.c_int, ctypes.c_double
            lib.oracle_tc_prefill.argtypes = [i, i, i, i, i, i, _D, _D, _D, _D, _D, _D, d,
                                              _D, _D, _D, _D, _D, _I32, _I64]
            lib.oracle_tc_decode.argtypes = [i, i, i, i, i, i, _D, _D, _D, _I64, _D, _D, _D,
                                             _D, _D, _D, d, _D]
            lib.oracle_tc_output_at.argtypes = [i, i, i, i, _D, _D, _D, d, d, d, d, i, _I64, _D]
            lib.oracle_tc_output_at.restype = None
            lib.oracle_delta.argtypes = [i, i, i, i, i, _D, _D, _D, _D, _D, _D, _D]
            lib.oracle_sparse_linattn.argtypes = [i, i, i, i, i, _D, _D, _D, _D, _D, _D]
            lib.oracle_sparse_linattn_output_at.argtypes = [i, i, i, _D, _D, _D, _D, i, _I64, _D]
            lib.oracle_sparse_linattn_output_at.restype = None
            lib.oracle_tc_backward.argtypes = [i, i, i, i, i, i, _D, _D, _D, _D, _D, _D, d, _D,
                                               _D, _D, _D, _D, _D, _D]
            lib.oracle_delta_backward.argtypes = [i, i, i, i, i, _D, _D, _D, _D, _D, _D, _D, _D, _D,
                                                  _D, _D, _D]
            lib.oracle_bdh_keys.argtypes = [i, i, i, i, i, _D, _D, d, _D]
            lib.oracle_bdh_keys.restype = None
            lib.oracle_set_threads.argtypes = [i]
            lib.oracle_set_threads.restype = None
            lib.oracle_get_threads.restype = i
            _lib = lib
    return _lib


def f64(x) -> np.ndarray:
    """Exact float64 copy of a torch tensor or array (bf16/fp32 upcast)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(a):
    return None if a is None else a.ctypes.data_as(_D)


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().oracle_get_threads())


def default_scale(d_k: int) -> float:
    return 1.0 / float(np.sqrt(d_k))


def tc_prefill(q, k, v, lam, eta, gate, W, scale=None, want_state=False, want_m=False,
               want_writes=False):
    """Tensor Cache layer over tokens 0..T-1 from an empty state.

    q,k [B,H,T,d_k], v [B,H,T,d_v], lam/eta/gate [H].  Returns a dict with
    ``y`` [B,H,T,d_v] and, on request, ``m`` (L2 read alone), the final state
    ``ring_k``/``ring_v``/``A`` and ``write_count``/``write_time`` [B,H,T].
    """
    q, k, v = f64(q), f64(k), f64(v)
    lam, eta, gate = f64(lam), f64(eta), f64(gate)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    W = int(W)
    scale = default_scale(dk) if scale is None else float(scale)
    out = {"y": np.zeros((B, H, T, dv))}
    m = np.zeros((B, H, T, dv)) if want_m else None
    rk = np.zeros((B, H, W, dk)) if want_state else None
    rv = np.zeros((B, H, W, dv)) if want_state else None
    A = np.zeros((B, H, dk, dv)) if want_state else None
    wc = np.zeros((B, H, T), dtype=np.int32) if want_writes else None
    wt = np.zeros((B, H, T), dtype=np.int64) if want_writes else None
    rc = _load().oracle_tc_prefill(B, H, T, dk, dv, W, _p(q), _p(k), _p(v), _p(lam), _p(eta),
                                   _p(gate), scale, _p(out["y"]), _p(m), _p(rk), _p(rv), _p(A),
                                   None if wc is None else wc.ctypes.data_as(_I32),
                                   None if wt is None else wt.ctypes.data_as(_I64))
    if rc != 0:
        raise MemoryError("oracle_tc_prefill failed to allocate")
    if want_m:
        out["m"] = m
    if want_state:
        out.update(ring_k=rk, ring_v=rv, A=A, pos=np.full((B,), T, dtype=np.int64))
    if want_writes:
        out.update(write_count=wc, write_time=wt)
    return out


def tc_decode(state, q, k, v, lam, eta, gate, scale=None):
    """Continue a Tensor Cache state for ``steps`` single-token steps.

    state: dict ring_k [S,H,W,d_k], ring_v [S,H,W,d_v], A [S,H,d_k,d_v],
    pos [S] (copied, not modified).  q,k [steps,S,H,d_k], v [steps,S,H,d_v].
    Returns (y [steps,S,H,d_v], new_state).
    """
    rk, rv, A = f64(state["ring_k"]).copy(), f64(state["ring_v"]).copy(), f64(state["A"]).copy()
    pos = np.ascontiguousarray(np.asarray(state["pos"], dtype=np.int64)).copy()
    q, k, v = f64(q), f64(k), f64(v)
    lam, eta, gate = f64(lam), f64(eta), f64(gate)
    steps, S, H, dk = q.shape
    dv = v.shape[-1]
    W = rk.shape[2]
    scale = default_scale(dk) if scale is None else float(scale)
    y = np.zeros((steps, S, H, dv))
    rc = _load().oracle_tc_decode(S, H, dk, dv, W, steps, _p(rk), _p(rv), _p(A),
                                  pos.ctypes.data_as(_I64), _p(q), _p(k), _p(v), _p(lam),
                                  _p(eta), _p(gate), scale, _p(y))
    if rc != 0:
        raise MemoryError("oracle_tc_decode failed to allocate")
    return y, dict(ring_k=rk, ring_v=rv, A=A, pos=pos)


def tc_output_at(q, k, v, lam, eta, gate, W, ts, scale=None):
    """Closed-form Tensor Cache output of one unit at positions ``ts``.

    q,k [T,d_k], v [T,d_v], scalars lam/eta/gate.  Returns [len(ts), d_v].
    """
    q, k, v = f64(q), f64(k), f64(v)
    T, dk = q.shape
    dv = v.shape[-1]
    ts = np.ascontiguousarray(np.asarray(ts, dtype=np.int64))
    scale = default_scale(dk) if scale is None else float(scale)
    y = np.zeros((len(ts), dv))
    _load().oracle_tc_output_at(T, dk, dv, int(W), _p(q), _p(k), _p(v), float(lam), float(eta),
                                float(gate), scale, len(ts), ts.ctypes.data_as(_I64), _p(y))
    return y


def delta(q, k, v, beta, S0=None, want_state=False):
    """DeltaNet delta rule; returns dict y [B,H,T,d_v] (+ S [B,H,d_k,d_v])."""
    q, k, v, beta = f64(q), f64(k), f64(v), f64(beta)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    S0 = None if S0 is None else f64(S0)
    S = np.zeros((B, H, dk, dv)) if want_state else None
    y = np.zeros((B, H, T, dv))
    rc = _load().oracle_delta(B, H, T, dk, dv, _p(q), _p(k), _p(v), _p(beta), _p(S0), _p(S), _p(y))
    if rc != 0:
        raise MemoryError("oracle_delta failed to allocate")
    out = {"y": y}
    if want_state:
        out["S"] = S
    return out


def sparse_linattn(q, k, v, S0=None, want_state=False):
    """BDH-style additive linear attention; returns dict y (+ S [B,H,N,d_v])."""
    q, k, v = f64(q), f64(k), f64(v)
    B, H, T, N = q.shape
    dv = v.shape[-1]
    S0 = None if S0 is None else f64(S0)
    S = np.zeros((B, H, N, dv)) if want_state else None
    y = np.zeros((B, H, T, dv))
    rc = _load().oracle_sparse_linattn(B, H, T, N, dv, _p(q), _p(k), _p(v), _p(S0), _p(S), _p(y))
    if rc != 0:
        raise MemoryError("oracle_sparse_linattn failed to allocate")
    out = {"y": y}
    if want_state:
        out["S"] = S
    return out


def sparse_linattn_output_at(q, k, v, ts, S0=None):
    """Closed-form additive read of one unit at positions ``ts``.

    q,k [T,N], v [T,d_v], S0 [N,d_v] or None.  Returns [len(ts), d_v].
    """
    q, k, v = f64(q), f64(k), f64(v)
    T, N = q.shape
    dv = v.shape[-1]
    S0 = None if S0 is None else f64(S0)
    ts = np.ascontiguousarray(np.asarray(ts, dtype=np.int64))
    y = np.zeros((len(ts), dv))
    _load().oracle_sparse_linattn_output_at(T, N, dv, _p(q), _p(k), _p(v), _p(S0), len(ts),
                                            ts.ctypes.data_as(_I64), _p(y))
    return y


def tc_backward(q, k, v, lam, eta, gate, W, dy, scale=None):
    """Gradient of L = sum <dy, y> through the Tensor Cache layer (prefill from
    an empty state).  Returns dict dq, dk [B,H,T,d_k], dv [B,H,T,d_v] and
    dlam, deta, dgate [H] (summed over the batch)."""
    q, k, v, dy = f64(q), f64(k), f64(v), f64(dy)
    lam, eta, gate = f64(lam), f64(eta), f64(gate)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    scale = default_scale(dk) if scale is None else float(scale)
    out = {"dq": np.zeros((B, H, T, dk)), "dk": np.zeros((B, H, T, dk)), "dv": np.zeros((B, H, T, dv)),
           "dlam": np.zeros(H), "deta": np.zeros(H), "dgate": np.zeros(H)}
    rc = _load().oracle_tc_backward(B, H, T, dk, dv, int(W), _p(q), _p(k), _p(v), _p(lam), _p(eta),
                                    _p(gate), scale, _p(dy), _p(out["dq"]), _p(out["dk"]), _p(out["dv"]),
                                    _p(out["dlam"]), _p(out["deta"]), _p(out["dgate"]))
    if rc != 0:
        raise MemoryError("oracle_tc_backward failed to allocate")
    return out


def delta_backward(q, k, v, beta, dy, S0=None, dS_T=None):
    """Gradient of L = sum <dy, o> (+ <dS_T, S_T>) through the delta rule.
    Returns dict dq, dk, dv, dbeta and dS0 (key-major [B,H,d_k,d_v])."""
    q, k, v, beta, dy = f64(q), f64(k), f64(v), f64(beta), f64(dy)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    S0 = None if S0 is None else f64(S0)
    dS_T = None if dS_T is None else f64(dS_T)
    out = {"dq": np.zeros((B, H, T, dk)), "dk": np.zeros((B, H, T, dk)), "dv": np.zeros((B, H, T, dv)),
           "dbeta": np.zeros((B, H, T)), "dS0": np.zeros((B, H, dk, dv))}
    rc = _load().oracle_delta_backward(B, H, T, dk, dv, _p(q), _p(k), _p(v), _p(beta), _p(S0), _p(dy),
                                       _p(dS_T), _p(out["dq"]), _p(out["dk"]), _p(out["dv"]),
                                       _p(out["dbeta"]), _p(out["dS0"]))
    if rc != 0:
        raise MemoryError("oracle_delta_backward failed to allocate")
    return out


def bdh_keys(x, U, theta):
    """BDH activations max(0, x U_h - theta): x [B,H,T,R], U [H,R,N];
    returns [B,H,T,N] float64."""
    x, U = f64(x), f64(U)
    B, H, T, R = x.shape
    N = U.shape[-1]
    out = np.zeros((B, H, T, N))
    _load().oracle_bdh_keys(B, H, T, R, N, _p(x), _p(U), float(theta), _p(out))
    return out
