"""ctypes binding for libopam.so: argument marshalling only.

Every function here checks tensor placement, shapes and element types
against the C header's contract (extents are taken from q, so a mismatched
k, v, state or output would otherwise be read or written out of bounds on
the device), passes raw device pointers, sizes and the current CUDA stream to
the C entry point of the same name, and turns a non-OK status into an
exception.  All arithmetic happens in the CUDA
kernels behind the C ABI; there is no fallback path.  PyTorch only allocates
device memory (outputs, state, workspace) and supplies the stream.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# OPAM_LIBRARY selects another build of the same library (for instance the
# debug-bounds build, libopam_debug.so); the default is the normal build.
LIB_PATH = os.environ.get("OPAM_LIBRARY") or os.path.join(_PKG, "libopam.so")

OPAM_F32, OPAM_BF16 = 0, 1
_STATUS = {0: "OK", -1: "INVALID_ARG", -2: "UNSUPPORTED", -3: "CUDA", -4: "TIMEOUT", -5: "WORKSPACE"}
OPAM_ERR_TIMEOUT, OPAM_ERR_WORKSPACE = -4, -5
STATUS_BYTES = 256  # OPAM_STATUS_BYTES in include/opam.h

# Every symbol the C header declares (checked by the CPU test-suite).
EXPORTS = (
    "tc_layer_forward_workspace_size", "tc_layer_forward", "tc_layer_forward_noalloc",
    "tc_layer_backward_workspace_size", "tc_layer_backward",
    "delta_rule_backward_workspace_size", "delta_rule_backward",
    "tc_window_forward_workspace_size", "tc_window_forward",
    "tc_decode_step_workspace_size", "tc_decode_step",
    "delta_rule_forward_workspace_size", "delta_rule_forward", "delta_decode_step",
    "sparse_linattn_forward_workspace_size", "sparse_linattn_forward",
    "sparse_linattn_keygen_forward_workspace_size", "sparse_linattn_keygen_forward",
    "opam_last_error", "opam_profile_events", "opam_kernel_launches", "opam_check_device_error", "opam_fp32_fma_probe",
    "opam_selftest_bounded_wait", "opam_selftest_bounds", "opam_debug_bounds_build",
)


class OpamError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


class TCStateStruct(ctypes.Structure):
    _fields_ = [("ring_k", ctypes.c_void_p), ("ring_v", ctypes.c_void_p),
                ("A", ctypes.c_void_p), ("pos", ctypes.c_void_p),
                ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("W", ctypes.c_int32),
                ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32), ("dtype", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libopam.so; raise if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m outer_product_associative_chunked_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        sp = ctypes.POINTER(TCStateStruct)
        L.opam_last_error.restype = ctypes.c_char_p
        L.opam_last_error.argtypes = []
        L.tc_layer_forward_workspace_size.restype = sz
        L.tc_layer_forward_workspace_size.argtypes = [i, i, i, i, i, i, i]
        L.tc_layer_forward.restype = i
        L.tc_layer_forward.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, vp, vp, vp, f, vp, sp, vp, sz, vp]
        L.tc_layer_forward_noalloc.restype = i
        L.tc_layer_forward_noalloc.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, vp, vp, vp, f, vp, sp, vp]
        L.tc_layer_backward_workspace_size.restype = sz
        L.tc_layer_backward_workspace_size.argtypes = [i, i, i, i, i, i, i]
        L.tc_layer_backward.restype = i
        L.tc_layer_backward.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, vp, vp, vp, f, vp, vp, vp, vp, vp, vp,
                                        vp, vp, sz, vp]
        L.delta_rule_backward_workspace_size.restype = sz
        L.delta_rule_backward_workspace_size.argtypes = [i, i, i, i, i, i]
        L.delta_rule_backward.restype = i
        L.delta_rule_backward.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                          sz, vp]
        L.tc_window_forward_workspace_size.restype = sz
        L.tc_window_forward_workspace_size.argtypes = [i, i, i, i, i, i, i]
        L.tc_window_forward.restype = i
        L.tc_window_forward.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, f, vp, vp, sz, vp]
        L.tc_decode_step_workspace_size.restype = sz
        L.tc_decode_step_workspace_size.argtypes = [sp]
        L.tc_decode_step.restype = i
        L.tc_decode_step.argtypes = [sp, vp, vp, vp, vp, vp, vp, f, vp, vp, sz, vp]
        L.delta_rule_forward_workspace_size.restype = sz
        L.delta_rule_forward_workspace_size.argtypes = [i, i, i, i, i, i, i]
        L.delta_rule_forward.restype = i
        L.delta_rule_forward.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp, vp, vp, vp, sz, vp]
        L.delta_decode_step.restype = i
        L.delta_decode_step.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, vp, vp]
        L.sparse_linattn_forward_workspace_size.restype = sz
        L.sparse_linattn_forward_workspace_size.argtypes = [i, i, i, i, i]
        L.sparse_linattn_forward.restype = i
        L.sparse_linattn_forward.argtypes = [vp, vp, vp, i, i, i, i, i, vp, vp, vp, vp, sz, vp]
        L.sparse_linattn_keygen_forward_workspace_size.restype = sz
        L.sparse_linattn_keygen_forward_workspace_size.argtypes = [i, i, i, i, i, i]
        L.sparse_linattn_keygen_forward.restype = i
        L.sparse_linattn_keygen_forward.argtypes = [vp, vp, vp, f, vp, i, i, i, i, i, i, vp, vp, vp, vp, sz, vp]
        L.opam_profile_events.restype = i
        L.opam_profile_events.argtypes = [vp, vp]
        L.opam_kernel_launches.restype = ctypes.c_uint64
        L.opam_kernel_launches.argtypes = []
        L.opam_fp32_fma_probe.restype = i
        L.opam_fp32_fma_probe.argtypes = [vp, i, i, ctypes.POINTER(ctypes.c_double), vp]
        L.opam_check_device_error.restype = i
        L.opam_check_device_error.argtypes = [vp, vp]
        L.opam_selftest_bounds.restype = i
        L.opam_selftest_bounds.argtypes = [i, vp, vp]
        L.opam_debug_bounds_build.restype = i
        L.opam_debug_bounds_build.argtypes = []
        L.opam_selftest_bounded_wait.restype = i
        L.opam_selftest_bounded_wait.argtypes = [i, ctypes.c_longlong, vp, vp]
        _lib = L
    return _lib


def last_error() -> str:
    return lib().opam_last_error().decode()


def profile_events(start=None, stop=None) -> None:
    """Have later calls on this thread record two torch.cuda.Events around
    their dominant kernel (None, None switches it off)."""
    lib().opam_profile_events(None if start is None else ctypes.c_void_p(start.cuda_event),
                              None if stop is None else ctypes.c_void_p(stop.cuda_event))


def fp32_fma_probe(out, blocks: int, iters: int, stream=None) -> float:
    """Enqueue the FP32 FMA rate probe (out: >= blocks*256 float32 on the
    device); returns the flops the launch performs."""
    _dev(out)
    if out.dtype != torch.float32 or out.numel() < blocks * 256:
        raise ValueError("fp32_fma_probe: out must hold blocks*256 float32")
    fl = ctypes.c_double(0.0)
    _check(lib().opam_fp32_fma_probe(_ptr(out), int(blocks), int(iters), ctypes.byref(fl), _stream(stream)))
    return fl.value


def kernel_launches() -> int:
    """Kernels libopam has launched in this process so far."""
    return int(lib().opam_kernel_launches())


def check_device_error(workspace=None, stream=None) -> None:
    """Synchronise `stream` (default: the current stream) and raise
    OpamError(CUDA) on a CUDA error there, or OpamError(TIMEOUT) if the most
    recent call that used `workspace` had a bounded wait run out.  With
    workspace None: the built-in scratch of tc_layer_forward_noalloc."""
    _check(lib().opam_check_device_error(_ptr(workspace), _stream(stream)))


# The workspace and stream of the latest call of each entry point made through
# this module on the calling thread, so that check_device_errors() can read
# their status words.  One per entry point is kept (not one per call), so no
# more memory than the latest calls' workspaces stays alive.
_recent = threading.local()


def _remember(name, workspace, stream):
    d = getattr(_recent, "calls", None)
    if d is None:
        d = _recent.calls = {}
    d[name] = (workspace, stream)


def check_device_errors() -> None:
    """check_device_error() for the latest call of every entry point made on
    this thread since the last check (and the no-alloc scratch); forgets them."""
    d = getattr(_recent, "calls", None) or {}
    _recent.calls = {}
    for ws, stream in d.values():
        _check(lib().opam_check_device_error(_ptr(ws), stream))
    _check(lib().opam_check_device_error(None, _stream(None)))


def selftest_bounded_wait(arrive: bool, limit_cycles: int = 1_000_000, workspace=None, stream=None):
    """Run the bounded-wait self-test kernel into `workspace` (a fresh status
    block if None, returned): with arrive=False its wait runs out after
    limit_cycles and check_device_error(workspace) raises TIMEOUT."""
    ws = torch.empty(STATUS_BYTES, dtype=torch.uint8, device="cuda") if workspace is None else workspace
    _check(lib().opam_selftest_bounded_wait(1 if arrive else 0, int(limit_cycles), _ptr(ws), _stream(stream)))
    return ws


def debug_bounds_build() -> bool:
    """True when the loaded library was built with its index checks on."""
    return bool(lib().opam_debug_bounds_build())


def selftest_bounds(n: int, workspace=None, stream=None):
    """Run the index-check self-test (thread i of one warp checks i < n) into
    `workspace` (a fresh status block if None, returned)."""
    ws = torch.empty(STATUS_BYTES, dtype=torch.uint8, device="cuda") if workspace is None else workspace
    _check(lib().opam_selftest_bounds(int(n), _ptr(ws), _stream(stream)))
    return ws


def _check(rc: int) -> None:
    if rc != 0:
        raise OpamError(rc, last_error())


def dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return OPAM_F32
    if dt == torch.bfloat16:
        return OPAM_BF16
    raise TypeError(f"unsupported element type {dt}; use float32 or bfloat16")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _workspace(nbytes: int, workspace, device):
    if nbytes == 0:
        raise OpamError(-1, last_error() or "invalid arguments")
    if workspace is None:
        return torch.empty(nbytes, dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise OpamError(OPAM_ERR_WORKSPACE, f"workspace holds {workspace.numel()} bytes, {nbytes} required")
    return workspace


def _expect(fn, name, t, shape, dtype, device):
    """Raise ValueError unless tensor `t` has exactly `shape` and `dtype` and
    sits on `device`."""
    if t is None:
        return
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or t.device != device:
        raise ValueError(f"{fn}: {name} is {tuple(t.shape)} {t.dtype} on {t.device}; expected "
                         f"{tuple(shape)} {dtype} on {device}")


def _ndim(fn, name, t, n):
    if t.dim() != n:
        raise ValueError(f"{fn}: {name} must have {n} dimensions, got {tuple(t.shape)}")


# ------------------------------------------------------------------ Tensor Cache
class TCState:
    """Caller-owned Tensor Cache streaming state (ring, A, pos) on the GPU."""

    def __init__(self, B, H, W, d_k, d_v, dtype=torch.bfloat16, device="cuda"):
        self.B, self.H, self.W, self.d_k, self.d_v, self.dtype = B, H, W, d_k, d_v, dtype
        self.ring_k = torch.zeros(B, H, W, d_k, dtype=dtype, device=device)
        self.ring_v = torch.zeros(B, H, W, d_v, dtype=dtype, device=device)
        self.A = torch.zeros(B, H, d_k, d_v, dtype=torch.float32, device=device)
        self.pos = torch.zeros(B, dtype=torch.int64, device=device)

    def struct(self) -> TCStateStruct:
        return TCStateStruct(self.ring_k.data_ptr(), self.ring_v.data_ptr(), self.A.data_ptr(),
                             self.pos.data_ptr(), self.B, self.H, self.W, self.d_k, self.d_v,
                             dtype_code(self.dtype))


def tc_layer_forward_workspace_size(B, H, T, d_k, d_v, W, dtype) -> int:
    return int(lib().tc_layer_forward_workspace_size(B, H, T, d_k, d_v, W, dtype_code(dtype)))


def _check_tc_prefill(fn, q, k, v, lam, eta, gate, out, state, W):
    """Shapes and dtypes of a Tensor Cache prefill against q [B,H,T,d_k]."""
    _ndim(fn, "q", q, 4)
    _ndim(fn, "v", v, 4)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dev, dt = q.device, q.dtype
    _expect(fn, "k", k, (B, H, T, dk), dt, dev)
    _expect(fn, "v", v, (B, H, T, dv), dt, dev)
    for name, t in (("lambda", lam), ("eta", eta), ("gate", gate)):
        _expect(fn, name, t, (H,), torch.float32, dev)
    _expect(fn, "out", out, (B, H, T, dv), dt, dev)
    if state is not None:
        if (state.B, state.H, state.W, state.d_k, state.d_v, state.dtype) != (B, H, int(W), dk, dv, dt):
            raise ValueError(f"{fn}: state is (B,H,W,d_k,d_v,dtype)=({state.B},{state.H},{state.W},"
                             f"{state.d_k},{state.d_v},{state.dtype}); the call has ({B},{H},{W},{dk},{dv},{dt})")
        _check_state_tensors(fn, state, dev)
    return B, H, T, dk, dv


def _check_state_tensors(fn, state, dev):
    B, H, W, dk, dv = state.B, state.H, state.W, state.d_k, state.d_v
    _dev(state.ring_k, state.ring_v, state.A, state.pos)
    _expect(fn, "state.ring_k", state.ring_k, (B, H, W, dk), state.dtype, dev)
    _expect(fn, "state.ring_v", state.ring_v, (B, H, W, dv), state.dtype, dev)
    _expect(fn, "state.A", state.A, (B, H, dk, dv), torch.float32, dev)
    _expect(fn, "state.pos", state.pos, (B,), torch.int64, dev)


def tc_layer_forward(q, k, v, lam, eta, gate, W, softmax_scale=0.0, out=None, state=None,
                     workspace=None, stream=None):
    """Tensor Cache prefill; q,k [B,H,T,d_k], v [B,H,T,d_v]; returns y [B,H,T,d_v]."""
    _dev(q, k, v, lam, eta, gate, out, workspace)
    B, H, T, dk, dv = _check_tc_prefill("tc_layer_forward", q, k, v, lam, eta, gate, out, state, W)
    dt = dtype_code(q.dtype)
    y = torch.empty(B, H, T, dv, dtype=q.dtype, device=q.device) if out is None else out
    ws = _workspace(tc_layer_forward_workspace_size(B, H, T, dk, dv, W, q.dtype), workspace, q.device)
    st = ctypes.byref(state.struct()) if state is not None else None
    s = _stream(stream)
    _check(lib().tc_layer_forward(_ptr(q), _ptr(k), _ptr(v), dt, B, H, T, dk, dv, int(W), _ptr(lam),
                                  _ptr(eta), _ptr(gate), float(softmax_scale), _ptr(y), st, _ptr(ws),
                                  ws.numel(), s))
    _remember("tc_layer_forward", ws, s)
    return y


STATIC_SCRATCH_BYTES = 64 << 20  # OPAM_STATIC_SCRATCH_BYTES in include/opam.h


def tc_layer_forward_noalloc(q, k, v, lam, eta, gate, W, out, softmax_scale=0.0, state=None,
                             stream=None):
    """tc_layer_forward for callers that cannot allocate device memory.

    For hosts that hand the library only input and output buffers (plugins
    inside an application that owns all device memory, services that forbid
    allocation after start-up).  ``out`` must be given; no workspace is taken:
    the library uses its built-in scratch of STATIC_SCRATCH_BYTES, and rejects
    larger problems with OpamError(WORKSPACE).  Calls sharing a device must
    not overlap on the GPU; make one call on a device outside stream capture
    before capturing any.  check_device_error(None) reads its status.
    """
    _dev(q, k, v, lam, eta, gate, out)
    if out is None:
        raise ValueError("tc_layer_forward_noalloc: out must be given")
    B, H, T, dk, dv = _check_tc_prefill("tc_layer_forward_noalloc", q, k, v, lam, eta, gate, out, state, W)
    st = ctypes.byref(state.struct()) if state is not None else None
    _check(lib().tc_layer_forward_noalloc(_ptr(q), _ptr(k), _ptr(v), dtype_code(q.dtype), B, H, T, dk, dv,
                                          int(W), _ptr(lam), _ptr(eta), _ptr(gate), float(softmax_scale),
                                          _ptr(out), st, _stream(stream)))
    return out


def tc_layer_backward_workspace_size(B, H, T, d_k, d_v, W, dtype) -> int:
    return int(lib().tc_layer_backward_workspace_size(B, H, T, d_k, d_v, W, dtype_code(dtype)))


def tc_layer_backward(q, k, v, lam, eta, gate, W, dy, softmax_scale=0.0, out=None, workspace=None,
                      stream=None):
    """Gradient of sum <dy, y> through tc_layer_forward.  Returns
    (dq, dk, dv, dlam, deta, dgate); ``out`` may give those six tensors."""
    fn = "tc_layer_backward"
    _dev(q, k, v, lam, eta, gate, dy, workspace)
    B, H, T, dk, dv = _check_tc_prefill(fn, q, k, v, lam, eta, gate, None, None, W)
    _expect(fn, "dy", dy, (B, H, T, dv), q.dtype, q.device)
    if out is None:
        out = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
               torch.empty(H, dtype=torch.float32, device=q.device), torch.empty(H, dtype=torch.float32, device=q.device),
               torch.empty(H, dtype=torch.float32, device=q.device))
    gq, gk, gv, glam, geta, ggate = out
    _dev(*out)
    _expect(fn, "dq", gq, (B, H, T, dk), q.dtype, q.device)
    _expect(fn, "dk", gk, (B, H, T, dk), q.dtype, q.device)
    _expect(fn, "dv", gv, (B, H, T, dv), q.dtype, q.device)
    for name, t in (("dlambda", glam), ("deta", geta), ("dgate", ggate)):
        _expect(fn, name, t, (H,), torch.float32, q.device)
    ws = _workspace(tc_layer_backward_workspace_size(B, H, T, dk, dv, W, q.dtype), workspace, q.device)
    s = _stream(stream)
    _check(lib().tc_layer_backward(_ptr(q), _ptr(k), _ptr(v), dtype_code(q.dtype), B, H, T, dk, dv, int(W),
                                   _ptr(lam), _ptr(eta), _ptr(gate), float(softmax_scale), _ptr(dy), _ptr(gq),
                                   _ptr(gk), _ptr(gv), _ptr(glam), _ptr(geta), _ptr(ggate), _ptr(ws), ws.numel(),
                                   s))
    _remember(fn, ws, s)
    return out


def tc_window_forward_workspace_size(B, H, T, d_k, d_v, W, dtype) -> int:
    return int(lib().tc_window_forward_workspace_size(B, H, T, d_k, d_v, W, dtype_code(dtype)))


def tc_window_forward(q, k, v, W, softmax_scale=0.0, out=None, workspace=None, stream=None):
    """Window-only variant (the ring alone, no L2 memory); q,k [B,H,T,d_k],
    v [B,H,T,d_v]; returns y [B,H,T,d_v]."""
    _dev(q, k, v, out, workspace)
    B, H, T, dk, dv = _check_tc_prefill("tc_window_forward", q, k, v, None, None, None, out, None, W)
    y = torch.empty(B, H, T, dv, dtype=q.dtype, device=q.device) if out is None else out
    ws = _workspace(tc_window_forward_workspace_size(B, H, T, dk, dv, W, q.dtype), workspace, q.device)
    s = _stream(stream)
    _check(lib().tc_window_forward(_ptr(q), _ptr(k), _ptr(v), dtype_code(q.dtype), B, H, T, dk, dv, int(W),
                                   float(softmax_scale), _ptr(y), _ptr(ws), ws.numel(), s))
    _remember("tc_window_forward", ws, s)
    return y


def tc_decode_step_workspace_size(state: TCState) -> int:
    return int(lib().tc_decode_step_workspace_size(ctypes.byref(state.struct())))


def tc_decode_step(state: TCState, q, k, v, lam, eta, gate, softmax_scale=0.0, out=None,
                   workspace=None, stream=None):
    """One decode step; q,k [B,H,d_k], v [B,H,d_v]; returns y [B,H,d_v]; updates state."""
    fn = "tc_decode_step"
    _dev(q, k, v, lam, eta, gate, out, workspace)
    B, H, dk, dv, dev = state.B, state.H, state.d_k, state.d_v, q.device
    _check_state_tensors(fn, state, dev)
    _expect(fn, "q", q, (B, H, dk), state.dtype, dev)
    _expect(fn, "k", k, (B, H, dk), state.dtype, dev)
    _expect(fn, "v", v, (B, H, dv), state.dtype, dev)
    for name, t in (("lambda", lam), ("eta", eta), ("gate", gate)):
        _expect(fn, name, t, (H,), torch.float32, dev)
    _expect(fn, "out", out, (B, H, dv), state.dtype, dev)
    y = torch.empty(B, H, dv, dtype=state.dtype, device=dev) if out is None else out
    st = state.struct()
    ws = _workspace(int(lib().tc_decode_step_workspace_size(ctypes.byref(st))), workspace, dev)
    s = _stream(stream)
    _check(lib().tc_decode_step(ctypes.byref(st), _ptr(q), _ptr(k), _ptr(v), _ptr(lam), _ptr(eta),
                                _ptr(gate), float(softmax_scale), _ptr(y), _ptr(ws), ws.numel(), s))
    _remember("tc_decode_step", ws, s)
    return y


# ------------------------------------------------------------------ DeltaNet
def delta_rule_forward_workspace_size(B, H, T, d_k, d_v, chunk, dtype) -> int:
    return int(lib().delta_rule_forward_workspace_size(B, H, T, d_k, d_v, chunk, dtype_code(dtype)))


def delta_rule_forward(q, k, v, beta, chunk=0, S0=None, S_out=None, out=None, workspace=None,
                       stream=None):
    """DeltaNet delta rule; q,k [B,H,T,d_k], v [B,H,T,d_v], beta [B,H,T] fp32."""
    fn = "delta_rule_forward"
    _dev(q, k, v, beta, S0, S_out, out, workspace)
    _ndim(fn, "q", q, 4)
    _ndim(fn, "v", v, 4)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dev, dt = q.device, q.dtype
    _expect(fn, "k", k, (B, H, T, dk), dt, dev)
    _expect(fn, "v", v, (B, H, T, dv), dt, dev)
    _expect(fn, "beta", beta, (B, H, T), torch.float32, dev)
    _expect(fn, "S0", S0, (B, H, dk, dv), torch.float32, dev)
    _expect(fn, "S_out", S_out, (B, H, dk, dv), torch.float32, dev)
    _expect(fn, "out", out, (B, H, T, dv), dt, dev)
    y = torch.empty(B, H, T, dv, dtype=q.dtype, device=q.device) if out is None else out
    ws = _workspace(delta_rule_forward_workspace_size(B, H, T, dk, dv, chunk, q.dtype), workspace,
                    q.device)
    s = _stream(stream)
    _check(lib().delta_rule_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), dtype_code(q.dtype), B, H,
                                    T, dk, dv, int(chunk), _ptr(S0), _ptr(S_out), _ptr(y), _ptr(ws),
                                    ws.numel(), s))
    _remember("delta_rule_forward", ws, s)
    return y


def delta_rule_backward_workspace_size(B, H, T, d_k, d_v, dtype) -> int:
    return int(lib().delta_rule_backward_workspace_size(B, H, T, d_k, d_v, dtype_code(dtype)))


def delta_rule_backward(q, k, v, beta, dy, S0=None, dS_T=None, want_dS0=False, out=None, workspace=None,
                        stream=None):
    """Gradient of sum <dy, o> (+ <dS_T, S_T>) through delta_rule_forward.
    Returns (dq, dk, dv, dbeta, dS0 or None)."""
    fn = "delta_rule_backward"
    _dev(q, k, v, beta, dy, S0, dS_T, workspace)
    _ndim(fn, "q", q, 4)
    _ndim(fn, "v", v, 4)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dev, dt = q.device, q.dtype
    _expect(fn, "k", k, (B, H, T, dk), dt, dev)
    _expect(fn, "v", v, (B, H, T, dv), dt, dev)
    _expect(fn, "beta", beta, (B, H, T), torch.float32, dev)
    _expect(fn, "dy", dy, (B, H, T, dv), dt, dev)
    _expect(fn, "S0", S0, (B, H, dk, dv), torch.float32, dev)
    _expect(fn, "dS_T", dS_T, (B, H, dk, dv), torch.float32, dev)
    if out is None:
        out = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(beta),
               torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev) if want_dS0 else None)
    gq, gk, gv, gb, gS0 = out
    _dev(*out)
    _expect(fn, "dq", gq, (B, H, T, dk), dt, dev)
    _expect(fn, "dk", gk, (B, H, T, dk), dt, dev)
    _expect(fn, "dv", gv, (B, H, T, dv), dt, dev)
    _expect(fn, "dbeta", gb, (B, H, T), torch.float32, dev)
    _expect(fn, "dS0", gS0, (B, H, dk, dv), torch.float32, dev)
    ws = _workspace(delta_rule_backward_workspace_size(B, H, T, dk, dv, dt), workspace, dev)
    s = _stream(stream)
    _check(lib().delta_rule_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), dtype_code(dt), B, H, T, dk, dv,
                                     _ptr(S0), _ptr(dy), _ptr(dS_T), _ptr(gq), _ptr(gk), _ptr(gv), _ptr(gb),
                                     _ptr(gS0), _ptr(ws), ws.numel(), s))
    _remember(fn, ws, s)
    return out


def delta_decode_step(S, q, k, v, beta, out=None, stream=None):
    """One DeltaNet decode step; S [B,H,d_k,d_v] fp32 key-major (updated in
    place), q,k [B,H,d_k], v [B,H,d_v], beta [B,H] fp32; returns y [B,H,d_v]."""
    fn = "delta_decode_step"
    _dev(S, q, k, v, beta, out)
    _ndim(fn, "q", q, 3)
    _ndim(fn, "v", v, 3)
    B, H, dk = q.shape
    dv = v.shape[-1]
    dev, dt = q.device, q.dtype
    _expect(fn, "k", k, (B, H, dk), dt, dev)
    _expect(fn, "v", v, (B, H, dv), dt, dev)
    _expect(fn, "S", S, (B, H, dk, dv), torch.float32, dev)
    _expect(fn, "beta", beta, (B, H), torch.float32, dev)
    _expect(fn, "out", out, (B, H, dv), dt, dev)
    y = torch.empty(B, H, dv, dtype=q.dtype, device=q.device) if out is None else out
    _check(lib().delta_decode_step(_ptr(S), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), dtype_code(q.dtype), B,
                                   H, dk, dv, _ptr(y), _stream(stream)))
    return y


# ------------------------------------------------------------------ BDH
def sparse_linattn_forward_workspace_size(B, H, T, N, d_v) -> int:
    return int(lib().sparse_linattn_forward_workspace_size(B, H, T, N, d_v))


def sparse_linattn_forward(q, k, v, S0=None, S_out=None, out=None, workspace=None, stream=None):
    """BDH-style additive linear attention; q,k [B,H,T,N] fp32, v [B,H,T,d_v] fp32."""
    fn = "sparse_linattn_forward"
    _dev(q, k, v, S0, S_out, out, workspace)
    _ndim(fn, "q", q, 4)
    _ndim(fn, "v", v, 4)
    B, H, T, N = q.shape
    dv = v.shape[-1]
    dev, f32 = q.device, torch.float32
    _expect(fn, "q", q, (B, H, T, N), f32, dev)
    _expect(fn, "k", k, (B, H, T, N), f32, dev)
    _expect(fn, "v", v, (B, H, T, dv), f32, dev)
    _expect(fn, "S0", S0, (B, H, N, dv), f32, dev)
    _expect(fn, "S_out", S_out, (B, H, N, dv), f32, dev)
    _expect(fn, "out", out, (B, H, T, dv), f32, dev)
    y = torch.empty(B, H, T, dv, dtype=torch.float32, device=q.device) if out is None else out
    ws = _workspace(sparse_linattn_forward_workspace_size(B, H, T, N, dv), workspace, q.device)
    s = _stream(stream)
    _check(lib().sparse_linattn_forward(_ptr(q), _ptr(k), _ptr(v), B, H, T, N, dv, _ptr(S0),
                                        _ptr(S_out), _ptr(y), _ptr(ws), ws.numel(), s))
    _remember("sparse_linattn_forward", ws, s)
    return y


def sparse_linattn_keygen_forward_workspace_size(B, H, T, R, N, d_v) -> int:
    return int(lib().sparse_linattn_keygen_forward_workspace_size(B, H, T, R, N, d_v))


def sparse_linattn_keygen_forward(xq, xk, U, theta, v, S0=None, S_out=None, out=None, workspace=None,
                                  stream=None):
    """BDH-style attention with q = ReLU(xq U_h - theta), k = ReLU(xk U_h - theta)
    generated on the GPU: xq, xk [B,H,T,R] bf16, U [H,R,N] bf16, v [B,H,T,d_v]
    fp32; returns y [B,H,T,d_v] fp32."""
    fn = "sparse_linattn_keygen_forward"
    _dev(xq, xk, U, v, S0, S_out, out, workspace)
    _ndim(fn, "xq", xq, 4)
    _ndim(fn, "U", U, 3)
    _ndim(fn, "v", v, 4)
    B, H, T, R = xq.shape
    N = U.shape[-1]
    dv = v.shape[-1]
    dev, f32, bf = xq.device, torch.float32, torch.bfloat16
    _expect(fn, "xq", xq, (B, H, T, R), bf, dev)
    _expect(fn, "xk", xk, (B, H, T, R), bf, dev)
    _expect(fn, "U", U, (H, R, N), bf, dev)
    _expect(fn, "v", v, (B, H, T, dv), f32, dev)
    _expect(fn, "S0", S0, (B, H, N, dv), f32, dev)
    _expect(fn, "S_out", S_out, (B, H, N, dv), f32, dev)
    _expect(fn, "out", out, (B, H, T, dv), f32, dev)
    y = torch.empty(B, H, T, dv, dtype=f32, device=dev) if out is None else out
    ws = _workspace(sparse_linattn_keygen_forward_workspace_size(B, H, T, R, N, dv), workspace, dev)
    s = _stream(stream)
    _check(lib().sparse_linattn_keygen_forward(_ptr(xq), _ptr(xk), _ptr(U), float(theta), _ptr(v), B, H, T, R, N,
                                               dv, _ptr(S0), _ptr(S_out), _ptr(y), _ptr(ws), ws.numel(), s))
    _remember(fn, ws, s)
    return y
