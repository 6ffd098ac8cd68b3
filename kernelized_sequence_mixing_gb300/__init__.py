"""GB300 (sm_103a) kernelized linear attention, phi(x) = elu(x) + 1.

A thin ctypes binding over the C ABI in include/linattn.h (liblinattn.so,
built in-tree by ``kernelized_sequence_mixing_gb300.build``).  This module
only marshals arguments: shapes, dtypes, the current CUDA stream and, for host
tensors, the host<->device copies around the call.  Every step of the
computation runs in the library's CUDA kernels; there is no CPU fallback, and
a missing library raises RuntimeError.

Functions (same names as the C entry points, minus the ``la_`` prefix):
  forward(q, k, v, causal=True, gamma=None, eps=1e-6, out=None)
  prefill_state(k, v, gamma=None, S=None, z=None)
  decode_step(q, k, v, S, z, gamma=None, eps=1e-6, out=None)
  forward_state(q, k, v, gamma=None, eps=1e-6, out=None, S=None, z=None)
  forward_gated(q, k, v, a, eps=1e-6, out=None, return_state=False, S=None, z=None)
  decode_gated(q, k, v, a, S, z, eps=1e-6, out=None)
  favor_features(x, W, out=None)
  forward_favor(q, k, v, W, causal=True, gamma=None, eps=1e-6, out=None)
  backward(q, k, v, do, gamma=None, eps=1e-6)
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import workloads  # noqa: F401  (seeded input generators)

__all__ = ["forward", "prefill_state", "decode_step", "forward_state",
           "forward_gated", "decode_gated", "favor_features", "forward_favor", "backward",
           "status_string",
           "device_wait_timeouts", "causal_kernel", "backward_kernel",
           "load_library", "library_path", "LinAttnError", "workloads"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "liblinattn.so")
_lib = None
_lock = threading.Lock()

LA_OK, LA_ERR_INVALID_ARG, LA_ERR_UNSUPPORTED, LA_ERR_CUDA = 0, 1, 2, 3
_DTYPES = {torch.float32: 0, torch.bfloat16: 1}


class LinAttnError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__(f"{fn}: {status_string(code)} (status {code})")


def library_path() -> str:
    """Path of the in-tree liblinattn.so that load_library() opens."""
    return _LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load liblinattn.so; raises RuntimeError if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"{_LIB_PATH} is missing: build it with "
                    "`python -m kernelized_sequence_mixing_gb300.build` "
                    "(or __graft_entry__.build()); there is no fallback path")
            lib = ctypes.CDLL(_LIB_PATH)
            P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            FP = ctypes.POINTER(ctypes.c_float)
            lib.la_forward.argtypes = [P, P, P, P, I, I, I, I, I, I, FP, F, I, P]
            lib.la_forward_host.argtypes = [P, P, P, P, I, I, I, I, I, I, FP, F, I, P]
            lib.la_forward_host.restype = I
            lib.la_forward.restype = I
            lib.la_prefill_state.argtypes = [P, P, P, P, I, I, I, I, I, FP, I, P]
            lib.la_prefill_state.restype = I
            lib.la_forward_state.argtypes = [P, P, P, P, P, P, I, I, I, I, I, FP, F,
                                             I, P]
            lib.la_forward_state.restype = I
            lib.la_decode_step.argtypes = [P, P, P, P, P, P, I, I, I, I, FP, F,
                                           I, P]
            lib.la_decode_step.restype = I
            lib.la_forward_gated.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, F,
                                             I, P]
            lib.la_forward_gated.restype = I
            lib.la_decode_gated.argtypes = [P, P, P, P, P, P, P, I, I, I, I, F, I, P]
            lib.la_decode_gated.restype = I
            lib.la_favor_features.argtypes = [P, P, P, I, I, I, I, P]
            lib.la_favor_features.restype = I
            lib.la_forward_favor.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, FP, F,
                                             I, P]
            lib.la_forward_favor.restype = I
            lib.la_backward.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, FP, F, I, P]
            lib.la_backward.restype = I
            lib.la_gated_kernel.argtypes = [I, I, I, I, I, I, I]
            lib.la_gated_kernel.restype = I
            lib.la_backward_launches.argtypes = [I, I, I, I, I, FP, I]
            lib.la_backward_launches.restype = I
            lib.la_backward_kernel.argtypes = [I, I, I, I, I, FP, I]
            lib.la_backward_kernel.restype = I
            lib.la_causal_kernel.argtypes = [I, I, I, I, I, FP, I]
            lib.la_causal_kernel.restype = I
            lib.la_wait_selftest.argtypes = [ctypes.c_longlong, ctypes.POINTER(I)]
            lib.la_wait_selftest.restype = I
            lib.la_device_wait_timeouts.argtypes = [I]
            lib.la_device_wait_timeouts.restype = I
            lib.la_status_string.argtypes = [I]
            lib.la_status_string.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def status_string(code: int) -> str:
    """The library's text for a status code (la_status_string)."""
    return load_library().la_status_string(int(code)).decode()


def causal_kernel(B, H, N, D, Dv, gamma=None, dtype=torch.bfloat16) -> str:
    """Which kernel a causal forward with these sizes runs: "tensor-core-128"
    (128-token chunks), "tensor-core" (64-token chunks) or "cuda-core"
    (host-only query)."""
    code = load_library().la_causal_kernel(B, H, N, D, Dv, _gamma_arg(gamma, H),
                                           _DTYPES[dtype])
    if code < 0:
        raise LinAttnError("la_causal_kernel", -code)
    return {2: "tensor-core-128", 1: "tensor-core"}.get(code, "cuda-core")


def device_wait_timeouts(reset: bool = False) -> int:
    """Count of device-side bounded waits that gave up on the current device
    (nonzero: some kernel abandoned its work).  Synchronise first."""
    return int(load_library().la_device_wait_timeouts(1 if reset else 0))


def _gamma_arg(gamma, H):
    if gamma is None:
        return None
    if isinstance(gamma, torch.Tensor):
        vals = gamma.detach().to("cpu", torch.float32).reshape(-1).tolist()
    elif isinstance(gamma, (int, float)):
        vals = [float(gamma)] * H
    else:
        vals = [float(x) for x in gamma]
    if len(vals) != H:
        raise ValueError(f"gamma needs {H} values (one per head), got {len(vals)}")
    return (ctypes.c_float * H)(*vals)


def _dtype_code(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}: use float32 or bfloat16")


def _stream(dev):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _check(fn, code):
    if code != LA_OK:
        raise LinAttnError(fn, code)


def _contig(name, t):
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# Device types whose memory the kernels may address.  The C entry points take
# plain pointers and cannot tell a host pointer or a short buffer from a good
# one, so every shape, dtype and device is checked here, before the call.
_DEVICE_TYPES = ("cuda",)


def _one_device(fn, named, allow_host=False):
    """All tensors of ``named`` [(name, tensor or None)] on one device, of a
    type the kernels can address (or the host, where ``allow_host``: the
    forward copies host tensors itself)."""
    present = [(n, t) for n, t in named if t is not None]
    devs = {t.device for _, t in present}
    if len(devs) > 1:
        where = ", ".join(f"{n} on {t.device}" for n, t in present)
        raise ValueError(f"{fn}: all tensors must be on one device ({where})")
    dev = next(iter(devs))
    if dev.type not in _DEVICE_TYPES and not allow_host:
        raise ValueError(f"{fn}: tensors must be CUDA tensors, got {dev}")
    return dev


def _expect(fn, name, t, shape, dtype):
    """A caller-provided buffer: exactly ``shape`` and ``dtype``, contiguous."""
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{fn}: {name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{fn}: {name} must be {dtype}, got {t.dtype}")
    _contig(name, t)


def _qkv(fn, q, k, v, extra=()):
    """q, k: [B, H, N, D]; v: [B, H, N, Dv]; one dtype (plus ``extra`` named
    tensors of that dtype), contiguous.  Returns (B, H, N, D, Dv)."""
    for n, t in (("q", q), ("k", k), ("v", v)) + tuple(extra):
        _contig(n, t)
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or v.shape[:3] != q.shape[:3]:
        raise ValueError(f"{fn}: expected q, k: [B, H, N, D] and v: [B, H, N, Dv]")
    if not all(t.dtype == q.dtype for t in (k, v) + tuple(t for _, t in extra)):
        names = ", ".join(["q", "k", "v"] + [n for n, _ in extra])
        raise TypeError(f"{fn}: {names} must share one dtype")
    _dtype_code(q)
    B, H, N, D = q.shape
    return B, H, N, D, v.shape[-1]


def _step_qkv(fn, q, k, v):
    """Decode-step inputs q, k: [B, H, D]; v: [B, H, Dv]; one dtype."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _contig(n, t)
    if q.dim() != 3 or k.shape != q.shape or v.dim() != 3 or v.shape[:2] != q.shape[:2]:
        raise ValueError(f"{fn}: expected q, k: [B, H, D] and v: [B, H, Dv]")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError(f"{fn}: q, k and v must share one dtype")
    _dtype_code(q)
    B, H, D = q.shape
    return B, H, D, v.shape[-1]


def forward(q, k, v, causal=True, gamma=None, eps=1e-6, out=None,
            device=None):
    """Linear attention over whole sequences.

    q, k: [B, H, N, D]; v: [B, H, N, Dv]; all float32 or all bfloat16,
    contiguous.  CUDA tensors are used in place on the current stream; host
    tensors go through la_forward_host on ``device`` (default cuda:0), which
    overlaps the copies with the kernels by groups of heads; the result is a
    host tensor (pinned), complete when this returns.  gamma: None, a float,
    or H per-head decays in [0, 1] (causal only).  Returns o: [B, H, N, Dv].
    """
    B, H, N, D, Dv = _qkv("forward", q, k, v)
    src = _one_device("forward", (("q", q), ("k", k), ("v", v), ("out", out)),
                      allow_host=True)
    if out is not None:
        _expect("forward", "out", out, (B, H, N, Dv), q.dtype)
    lib = load_library()
    host = src.type != "cuda"
    dev = torch.device(device or "cuda:0") if host else q.device
    dt = _dtype_code(q)
    g = _gamma_arg(gamma, H)
    with torch.cuda.device(dev):
        if host:
            qh, kh, vh = (t if t.is_pinned() else t.pin_memory() for t in (q, k, v))
            res = out if out is not None else torch.empty(
                (B, H, N, Dv), dtype=q.dtype, pin_memory=True)
            _check("la_forward_host", lib.la_forward_host(
                _ptr(qh), _ptr(kh), _ptr(vh), _ptr(res), B, H, N, D, Dv,
                1 if causal else 0, g, float(eps), dt, _stream(dev)))
            torch.cuda.current_stream(dev).synchronize()
            return res
        od = out if out is not None else torch.empty(
            (B, H, N, Dv), dtype=q.dtype, device=dev)
        _check("la_forward", lib.la_forward(
            _ptr(q), _ptr(k), _ptr(v), _ptr(od), B, H, N, D, Dv,
            1 if causal else 0, g, float(eps), dt, _stream(dev)))
        return od


def prefill_state(k, v, gamma=None, S=None, z=None):
    """State after a causal pass: S = sum_j gamma^(N-1-j) phi(k_j) v_j^T,
    z likewise.  k: [B, H, N, D], v: [B, H, N, Dv] CUDA tensors.  Returns
    (S [B, H, D, Dv] fp32, z [B, H, D] fp32), written into S, z if given."""
    _contig("k", k)
    _contig("v", v)
    if k.dim() != 4 or v.dim() != 4 or v.shape[:3] != k.shape[:3]:
        raise ValueError("prefill_state: expected k: [B, H, N, D] and v: [B, H, N, Dv]")
    if k.dtype != v.dtype:
        raise TypeError("prefill_state: k and v must share one dtype")
    _dtype_code(k)
    B, H, N, D = k.shape
    Dv = v.shape[-1]
    dev = _one_device("prefill_state", (("k", k), ("v", v), ("S", S), ("z", z)))
    if S is not None:
        _expect("prefill_state", "S", S, (B, H, D, Dv), torch.float32)
    if z is not None:
        _expect("prefill_state", "z", z, (B, H, D), torch.float32)
    lib = load_library()
    with torch.cuda.device(dev):
        if S is None:
            S = torch.empty((B, H, D, Dv), dtype=torch.float32, device=dev)
        if z is None:
            z = torch.empty((B, H, D), dtype=torch.float32, device=dev)
        _check("la_prefill_state", lib.la_prefill_state(
            _ptr(k), _ptr(v), _ptr(S), _ptr(z), B, H, N, D, Dv,
            _gamma_arg(gamma, H), _dtype_code(k), _stream(dev)))
    return S, z


def forward_state(q, k, v, gamma=None, eps=1e-6, out=None, S=None, z=None):
    """Causal forward that also returns the state after the last token:
    (o [B, H, N, Dv], S [B, H, D, Dv] fp32, z [B, H, D] fp32), the state the
    decode loop continues from.  q, k: [B, H, N, D]; v: [B, H, N, Dv] CUDA
    tensors of one dtype; out, S, z: optional destinations."""
    fn = "forward_state"
    B, H, N, D, Dv = _qkv(fn, q, k, v)
    dev = _one_device(fn, (("q", q), ("k", k), ("v", v), ("out", out), ("S", S), ("z", z)))
    if out is not None:
        _expect(fn, "out", out, (B, H, N, Dv), q.dtype)
    if S is not None:
        _expect(fn, "S", S, (B, H, D, Dv), torch.float32)
    if z is not None:
        _expect(fn, "z", z, (B, H, D), torch.float32)
    lib = load_library()
    with torch.cuda.device(dev):
        o = out if out is not None else torch.empty((B, H, N, Dv), dtype=q.dtype, device=dev)
        if S is None:
            S = torch.empty((B, H, D, Dv), dtype=torch.float32, device=dev)
        if z is None:
            z = torch.empty((B, H, D), dtype=torch.float32, device=dev)
        _check("la_forward_state", lib.la_forward_state(
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(S), _ptr(z), B, H, N, D, Dv,
            _gamma_arg(gamma, H), float(eps), _dtype_code(q), _stream(dev)))
    return o, S, z


def decode_step(q, k, v, S, z, gamma=None, eps=1e-6, out=None):
    """One recurrent step in place on (S, z): update with (k, v), then read
    out with q.  q, k: [B, H, D]; v: [B, H, Dv]; S: [B, H, D, Dv] fp32;
    z: [B, H, D] fp32 (all CUDA).  Returns o: [B, H, Dv]."""
    fn = "decode_step"
    B, H, D, Dv = _step_qkv(fn, q, k, v)
    dev = _one_device(fn, (("q", q), ("k", k), ("v", v), ("S", S), ("z", z), ("out", out)))
    _expect(fn, "S", S, (B, H, D, Dv), torch.float32)
    _expect(fn, "z", z, (B, H, D), torch.float32)
    if out is not None:
        _expect(fn, "out", out, (B, H, Dv), q.dtype)
    lib = load_library()
    with torch.cuda.device(dev):
        if out is None:
            out = torch.empty((B, H, Dv), dtype=q.dtype, device=dev)
        _check("la_decode_step", lib.la_decode_step(
            _ptr(q), _ptr(k), _ptr(v), _ptr(S), _ptr(z), _ptr(out), B, H, D,
            Dv, _gamma_arg(gamma, H), float(eps), _dtype_code(q),
            _stream(dev)))
    return out


def forward_gated(q, k, v, a, eps=1e-6, out=None, return_state=False, S=None, z=None):
    """Gated causal forward: S_t = diag(a_t) S_(t-1) + phi(k_t) v_t^T,
    z_t = a_t * z_(t-1) + phi(k_t), o_t = phi(q_t)^T S_t / (phi(q_t).z_t + eps).
    q, k: [B, H, N, D]; v: [B, H, N, Dv] CUDA tensors of one dtype; a:
    [B, H, N, D] float32 gates in [0, 1] on the same device.  Returns o, or
    (o, S [B, H, D, Dv] fp32, z [B, H, D] fp32) with the state after the last
    token when return_state is true (or S, z are given)."""
    fn = "forward_gated"
    B, H, N, D, Dv = _qkv(fn, q, k, v)
    _expect(fn, "a", a, (B, H, N, D), torch.float32)
    dev = _one_device(fn, (("q", q), ("k", k), ("v", v), ("a", a), ("out", out), ("S", S),
                           ("z", z)))
    if out is not None:
        _expect(fn, "out", out, (B, H, N, Dv), q.dtype)
    if S is not None:
        _expect(fn, "S", S, (B, H, D, Dv), torch.float32)
    if z is not None:
        _expect(fn, "z", z, (B, H, D), torch.float32)
    lib = load_library()
    want_state = return_state or S is not None or z is not None
    with torch.cuda.device(dev):
        o = out if out is not None else torch.empty((B, H, N, Dv), dtype=q.dtype, device=dev)
        if want_state:
            if S is None:
                S = torch.empty((B, H, D, Dv), dtype=torch.float32, device=dev)
            if z is None:
                z = torch.empty((B, H, D), dtype=torch.float32, device=dev)
        _check("la_forward_gated", lib.la_forward_gated(
            _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(o),
            _ptr(S) if want_state else None, _ptr(z) if want_state else None,
            B, H, N, D, Dv, float(eps), _dtype_code(q), _stream(dev)))
    return (o, S, z) if want_state else o


def decode_gated(q, k, v, a, S, z, eps=1e-6, out=None):
    """One gated recurrent step in place on (S, z): S <- diag(a) S +
    phi(k) v^T, z <- a * z + phi(k), then read out with q.  q, k, a: [B, H, D]
    (a float32); v: [B, H, Dv]; S: [B, H, D, Dv] fp32; z: [B, H, D] fp32 (all
    CUDA).  Returns o: [B, H, Dv]."""
    fn = "decode_gated"
    B, H, D, Dv = _step_qkv(fn, q, k, v)
    dev = _one_device(fn, (("q", q), ("k", k), ("v", v), ("a", a), ("S", S), ("z", z),
                           ("out", out)))
    _expect(fn, "a", a, (B, H, D), torch.float32)
    _expect(fn, "S", S, (B, H, D, Dv), torch.float32)
    _expect(fn, "z", z, (B, H, D), torch.float32)
    if out is not None:
        _expect(fn, "out", out, (B, H, Dv), q.dtype)
    lib = load_library()
    with torch.cuda.device(dev):
        if out is None:
            out = torch.empty((B, H, Dv), dtype=q.dtype, device=dev)
        _check("la_decode_gated", lib.la_decode_gated(
            _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(S), _ptr(z), _ptr(out), B, H, D,
            Dv, float(eps), _dtype_code(q), _stream(dev)))
    return out


def favor_features(x, W, out=None):
    """Performer random features phi(x) = r^(-1/2) exp(W x - |x|^2 / 2) of
    every row of x [..., D] with the directions W [r, D] (same dtype, CUDA).
    Returns [..., r]."""
    fn = "favor_features"
    _contig("x", x)
    _contig("W", W)
    if x.dim() < 1 or W.dim() != 2 or W.shape[1] != x.shape[-1]:
        raise ValueError(f"{fn}: W must be [r, D] for x [..., D]")
    if W.dtype != x.dtype:
        raise TypeError(f"{fn}: W must have the dtype of x")
    _dtype_code(x)
    D, r = x.shape[-1], W.shape[0]
    rows = x.numel() // D if D else 0
    dev = _one_device(fn, (("x", x), ("W", W), ("out", out)))
    if out is not None:
        _expect(fn, "out", out, tuple(x.shape[:-1]) + (r,), x.dtype)
    lib = load_library()
    with torch.cuda.device(dev):
        if out is None:
            out = torch.empty(x.shape[:-1] + (r,), dtype=x.dtype, device=dev)
        _check("la_favor_features", lib.la_favor_features(
            _ptr(x), _ptr(W), _ptr(out), rows, D, r, _dtype_code(x), _stream(dev)))
    return out


def forward_favor(q, k, v, W, causal=True, gamma=None, eps=1e-6, out=None):
    """Performer attention: the random features of q and k with the
    directions W [r, D], then linear attention over them (causal with
    optional per-head decay, or non-causal).  q, k: [B, H, N, D]; v:
    [B, H, N, Dv]; all CUDA tensors of one dtype.  Returns o [B, H, N, Dv]."""
    fn = "forward_favor"
    B, H, N, D, Dv = _qkv(fn, q, k, v, extra=(("W", W),))
    if W.dim() != 2 or W.shape[1] != D:
        raise ValueError(f"{fn}: W must be [r, D]")
    r = W.shape[0]
    dev = _one_device(fn, (("q", q), ("k", k), ("v", v), ("W", W), ("out", out)))
    if out is not None:
        _expect(fn, "out", out, (B, H, N, Dv), q.dtype)
    lib = load_library()
    with torch.cuda.device(dev):
        if out is None:
            out = torch.empty((B, H, N, Dv), dtype=q.dtype, device=dev)
        _check("la_forward_favor", lib.la_forward_favor(
            _ptr(q), _ptr(k), _ptr(v), _ptr(W), _ptr(out), B, H, N, D, Dv, r,
            1 if causal else 0, _gamma_arg(gamma, H), float(eps), _dtype_code(q),
            _stream(dev)))
    return out


def backward(q, k, v, do, gamma=None, eps=1e-6, dq=None, dk=None, dv=None):
    """Gradients (dq, dk, dv) of the causal forward o = forward(q, k, v,
    causal=True, gamma, eps) for the upstream gradient do = dL/do.  q, k:
    [B, H, N, D]; v, do: [B, H, N, Dv]; CUDA tensors of one dtype."""
    fn = "backward"
    B, H, N, D, Dv = _qkv(fn, q, k, v, extra=(("do", do),))
    if do.shape != v.shape:
        raise ValueError(f"{fn}: do must have the shape of v")
    dev = _one_device(fn, (("q", q), ("k", k), ("v", v), ("do", do), ("dq", dq), ("dk", dk),
                           ("dv", dv)))
    for n, t, shape in (("dq", dq, q.shape), ("dk", dk, k.shape), ("dv", dv, v.shape)):
        if t is not None:
            _expect(fn, n, t, shape, q.dtype)
    lib = load_library()
    with torch.cuda.device(dev):
        dq = torch.empty_like(q) if dq is None else dq
        dk = torch.empty_like(k) if dk is None else dk
        dv = torch.empty_like(v) if dv is None else dv
        _check("la_backward", lib.la_backward(
            _ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, D, Dv,
            _gamma_arg(gamma, H), float(eps), _dtype_code(q), _stream(dev)))
    return dq, dk, dv


def backward_launches(B, H, N, D, Dv, gamma=None, dtype=torch.bfloat16) -> int:
    """Kernels one backward() call with these arguments launches on the
    current device."""
    n = load_library().la_backward_launches(B, H, N, D, Dv, _gamma_arg(gamma, H), _DTYPES[dtype])
    if n < 0:
        raise LinAttnError("la_backward_launches", -n)
    return int(n)


def backward_kernel(B, H, N, D, Dv, gamma=None, dtype=torch.bfloat16) -> str:
    """Which kernels backward() runs: "tensor-core" (bf16, Dv = 64, every
    decay >= 0.35) or "cuda-core".  Host-only query."""
    code = load_library().la_backward_kernel(B, H, N, D, Dv, _gamma_arg(gamma, H), _DTYPES[dtype])
    if code < 0:
        raise LinAttnError("la_backward_kernel", -code)
    return "tensor-core" if code == 1 else "cuda-core"


def gated_kernel(B, H, N, D, Dv, dtype=torch.bfloat16, want_state=False) -> str:
    """Which form forward_gated runs: "tensor-core" (it still falls back to
    the CUDA-core form at run time when some chunk's gates forget harder
    than 2^-93) or "cuda-core"; the final state does not change the choice.
    Host-only query."""
    code = load_library().la_gated_kernel(B, H, N, D, Dv, _DTYPES[dtype], 1 if want_state else 0)
    if code < 0:
        raise LinAttnError("la_gated_kernel", -code)
    return "tensor-core" if code == 1 else "cuda-core"


def wait_selftest(cycles=2_000_000) -> bool:
    """Run the kernels' bounded wait on a barrier nothing arrives on, with a
    short limit: True if it gave up (and counted itself in
    device_wait_timeouts), as it should.  Synchronises the device."""
    gave_up = ctypes.c_int(0)
    _check("la_wait_selftest", load_library().la_wait_selftest(int(cycles), ctypes.byref(gave_up)))
    return bool(gave_up.value)
