"""fp64 CPU oracle for kernelized linear attention (phi = elu + 1).

TEST INFRASTRUCTURE ONLY: imported by the test suite, by the smoke check and
by the CPU-baseline leg of the benchmark, never by the library.  It shares no
code with the CUDA path; the arithmetic lives in ``linattn_oracle.c`` (plain C,
fp64, one unit per thread) and this module only marshals numpy arrays.

What each function computes, with the passage it follows:

* ``phi``         -- elu(x) + 1 with alpha = 1: x + 1 for x > 0, exp(x) else.
                     "Linear Attention Mechanisms" (dileepadev.github.io),
                     "Choosing the Feature Map", ELU-based features.
* ``causal``      -- the recurrence S_i = g S_{i-1} + phi(k_i) v_i^T,
                     z_i = g z_{i-1} + phi(k_i), o_i = phi(q_i)^T S_i /
                     (phi(q_i).z_i + eps).  Same page, "Recurrent
                     Reformulation"; decay from "Gating and Selective State
                     Updates" (RetNet) and "Attention-Free / Sub-Quadratic
                     Architectures", "Evolution: add decay/gating".
* ``noncausal``   -- S = sum_j phi(k_j) v_j^T, z = sum_j phi(k_j) once, then
                     the same read-out for every query.  "The Kernel Trick for
                     Attention"; eps as in the NumPy listing of "Linear
                     Attention Mechanisms" (sadullah.online).
* ``prefill``     -- the (S, z) left by ``causal`` after the last token.
* ``decode_step`` -- one iteration of the causal loop on a given (S, z).
* ``gated``       -- the causal loop with a data-dependent gate per step and
                     key feature in place of gamma: S_i = G_i (.) S_{i-1} +
                     phi(k_i) v_i^T with G_i = a_i 1^T, z gated alike.  Same
                     page, "Gating and Selective State Updates" (Gated Linear
                     Attention); "Evolution: add decay/gating".

Pins (tests/test_oracle.py) check every function against things other than
itself: a quadratic masked brute force, an exact rational evaluation, a
restatement of the pages' NumPy listing, closed forms and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "linattn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle into oracle/liboracle.so with the host gcc.

    -ffp-contract=off keeps every multiply and add separately rounded, so x86
    and Arm hosts give the same fp64 results.
    """
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
           "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            lib.oracle_phi.argtypes = [f64]
            lib.oracle_phi.restype = f64
            lib.oracle_causal.argtypes = [P, P, P, P, f64, i64, i64, i32, i32,
                                          P, P, P, i32, i32]
            lib.oracle_causal.restype = i32
            lib.oracle_noncausal.argtypes = [P, P, P, f64, i64, i64, i32, i32,
                                             P, P, P, i32]
            lib.oracle_noncausal.restype = i32
            lib.oracle_decode_step.argtypes = [P, P, P, P, f64, i64, i32, i32,
                                               P, P, P, i32]
            lib.oracle_decode_step.restype = i32
            lib.oracle_gated.argtypes = [P, P, P, P, f64, i64, i64, i32, i32,
                                         P, P, P, i32]
            lib.oracle_gated.restype = i32
            _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _f32(a, ndim):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    if a.ndim != ndim:
        raise ValueError(f"expected a {ndim}-d array, got shape {a.shape}")
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _units(x):
    """Fold leading dims: [..., N, D] -> [U, N, D]."""
    lead = x.shape[:-2]
    return int(np.prod(lead)) if lead else 1, lead


def _gamma_units(gamma, lead, U):
    """gamma: None (all 1), a scalar, or an array broadcastable to lead dims
    (e.g. one value per head for [B, H, ...] inputs).  Returned per unit in
    fp64, widened from the fp32 value the library also receives."""
    if gamma is None:
        return None
    g = np.asarray(gamma, dtype=np.float32).astype(np.float64)
    g = np.broadcast_to(g, lead if lead else ()).reshape(-1) if g.ndim else \
        np.full(U, float(g))
    return np.ascontiguousarray(g.reshape(U))


def phi(x):
    """phi(x) = elu(x) + 1 evaluated by the C oracle, element by element."""
    lib = _load()
    x = np.asarray(x, dtype=np.float64)
    return np.vectorize(lib.oracle_phi, otypes=[np.float64])(x)


def causal(q, k, v, gamma=None, eps=1e-6, return_state=False, state=None,
           nthreads=None):
    """Causal linear attention, token-by-token recurrence in fp64.

    q, k: [..., N, D]; v: [..., N, Dv] (any float dtype; widened to fp32 then
    fp64 -- bf16 and fp32 widen exactly).  gamma per leading unit (see
    ``_gamma_units``).  ``state`` = (S [..., D, Dv], z [..., D]) starts the
    recurrence from a given state.  Returns o [..., N, Dv] fp64, plus (S, z)
    after the last token if ``return_state``.
    """
    lib = _load()
    q = _f32(q, np.ndim(q)); k = _f32(k, q.ndim); v = _f32(v, q.ndim)
    N, D = q.shape[-2], q.shape[-1]
    Dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:-1] != q.shape[:-1]:
        raise ValueError("shape mismatch")
    U, lead = _units(q)
    g = _gamma_units(gamma, lead, U)
    o = np.empty(q.shape[:-1] + (Dv,), dtype=np.float64)
    S = np.zeros(lead + (D, Dv), dtype=np.float64)
    z = np.zeros(lead + (D,), dtype=np.float64)
    if state is not None:
        S[...] = np.asarray(state[0], dtype=np.float64)
        z[...] = np.asarray(state[1], dtype=np.float64)
    rc = lib.oracle_causal(_ptr(q), _ptr(k), _ptr(v), _ptr(g), float(eps), U,
                           N, D, Dv, _ptr(o), _ptr(S), _ptr(z),
                           1 if state is not None else 0,
                           nthreads or default_threads())
    if rc:
        raise RuntimeError("oracle_causal rejected its arguments")
    return (o, S, z) if return_state else o


def noncausal(q, k, v, eps=1e-6, return_state=False, nthreads=None):
    """Non-causal linear attention in fp64: S, z over all keys, then o."""
    lib = _load()
    q = _f32(q, np.ndim(q)); k = _f32(k, q.ndim); v = _f32(v, q.ndim)
    N, D = q.shape[-2], q.shape[-1]
    Dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:-1] != q.shape[:-1]:
        raise ValueError("shape mismatch")
    U, lead = _units(q)
    o = np.empty(q.shape[:-1] + (Dv,), dtype=np.float64)
    S = np.empty(lead + (D, Dv), dtype=np.float64)
    z = np.empty(lead + (D,), dtype=np.float64)
    rc = lib.oracle_noncausal(_ptr(q), _ptr(k), _ptr(v), float(eps), U, N, D,
                              Dv, _ptr(o), _ptr(S), _ptr(z),
                              nthreads or default_threads())
    if rc:
        raise RuntimeError("oracle_noncausal rejected its arguments")
    return (o, S, z) if return_state else o


def prefill(k, v, gamma=None, nthreads=None):
    """State (S [..., D, Dv], z [..., D]) after running the causal recurrence
    over all N tokens: S = sum_j gamma^(N-1-j) phi(k_j) v_j^T, likewise z."""
    lib = _load()
    k = _f32(k, np.ndim(k)); v = _f32(v, k.ndim)
    N, D = k.shape[-2], k.shape[-1]
    Dv = v.shape[-1]
    U, lead = _units(k)
    g = _gamma_units(gamma, lead, U)
    S = np.zeros(lead + (D, Dv), dtype=np.float64)
    z = np.zeros(lead + (D,), dtype=np.float64)
    rc = lib.oracle_causal(None, _ptr(k), _ptr(v), _ptr(g), 0.0, U, N, D, Dv,
                           None, _ptr(S), _ptr(z), 0,
                           nthreads or default_threads())
    if rc:
        raise RuntimeError("oracle_causal rejected its arguments")
    return S, z


def decode_step(q, k, v, S, z, gamma=None, eps=1e-6, nthreads=None):
    """One recurrent step: q, k [..., D], v [..., Dv]; S [..., D, Dv] and
    z [..., D] (fp64) are returned updated (copies), with o [..., Dv]."""
    lib = _load()
    q = _f32(q, np.ndim(q)); k = _f32(k, q.ndim); v = _f32(v, q.ndim)
    D, Dv = q.shape[-1], v.shape[-1]
    lead = q.shape[:-1]
    U = int(np.prod(lead)) if lead else 1
    S = np.array(S, dtype=np.float64, copy=True, order="C")
    z = np.array(z, dtype=np.float64, copy=True, order="C")
    if S.shape != lead + (D, Dv) or z.shape != lead + (D,):
        raise ValueError("state shape mismatch")
    g = _gamma_units(gamma, lead, U)
    o = np.empty(lead + (Dv,), dtype=np.float64)
    rc = lib.oracle_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), float(eps),
                                U, D, Dv, _ptr(S), _ptr(z), _ptr(o),
                                nthreads or default_threads())
    if rc:
        raise RuntimeError("oracle_decode_step rejected its arguments")
    return o, S, z


def gated(q, k, v, a, eps=1e-6, return_state=False, nthreads=None):
    """Gated causal linear attention in fp64: q, k, a [..., N, D];
    v [..., N, Dv]; a holds the gate a_i[d] of each step and key feature
    (fp32 values, widened).  Returns o [..., N, Dv], plus (S, z) after the
    last token if ``return_state``."""
    lib = _load()
    q = _f32(q, np.ndim(q)); k = _f32(k, q.ndim); v = _f32(v, q.ndim)
    a = _f32(a, q.ndim)
    N, D = q.shape[-2], q.shape[-1]
    Dv = v.shape[-1]
    if k.shape != q.shape or a.shape != q.shape or v.shape[:-1] != q.shape[:-1]:
        raise ValueError("shape mismatch")
    U, lead = _units(q)
    o = np.empty(q.shape[:-1] + (Dv,), dtype=np.float64)
    S = np.zeros(lead + (D, Dv), dtype=np.float64)
    z = np.zeros(lead + (D,), dtype=np.float64)
    rc = lib.oracle_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(a), float(eps), U, N,
                          D, Dv, _ptr(o), _ptr(S), _ptr(z),
                          nthreads or default_threads())
    if rc:
        raise RuntimeError("oracle_gated rejected its arguments")
    return (o, S, z) if return_state else o
