"""The Python binding's argument checks, on CPU.  The C entry points take
plain pointers and cannot see a buffer's size or device, so the binding
checks every shape, dtype, device and layout before it loads the library.
These tests use meta tensors (no storage) and replace the library loader by
a sentinel: a call whose arguments pass every check reaches the sentinel, a
bad one raises ValueError or TypeError first, and nothing is ever launched."""
import pytest
import torch

import kernelized_sequence_mixing_gb300 as la

B, H, N, D, DV, R = 2, 3, 16, 64, 128, 128
BF, F32 = torch.bfloat16, torch.float32


class Reached(Exception):
    """The call passed the binding's checks and asked for the library."""


@pytest.fixture(autouse=True)
def no_library(monkeypatch):
    def stop():
        raise Reached

    monkeypatch.setattr(la, "load_library", stop)
    # meta tensors stand in for device tensors
    monkeypatch.setattr(la, "_DEVICE_TYPES", ("cuda", "meta"))


def T(*shape, dtype=BF, device="meta"):
    return torch.empty(shape, dtype=dtype, device=device)


def host(t):
    """An empty host tensor shaped like ``t``."""
    return torch.empty(t.shape, dtype=t.dtype)


def seq():
    return T(B, H, N, D), T(B, H, N, D), T(B, H, N, DV)


def step():
    return T(B, H, D), T(B, H, D), T(B, H, DV)


def state():
    return T(B, H, D, DV, dtype=F32), T(B, H, D, dtype=F32)


def passes(fn, *a, **kw):
    with pytest.raises(Reached):
        fn(*a, **kw)


def fails(exc, fn, *a, **kw):
    with pytest.raises(exc):
        fn(*a, **kw)


def test_good_calls_reach_the_library():
    q, k, v = seq()
    S, z = state()
    passes(la.forward, q, k, v)
    passes(la.forward, q, k, v, out=T(B, H, N, DV))
    hq, hk, hv = (host(t) for t in seq())
    passes(la.forward, hq, hk, hv, out=torch.empty(B, H, N, DV, dtype=BF))  # host buffers
    passes(la.prefill_state, k, v)
    passes(la.prefill_state, k, v, S=S, z=z)
    passes(la.forward_state, q, k, v, out=T(B, H, N, DV), S=S, z=z)
    passes(la.decode_step, *step(), S, z, out=T(B, H, DV))
    passes(la.forward_gated, q, k, v, T(B, H, N, D, dtype=F32), return_state=True)
    passes(la.forward_gated, q, k, v, T(B, H, N, D, dtype=F32), S=S, z=z)
    passes(la.decode_gated, *step(), T(B, H, D, dtype=F32), S, z, out=T(B, H, DV))
    passes(la.favor_features, T(5, 7, D), T(R, D), out=T(5, 7, R))
    passes(la.forward_favor, q, k, v, T(R, D), out=T(B, H, N, DV))
    passes(la.backward, q, k, v, T(B, H, N, DV), dq=T(B, H, N, D), dk=T(B, H, N, D),
           dv=T(B, H, N, DV))


def test_forward_checks():
    q, k, v = seq()
    fails(ValueError, la.forward, q, k, v, out=T(B, H, N, D))          # Dv = 128, not 64
    fails(TypeError, la.forward, q, k, v, out=T(B, H, N, DV, dtype=F32))
    fails(ValueError, la.forward, q, k, v, out=T(B, H, DV, N).transpose(2, 3))
    fails(ValueError, la.forward, q, k, v[0])                          # v not 4-D
    fails(ValueError, la.forward, q, k[:, :, :8], v)                   # k shorter than q
    fails(TypeError, la.forward, q, k, T(B, H, N, DV, dtype=F32))      # mixed dtypes
    fails(TypeError, la.forward, *(t.to(torch.float16) for t in (q, k, v)))
    # a host tensor beside device tensors, either way round
    fails(ValueError, la.forward, q, host(k), v)
    fails(ValueError, la.forward, q, k, v, out=torch.empty(B, H, N, DV, dtype=BF))


def test_state_checks():
    q, k, v = seq()
    S, z = state()
    fails(ValueError, la.prefill_state, k, v, S=T(B, H, DV, D, dtype=F32))  # transposed
    fails(TypeError, la.prefill_state, k, v, z=T(B, H, D, dtype=torch.float64))
    fails(ValueError, la.prefill_state, k[0], v[0])
    fails(TypeError, la.forward_state, q, k, v, S=T(B, H, D, DV, dtype=BF), z=z)
    fails(ValueError, la.forward_state, q, k, v, out=T(B, H, N + 1, DV), S=S, z=z)
    fails(ValueError, la.forward_state, q, k, v, S=S, z=torch.empty(B, H, D))  # host z


def test_decode_checks():
    S, z = state()
    q, k, v = step()
    fails(ValueError, la.decode_step, q, k, v, S[:, :1], z)
    fails(ValueError, la.decode_step, q, k, v, S, z[..., :-1])
    fails(TypeError, la.decode_step, q, k, v, S.to(BF), z)
    fails(ValueError, la.decode_step, q, k, T(B, H + 1, DV), S, z)
    fails(ValueError, la.decode_step, q, k, v, S, z, out=T(B, H, D))
    fails(ValueError, la.decode_step, *seq(), S, z)                    # sequence inputs
    # the decode step has no host path
    hq, hk, hv = (host(t) for t in (q, k, v))
    fails(ValueError, la.decode_step, hq, hk, hv, host(S), host(z))
    fails(ValueError, la.decode_gated, q, k, v, T(B, H, N, D, dtype=F32), S, z)
    fails(TypeError, la.decode_gated, q, k, v, T(B, H, D), S, z)          # bf16 gates
    fails(ValueError, la.decode_gated, q, k, v, T(B, H, D, dtype=F32), S, z, out=T(B, DV))


def test_gated_checks():
    q, k, v = seq()
    S, z = state()
    a = T(B, H, N, D, dtype=F32)
    fails(TypeError, la.forward_gated, q, k, v, a.to(BF))
    fails(ValueError, la.forward_gated, q, k, v, a[:, :, :-1])
    fails(ValueError, la.forward_gated, q, k, v, a, S=S[..., :-1], z=z)
    fails(ValueError, la.forward_gated, q, k, v, a, out=T(B, H, N, D))
    fails(ValueError, la.forward_gated, q, k, v, host(a))


def test_favor_checks():
    q, k, v = seq()
    W = T(R, D)
    fails(ValueError, la.favor_features, T(5, D), W, out=T(5, R + 1))
    fails(TypeError, la.favor_features, T(5, D), W.to(F32))
    fails(ValueError, la.favor_features, T(5, D + 1), W)
    fails(ValueError, la.forward_favor, q, k, v, T(R, D + 64))
    fails(TypeError, la.forward_favor, q, k, v, W.to(F32))
    fails(ValueError, la.forward_favor, q, k, v, W, out=T(B, H, N, R + 8))


def test_backward_checks():
    q, k, v = seq()
    do = T(B, H, N, DV)
    fails(ValueError, la.backward, q, k, v, T(B, H, N, D))              # do not shaped as v
    fails(TypeError, la.backward, q, k, v, do.to(F32))
    fails(ValueError, la.backward, q, k, v, do, dq=T(B, H, N, DV))
    fails(TypeError, la.backward, q, k, v, do, dv=T(B, H, N, DV, dtype=F32))
    fails(ValueError, la.backward, q, k, v, do, dk=torch.empty(B, H, N, D, dtype=BF))
