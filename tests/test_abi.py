"""The C ABI without a GPU: the library loads, exports every symbol that
include/*.h declares, and rejects bad arguments before any CUDA call (so
these tests never touch a device)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OK, INVALID, UNSUPPORTED, CUDA_ERR = 0, 1, 2, 3
F32, BF16 = 0, 1
A = 0x10000          # a 16-byte aligned fake device address (never touched)
STEP = 0x10000000    # distance between fake buffers (no overlap)


@pytest.fixture(scope="module")
def lib():
    from kernelized_sequence_mixing_gb300 import build
    build.build()
    import kernelized_sequence_mixing_gb300 as la
    return la.load_library()


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        names.update(re.findall(r"LA_API\s+[\w\s\*]*?\b(la_\w+)\s*\(", src))
    return sorted(names)


def test_header_declares_entry_points():
    syms = declared_symbols()
    for s in ("la_forward", "la_forward_host", "la_forward_state", "la_prefill_state", "la_decode_step",
              "la_forward_gated", "la_decode_gated", "la_favor_features", "la_forward_favor",
              "la_backward", "la_backward_launches", "la_backward_kernel", "la_gated_kernel", "la_wait_selftest",
              "la_status_string", "la_causal_kernel",
              "la_device_wait_timeouts"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, text in ((OK, "ok"), (INVALID, "invalid argument"),
                       (UNSUPPORTED, "unsupported"), (CUDA_ERR, "CUDA")):
        assert text in lib.la_status_string(code).decode()


def fwd(lib, q=A, k=A + STEP, v=A + 2 * STEP, o=A + 3 * STEP, B=1, H=2, N=8,
        D=64, Dv=64, causal=1, gamma=None, eps=1e-6, dt=BF16):
    g = None if gamma is None else (ctypes.c_float * len(gamma))(*gamma)
    return lib.la_forward(q, k, v, o, B, H, N, D, Dv, causal, g, eps, dt, None)


def test_forward_rejects_bad_arguments(lib):
    assert fwd(lib, q=None) == INVALID
    assert fwd(lib, o=0) == INVALID
    assert fwd(lib, q=A + 8) == INVALID          # misaligned
    assert fwd(lib, v=A + 2 * STEP + 4) == INVALID
    assert fwd(lib, B=-1) == INVALID
    assert fwd(lib, D=0) == INVALID
    assert fwd(lib, eps=-1e-6) == INVALID
    assert fwd(lib, eps=float("nan")) == INVALID
    assert fwd(lib, eps=float("inf")) == INVALID
    assert fwd(lib, gamma=[0.5, 1.5]) == INVALID
    assert fwd(lib, gamma=[0.5, float("nan")]) == INVALID
    assert fwd(lib, gamma=[-0.1, 1.0]) == INVALID
    assert fwd(lib, causal=0, gamma=[0.5, 1.0]) == INVALID
    assert fwd(lib, dt=7) == INVALID
    # aliasing: o overlaps q (same start, or partial overlap)
    assert fwd(lib, o=A) == INVALID
    assert fwd(lib, o=A + 1024) == INVALID


def test_forward_unsupported_shapes(lib):
    assert fwd(lib, D=96) == UNSUPPORTED
    assert fwd(lib, Dv=256) == UNSUPPORTED
    assert fwd(lib, D=32, dt=F32) == UNSUPPORTED
    g = [1.0] * 257
    assert fwd(lib, H=257, gamma=g) == UNSUPPORTED
    assert fwd(lib, B=1 << 16, H=256, N=1 << 16, gamma=[1.0] * 256) == UNSUPPORTED


def test_forward_empty_calls_are_noops(lib):
    assert fwd(lib, N=0, q=None, k=None, v=None, o=None) == OK
    assert fwd(lib, B=0, q=None, k=None, v=None, o=None) == OK
    assert fwd(lib, H=0, q=None, k=None, v=None, o=None) == OK
    # gamma of 1 is accepted non-causally
    assert fwd(lib, N=0, causal=0, gamma=[1.0, 1.0]) == OK


def test_prefill_rejects_bad_arguments(lib):
    P = lib.la_prefill_state
    assert P(A, A + STEP, None, A + 3 * STEP, 1, 2, 8, 64, 64, None, BF16, None) == INVALID
    assert P(A, A + STEP, A + 2 * STEP, A + 2 * STEP, 1, 2, 8, 64, 64, None, BF16, None) == INVALID
    assert P(A, A + STEP, A, A + 3 * STEP, 1, 2, 8, 64, 64, None, BF16, None) == INVALID
    assert P(A, A + STEP, A + 2 * STEP + 4, A + 3 * STEP, 1, 2, 8, 64, 64, None, BF16, None) == INVALID
    bad = (ctypes.c_float * 2)(2.0, 1.0)
    assert P(A, A + STEP, A + 2 * STEP, A + 3 * STEP, 1, 2, 8, 64, 64, bad, BF16, None) == INVALID
    assert P(A, A + STEP, A + 2 * STEP, A + 3 * STEP, 1, 2, 8, 48, 64, None, BF16, None) == UNSUPPORTED
    assert P(None, None, None, None, 0, 2, 8, 64, 64, None, BF16, None) == OK


def test_forward_state_rejects_bad_arguments(lib):
    Fs = lib.la_forward_state
    q, k, v, o, S, z = (A + i * STEP for i in range(6))

    def call(qq=q, kk=k, vv=v, oo=o, SS=S, zz=z, B=1, H=2, N=8, D=128, Dv=128, eps=1e-6,
             g=None, dt=BF16):
        return Fs(qq, kk, vv, oo, SS, zz, B, H, N, D, Dv, g, eps, dt, None)

    assert call(SS=None) == INVALID
    assert call(zz=None) == INVALID
    assert call(SS=S + 8) == INVALID            # misaligned state
    assert call(zz=S + 64) == INVALID           # z inside S
    assert call(SS=q) == INVALID                # S aliases q
    assert call(zz=o + 16) == INVALID           # z inside o
    assert call(oo=v) == INVALID                # o aliases v
    assert call(qq=None) == INVALID
    assert call(eps=-1.0) == INVALID
    assert call(g=(ctypes.c_float * 2)(0.5, 1.5)) == INVALID
    assert call(D=96) == UNSUPPORTED
    assert call(B=0, qq=None, kk=None, vv=None, oo=None, SS=None, zz=None) == OK


def test_decode_rejects_bad_arguments(lib):
    Dc = lib.la_decode_step
    ptrs = [A + i * STEP for i in range(6)]

    def call(p=ptrs, B=2, H=2, D=128, Dv=128, eps=1e-6, g=None, dt=BF16):
        return Dc(*p, B, H, D, Dv, g, eps, dt, None)

    assert call(p=[None] + ptrs[1:]) == INVALID
    assert call(eps=-1.0) == INVALID
    assert call(p=ptrs[:5] + [ptrs[3]]) == INVALID      # o aliases S
    assert call(p=ptrs[:4] + [ptrs[3] + 64, ptrs[5]]) == INVALID  # z inside S
    assert call(p=ptrs[:3] + [ptrs[0]] + ptrs[4:]) == INVALID     # S aliases q
    assert call(p=ptrs[:5] + [ptrs[5] + 2]) == INVALID  # misaligned o
    assert call(D=100) == UNSUPPORTED
    assert call(g=(ctypes.c_float * 2)(1.0, -0.5)) == INVALID
    assert call(B=0, p=[None] * 6) == OK


def test_forward_gated_rejects_bad_arguments(lib):
    Fg = lib.la_forward_gated
    Fg.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_int,
                                                                ctypes.c_void_p]
    q, k, v, a, o, S, z = (A + i * STEP for i in range(7))

    def call(qq=q, kk=k, vv=v, aa=a, oo=o, SS=S, zz=z, B=1, H=2, N=8, D=128, Dv=128,
             eps=1e-6, dt=BF16):
        return Fg(qq, kk, vv, aa, oo, SS, zz, B, H, N, D, Dv, eps, dt, None)

    assert call(SS=None) == INVALID             # S without z
    assert call(zz=None) == INVALID             # z without S
    assert call(aa=None) == INVALID             # no gates
    assert call(aa=a + 4) == INVALID            # misaligned gates
    assert call(oo=a + 64) == INVALID           # o inside the gates
    assert call(SS=a) == INVALID                # S aliases the gates
    assert call(zz=o + 16) == INVALID           # z inside o
    assert call(oo=q) == INVALID                # o aliases q
    assert call(eps=float("nan")) == INVALID
    assert call(D=96) == UNSUPPORTED
    assert call(dt=7) == INVALID
    assert call(B=0, qq=None, kk=None, vv=None, aa=None, oo=None, SS=None, zz=None) == OK


def test_decode_gated_rejects_bad_arguments(lib):
    Dg = lib.la_decode_gated
    Dg.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_int] * 4 + [ctypes.c_float, ctypes.c_int,
                                                                ctypes.c_void_p]
    ptrs = [A + i * STEP for i in range(7)]     # q, k, v, a, S, z, o

    def call(p=ptrs, B=2, H=2, D=128, Dv=128, eps=1e-6, dt=BF16):
        return Dg(*p, B, H, D, Dv, eps, dt, None)

    assert call(p=ptrs[:3] + [None] + ptrs[4:]) == INVALID       # no gates
    assert call(p=ptrs[:4] + [ptrs[3]] + ptrs[5:]) == INVALID    # S aliases a
    assert call(p=ptrs[:6] + [ptrs[4] + 32]) == INVALID          # o inside S
    assert call(p=ptrs[:3] + [ptrs[3] + 8] + ptrs[4:]) == INVALID  # misaligned a
    assert call(eps=-1.0) == INVALID
    assert call(Dv=32) == UNSUPPORTED
    assert call(B=0, p=[None] * 7) == OK


def test_favor_rejects_bad_arguments(lib):
    Ff = lib.la_favor_features
    Ff.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 + [ctypes.c_void_p]
    x, W, f = A, A + STEP, A + 2 * STEP
    assert Ff(x, W, None, 100, 128, 128, BF16, None) == INVALID
    assert Ff(x, W, x + 256, 100, 128, 128, BF16, None) == INVALID   # phi overlaps x
    assert Ff(x, W + 8, f, 100, 128, 128, BF16, None) == INVALID     # misaligned W
    assert Ff(x, W, f, 100, 96, 128, BF16, None) == UNSUPPORTED
    assert Ff(x, W, f, 100, 128, 32, BF16, None) == UNSUPPORTED
    assert Ff(x, W, f, -1, 128, 128, BF16, None) == INVALID
    assert Ff(None, None, None, 0, 128, 128, BF16, None) == OK
    Fw = lib.la_forward_favor
    Fw.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 7 + [ctypes.c_void_p, ctypes.c_float,
                                                                ctypes.c_int, ctypes.c_void_p]
    q, k, v, Wd, o = (A + i * STEP for i in range(5))

    def call(qq=q, kk=k, vv=v, WW=Wd, oo=o, B=1, H=2, N=8, D=128, Dv=128, r=128, causal=1,
             g=None, eps=1e-6, dt=BF16):
        return Fw(qq, kk, vv, WW, oo, B, H, N, D, Dv, r, causal, g, eps, dt, None)

    assert call(WW=None) == INVALID
    assert call(oo=Wd) == INVALID               # o aliases W
    assert call(r=100) == UNSUPPORTED
    assert call(r=0) == INVALID
    assert call(causal=0, g=(ctypes.c_float * 2)(0.5, 1.0)) == INVALID
    assert call(eps=-1.0) == INVALID
    assert call(B=0, qq=None, kk=None, vv=None, WW=None, oo=None) == OK


def test_wait_selftest_rejects_bad_arguments(lib):
    St = lib.la_wait_selftest
    St.argtypes = [ctypes.c_longlong, ctypes.POINTER(ctypes.c_int)]
    g = ctypes.c_int(0)
    assert St(0, ctypes.byref(g)) == INVALID
    assert St(5_000_000_000, ctypes.byref(g)) == INVALID
    assert St(1000, None) == INVALID


def test_gated_kernel_dispatch(lib):
    Gk = lib.la_gated_kernel
    assert Gk(2, 4, 1000, 128, 128, BF16, 0) == 1      # tensor cores
    assert Gk(2, 4, 1000, 128, 128, BF16, 1) == 1      # with the final state too
    assert Gk(1, 4, 1000, 128, 128, BF16, 0) == 0      # B*H < 8
    assert Gk(2, 4, 1000, 64, 128, BF16, 0) == 0       # D = 64
    assert Gk(2, 4, 1000, 128, 128, F32, 0) == 0       # fp32
    assert Gk(2, 4, 1000, 96, 128, BF16, 0) == -UNSUPPORTED


def test_backward_rejects_bad_arguments(lib):
    Fb = lib.la_backward
    Fb.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_int] * 5 + [ctypes.c_void_p, ctypes.c_float,
                                                                ctypes.c_int, ctypes.c_void_p]
    q, k, v, do, dq, dk, dv = (A + i * STEP for i in range(7))

    def call(p=(q, k, v, do, dq, dk, dv), B=1, H=2, N=8, D=64, Dv=64, g=None, eps=1e-6, dt=F32):
        return Fb(*p, B, H, N, D, Dv, g, eps, dt, None)

    assert call(p=(q, k, v, None, dq, dk, dv)) == INVALID      # no upstream gradient
    assert call(p=(q, k, v, do, q, dk, dv)) == INVALID         # dq aliases q
    assert call(p=(q, k, v, do, dq, dq + 64, dv)) == INVALID   # dk inside dq
    assert call(p=(q, k, v, do + 4, dq, dk, dv)) == INVALID    # misaligned
    assert call(eps=-1.0) == INVALID
    assert call(g=(ctypes.c_float * 2)(0.5, 2.0)) == INVALID
    assert call(D=32) == UNSUPPORTED
    assert call(B=0, p=(None,) * 7) == OK


def test_backward_launches_rejects_bad_sizes(lib):
    """Host-only paths of the launch count: invalid and unsupported sizes
    give the negated status, an empty call launches nothing.  (Valid sizes
    read the device's SM count, so they are left to the GPU tests.)"""
    L = lib.la_backward_launches
    L.argtypes = [ctypes.c_int] * 5 + [ctypes.c_void_p, ctypes.c_int]
    assert L(-1, 2, 8, 64, 64, None, F32) == -INVALID
    assert L(1, 2, 8, 0, 64, None, F32) == -INVALID
    assert L(1, 2, 8, 96, 64, None, F32) == -UNSUPPORTED
    assert L(1, 300, 8, 64, 64, None, F32) == -UNSUPPORTED               # more heads than supported
    assert L(1 << 16, 1 << 8, 1 << 8, 64, 64, None, F32) == -UNSUPPORTED  # 2^32 tokens
    assert L(1, 2, 8, 64, 64, None, 7) == -INVALID                      # unknown dtype
    assert L(1, 2, 8, 64, 64, (ctypes.c_float * 2)(0.5, 1.5), BF16) == -INVALID
    assert L(0, 2, 8, 64, 64, None, F32) == 0
    assert L(1, 2, 0, 128, 128, None, BF16) == 0


def test_backward_kernel_dispatch(lib):
    """Host-only: the tensor-core backward takes bf16 with Dv = 64 and every
    decay inside the 64-token chunk kernel's envelope."""
    K = lib.la_backward_kernel
    K.argtypes = [ctypes.c_int] * 5 + [ctypes.c_void_p, ctypes.c_int]
    g = lambda *x: (ctypes.c_float * len(x))(*x)  # noqa: E731
    assert K(4, 8, 4096, 64, 64, None, BF16) == 1
    assert K(1, 2, 333, 128, 64, g(0.9, 1.0), BF16) == 1
    assert K(1, 2, 333, 128, 64, g(0.35, 1.0), BF16) == 1
    assert K(1, 2, 333, 128, 64, g(0.34, 1.0), BF16) == 0   # decay too strong
    assert K(1, 2, 333, 64, 128, None, BF16) == 0           # Dv = 128
    assert K(4, 8, 4096, 64, 64, None, F32) == 0            # fp32 inputs
    assert K(1, 2, 8, 96, 64, None, BF16) == -UNSUPPORTED


def test_causal_kernel_dispatch(lib):
    K = lib.la_causal_kernel
    g = lambda *x: (ctypes.c_float * len(x))(*x)  # noqa: E731
    assert K(2, 16, 16384, 128, 128, None, BF16) == 2           # 128-token chunks
    assert K(2, 16, 16384, 128, 128, g(*[0.96875] * 16), BF16) == 2
    assert K(1, 2, 100, 128, 128, g(0.6, 1.0), BF16) == 1       # too strong for 128
    assert K(4, 8, 4096, 64, 64, None, BF16) == 1
    assert K(1, 2, 100, 64, 128, g(0.35, 1.0), BF16) == 1
    assert K(1, 2, 100, 64, 128, g(0.34, 1.0), BF16) == 0   # strong decay
    assert K(1, 2, 100, 64, 128, g(0.0, 1.0), BF16) == 0
    assert K(1, 1, 256, 64, 64, None, F32) == 0             # fp32 inputs
    assert K(1, 1, 256, 96, 64, None, BF16) == -UNSUPPORTED
    assert K(1, 2, 256, 64, 64, g(1.5, 1.0), BF16) == -INVALID
    assert K(256, 256, 1, 64, 64, None, BF16) == 1          # one-dimensional grid


def test_forward_host_rejects_bad_arguments(lib):
    """Host-only: la_forward_host validates like la_forward before any CUDA
    call (host pointers need no alignment)."""
    F = lib.la_forward_host
    F.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 6 + [ctypes.c_void_p, ctypes.c_float,
                                                               ctypes.c_int, ctypes.c_void_p]
    q, k, v, o = (A + i * STEP for i in range(4))

    def call(p=(q, k, v, o), B=1, H=2, N=8, D=64, Dv=64, causal=1, g=None, eps=1e-6, dt=BF16):
        return F(*p, B, H, N, D, Dv, causal, g, eps, dt, None)

    assert call(p=(q, k, v, None)) == INVALID
    assert call(p=(q, k, v, q)) == INVALID                   # o aliases q
    assert call(eps=float("nan")) == INVALID
    assert call(causal=0, g=(ctypes.c_float * 2)(0.5, 1.0)) == INVALID
    assert call(D=96) == UNSUPPORTED
    assert call(B=0, p=(None,) * 4) == OK                    # empty: nothing to do
