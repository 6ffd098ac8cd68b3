"""la_forward_noncausal_static: the non-causal forward that allocates nothing.

Some callers cannot let a library allocate device memory (an application
that reserves HBM up front in its own allocator, a latency-critical loop that
must not stall or fail on a full memory pool).  This entry point keeps its
scratch in a fixed array inside the library.  The GPU test calls it through
the C ABI, on two calls in a row with different inputs (so that leftovers in
the shared scratch from the first call would show up in the second), and
checks each result against the fp64 oracle (every head of the small cases,
sampled whole heads of the full-size workload) and against the regular
(allocating) non-causal forward.  This file is named to be collected last.
"""
import ctypes

import pytest
import torch

from helpers import TOL, max_row_error, record, to_np

OK, INVALID, UNSUPPORTED = 0, 1, 2
F32, BF16 = 0, 1


@pytest.fixture(scope="module")
def lib():
    from kernelized_sequence_mixing_gb300 import build
    build.build()
    import kernelized_sequence_mixing_gb300 as la
    L = la.load_library()
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.la_forward_noncausal_static.argtypes = [P, P, P, P, I, I, I, I, I, F, I, P]
    L.la_forward_noncausal_static.restype = I
    L.la_forward_noncausal_static_limit.argtypes = []
    L.la_forward_noncausal_static_limit.restype = ctypes.c_size_t
    return L


def test_static_entry_point_rejects_before_touching_the_device(lib):
    """Host-only: sizes beyond the scratch, and bad arguments, are refused
    before any CUDA call."""
    A, S = 0x10000, 0x10000000
    call = lambda B, H, N, D=128, Dv=128, eps=1e-6, q=A: lib.la_forward_noncausal_static(  # noqa: E731
        q, A + S, A + 2 * S, A + 3 * S, B, H, N, D, Dv, eps, BF16, None)
    limit = lib.la_forward_noncausal_static_limit()
    assert limit == 32 << 20
    per_head = (128 * 128 + 128) * 4
    too_many = limit // per_head + 1                 # heads whose states alone overflow
    assert call(too_many // 256 + 1, 256, 16) == UNSUPPORTED
    assert call(1, 2, 16, D=96) == UNSUPPORTED
    assert call(1, 2, 16, eps=-1.0) == INVALID
    assert call(1, 2, 16, q=None) == INVALID
    assert call(1, 2, 0, q=None) == OK               # empty: nothing to do


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,shape", [
    (torch.bfloat16, (2, 4, 9000, 64, 128)),   # split reduction (partials in scratch)
    (torch.float32, (1, 3, 777, 128, 64)),     # one split
    (torch.bfloat16, (8, 16, 65536, 64, 64)),  # the full non-causal workload
])
def test_static_entry_point_matches_oracle(lib, oracle_mod, dtype, shape):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kernelized_sequence_mixing_gb300 as la
    from kernelized_sequence_mixing_gb300.workloads import make_qkv
    B, H, N, D, Dv = shape
    dt = F32 if dtype == torch.float32 else BF16
    stream = torch.cuda.current_stream()
    # the oracle on whole heads: all of them for the small cases, eight spread
    # over batch entries and head indices for the full-size workload
    units = ([(b, h) for b in range(B) for h in range(H)] if B * H <= 16 else
             [(b, (3 * b + 1) % H) for b in range(B)])
    bs = [u[0] for u in units]
    hs = [u[1] for u in units]
    for seed in (11, 12):  # two calls in a row sharing the scratch
        qc, kc, vc = make_qkv(B, H, N, D, Dv, dtype, seed, 0.5)
        q, k, v = qc.cuda(), kc.cuda(), vc.cuda()
        o = torch.empty((B, H, N, Dv), dtype=dtype, device="cuda")
        rc = lib.la_forward_noncausal_static(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, H, N, D,
            Dv, 1e-6, dt, ctypes.c_void_p(stream.cuda_stream))
        assert rc == OK, rc
        alloc = la.forward(q, k, v, causal=False, eps=1e-6)
        torch.cuda.synchronize()
        got = to_np(o)
        ref = oracle_mod.noncausal(to_np(qc[bs, hs]), to_np(kc[bs, hs]), to_np(vc[bs, hs]),
                                   eps=1e-6)
        err = record(f"allocation-free non-causal {'fp32' if dt == F32 else 'bf16'} vs oracle",
                     max(max_row_error(got[b, h], ref[i]) for i, (b, h) in enumerate(units)),
                     TOL[dtype])
        assert err < TOL[dtype], (seed, err)
        err2 = max_row_error(got, to_np(alloc))
        assert err2 < TOL[dtype], (seed, err2)
