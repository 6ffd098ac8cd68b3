"""GPU parity of the backward pass against the fp64 gradient oracle
(oracle/backward.py), on seeded inputs and upstream gradients.

Errors are normwise per row (one token of one (batch, head) unit), measured
against the larger of the row's own size and the size of the terms summed
into it: max over rows i of ||x_i - r_i||_inf / max(||r_i||_inf, ||T_i||_inf),
where T is the same gradient summed over the absolute values of its terms.
The rounding error of an fp32 sum is bounded by the unit roundoff times the
sum of |terms|, and a gradient row can be a near-total cancellation of large
terms (dq of a single token: the output depends on q only through eps, so
gt . v - c is almost exactly 0), so the error bound of a row scales with its
T_i, not with its result.  fp32 inputs: 2e-4.  bf16 inputs on the fp32
CUDA-core kernels: 1e-2 (the inputs are widened exactly, the arithmetic is
fp32 and the gradients are rounded once to bf16).  bf16 inputs on the tensor
cores: 2e-2, the bound the bf16 forward kernels are held to, for the same
arithmetic (bf16 matrix-multiply operands, fp32 accumulation).  A term of a
gradient sum there carries the bf16 roundings of its two mapped operands,
the masked product P, the value operand and the output (up to six), plus
the relative error of the normaliser d_i that gt_i = dO_i / d_i inherits
from the forward product (up to four more): about 10 * 2^-9 = 2e-2 of the
row's term scale when every rounding falls the same way."""
import numpy as np
import pytest
import torch

from helpers import record, to_np

pytestmark = pytest.mark.gpu

BWD_TOL = {torch.float32: 2e-4, torch.bfloat16: 1e-2}
BWD_TOL_TC = 2e-2  # bf16 operands on tensor cores (see the module docstring)


@pytest.fixture(scope="module")
def la():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kernelized_sequence_mixing_gb300 import build
    build.build()
    import kernelized_sequence_mixing_gb300 as m
    return m


@pytest.fixture(scope="module")
def bw():
    from oracle import backward
    return backward


def row_err(x, r, scale):
    """max over rows i of ||x_i - r_i||_inf / max(||r_i||_inf, ||T_i||_inf);
    x, r, scale (T) [..., N, C]."""
    x = np.asarray(x, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    den = np.maximum(np.abs(r).max(axis=-1),
                     np.abs(np.asarray(scale, dtype=np.float64)).max(axis=-1))
    return float((np.abs(x - r).max(axis=-1) / np.maximum(den, 1e-30)).max())


def term_sizes(q, k, v, do, gamma, eps):
    """Per unit, the gradients' sums taken over absolute values of their
    terms (|dL/dw_ij| <= |gt_i| . |v_j| + |c_i|): the scale of their fp32
    rounding error.  q, k [N, D]; v, do [N, Dv]; fp64."""
    q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    fq = np.where(q > 0, q + 1, np.exp(np.minimum(q, 0)))
    fk = np.where(k > 0, k + 1, np.exp(np.minimum(k, 0)))
    N = q.shape[0]
    i, j = np.arange(N)[:, None], np.arange(N)[None, :]
    g = 1.0 if gamma is None else float(np.float32(gamma))
    G = np.where(j <= i, np.power(g, np.where(j <= i, i - j, 0).astype(np.float64)), 0.0)
    Wm = (fq @ fk.T) * G
    d = Wm.sum(1) + eps
    o = (Wm @ v) / d[:, None]
    gt = do / d[:, None]
    c = np.abs(np.sum(gt * o, axis=1))
    T = (np.abs(gt) @ np.abs(v).T + c[:, None]) * G
    return (T @ fk) * np.minimum(fq, 1), (T.T @ fq) * np.minimum(fk, 1), Wm.T @ np.abs(gt)


def inputs(B, H, N, D, Dv, dtype, seed):
    from kernelized_sequence_mixing_gb300.workloads import make_qkv
    q, k, v = make_qkv(B, H, N, D, Dv, dtype, seed, 0.5)
    g = torch.Generator().manual_seed(seed + 99)
    do = torch.randn((B, H, N, Dv), generator=g).to(dtype)
    return q, k, v, do


BWD_CASES = [
    # (B, H, N, D, Dv, gammas)
    (1, 1, 1, 64, 64, None),
    (1, 2, 63, 64, 128, None),
    (2, 2, 333, 128, 64, [0.9, 1.0]),
    (1, 3, 700, 128, 128, [0.5, 0.97, 0.999]),
    (1, 1, 1000, 64, 64, [0.0]),
    # bf16 on tensor cores: several sequence parts per head (few heads, long
    # sequences, ragged ends), the decay envelope's edge, D = 128
    (1, 2, 3001, 64, 64, [0.35, 0.999]),
    (1, 3, 2050, 128, 64, [1.0, 0.9, 0.5]),
    (2, 3, 65, 64, 64, [0.97, 1.0, 0.6]),
]


def expect_path(dtype, Dv, gammas):
    tc = dtype == torch.bfloat16 and Dv == 64 and (gammas is None or min(gammas) >= 0.35)
    return "tensor-core" if tc else "cuda-core"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: "x".join(map(str, c[:5])))
def test_backward(la, bw, dtype, case):
    B, H, N, D, Dv, gl = case
    q, k, v, do = inputs(B, H, N, D, Dv, dtype, N + D + Dv)
    g = None if gl is None else torch.tensor([gl[h % len(gl)] for h in range(H)],
                                             dtype=torch.float32)
    assert la.backward_kernel(B, H, N, D, Dv, gamma=g, dtype=dtype) == expect_path(dtype, Dv, gl)
    dq, dk, dv = la.backward(q.cuda(), k.cuda(), v.cuda(), do.cuda(), gamma=g)
    torch.cuda.synchronize()
    gu = None if g is None else np.tile(g.numpy(), B).reshape(B, H)
    rq, rk, rv = bw.causal_backward_units(to_np(q), to_np(k), to_np(v), to_np(do), gu, 1e-6)
    sizes = [np.zeros_like(r) for r in (rq, rk, rv)]
    for b in range(B):
        for h in range(H):
            ts = term_sizes(to_np(q[b, h]), to_np(k[b, h]), to_np(v[b, h]), to_np(do[b, h]),
                            None if gu is None else gu[b, h], 1e-6)
            for arr, t in zip(sizes, ts):
                arr[b, h] = t
    path = expect_path(dtype, Dv, gl)
    tol = BWD_TOL_TC if path == "tensor-core" else BWD_TOL[dtype]
    for name, got, ref, sz in (("dq", dq, rq, sizes[0]), ("dk", dk, rk, sizes[1]),
                               ("dv", dv, rv, sizes[2])):
        err = record(f"backward {name} {'fp32' if dtype == torch.float32 else 'bf16'} ({path})",
                     row_err(to_np(got), ref, sz), tol)
        assert err < tol, (name, err)


def test_backward_repeatable_and_empty(la):
    q, k, v, do = inputs(1, 2, 500, 64, 64, torch.bfloat16, 3)
    a1 = la.backward(q.cuda(), k.cuda(), v.cuda(), do.cuda())
    a2 = la.backward(q.cuda(), k.cuda(), v.cuda(), do.cuda())
    assert all(torch.equal(x, y) for x, y in zip(a1, a2))
    e = torch.empty((1, 2, 0, 64), dtype=torch.bfloat16, device="cuda")
    dq, dk, dv = la.backward(e, e, e, e)
    assert dq.numel() == 0


def test_backward_bf16_n4096_sampled_units(la, bw):
    """The backward workload at full size (B4 H8 N4096 D=Dv=64), in the
    launch configuration the benchmark times; whole units sampled."""
    from kernelized_sequence_mixing_gb300.workloads import WORKLOADS, workload_inputs, workload_upstream
    w = WORKLOADS["backward_bf16_n4096"]
    assert la.backward_kernel(w.B, w.H, w.N, w.D, w.Dv, dtype=w.dtype) == "tensor-core"
    q, k, v = workload_inputs(w)
    do = workload_upstream(w)
    dq, dk, dv = la.backward(q.cuda(), k.cuda(), v.cuda(), do.cuda(), eps=w.eps)
    torch.cuda.synchronize()
    for b, h in ((0, 0), (1, 2), (2, 7), (3, 5)):
        args = (to_np(q[b, h]), to_np(k[b, h]), to_np(v[b, h]), to_np(do[b, h]), None, w.eps)
        refs = bw.causal_backward(*args)
        for name, got, ref, sz in zip(("dq", "dk", "dv"), (dq, dk, dv), refs, term_sizes(*args)):
            err = record(f"backward_bf16_n4096 {name} (sampled units)",
                         row_err(to_np(got[b, h]), ref, sz), BWD_TOL_TC)
            assert err < BWD_TOL_TC, (b, h, name, err)
