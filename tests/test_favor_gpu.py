"""GPU parity of the Performer path against the fp64 oracle (oracle/favor.py):
the random-feature map alone (element by element; the features are
positive, so element-wise relative error is well posed) and the attention
over it, causal and non-causal, on seeded inputs and directions."""
import numpy as np
import pytest
import torch

from helpers import TOL, max_row_error, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def la():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kernelized_sequence_mixing_gb300 import build
    build.build()
    import kernelized_sequence_mixing_gb300 as m
    return m


@pytest.fixture(scope="module")
def fv():
    from oracle import favor
    return favor


def qkv(B, H, N, D, Dv, dtype, seed):
    from kernelized_sequence_mixing_gb300.workloads import make_qkv
    return make_qkv(B, H, N, D, Dv, dtype, seed, D ** -0.25)


def directions(r, D, dtype, seed, orthogonal=True):
    from kernelized_sequence_mixing_gb300.workloads import favor_matrix
    return favor_matrix(r, D, seed, orthogonal, dtype)


# element-wise relative bounds on phi: fp32 arithmetic throughout, or exact
# bf16 products with fp32 sums and one bf16 rounding of phi
FEAT_TOL = {torch.float32: 1e-4, torch.bfloat16: 8e-3}


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("D,r", [(64, 64), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("rows", [1, 129, 1000])
def test_favor_features(la, fv, dtype, D, r, rows):
    x = qkv(1, 1, rows, D, 64, dtype, rows + D)[0].reshape(rows, D)
    W = directions(r, D, dtype, 3 * r + D)
    f = la.favor_features(x.cuda(), W.cuda())
    ref = fv.favor_features(to_np(x), to_np(W))
    rel = np.abs(to_np(f) - ref) / ref
    assert rel.max() < FEAT_TOL[dtype], rel.max()


def test_favor_features_iid_and_tiles_of_q_and_k(la, fv):
    """Many tiles (several per CTA of the persistent kernel), iid directions."""
    x = qkv(2, 4, 3001, 128, 64, torch.bfloat16, 1)[0]
    W = directions(128, 128, torch.bfloat16, 2, orthogonal=False)
    f = la.favor_features(x.cuda(), W.cuda())
    ref = fv.favor_features(to_np(x), to_np(W))
    assert (np.abs(to_np(f) - ref) / ref).max() < FEAT_TOL[torch.bfloat16]


FAVOR_CASES = [
    # (B, H, N, D, Dv, r, causal, gammas)
    (1, 2, 333, 64, 64, 64, True, None),
    (2, 3, 700, 128, 128, 128, True, [0.9, 0.99, 1.0]),
    (1, 2, 1000, 128, 64, 64, True, None),
    (1, 1, 1, 64, 128, 128, True, None),
    (2, 2, 500, 64, 64, 128, False, None),
    (1, 3, 2000, 128, 128, 128, False, None),
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("case", FAVOR_CASES, ids=lambda c: "x".join(map(str, c[:6])) + ("c" if c[6] else "n"))
def test_forward_favor(la, fv, dtype, case):
    B, H, N, D, Dv, r, causal, gl = case
    q, k, v = qkv(B, H, N, D, Dv, dtype, 7 * N + r)
    W = directions(r, D, dtype, N)
    g = None if gl is None else torch.tensor([gl[h % len(gl)] for h in range(H)],
                                             dtype=torch.float32)
    o = la.forward_favor(q.cuda(), k.cuda(), v.cuda(), W.cuda(), causal=causal, gamma=g)
    gn = None if g is None else g.numpy()[None, :]
    ref = fv.favor(to_np(q), to_np(k), to_np(v), to_np(W), causal=causal, gamma=gn)
    err = max_row_error(to_np(o), ref)
    assert err < TOL[dtype], err


def test_favor_bf16_n16384_sampled_heads(la, fv):
    """The Performer workload at full size, in the launch configuration the
    benchmark times; whole (b, h) units sampled."""
    from kernelized_sequence_mixing_gb300.workloads import (
        WORKLOADS, workload_favor_matrix, workload_inputs)
    w = WORKLOADS["favor_bf16_n16384"]
    q, k, v = workload_inputs(w)
    W = workload_favor_matrix(w)
    o = la.forward_favor(q.cuda(), k.cuda(), v.cuda(), W.cuda(), causal=True, eps=w.eps)
    torch.cuda.synchronize()
    for b, h in ((0, 0), (1, 7)):
        ref = fv.favor(to_np(q[b, h]), to_np(k[b, h]), to_np(v[b, h]), to_np(W), causal=True,
                       eps=w.eps)
        err = max_row_error(to_np(o[b, h]), ref)
        assert err < 2e-2, (b, h, err)
