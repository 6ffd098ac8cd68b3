"""GPU parity of the gated forms (gated linear attention: one gate per key
feature and token) against the fp64 oracle, on the same seeded inputs.

Small cases run in full: several 64-token chunks, a ragged tail, one and many
sequence parts, and gates that cover both chunk paths (mild gates keep every
chunk on the factorised path; gates drawn from [0, 1] with exact zeros push
chunks onto the token recurrence).  The full-size gated workload is compared
on sampled heads.  Errors are per-row normwise (helpers.TOL).
"""
import numpy as np
import pytest
import torch

from helpers import TOL, max_row_error, state_error, to_np

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
def ora(oracle_mod):
    return oracle_mod


def inputs(B, H, N, D, Dv, dtype, seed, gates):
    from kernelized_sequence_mixing_gb300.workloads import make_gates, make_qkv
    q, k, v = make_qkv(B, H, N, D, Dv, dtype, seed, 0.5)
    if gates == "mild":
        a = make_gates(B, H, N, D, seed + 1, 0.9, 1.0)
    elif gates == "strong":     # per-chunk products down to ~2^-53, no fallback
        a = make_gates(B, H, N, D, seed + 1, 0.5, 1.0)
    elif gates == "wide":       # strong forgetting: exact zeros and ones
        a = make_gates(B, H, N, D, seed + 1, 0.0, 1.0, zero_frac=0.01, one_frac=0.05)
    elif gates == "ones":
        a = torch.ones((B, H, N, D), dtype=torch.float32)
    else:
        raise ValueError(gates)
    return q, k, v, a


GATED_SMALL = [
    # (B, H, N, D, Dv)
    (1, 1, 1, 64, 64),
    (1, 2, 63, 128, 128),
    (2, 3, 333, 64, 128),
    (1, 2, 1000, 128, 64),
    (1, 1, 4099, 128, 128),
    (4, 40, 130, 64, 64),      # many (b, h): three parts of one chunk each
    (4, 40, 50, 64, 64),       # one chunk: one part, no state pass
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("gates", ["mild", "wide", "ones"])
@pytest.mark.parametrize("shape", GATED_SMALL, ids=lambda s: "x".join(map(str, s)))
def test_gated_small(la, ora, dtype, gates, shape):
    B, H, N, D, Dv = shape
    q, k, v, a = inputs(B, H, N, D, Dv, dtype, 11 * N + D, gates)
    o, S, z = la.forward_gated(q.cuda(), k.cuda(), v.cuda(), a.cuda(), eps=1e-6,
                               return_state=True)
    torch.cuda.synchronize()
    ref, S_ref, z_ref = ora.gated(to_np(q), to_np(k), to_np(v), a.numpy(), eps=1e-6,
                                  return_state=True)
    tol = TOL[dtype]
    err = max_row_error(to_np(o), ref)
    assert err < tol, err
    # the state is accumulated in fp32 from the inputs as given: fp32 bound
    assert state_error(to_np(S), S_ref) < 1e-4
    assert state_error(to_np(z)[..., None], z_ref[..., None]) < 1e-4
    # without the state the output is the same
    o2 = la.forward_gated(q.cuda(), k.cuda(), v.cuda(), a.cuda(), eps=1e-6)
    assert torch.equal(o, o2)


# The tensor-core form: bf16, D = Dv = 128, B*H >= 8, no final state.  Wide
# gates (exact zeros) make it fall back to the CUDA-core form at run time.
GATED_TC = [
    (2, 4, 1000, 128, 128),
    (1, 8, 333, 128, 128),
    (4, 4, 128, 128, 128),
    (1, 8, 1, 128, 128),
    (2, 8, 4099, 128, 128),
]


@pytest.mark.parametrize("gates", ["mild", "strong", "ones", "wide"])
@pytest.mark.parametrize("shape", GATED_TC, ids=lambda s: "x".join(map(str, s)))
def test_gated_tensor_core(la, ora, gates, shape):
    B, H, N, D, Dv = shape
    assert la.gated_kernel(B, H, N, D, Dv) == "tensor-core"
    assert la.gated_kernel(B, H, N, D, Dv, want_state=True) == "tensor-core"
    q, k, v, a = inputs(B, H, N, D, Dv, torch.bfloat16, 13 * N + H, gates)
    o = la.forward_gated(q.cuda(), k.cuda(), v.cuda(), a.cuda(), eps=1e-6)
    torch.cuda.synchronize()
    ref, S_ref, z_ref = ora.gated(to_np(q), to_np(k), to_np(v), a.numpy(), eps=1e-6,
                                  return_state=True)
    err = max_row_error(to_np(o), ref)
    assert err < 2e-2, err
    # the same call with the final state: the same output, and the state
    # (summed from bf16 operands like the output on the tensor-core form,
    # so held to the bf16 bound)
    o2, S, z = la.forward_gated(q.cuda(), k.cuda(), v.cuda(), a.cuda(), eps=1e-6,
                                return_state=True)
    assert torch.equal(o, o2)
    eS = state_error(to_np(S), S_ref)
    ez = state_error(to_np(z)[..., None], z_ref[..., None])
    assert eS < 2e-2 and ez < 2e-2, (eS, ez)


def test_gated_ones_equals_ungated_forward(la, ora):
    """a = 1 everywhere is plain causal linear attention; the fp32 CUDA-core
    forward and the gated forward agree to fp32 rounding."""
    B, H, N, D, Dv = 1, 2, 700, 128, 128
    q, k, v, a = inputs(B, H, N, D, Dv, torch.float32, 3, "ones")
    og = la.forward_gated(q.cuda(), k.cuda(), v.cuda(), a.cuda())
    oc = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=True)
    assert max_row_error(to_np(og), to_np(oc)) < 1e-5


def test_gated_constant_gate_equals_decayed_forward(la, ora):
    """a_t[d] = gamma_h for every t and d is the fixed per-head decay."""
    B, H, N, D, Dv = 2, 3, 500, 64, 64
    from kernelized_sequence_mixing_gb300.workloads import make_qkv
    q, k, v = make_qkv(B, H, N, D, Dv, torch.float32, 8, 0.5)
    g = torch.tensor([0.5, 0.9, 0.999], dtype=torch.float32)
    a = g.view(1, H, 1, 1).expand(B, H, N, D).contiguous()
    og = la.forward_gated(q.cuda(), k.cuda(), v.cuda(), a.cuda())
    oc = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=True, gamma=g)
    ref = ora.causal(to_np(q), to_np(k), to_np(v), gamma=g.numpy())
    assert max_row_error(to_np(og), ref) < 1e-4
    assert max_row_error(to_np(og), to_np(oc)) < 2e-4


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("gates", ["mild", "wide"])
def test_gated_forward_then_decode(la, ora, dtype, gates):
    """forward_gated over N tokens, then M gated decode steps from its state,
    reproduce the oracle's rows N..N+M-1 and its final state."""
    B, H, N, M, D, Dv = 2, 4, 300, 9, 128, 64
    q, k, v, a = inputs(B, H, N + M, D, Dv, dtype, 21, gates)
    qd, kd, vd, ad = q.cuda(), k.cuda(), v.cuda(), a.cuda()
    _, S, z = la.forward_gated(qd[:, :, :N].contiguous(), kd[:, :, :N].contiguous(),
                               vd[:, :, :N].contiguous(), ad[:, :, :N].contiguous(),
                               return_state=True)
    ref, S_ref, z_ref = ora.gated(to_np(q), to_np(k), to_np(v), a.numpy(),
                                  return_state=True)
    for t in range(M):
        o = la.decode_gated(qd[:, :, N + t].contiguous(), kd[:, :, N + t].contiguous(),
                            vd[:, :, N + t].contiguous(), ad[:, :, N + t].contiguous(), S, z)
        err = max_row_error(to_np(o), ref[:, :, N + t])
        assert err < TOL[dtype], (t, err)
    assert state_error(to_np(S), S_ref) < 1e-4
    assert state_error(to_np(z)[..., None], z_ref[..., None]) < 1e-4


def test_gated_empty_and_single_token(la, ora):
    q, k, v, a = inputs(1, 2, 1, 64, 64, torch.bfloat16, 1, "wide")
    o, S, z = la.forward_gated(q.cuda(), k.cuda(), v.cuda(), a.cuda(), return_state=True)
    ref = ora.gated(to_np(q), to_np(k), to_np(v), a.numpy())
    assert max_row_error(to_np(o), ref) < 2e-2
    e = torch.empty((1, 2, 0, 64), dtype=torch.bfloat16, device="cuda")
    ea = torch.empty((1, 2, 0, 64), dtype=torch.float32, device="cuda")
    o0, S0, z0 = la.forward_gated(e, e, e, ea, return_state=True)
    torch.cuda.synchronize()
    assert o0.numel() == 0 and not S0.any() and not z0.any()


def test_gated_repeatable(la):
    q, k, v, a = inputs(1, 4, 2000, 128, 128, torch.bfloat16, 5, "wide")
    args = [t.cuda() for t in (q, k, v, a)]
    o1 = la.forward_gated(*args)
    o2 = la.forward_gated(*args)
    assert torch.equal(o1, o2)


def test_gated_bf16_n16384_sampled_heads(la, ora):
    """The gated workload at full size, in the launch configuration the
    benchmark times; whole (b, h) units sampled from both batch entries."""
    from kernelized_sequence_mixing_gb300.workloads import (
        WORKLOADS, workload_gates, workload_inputs)
    w = WORKLOADS["gla_bf16_n16384"]
    q, k, v = workload_inputs(w)
    a = workload_gates(w)
    o = la.forward_gated(q.cuda(), k.cuda(), v.cuda(), a.cuda(), eps=w.eps)
    torch.cuda.synchronize()
    for b, h in ((0, 0), (1, 9), (1, 15)):
        ref = ora.gated(to_np(q[b, h]), to_np(k[b, h]), to_np(v[b, h]), a[b, h].numpy(),
                        eps=w.eps)
        err = max_row_error(to_np(o[b, h]), ref)
        assert err < 2e-2, (b, h, err)


def test_decode_gated_h32_full_sampled(la, ora):
    """The gated decode workload's shape (256 sequences x H32, D = Dv = 128),
    from a zero state: M gated steps over all units, sampled units followed
    by the oracle's gated recurrence over the same M tokens."""
    from kernelized_sequence_mixing_gb300.workloads import (
        WORKLOADS, decode_step_gates, decode_step_inputs)
    w = WORKLOADS["decode_gated_bf16_h32"]
    M = 6
    S = torch.zeros((w.B, w.H, w.D, w.Dv), dtype=torch.float32, device="cuda")
    z = torch.zeros((w.B, w.H, w.D), dtype=torch.float32, device="cuda")
    units = [(0, 0), (77, 13), (255, 31)]
    qs, ks, vs, as_, outs = [], [], [], [], []
    for t in range(M):
        q, k, v = decode_step_inputs(w, t)
        a = decode_step_gates(w, t)
        o = la.decode_gated(q.cuda(), k.cuda(), v.cuda(), a.cuda(), S, z, eps=w.eps)
        qs.append(q); ks.append(k); vs.append(v); as_.append(a); outs.append(o.cpu())
    torch.cuda.synchronize()
    for b, h in units:
        seq = lambda xs: np.stack([to_np(x[b, h]) for x in xs])  # noqa: E731
        ref, S_ref, z_ref = ora.gated(seq(qs), seq(ks), seq(vs), seq(as_), eps=w.eps,
                                      return_state=True)
        got = seq(outs)
        assert max_row_error(got, ref) < 2e-2
        assert state_error(to_np(S[b, h]), S_ref) < 1e-4
        assert state_error(to_np(z[b, h])[None], z_ref[None]) < 1e-4
