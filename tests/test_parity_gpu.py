"""GPU parity: the CUDA path against the fp64 oracle on the same seeded inputs.

Small cases are compared in full (several chunk tiles plus a ragged tail);
the full-size workloads, run in the same launch configuration the benchmark
times, are compared on whole sampled heads.  Errors are per-row normwise
(see helpers.TOL): 1e-4 for fp32 inputs, 2e-2 for bf16 inputs.  Each test
records its worst error, printed with its tolerance at the end of the run.
"""
import numpy as np
import pytest
import torch

from helpers import TOL, max_row_error, record, state_error, to_np

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


def gen(B, H, N, D, Dv, dtype, seed, scale=0.5):
    from kernelized_sequence_mixing_gb300.workloads import make_qkv
    return make_qkv(B, H, N, D, Dv, dtype, seed, scale)


def dtype_name(dtype):
    return "fp32" if dtype == torch.float32 else "bf16"


def gammas_for(H, kind):
    if kind is None:
        return None
    if kind == "mix":    # includes decays too strong for the tensor-core path
        base = [0.0, 0.5, 0.9, 0.96875, 0.999, 1.0]
        return torch.tensor([base[h % len(base)] for h in range(H)],
                            dtype=torch.float32)
    if kind == "mild":   # every decay inside the tensor-core envelope
        base = [0.35, 0.75, 0.96875, 0.999, 1.0, 0.5]
        return torch.tensor([base[h % len(base)] for h in range(H)],
                            dtype=torch.float32)
    if kind == "retnet":
        from kernelized_sequence_mixing_gb300.workloads import retnet_gammas
        return retnet_gammas(H)
    return torch.full((H,), float(kind), dtype=torch.float32)


# --------------------------------------------------------------------------
# causal forward

CAUSAL_SMALL = [
    # (B, H, N, D, Dv)
    (1, 1, 1, 64, 64),
    (1, 2, 63, 64, 64),
    (2, 1, 64, 64, 128),
    (1, 3, 65, 128, 64),
    (1, 2, 200, 128, 128),
    (2, 2, 1000, 64, 64),
    (1, 2, 1337, 128, 128),
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16],
                         ids=["f32", "bf16"])
@pytest.mark.parametrize("gkind", [None, "mix", "mild"])
@pytest.mark.parametrize("shape", CAUSAL_SMALL, ids=lambda s: "x".join(map(str, s)))
def test_causal_small(la, ora, dtype, gkind, shape):
    B, H, N, D, Dv = shape
    q, k, v = gen(B, H, N, D, Dv, dtype, seed=N + D + 7 * H)
    g = gammas_for(H, gkind)
    path = la.causal_kernel(B, H, N, D, Dv, gamma=g, dtype=dtype)
    # "mix" always holds 0.0 for head 0, which sends the call to the CUDA
    # cores; "mild" holds 0.35 and 0.5, too strong for 128-token chunks
    tc_expected = dtype == torch.bfloat16 and gkind != "mix"
    c128 = tc_expected and (D, Dv) == (128, 128) and gkind is None
    assert path == ("tensor-core-128" if c128 else
                    "tensor-core" if tc_expected else "cuda-core"), path
    o = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=True, gamma=g, eps=1e-6)
    torch.cuda.synchronize()
    ref = ora.causal(to_np(q), to_np(k), to_np(v),
                     gamma=None if g is None else g.numpy(), eps=1e-6)
    err = record(f"causal small {dtype_name(dtype)}", max_row_error(to_np(o), ref), TOL[dtype])
    assert err < TOL[dtype], err


# The tensor-core path cuts each (batch, head) into parts (at most one wave of
# CTAs) and rescales its state once per decay window.  Many heads give one
# part per head and windows of one chunk (gamma = 0.35 / 0.5) or several
# (0.9, 0.99); fewer heads give several multi-chunk parts, so the state
# crosses parts and windows (20 heads x 64 chunks: 5 parts of 12-13 chunks,
# skewed toward the front; 16 heads x 128 chunks: 7 skewed parts of 15-22).
CAUSAL_PARTS = [
    # (B, H, N, D, Dv, gammas)
    (8, 76, 700, 64, 64, [0.35, 0.5, 0.9, 0.99]),
    (2, 100, 2560, 64, 64, [0.5, 0.9, 0.99, 1.0]),
    (1, 40, 1500, 128, 128, [0.6, 0.97, 1.0, 0.85]),
    (2, 10, 4096, 128, 64, [0.5, 0.35, 0.9, 0.999, 1.0]),
    (1, 16, 8192, 64, 64, [0.4, 0.8, 0.95, 1.0]),
]


@pytest.mark.parametrize("case", CAUSAL_PARTS, ids=lambda c: "x".join(map(str, c[:5])))
def test_causal_parts_and_windows(la, ora, case):
    B, H, N, D, Dv, gl = case
    q, k, v = gen(B, H, N, D, Dv, torch.bfloat16, seed=H + N)
    g = torch.tensor([gl[h % len(gl)] for h in range(H)], dtype=torch.float32)
    assert la.causal_kernel(B, H, N, D, Dv, gamma=g, dtype=torch.bfloat16) == "tensor-core"
    o = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=True, gamma=g, eps=1e-6)
    torch.cuda.synchronize()
    ref = ora.causal(to_np(q), to_np(k), to_np(v), gamma=g.numpy(), eps=1e-6)
    err = record("causal parts and windows (64-token kernel)", max_row_error(to_np(o), ref), 2e-2)
    assert err < 2e-2, err


# The 128-token-chunk kernel (bf16, D = Dv = 128, every gamma >= 0.61): one
# token, ragged single chunks, a chunk plus one token, windows of one chunk
# (gamma = 0.61) and of several, several parts per head (few heads) with the
# state crossing parts and windows, one part per head (many heads).
CAUSAL128 = [
    # (B, H, N, gammas)
    (1, 1, 1, None),
    (1, 2, 127, [0.61, 1.0]),
    (2, 3, 129, [0.7, 0.9, 1.0]),
    (1, 2, 1000, [0.61, 0.999]),
    (1, 8, 5000, [0.8, 0.97, 1.0, 0.9]),
    (1, 3, 20000, [0.61, 0.99, 1.0]),
    (2, 76, 700, [0.75, 0.96875, 1.0, 0.999]),
]


@pytest.mark.parametrize("case", CAUSAL128, ids=lambda c: "x".join(map(str, c[:3])))
def test_causal_chunk128(la, ora, case):
    B, H, N, gl = case
    D = Dv = 128
    q, k, v = gen(B, H, N, D, Dv, torch.bfloat16, seed=3 * H + N)
    g = None if gl is None else torch.tensor([gl[h % len(gl)] for h in range(H)],
                                             dtype=torch.float32)
    assert la.causal_kernel(B, H, N, D, Dv, gamma=g, dtype=torch.bfloat16) == "tensor-core-128"
    o = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=True, gamma=g, eps=1e-6)
    torch.cuda.synchronize()
    ref = ora.causal(to_np(q), to_np(k), to_np(v),
                     gamma=None if g is None else g.numpy(), eps=1e-6)
    err = record("causal 128-token kernel", max_row_error(to_np(o), ref), 2e-2)
    assert err < 2e-2, err


def test_causal_f32_n256_full(la, ora):
    """fp32, gamma = 1, B1 H1 N256 D=Dv=64, N(0,1) from seed 0."""
    from kernelized_sequence_mixing_gb300.workloads import (WORKLOADS,
                                                            workload_inputs)
    w = WORKLOADS["causal_f32_n256"]
    q, k, v = workload_inputs(w)
    o = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=True, eps=w.eps)
    ref = ora.causal(to_np(q), to_np(k), to_np(v), eps=w.eps)
    assert o.shape == (1, 1, 256, 64) and o.dtype == torch.float32
    err = record("causal_f32_n256 (every row)", max_row_error(to_np(o), ref), 1e-4)
    assert err < 1e-4


def test_causal_bf16_n4096_full(la, ora):
    """bf16, gamma = 1, B4 H8 N4096 D=Dv=64: every row of every head."""
    from kernelized_sequence_mixing_gb300.workloads import (WORKLOADS,
                                                            workload_inputs)
    w = WORKLOADS["causal_bf16_n4096"]
    q, k, v = workload_inputs(w)
    o = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=True, eps=w.eps)
    ref = ora.causal(to_np(q), to_np(k), to_np(v), eps=w.eps)
    err = record("causal_bf16_n4096 (every row)", max_row_error(to_np(o), ref), 2e-2)
    assert err < 2e-2


def test_causal_decay_bf16_n16384_all_heads(la, ora):
    """The benchmarked workload (B2 H16 N16384 D=Dv=128, per-head RetNet
    decay), one launch at full size, in the benchmark's launch configuration
    (four sequence parts per head): every row of all 32 heads against the
    oracle, so every part boundary and look-back chain is compared."""
    from kernelized_sequence_mixing_gb300.workloads import (WORKLOADS,
                                                            workload_inputs)
    w = WORKLOADS["causal_decay_bf16_n16384"]
    q, k, v = workload_inputs(w)
    g = w.gamma()
    o = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=True, gamma=g,
                   eps=w.eps)
    o = to_np(o)
    assert np.isfinite(o).all()
    ref = ora.causal(to_np(q), to_np(k), to_np(v), gamma=g.numpy(), eps=w.eps)
    worst = 0.0
    for b in range(w.B):
        for h in range(w.H):
            err = max_row_error(o[b, h], ref[b, h])
            worst = max(worst, err)
            assert err < 2e-2, (b, h, err)
    record("causal_decay_bf16_n16384 (all 32 heads, every row)", worst, 2e-2)


def test_causal_empty_and_host_buffers(la, ora):
    q, k, v = gen(1, 2, 0, 64, 64, torch.bfloat16, 1)
    o = la.forward(q.cuda(), k.cuda(), v.cuda())
    assert o.shape == (1, 2, 0, 64)
    # host tensors (la_forward_host: groups of heads whose copies overlap the
    # kernels): the oracle's result within tolerance, and the device path's
    q, k, v = gen(1, 2, 300, 64, 128, torch.bfloat16, 2)
    o_host = la.forward(q, k, v, gamma=[0.9, 1.0])
    o_dev = la.forward(q.cuda(), k.cuda(), v.cuda(), gamma=[0.9, 1.0])
    assert o_host.device.type == "cpu"
    ref = ora.causal(to_np(q), to_np(k), to_np(v), gamma=[0.9, 1.0])
    assert max_row_error(to_np(o_host), ref) < 2e-2
    assert max_row_error(to_np(o_host), to_np(o_dev)) < 2e-2


# Host buffers through la_forward_host: several batch entries and head
# groups, decays per head (each group keeps its own), causal and non-causal,
# both dtypes; pinned inputs and a pinned output buffer as the benchmark's
# end-to-end leg passes them.
HOST_CASES = [
    # (B, H, N, D, Dv, dtype, causal, gammas)
    (2, 16, 1000, 128, 128, torch.bfloat16, True, "retnet"),
    (3, 5, 777, 64, 64, torch.bfloat16, False, None),
    (2, 3, 300, 64, 128, torch.float32, True, "mix"),
]


@pytest.mark.parametrize("case", HOST_CASES, ids=lambda c: "x".join(map(str, c[:5])) + ("c" if c[6] else "n"))
def test_forward_host_buffers(la, ora, case):
    B, H, N, D, Dv, dtype, causal, gk = case
    q, k, v = gen(B, H, N, D, Dv, dtype, seed=B + H + N)
    g = gammas_for(H, gk)
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    out = torch.empty((B, H, N, Dv), dtype=dtype, pin_memory=True)
    o = la.forward(qh, kh, vh, causal=causal, gamma=g, out=out)
    assert o.data_ptr() == out.data_ptr() and o.device.type == "cpu"
    gn = None if g is None else g.numpy()
    ref = (ora.causal(to_np(q), to_np(k), to_np(v), gamma=gn) if causal else
           ora.noncausal(to_np(q), to_np(k), to_np(v)))
    err = record(f"host buffers {dtype_name(dtype)}", max_row_error(to_np(o), ref), TOL[dtype])
    assert err < TOL[dtype], err


def test_causal_repeatable(la):
    q, k, v = (t.cuda() for t in gen(2, 2, 777, 128, 128, torch.bfloat16, 3))
    a = la.forward(q, k, v, gamma=[0.95, 0.5])
    b = la.forward(q, k, v, gamma=[0.95, 0.5])
    assert torch.equal(a, b)


# --------------------------------------------------------------------------
# non-causal forward

NONCAUSAL_SMALL = [
    (1, 1, 1, 64, 64),
    (1, 2, 100, 64, 128),
    (2, 1, 4096, 128, 64),
    (1, 2, 4097, 128, 128),
    (1, 1, 10000, 64, 64),
    # more (batch, head) work items than resident CTAs: a CTA's later items
    # belong to other heads (the persistent passes replace [S | z] and start
    # a new record mid-loop), with a ragged last tile
    (8, 80, 333, 64, 64),
    (4, 90, 129, 128, 128),
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16],
                         ids=["f32", "bf16"])
@pytest.mark.parametrize("shape", NONCAUSAL_SMALL, ids=lambda s: "x".join(map(str, s)))
def test_noncausal_small(la, ora, dtype, shape):
    B, H, N, D, Dv = shape
    q, k, v = gen(B, H, N, D, Dv, dtype, seed=3 * N + D)
    o = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=False)
    ref = ora.noncausal(to_np(q), to_np(k), to_np(v), eps=1e-6)
    err = record(f"non-causal small {dtype_name(dtype)}", max_row_error(to_np(o), ref), TOL[dtype])
    assert err < TOL[dtype]


def test_noncausal_equals_last_causal_row(la):
    q, k, v = (t.cuda() for t in gen(1, 2, 999, 64, 64, torch.float32, 5))
    on = la.forward(q, k, v, causal=False)
    oc = la.forward(q, k, v, causal=True)
    err = max_row_error(to_np(on[:, :, -1]), to_np(oc[:, :, -1]))
    assert err < 1e-4


def test_noncausal_repeatable(la):
    q, k, v = (t.cuda() for t in gen(2, 2, 9000, 64, 64, torch.bfloat16, 6))
    assert torch.equal(la.forward(q, k, v, causal=False),
                       la.forward(q, k, v, causal=False))


def test_noncausal_bf16_n65536_sampled_heads(la, ora):
    """Full-size non-causal workload (B8 H16 N65536 D=Dv=64), in the launch
    configuration the benchmark times; 32 of the 128 heads compared whole
    (every batch entry, every head index)."""
    from kernelized_sequence_mixing_gb300.workloads import (WORKLOADS,
                                                            workload_inputs)
    w = WORKLOADS["noncausal_bf16_n65536"]
    q, k, v = workload_inputs(w)
    o = to_np(la.forward(q.cuda(), k.cuda(), v.cuda(), causal=False,
                         eps=w.eps))
    assert np.isfinite(o).all()
    units = [(b, (5 * b + j) % w.H) for b in range(w.B) for j in range(0, w.H, 4)]
    assert len(units) == 32 and len(set(units)) == 32
    bs = [u[0] for u in units]
    hs = [u[1] for u in units]
    ref = ora.noncausal(to_np(q[bs, hs]), to_np(k[bs, hs]), to_np(v[bs, hs]), eps=w.eps)
    worst = 0.0
    for i, (b, h) in enumerate(units):
        err = max_row_error(o[b, h], ref[i])
        worst = max(worst, err)
        assert err < 2e-2, (b, h, err)
    record("noncausal_bf16_n65536 (32 of 128 heads, every row)", worst, 2e-2)


# --------------------------------------------------------------------------
# prefill and decode

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16],
                         ids=["f32", "bf16"])
@pytest.mark.parametrize("gkind", [None, "mix"])
@pytest.mark.parametrize("N,D,Dv", [(0, 64, 64), (1, 64, 128), (300, 128, 64),
                                    (5000, 128, 128)])
def test_prefill_state(la, ora, dtype, gkind, N, D, Dv):
    B, H = 1, 3
    q, k, v = gen(B, H, N, D, Dv, dtype, seed=N + 11)
    g = gammas_for(H, gkind)
    S, z = la.prefill_state(k.cuda(), v.cuda(), gamma=g)
    S_ref, z_ref = ora.prefill(to_np(k), to_np(v),
                               gamma=None if g is None else g.numpy())
    if N == 0:
        assert not S.any() and not z.any()
        return
    tol = 1e-4  # fp32 sums of up to 5000 terms
    eS = record("prefill state S", state_error(to_np(S), S_ref), tol)
    ez = record("prefill state z", state_error(to_np(z)[..., None], z_ref[..., None]), tol)
    assert eS < tol and ez < tol, (eS, ez)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16],
                         ids=["f32", "bf16"])
@pytest.mark.parametrize("gkind", [None, "mix"])
@pytest.mark.parametrize("D,Dv", [(64, 64), (128, 64), (64, 128), (128, 128)])
def test_prefill_then_decode_matches_causal(la, ora, dtype, gkind, D, Dv):
    """prefill(N) then M decode steps reproduce causal rows N..N+M-1."""
    B, H, N, M = 2, 6, 70, 12
    q, k, v = gen(B, H, N + M, D, Dv, dtype, seed=D + Dv)
    g = gammas_for(H, gkind)
    gn = None if g is None else g.numpy()
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    S, z = la.prefill_state(kd[:, :, :N].contiguous(), vd[:, :, :N].contiguous(),
                            gamma=g)
    ref_full, S_end, z_end = ora.causal(to_np(q), to_np(k), to_np(v), gamma=gn,
                                        return_state=True)
    for t in range(M):
        o = la.decode_step(qd[:, :, N + t].contiguous(), kd[:, :, N + t].contiguous(),
                           vd[:, :, N + t].contiguous(), S, z, gamma=g)
        err = max_row_error(to_np(o), ref_full[:, :, N + t])
        assert err < TOL[dtype], (t, err)
    assert state_error(to_np(S), S_end) < 1e-4
    assert state_error(to_np(z)[..., None], z_end[..., None]) < 1e-4
    # the GPU's own causal forward agrees too
    oc = la.forward(qd, kd, vd, gamma=g)
    assert max_row_error(to_np(o), to_np(oc[:, :, -1])) < 2 * TOL[dtype]


def test_decode_state_roundtrip(la):
    """A state copied out and back in continues identically (resume)."""
    B, H, D, Dv = 2, 4, 128, 128
    q, k, v = gen(B, H, 2, D, Dv, torch.bfloat16, 9)
    S = torch.rand(B, H, D, Dv, device="cuda")
    z = torch.rand(B, H, D, device="cuda") + 1
    S2, z2 = S.cpu().cuda(), z.cpu().cuda()
    args = [t[:, :, 0].contiguous().cuda() for t in (q, k, v)]
    o1 = la.decode_step(*args, S, z)
    o2 = la.decode_step(*args, S2, z2)
    assert torch.equal(o1, o2) and torch.equal(S, S2) and torch.equal(z, z2)


def test_decode_bf16_h32_full(la, ora):
    """The decode workload: 256 sequences x H32, D=Dv=128, fp32 state from a
    512-token prefill, then 1024 steps with fresh seeded inputs.  64 sampled
    (sequence, head) units (eight sequences x eight heads, spread over both
    ranges) are followed by the oracle through every step; outputs are gated
    at steps 0..7, every 128th and the last, and the final states are
    compared."""
    from kernelized_sequence_mixing_gb300.workloads import (
        WORKLOADS, decode_step_inputs, workload_inputs)
    w = WORKLOADS["decode_bf16_h32"]
    q, k, v = workload_inputs(w)
    S, z = la.prefill_state(k.cuda(), v.cuda())
    units = [(b, h) for b in (0, 17, 64, 101, 128, 170, 213, 255)
             for h in (0, 5, 9, 14, 16, 22, 27, 31)]
    bs = [u[0] for u in units]
    hs = [u[1] for u in units]
    Sr, zr = ora.prefill(to_np(k[bs, hs]), to_np(v[bs, hs]))
    e0 = record("decode_bf16_h32 prefill state (64 units)", state_error(to_np(S[bs, hs]), Sr), 1e-4)
    assert e0 < 1e-4
    gate = set(range(8)) | set(range(0, w.steps, 128)) | {w.steps - 1}
    worst = 0.0
    for t in range(w.steps):
        qt, kt, vt = decode_step_inputs(w, t)
        o = la.decode_step(qt.cuda(), kt.cuda(), vt.cuda(), S, z, eps=w.eps)
        orf, Sr, zr = ora.decode_step(to_np(qt[bs, hs]), to_np(kt[bs, hs]),
                                      to_np(vt[bs, hs]), Sr, zr, eps=w.eps)
        if t in gate:
            err = max_row_error(to_np(o[bs, hs]), orf)
            worst = max(worst, err)
            assert err < 2e-2, (t, err)
    record("decode_bf16_h32 outputs (64 units, gated steps)", worst, 2e-2)
    eS = record("decode_bf16_h32 final S (64 units)", state_error(to_np(S[bs, hs]), Sr), 1e-4)
    ez = record("decode_bf16_h32 final z (64 units)",
                state_error(to_np(z[bs, hs])[..., None], zr[..., None]), 1e-4)
    assert eS < 1e-4 and ez < 1e-4, (eS, ez)


# The causal forward that also returns the final state: the fused path of
# the 128-token kernel (the last part's CTA writes S, z; one part, a few
# parts, many parts, one token) and the composed path (forward, then the
# prefill reduction) of the 64-token and CUDA-core kernels.
FORWARD_STATE = [
    # (B, H, N, D, Dv, dtype, gammas)
    (1, 2, 1000, 128, 128, torch.bfloat16, [0.61, 0.999]),
    (1, 3, 20000, 128, 128, torch.bfloat16, [0.9, 0.99, 1.0]),
    (2, 76, 700, 128, 128, torch.bfloat16, [0.75, 0.97, 1.0, 0.999]),
    (1, 1, 1, 128, 128, torch.bfloat16, None),
    (1, 2, 333, 64, 64, torch.bfloat16, [0.9, 1.0]),
    (1, 2, 300, 64, 128, torch.float32, [0.5, 1.0]),
]


@pytest.mark.parametrize("case", FORWARD_STATE,
                         ids=lambda c: "x".join(map(str, c[:5])) + ("-f32" if c[5] == torch.float32 else ""))
def test_forward_state(la, ora, case):
    B, H, N, D, Dv, dtype, gl = case
    q, k, v = gen(B, H, N, D, Dv, dtype, seed=5 * H + N)
    g = None if gl is None else torch.tensor([gl[h % len(gl)] for h in range(H)],
                                             dtype=torch.float32)
    o, S, z = la.forward_state(q.cuda(), k.cuda(), v.cuda(), gamma=g, eps=1e-6)
    torch.cuda.synchronize()
    gn = None if g is None else g.numpy()
    ref = ora.causal(to_np(q), to_np(k), to_np(v), gamma=gn, eps=1e-6)
    S_ref, z_ref = ora.prefill(to_np(k), to_np(v), gamma=gn)
    tol = TOL[dtype]
    eo = record(f"forward with state: o {dtype_name(dtype)}", max_row_error(to_np(o), ref), tol)
    assert eo < tol
    eS = record(f"forward with state: S {dtype_name(dtype)}", state_error(to_np(S), S_ref), tol)
    ez = record(f"forward with state: z {dtype_name(dtype)}",
                state_error(to_np(z)[..., None], z_ref[..., None]), tol)
    # the fused state sums bf16 operands like the output: the bf16 bound
    assert eS < tol and ez < tol, (eS, ez)
    # and it equals the forward's own output path: la.forward gives the same o
    o2 = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=True, gamma=g, eps=1e-6)
    assert torch.equal(o, o2)


def test_tensor_core_and_cuda_core_paths_agree(la, ora):
    """The same bf16 problem through both causal kernels (a strong decay on a
    spare head forces the CUDA-core kernel) against the oracle."""
    B, H, N, D, Dv = 1, 3, 777, 128, 128
    q, k, v = gen(B, H, N, D, Dv, torch.bfloat16, 77)
    g_128 = torch.tensor([0.9, 0.99, 1.0])
    g_64 = torch.tensor([0.9, 0.99, 0.5])
    g_cc = torch.tensor([0.9, 0.99, 0.1])
    assert la.causal_kernel(B, H, N, D, Dv, g_128) == "tensor-core-128"
    assert la.causal_kernel(B, H, N, D, Dv, g_64) == "tensor-core"
    assert la.causal_kernel(B, H, N, D, Dv, g_cc) == "cuda-core"
    outs = [to_np(la.forward(q.cuda(), k.cuda(), v.cuda(), gamma=g))
            for g in (g_128, g_64, g_cc)]
    ref = ora.causal(to_np(q), to_np(k), to_np(v), gamma=g_128.numpy())
    for h in range(2):
        for o in outs:
            assert max_row_error(o[0, h], ref[0, h]) < 2e-2
        for o in outs[:2]:
            assert max_row_error(o[0, h], outs[2][0, h]) < 2e-2


def test_zz_no_device_wait_timeouts(la):
    """No tensor-core kernel gave up a bounded wait during this module."""
    torch.cuda.synchronize()
    assert la.device_wait_timeouts() == 0
