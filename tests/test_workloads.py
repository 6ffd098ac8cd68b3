"""The seeded input generators on CPU, against the recipe they state: the
per-head RetNet decays, the gate range and the exact 0 / 1 rates, the seed
offsets of each workload's extra inputs, determinism, shapes and dtypes, and
the sizes of the registered workloads."""
import torch
import pytest

from kernelized_sequence_mixing_gb300 import workloads as wl
from kernelized_sequence_mixing_gb300.workloads import WORKLOADS


def test_retnet_gammas_are_exact_powers_of_two_below_one():
    g = wl.retnet_gammas(16)
    assert g.dtype == torch.float32 and g.shape == (16,)
    # h = 0, 4, 8, 12: 1 - 2^-5, 1 - 2^-6, 1 - 2^-7, 1 - 2^-8, all exact in fp32
    for h, e in ((0, 5), (4, 6), (8, 7), (12, 8)):
        assert g[h].item() == 1.0 - 2.0 ** -e
    # between them, 1 - 2^(-5 - h/4) rounded once to fp32
    for h in range(16):
        want = 1.0 - 2.0 ** (-5.0 - h / 4.0)
        assert abs(g[h].item() - want) <= 2.0 ** -24
    assert torch.all(g[1:] > g[:-1]) and g[0] >= 0.96875 and g[-1] < 1.0


def test_make_qkv_is_seeded_and_shaped():
    q, k, v = wl.make_qkv(2, 3, 5, 64, 128, torch.bfloat16, seed=9, scale=0.5)
    assert q.shape == k.shape == (2, 3, 5, 64) and v.shape == (2, 3, 5, 128)
    assert q.dtype == k.dtype == v.dtype == torch.bfloat16
    q2, k2, v2 = wl.make_qkv(2, 3, 5, 64, 128, torch.bfloat16, seed=9, scale=0.5)
    assert torch.equal(q, q2) and torch.equal(k, k2) and torch.equal(v, v2)
    q3, _, _ = wl.make_qkv(2, 3, 5, 64, 128, torch.bfloat16, seed=10, scale=0.5)
    assert not torch.equal(q, q3)
    # q, k and v are three different draws of one stream
    assert not torch.equal(q, k)
    # the scale is applied before the single rounding: 0.5 x is exact in bf16
    qf, _, _ = wl.make_qkv(2, 3, 5, 64, 128, torch.float32, seed=9, scale=1.0)
    assert torch.equal(q, (qf * 0.5).to(torch.bfloat16))


def test_gates_range_and_exact_rates():
    a = wl.make_gates(2, 4, 256, 64, seed=3, lo=0.5, hi=1.0)
    assert a.dtype == torch.float32 and a.shape == (2, 4, 256, 64)
    assert a.min() >= 0.5 and a.max() < 1.0
    # uniform: mean near 0.75 over 131,072 draws
    assert abs(a.mean().item() - 0.75) < 0.005
    b = wl.make_gates(2, 4, 256, 64, seed=3, lo=0.5, hi=1.0, zero_frac=0.1, one_frac=0.05)
    zeros = (b == 0).float().mean().item()
    ones = (b == 1).float().mean().item()
    assert abs(zeros - 0.1 * 0.95) < 0.01     # zeros set first, then some become ones
    assert abs(ones - 0.05) < 0.005
    rest = b[(b != 0) & (b != 1)]
    assert rest.min() >= 0.5 and rest.max() < 1.0
    assert torch.equal(b, wl.make_gates(2, 4, 256, 64, seed=3, lo=0.5, hi=1.0,
                                        zero_frac=0.1, one_frac=0.05))


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_registered_workload_sizes(name):
    w = WORKLOADS[name]
    assert w.name == name
    assert w.D in (64, 128) and w.Dv in (64, 128)
    assert w.B * w.H * w.N < 2 ** 31
    if w.decayed:
        assert w.causal and torch.all(w.gamma() >= 0.61)   # the 128-token kernel's range
    else:
        assert w.gamma() is None


def test_the_five_configurations():
    want = {
        "causal_f32_n256": (True, 1, 1, 256, 64, 64, torch.float32, 1.0, 0, False),
        "causal_bf16_n4096": (True, 4, 8, 4096, 64, 64, torch.bfloat16, 0.5, 1, False),
        "causal_decay_bf16_n16384": (True, 2, 16, 16384, 128, 128, torch.bfloat16, 0.5, 2,
                                     True),
        "noncausal_bf16_n65536": (False, 8, 16, 65536, 64, 64, torch.bfloat16, 0.5, 3,
                                  False),
        "decode_bf16_h32": (True, 256, 32, 512, 128, 128, torch.bfloat16, 0.5, 4, False),
    }
    for name, t in want.items():
        w = WORKLOADS[name]
        assert (w.causal, w.B, w.H, w.N, w.D, w.Dv, w.dtype, w.scale, w.seed,
                w.decayed) == t, name
    d = WORKLOADS["decode_bf16_h32"]
    assert d.steps == 1024 and d.step_seed0 == 1000


def test_extra_inputs_use_their_seed_offsets():
    g = WORKLOADS["gla_bf16_n16384"]
    small = wl.Workload("t", True, 1, 2, 8, 64, 64, torch.bfloat16, 0.5, 5, gated=True)
    assert torch.equal(wl.workload_gates(small), wl.make_gates(1, 2, 8, 64, 6, 0.9, 1.0))
    assert g.gate_lo == 0.9 and g.seed == 5
    f = WORKLOADS["favor_bf16_n16384"]
    assert f.favor_r == 128 and f.scale == 128 ** -0.25
    assert torch.equal(wl.workload_favor_matrix(f),
                       wl.favor_matrix(128, 128, 8, True, torch.bfloat16))
    b = WORKLOADS["backward_bf16_n4096"]
    small_b = wl.Workload("t", True, 1, 2, 8, 64, 64, torch.bfloat16, 0.5, 7, backward=True)
    up = wl.workload_upstream(small_b)
    gen = torch.Generator().manual_seed(10)
    assert torch.equal(up, torch.randn((1, 2, 8, 64), generator=gen).to(torch.bfloat16))
    assert b.backward and b.seed == 7
    dg = WORKLOADS["decode_gated_bf16_h32"]
    small_d = wl.Workload("t", True, 2, 3, 4, 64, 64, torch.bfloat16, 0.5, 4, steps=8,
                          step_seed0=1000, gated=True)
    a5 = wl.decode_step_gates(small_d, 5)
    assert a5.shape == (2, 3, 64) and a5.is_contiguous()
    assert torch.equal(a5, wl.make_gates(2, 3, 1, 64, 51005, 0.9, 1.0)[:, :, 0])
    assert dg.steps == 1024 and dg.gated


def test_decode_step_inputs_follow_the_step_seed():
    d = wl.Workload("t", True, 2, 3, 4, 64, 128, torch.bfloat16, 0.5, 4, steps=8,
                    step_seed0=1000)
    q, k, v = wl.decode_step_inputs(d, 3)
    assert q.shape == k.shape == (2, 3, 64) and v.shape == (2, 3, 128)
    qq, kk, vv = wl.make_qkv(2, 3, 1, 64, 128, torch.bfloat16, 1003, 0.5)
    assert torch.equal(q, qq[:, :, 0]) and torch.equal(v, vv[:, :, 0])
