"""Pins of the gradient oracle (oracle/backward.py) to what it does not
compute itself: central finite differences of the C forward oracle (a
different program: the token recurrence), on tiny inputs, for every input
and several decays."""
import numpy as np
import pytest

from oracle import backward as bw


def loss_grad_fd(oracle_mod, q, k, v, do, gamma, eps, which, h=1e-6):
    """dL/d(which) by central differences of L = sum(do * o), o from the C
    oracle's token recurrence (fp64 arithmetic on fp32-widened inputs, so the
    inputs are perturbed in steps fp32 can hold)."""
    args = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
    x = args[which]
    g = np.zeros_like(x, dtype=np.float64)
    gam = None if gamma is None else np.array([gamma], dtype=np.float32)
    for idx in np.ndindex(*x.shape):
        old = x[idx]
        vals = []
        for s in (+1, -1):
            x[idx] = np.float32(old + s * h)
            step = float(np.float64(x[idx]) - np.float64(old))
            o = oracle_mod.causal(args["q"][None], args["k"][None], args["v"][None],
                                  gamma=gam, eps=eps)[0]
            vals.append((np.sum(do * o), step))
        x[idx] = old
        (lp, sp), (lm, sm) = vals
        g[idx] = (lp - lm) / (sp - sm)
    return g


@pytest.mark.parametrize("gamma", [None, 0.8])
@pytest.mark.parametrize("N,D,Dv", [(1, 3, 2), (6, 4, 3), (11, 3, 5)])
def test_backward_matches_finite_differences(oracle_mod, gamma, N, D, Dv):
    rng = np.random.default_rng(10 * N + D)
    q = rng.normal(size=(N, D)).astype(np.float32)
    k = rng.normal(size=(N, D)).astype(np.float32)
    v = rng.normal(size=(N, Dv)).astype(np.float32)
    do = rng.normal(size=(N, Dv))
    eps = 0.3  # a sizeable eps, so its place in the quotient is pinned too
    dq, dk, dv = bw.causal_backward(q, k, v, do, gamma, eps)
    for name, got in (("q", dq), ("k", dk), ("v", dv)):
        fd = loss_grad_fd(oracle_mod, q, k, v, do, gamma, eps, name, h=2e-3)
        err = np.abs(got - fd).max() / max(np.abs(fd).max(), 1e-12)
        assert err < 2e-4, (name, err)


def test_backward_forward_equals_c_oracle(oracle_mod):
    """The quadratic forward inside the gradient oracle is the C oracle's
    recurrence (a consistency check on the weights it differentiates)."""
    rng = np.random.default_rng(3)
    q, k, v = (rng.normal(size=(40, 6)).astype(np.float32) for _ in range(3))
    for gamma in (None, 0.5, 0.97):
        o = bw.causal_forward(q, k, v, gamma, 1e-6)
        gam = None if gamma is None else np.array([gamma], dtype=np.float32)
        ref = oracle_mod.causal(q[None], k[None], v[None], gamma=gam)[0]
        assert np.abs(o - ref).max() < 1e-12 * np.abs(ref).max()


def test_backward_of_constant_values_is_zero_for_q_and_k():
    """With every v_j equal, o_i = v (times sum w / (sum w + eps)); with
    eps = 0 the output does not depend on q or k at all."""
    rng = np.random.default_rng(4)
    q, k = rng.normal(size=(9, 4)), rng.normal(size=(9, 4))
    v = np.tile(rng.normal(size=(1, 3)), (9, 1))
    do = rng.normal(size=(9, 3))
    dq, dk, dv = bw.causal_backward(q, k, v, do, 0.9, eps=0.0)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12
    # and dv sums to the upstream gradient row sums (o is a convex mix of v)
    assert np.allclose(dv.sum(0), do.sum(0), rtol=1e-12, atol=1e-12)


def test_backward_units_takes_one_decay_per_head(oracle_mod):
    """The batched wrapper over [B, H, N, D] inputs with one decay per head:
    every unit's gradient equals central differences of the C oracle run on
    the whole batch with the same per-head decays.  The decays differ from
    head to head, so a unit paired with another head's decay fails."""
    rng = np.random.default_rng(12)
    B, H, N, D, Dv = 2, 3, 5, 3, 2
    q = rng.normal(size=(B, H, N, D)).astype(np.float32)
    k = rng.normal(size=(B, H, N, D)).astype(np.float32)
    v = rng.normal(size=(B, H, N, Dv)).astype(np.float32)
    do = rng.normal(size=(B, H, N, Dv))
    gam = np.array([0.5, 0.8, 1.0], dtype=np.float32)
    eps, h = 0.3, 2e-3
    got = dict(zip("qkv", bw.causal_backward_units(q, k, v, do, gam, eps)))
    args = {"q": q, "k": k, "v": v}
    for name in "qkv":
        x = args[name]
        fd = np.zeros(x.shape)
        for idx in np.ndindex(*x.shape):
            old = x[idx]
            vals = []
            for s in (+1, -1):
                x[idx] = np.float32(old + s * h)
                step = float(np.float64(x[idx]) - np.float64(old))
                o = oracle_mod.causal(q, k, v, gamma=gam, eps=eps)
                vals.append((np.sum(do * o), step))
            x[idx] = old
            (lp, sp), (lm, sm) = vals
            fd[idx] = (lp - lm) / (sp - sm)
        err = np.abs(got[name] - fd).max() / np.abs(fd).max()
        assert err < 2e-4, (name, err)
