"""Pins of the Performer oracle (oracle/favor.py) to facts it does not
compute itself: the unbiasedness the pages state for the feature map (Monte
Carlo over many random directions), the softmax-attention limit, a closed
form at W = 0, and a quadratic brute force of the attention over features."""
import numpy as np
import pytest
import torch

from oracle import favor as fv


def draw(seed, r, D, orthogonal):
    from kernelized_sequence_mixing_gb300.workloads import favor_matrix
    return favor_matrix(r, D, seed, orthogonal, dtype=torch.float64).numpy()


@pytest.mark.parametrize("orthogonal", [False, True])
def test_feature_map_is_unbiased_for_exp_qk(orthogonal):
    """E[phi(q).phi(k)] = exp(q.k) ("Choosing the Feature Map"): with 2^17
    directions the Monte Carlo mean sits within a few standard errors."""
    rng = np.random.default_rng(0)
    D, r = 6, 1 << 17
    W = draw(1, r, D, orthogonal)
    for _ in range(3):
        q = rng.normal(size=D) * 0.35
        k = rng.normal(size=D) * 0.35
        prods = fv.favor_features(q, W) * fv.favor_features(k, W) * r   # r samples
        est, se = prods.mean(), prods.std() / np.sqrt(r)
        assert abs(est - np.exp(q @ k)) < 5 * se + 1e-12, (est, np.exp(q @ k), se)


def test_feature_map_without_norm_term_would_be_biased():
    """Guard on the pin above: dropping -|x|^2/2 moves the estimate by far
    more than its standard error, so the pin separates the two readings."""
    rng = np.random.default_rng(1)
    D, r = 6, 1 << 16
    W = draw(2, r, D, False)
    q, k = rng.normal(size=D) * 0.5, rng.normal(size=D) * 0.5
    wrong = np.exp(q @ W.T) * np.exp(k @ W.T)
    assert abs(wrong.mean() - np.exp(q @ k)) > 20 * wrong.std() / np.sqrt(r)


def test_orthogonal_rows_and_marginal_norms():
    W = draw(3, 256, 64, True)
    for b in range(4):
        blk = W[64 * b:64 * (b + 1)]
        G = blk @ blk.T
        off = G - np.diag(np.diag(G))
        assert np.abs(off).max() < 1e-9 * np.abs(np.diag(G)).max()
    # squared row norms are chi-square with 64 degrees of freedom
    n2 = (W * W).sum(1)
    assert abs(n2.mean() - 64) < 4 * np.sqrt(2 * 64 / 256)


def test_zero_directions_give_the_gaussian_closed_form():
    """W = 0: every feature is exp(-|x|^2/2)/sqrt(r)."""
    x = np.random.default_rng(4).normal(size=(5, 7))
    f = fv.favor_features(x, np.zeros((16, 7)))
    ref = np.exp(-0.5 * (x * x).sum(1))[:, None] / 4.0
    assert np.allclose(f, np.broadcast_to(ref, f.shape), rtol=1e-15, atol=0)


def test_one_direction_fixes_each_feature_to_its_row():
    """W zero but for row j = c e_m: feature j is exp(c x_m - |x|^2/2)/sqrt(r)
    and every other feature exp(-|x|^2/2)/sqrt(r), so feature j belongs to
    row j of W.  D = r, so that a transposed W gives wrong values rather than
    a shape error."""
    r = D = 6
    x = np.random.default_rng(31).normal(size=(5, D))
    base = np.exp(-0.5 * (x * x).sum(1)) / np.sqrt(r)
    for j, m, c in ((0, 3, 0.7), (4, 1, -1.3), (5, 5, 0.4)):
        W = np.zeros((r, D))
        W[j, m] = c
        f = fv.favor_features(x, W)
        ref = np.repeat(base[:, None], r, axis=1)
        ref[:, j] = base * np.exp(c * x[:, m])
        assert np.allclose(f, ref, rtol=1e-14, atol=0)


def test_many_features_approach_softmax_attention():
    """With many random features, non-causal Performer attention approaches
    exact softmax attention softmax(q k^T) V (eps = 0)."""
    rng = np.random.default_rng(5)
    N, D, Dv, r = 8, 4, 3, 1 << 17
    q = rng.normal(size=(N, D)) * 0.3
    k = rng.normal(size=(N, D)) * 0.3
    v = rng.normal(size=(N, Dv))
    W = draw(6, r, D, True)
    o = fv.favor(q, k, v, W, causal=False, eps=0.0)
    s = np.exp(q @ k.T)
    ref = (s / s.sum(1, keepdims=True)) @ v
    assert np.abs(o - ref).max() < 0.02 * np.abs(ref).max()
    # and the causal form approaches the causally masked softmax
    oc = fv.favor(q, k, v, W, causal=True, eps=0.0)
    sm = np.tril(s)
    refc = (sm / sm.sum(1, keepdims=True)) @ v
    assert np.abs(oc - refc).max() < 0.02 * np.abs(refc).max()


@pytest.mark.parametrize("gamma", [None, 0.7])
def test_causal_features_match_quadratic_brute_force(gamma):
    rng = np.random.default_rng(7)
    U, N, r, Dv = 2, 13, 5, 4
    fq = rng.uniform(0.1, 2.0, size=(U, N, r))
    fk = rng.uniform(0.1, 2.0, size=(U, N, r))
    v = rng.normal(size=(U, N, Dv))
    g = 1.0 if gamma is None else gamma
    o, S, z = fv.causal_features(fq, fk, v, gamma=gamma, eps=0.25, return_state=True)
    for u in range(U):
        for i in range(N):
            w = np.array([g ** (i - j) * (fq[u, i] @ fk[u, j]) for j in range(i + 1)])
            ref = (w @ v[u, :i + 1]) / (w.sum() + 0.25)
            assert np.abs(o[u, i] - ref).max() < 1e-12 * np.abs(ref).max()
        Sref = sum(g ** (N - 1 - j) * np.outer(fk[u, j], v[u, j]) for j in range(N))
        assert np.abs(S[u] - Sref).max() < 1e-12 * np.abs(Sref).max()


def test_noncausal_equals_last_causal_row():
    rng = np.random.default_rng(8)
    fq = rng.uniform(0.1, 2.0, size=(9, 5))
    fk = rng.uniform(0.1, 2.0, size=(9, 5))
    v = rng.normal(size=(9, 3))
    on = fv.noncausal_features(fq, fk, v)
    oc = fv.causal_features(np.broadcast_to(fq[-1], fq.shape), fk, v)
    assert np.abs(on[-1] - oc[-1]).max() < 1e-13
