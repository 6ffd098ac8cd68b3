"""Pins for the fp64 oracle (CPU only).

Each test checks the oracle against something other than itself: exact
rational arithmetic on hand-worked examples, a quadratic masked brute force
(a different formula from the oracle's recurrence), a restatement of the NumPy
listing on "Linear Attention Mechanisms" (sadullah.online), closed forms and
invariants.  The cases mix D != Dv, gamma in {0, 1/2, 0.9, 1}, negative inputs
(exp branch of phi) and nonzero eps, so that a dropped term, a wrong sign or
index, a transposed state or a misplaced decay fails at least one of them.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.txt")


# --------------------------------------------------------------------------
# independent restatements used as pins (no oracle code involved)

def phi_np(x):
    """elu(x) + 1 with alpha = 1, written from its definition."""
    x = np.asarray(x, dtype=np.float64)
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def brute_causal(q, k, v, gamma, eps):
    """Quadratic masked form: o = ((phiQ phiK^T) * M * G) V / rowsum + eps,
    M_ij = [j <= i], G_ij = gamma^(i-j) (gamma^0 = 1, also for gamma = 0).
    "Linear Attention Mechanisms" (dileepadev.github.io), "The Kernel Trick
    for Attention" plus the causal mask ("Attention-Free / Sub-Quadratic
    Architectures", "The recurrent form (causal)") and the RetNet weight
    ("Gating and Selective State Updates")."""
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    N = q.shape[0]
    gamma = float(np.float32(gamma))  # the library and the oracle take fp32
    A = phi_np(q) @ phi_np(k).T
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    expo = np.where(j <= i, i - j, 0)
    G = np.where(j <= i, np.power(float(gamma), expo), 0.0)
    P = A * G
    return (P @ v) / (P.sum(axis=1, keepdims=True) + eps)


def listing_noncausal(Q, K, V, eps=1e-6):
    """The non-causal reassociated form as the NumPy listing on "Linear
    Attention Mechanisms" (sadullah.online), "The linear attention trick",
    describes it: map Q and K, form the d x d_v product of the mapped keys
    with the values, read it out with the mapped queries and divide by the
    mapped queries' product with the column sums of the mapped keys plus
    1e-6."""
    fq = phi_np(Q)
    fk = phi_np(K)
    kv = fk.T @ np.asarray(V, dtype=np.float64)
    colsum = fk.sum(axis=0)[:, None]
    return (fq @ kv) / (fq @ colsum + eps)


def rng_inputs(seed, N, D, Dv, scale=1.0):
    r = np.random.default_rng(seed)
    q = (r.standard_normal((N, D)) * scale).astype(np.float32)
    k = (r.standard_normal((N, D)) * scale).astype(np.float32)
    v = (r.standard_normal((N, Dv)) * scale).astype(np.float32)
    return q, k, v


def rel_err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# --------------------------------------------------------------------------
# phi

def test_phi_special_values(oracle_mod):
    phi = oracle_mod.phi
    assert phi(0.0) == 1.0
    for x in (1e-300, 0.25, 0.5, 1.0, 3.0, 1e6):
        assert phi(x) == x + 1.0
    for x in (-1e-12, -0.5, -1.0, -7.25, -40.0, -745.0):
        assert phi(x) == math.exp(x)
    assert phi(-1e-300) == 1.0  # continuous at 0 from below
    xs = np.linspace(-30, 30, 601)
    assert np.all(phi(xs) > 0)


# --------------------------------------------------------------------------
# exact hand-worked fixtures

def _parse_matrix(s):
    return [[Fraction(e.strip()) for e in row.split(",")] for row in s.split(";")]


def load_golden():
    cases, cur = [], None
    with open(GOLDEN) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {"name": rest}
            elif key == "end":
                cases.append(cur)
                cur = None
            elif key in ("q", "k", "v", "o", "a", "S", "z"):
                cur[key] = _parse_matrix(rest)
            elif key in ("gamma", "eps"):
                cur[key] = Fraction(rest)
            elif key in ("causal", "gated"):
                cur[key] = bool(int(rest))
    return cases


def exact_quadratic(case):
    """Exact rational evaluation of the weighted-sum form, inputs >= 0 only
    for q and k (phi(x) = x + 1 exactly)."""
    q, k, v = case["q"], case["k"], case["v"]
    g, eps, causal = case["gamma"], case["eps"], case["causal"]
    N = len(q)
    out = []
    for i in range(N):
        fq = [x + 1 for x in q[i]]
        num = [Fraction(0)] * len(v[0])
        den = Fraction(0)
        for j in range(N):
            if causal and j > i:
                continue
            fk = [x + 1 for x in k[j]]
            w = sum(a * b for a, b in zip(fq, fk))
            if causal:
                w *= g ** (i - j) if i > j else 1
            num = [n + w * x for n, x in zip(num, v[j])]
            den += w
        out.append([n / (den + eps) for n in num])
    return out


def exact_gated(case):
    """Exact rational evaluation of the gated recurrence's weighted-sum form:
    w_ts = sum_d phi(q_t)[d] phi(k_s)[d] prod_(u=s+1..t) a_u[d] (s <= t), and
    the final state S[d] = sum_s prod_(u=s+1..N-1) a_u[d] phi(k_s)[d] v_s."""
    q, k, v, a, eps = case["q"], case["k"], case["v"], case["a"], case["eps"]
    N, D, Dv = len(q), len(q[0]), len(v[0])

    def carry(s, t):  # prod_(u = s+1 .. t) a_u, per feature
        p = [Fraction(1)] * D
        for u in range(s + 1, t + 1):
            p = [x * y for x, y in zip(p, a[u])]
        return p

    out = []
    for t in range(N):
        fq = [x + 1 for x in q[t]]
        num, den = [Fraction(0)] * Dv, Fraction(0)
        for s in range(t + 1):
            fk = [x + 1 for x in k[s]]
            w = sum(x * y * c for x, y, c in zip(fq, fk, carry(s, t)))
            num = [n + w * x for n, x in zip(num, v[s])]
            den += w
        out.append([n / (den + eps) for n in num])
    S = [[Fraction(0)] * Dv for _ in range(D)]
    z = [Fraction(0)] * D
    for s in range(N):
        fk = [x + 1 for x in k[s]]
        c = carry(s, N - 1)
        for d in range(D):
            z[d] += c[d] * fk[d]
            S[d] = [x + c[d] * fk[d] * y for x, y in zip(S[d], v[s])]
    return out, S, [z]


@pytest.mark.parametrize("case", load_golden(), ids=lambda c: c["name"])
def test_hand_worked_examples(oracle_mod, case):
    as_f32 = lambda m: np.array(m, dtype=np.float64).astype(np.float32)  # noqa: E731
    as_f64 = lambda m: np.array([[float(x) for x in row] for row in m])  # noqa: E731
    if case.get("gated"):
        # the hand-derived values agree with exact rational arithmetic
        o, S, z = exact_gated(case)
        assert (o, S, z) == (case["o"], case["S"], case["z"])
        got, gS, gz = oracle_mod.gated(as_f32(case["q"]), as_f32(case["k"]), as_f32(case["v"]),
                                       as_f32(case["a"]), eps=float(case["eps"]),
                                       return_state=True)
        np.testing.assert_allclose(got, as_f64(case["o"]), rtol=1e-15, atol=1e-15)
        np.testing.assert_allclose(gS, as_f64(case["S"]), rtol=1e-15, atol=1e-15)
        np.testing.assert_allclose(gz, as_f64(case["z"])[0], rtol=1e-15, atol=1e-15)
        return
    # the fixture's hand-derived values agree with exact rational arithmetic
    assert exact_quadratic(case) == case["o"]
    q = np.array(case["q"], dtype=np.float64).astype(np.float32)
    k = np.array(case["k"], dtype=np.float64).astype(np.float32)
    v = np.array(case["v"], dtype=np.float64).astype(np.float32)
    if case["causal"]:
        o = oracle_mod.causal(q, k, v, gamma=float(case["gamma"]),
                              eps=float(case["eps"]))
    else:
        assert case["gamma"] == 1
        o = oracle_mod.noncausal(q, k, v, eps=float(case["eps"]))
    expect = np.array([[float(x) for x in row] for row in case["o"]])
    np.testing.assert_allclose(o, expect, rtol=1e-15, atol=1e-15)


# --------------------------------------------------------------------------
# brute force on tiny random inputs (exp branch exercised: negative inputs)

@pytest.mark.parametrize("gamma", [0.0, 0.5, 0.9, 1.0])
@pytest.mark.parametrize("N,D,Dv", [(1, 3, 5), (7, 4, 6), (33, 8, 3),
                                    (64, 5, 8)])
def test_causal_matches_quadratic_brute_force(oracle_mod, gamma, N, D, Dv):
    q, k, v = rng_inputs(100 + N + D, N, D, Dv)
    for eps in (0.0, 1e-6, 0.5):
        o = oracle_mod.causal(q, k, v, gamma=gamma, eps=eps)
        ref = brute_causal(q, k, v, gamma, eps)
        assert rel_err(o, ref) < 1e-12, (eps, rel_err(o, ref))


def test_causal_batched_units_and_per_head_gamma(oracle_mod):
    B, H, N, D, Dv = 2, 3, 20, 4, 5
    r = np.random.default_rng(7)
    q = r.standard_normal((B, H, N, D)).astype(np.float32)
    k = r.standard_normal((B, H, N, D)).astype(np.float32)
    v = r.standard_normal((B, H, N, Dv)).astype(np.float32)
    gam = np.array([0.25, 0.8, 1.0], dtype=np.float32)
    for nthreads in (1, 4):
        o = oracle_mod.causal(q, k, v, gamma=gam, eps=1e-6, nthreads=nthreads)
        for b in range(B):
            for h in range(H):
                ref = brute_causal(q[b, h], k[b, h], v[b, h], float(gam[h]),
                                   1e-6)
                assert rel_err(o[b, h], ref) < 1e-12


def test_decayed_state_closed_form(oracle_mod):
    """S = sum_j gamma^(N-1-j) phi(k_j) v_j^T and z likewise."""
    N, D, Dv, g = 40, 6, 3, 0.7
    _, k, v = rng_inputs(5, N, D, Dv)
    S, z = oracle_mod.prefill(k, v, gamma=g)
    w = float(np.float32(g)) ** (N - 1 - np.arange(N))
    fk = phi_np(k)
    S_ref = (fk * w[:, None]).T @ v.astype(np.float64)
    z_ref = (fk * w[:, None]).sum(axis=0)
    assert rel_err(S, S_ref) < 1e-13
    assert rel_err(z, z_ref) < 1e-13


# --------------------------------------------------------------------------
# the pages' non-causal listing, and non-causal invariants

@pytest.mark.parametrize("N,D,Dv", [(1, 2, 2), (50, 8, 8), (129, 6, 10)])
def test_noncausal_matches_listing(oracle_mod, N, D, Dv):
    q, k, v = rng_inputs(11 + N, N, D, Dv)
    o = oracle_mod.noncausal(q, k, v, eps=1e-6)
    assert rel_err(o, listing_noncausal(q, k, v, 1e-6)) < 1e-12


def test_noncausal_key_value_permutation_invariance(oracle_mod):
    q, k, v = rng_inputs(3, 61, 7, 5)
    perm = np.random.default_rng(0).permutation(61)
    o1 = oracle_mod.noncausal(q, k, v)
    o2 = oracle_mod.noncausal(q, k[perm], v[perm])
    assert rel_err(o2, o1) < 1e-13


def test_noncausal_equals_last_causal_row(oracle_mod):
    q, k, v = rng_inputs(4, 45, 8, 8)
    oc = oracle_mod.causal(q, k, v, gamma=1.0)
    on = oracle_mod.noncausal(q, k, v)
    assert rel_err(on[-1], oc[-1]) < 1e-13
    # and only the last row: earlier rows differ
    assert rel_err(on[0], oc[0]) > 1e-3


# --------------------------------------------------------------------------
# closed forms / invariants of the causal form

def test_constant_values_give_constant_output(oracle_mod):
    N, D, Dv = 30, 5, 4
    q, k, _ = rng_inputs(9, N, D, Dv)
    c = np.array([1.5, -2.0, 0.25, 3.0], dtype=np.float32)
    v = np.tile(c, (N, 1))
    for g in (1.0, 0.6):
        o = oracle_mod.causal(q, k, v, gamma=g, eps=0.0)
        assert np.max(np.abs(o - c[None, :])) < 1e-13
        # with eps: o = c * den / (den + eps)
        eps = 0.3
        o = oracle_mod.causal(q, k, v, gamma=g, eps=eps)
        P = brute_causal(q, k, np.ones((N, 1), np.float32), g, 0.0)  # = 1
        assert np.allclose(P, 1.0)
        fq, fk = phi_np(q), phi_np(k)
        i = np.arange(N)[:, None]
        j = np.arange(N)[None, :]
        g32 = float(np.float32(g))
        den = ((fq @ fk.T) * np.where(j <= i, g32 ** np.maximum(i - j, 0),
                                      0.0)).sum(1)
        assert rel_err(o, c[None, :] * (den / (den + eps))[:, None]) < 1e-13


def test_gamma_one_matches_undecayed(oracle_mod):
    q, k, v = rng_inputs(12, 25, 6, 7)
    assert np.array_equal(oracle_mod.causal(q, k, v, gamma=1.0),
                          oracle_mod.causal(q, k, v, gamma=None))


def test_gamma_zero_closed_form(oracle_mod):
    q, k, v = rng_inputs(13, 25, 6, 7)
    eps = 0.1
    a = (phi_np(q) * phi_np(k)).sum(1)
    ref = v.astype(np.float64) * (a / (a + eps))[:, None]
    o = oracle_mod.causal(q, k, v, gamma=0.0, eps=eps)
    assert rel_err(o, ref) < 1e-14
    # row 0 has the same value at any gamma
    for g in (0.3, 1.0):
        o = oracle_mod.causal(q, k, v, gamma=g, eps=eps)
        assert rel_err(o[0], ref[0]) < 1e-14


def test_output_linear_in_values(oracle_mod):
    q, k, v1 = rng_inputs(14, 30, 5, 6)
    _, _, v2 = rng_inputs(15, 30, 5, 6)
    a, b = 0.75, -1.25
    for g in (1.0, 0.8):
        o1 = oracle_mod.causal(q, k, v1, gamma=g)
        o2 = oracle_mod.causal(q, k, v2, gamma=g)
        o12 = oracle_mod.causal(q, k, (a * v1.astype(np.float64)
                                       + b * v2).astype(np.float32), gamma=g)
        # the fp32 rounding of the combined values is the only difference
        v12 = (a * v1.astype(np.float64) + b * v2).astype(np.float32)
        ref = brute_causal(q, k, v12, g, 1e-6)
        assert rel_err(o12, ref) < 1e-12
        assert rel_err(o12, a * o1 + b * o2) < 1e-6


@pytest.mark.parametrize("gamma", [1.0, 0.9])
def test_prefill_then_decode_equals_causal(oracle_mod, gamma):
    """prefill(N) followed by M single-token steps reproduces rows N..N+M-1 of
    one causal pass over N+M tokens, and the same final state."""
    N, M, D, Dv = 17, 9, 6, 4
    q, k, v = rng_inputs(21, N + M, D, Dv)
    o_full, S_full, z_full = oracle_mod.causal(q, k, v, gamma=gamma,
                                               return_state=True)
    S, z = oracle_mod.prefill(k[:N], v[:N], gamma=gamma)
    _, S_pre, z_pre = oracle_mod.causal(q[:N], k[:N], v[:N], gamma=gamma,
                                        return_state=True)
    assert np.array_equal(S, S_pre) and np.array_equal(z, z_pre)
    for t in range(M):
        o, S, z = oracle_mod.decode_step(q[N + t], k[N + t], v[N + t], S, z,
                                         gamma=gamma)
        assert rel_err(o, o_full[N + t]) < 1e-13
    assert rel_err(S, S_full) < 1e-13 and rel_err(z, z_full) < 1e-13


def test_state_in_continues_sequence(oracle_mod):
    q, k, v = rng_inputs(22, 40, 5, 5)
    o_full = oracle_mod.causal(q, k, v, gamma=0.95)
    _, S, z = oracle_mod.causal(q[:23], k[:23], v[:23], gamma=0.95,
                                return_state=True)
    o_tail = oracle_mod.causal(q[23:], k[23:], v[23:], gamma=0.95,
                               state=(S, z))
    assert rel_err(o_tail, o_full[23:]) < 1e-13


def test_decode_step_closed_forms(oracle_mod):
    """gamma = 0 forgets the carried state: S' = phi(k) v^T, z' = phi(k) and
    o = v a / (a + eps) with a = phi(q).phi(k), whatever (S, z) held; v = 0
    leaves S' = gamma S exactly (the update adds phi(k) 0^T)."""
    D, Dv, eps = 5, 3, 0.25
    q, k, v = rng_inputs(23, 1, D, Dv)
    rng = np.random.default_rng(24)
    S0 = rng.uniform(0.5, 2.0, (D, Dv))
    z0 = rng.uniform(0.5, 2.0, D)
    o, S, z = oracle_mod.decode_step(q[0], k[0], v[0], S0.copy(), z0.copy(),
                                     gamma=0.0, eps=eps)
    fq, fk = phi_np(q[0]), phi_np(k[0])
    a = float(fq @ fk)
    assert rel_err(o, v[0].astype(np.float64) * (a / (a + eps))) < 1e-14
    assert rel_err(S, np.outer(fk, v[0])) < 1e-15 and rel_err(z, fk) < 1e-15
    _, S, _ = oracle_mod.decode_step(q[0], k[0], np.zeros(Dv, np.float32),
                                     S0.copy(), z0.copy(), gamma=0.75, eps=eps)
    assert np.array_equal(S, 0.75 * S0)


@pytest.mark.parametrize("gamma", [1.0, 0.8])
def test_one_token_continuation_equals_decode_step(oracle_mod, gamma):
    """A causal pass over one token that starts from a given (S, z) and a
    decode step on the same (S, z) are the same recurrence step, reached
    through different entry points."""
    N, D, Dv = 12, 4, 6
    q, k, v = rng_inputs(25, N + 1, D, Dv)
    _, S, z = oracle_mod.causal(q[:N], k[:N], v[:N], gamma=gamma,
                                return_state=True)
    o_c, S_c, z_c = oracle_mod.causal(q[N:], k[N:], v[N:], gamma=gamma,
                                      state=(S.copy(), z.copy()),
                                      return_state=True)
    o_d, S_d, z_d = oracle_mod.decode_step(q[N], k[N], v[N], S.copy(),
                                           z.copy(), gamma=gamma)
    assert rel_err(o_c[0], o_d) < 1e-15
    assert rel_err(S_c, S_d) < 1e-15 and rel_err(z_c, z_d) < 1e-15


def test_empty_sequence(oracle_mod):
    q = np.zeros((0, 4), np.float32)
    v = np.zeros((0, 3), np.float32)
    assert oracle_mod.causal(q, q, v).shape == (0, 3)
    S, z = oracle_mod.prefill(q, v)
    assert not S.any() and not z.any()


# --------------------------------------------------------------------------
# gated form (per-step, per-key-feature gate G_i = a_i 1^T)

def brute_gated(q, k, v, a, eps):
    """Quadratic form of the gated recurrence, written from its definition:
    o_t = sum_(s <= t) w_ts v_s / (sum_(s <= t) w_ts + eps) with
    w_ts = sum_d phi(q_t)[d] phi(k_s)[d] prod_(u = s+1..t) a_u[d] (the
    product of the gates applied to the state after step s).  "Linear
    Attention Mechanisms" (dileepadev.github.io), "Gating and Selective State
    Updates", S_t = G_t (.) S_(t-1) + phi(k_t) v_t^T, unrolled."""
    q, k, v, a = (np.asarray(x, dtype=np.float64) for x in (q, k, v, a))
    N, D = q.shape
    fq, fk = phi_np(q), phi_np(k)
    o = np.zeros((N, v.shape[1]))
    for t in range(N):
        w = np.zeros(t + 1)
        for s in range(t + 1):
            prod = np.ones(D)
            for u in range(s + 1, t + 1):
                prod = prod * a[u]
            w[s] = float(np.sum(fq[t] * fk[s] * prod))
        o[t] = (w @ v[: t + 1]) / (w.sum() + eps)
    return o


def gate_inputs(seed, N, D, lo=0.0, hi=1.0):
    r = np.random.default_rng(seed)
    return r.uniform(lo, hi, size=(N, D)).astype(np.float32)


@pytest.mark.parametrize("N,D,Dv", [(1, 3, 2), (9, 4, 5), (24, 6, 3)])
def test_gated_matches_quadratic_brute_force(oracle_mod, N, D, Dv):
    q, k, v = rng_inputs(300 + N, N, D, Dv)
    for lo in (0.0, 0.5, 0.9):
        a = gate_inputs(400 + N, N, D, lo, 1.0)
        for eps in (0.0, 1e-6):
            o = oracle_mod.gated(q, k, v, a, eps=eps)
            assert rel_err(o, brute_gated(q, k, v, a, eps)) < 1e-12


def test_gated_constant_gate_is_the_decayed_form(oracle_mod):
    """a_i[d] = gamma for every step and feature is the RetNet decay; a = 1
    is plain linear attention (the pages' G_t = 1 case)."""
    q, k, v = rng_inputs(21, 40, 6, 5)
    for g in (1.0, 0.9, 0.5):
        a = np.full((40, 6), g, np.float32)
        assert rel_err(oracle_mod.gated(q, k, v, a), brute_causal(q, k, v, g, 1e-6)) < 1e-12


def test_gated_zero_gate_overwrites_the_state(oracle_mod):
    """G_t = 0 overwrites the state (the pages' forget case): the output at
    t depends on token t alone, o_t = v_t A / (A + eps), A = phi(q_t).phi(k_t),
    and the state after t is phi(k_t) v_t^T."""
    q, k, v = rng_inputs(22, 12, 5, 4)
    a = gate_inputs(23, 12, 5, 0.2, 1.0)
    a[7] = 0.0
    o, S, z = oracle_mod.gated(q[:8], k[:8], v[:8], a[:8], eps=1e-6, return_state=True)
    A = float(phi_np(q[7]) @ phi_np(k[7]))
    assert rel_err(o[7], v[7].astype(np.float64) * A / (A + 1e-6)) < 1e-13
    assert rel_err(S, np.outer(phi_np(k[7]), v[7].astype(np.float64))) < 1e-15
    assert rel_err(z, phi_np(k[7])) < 1e-15


def test_gated_feature_gates_act_per_row_of_the_state(oracle_mod):
    """A gate that is 0 on one key feature and 1 elsewhere clears exactly
    that row of S and entry of z, and leaves the rest as in the ungated sum."""
    q, k, v = rng_inputs(24, 10, 4, 3)
    a = np.ones((10, 4), np.float32)
    a[9, 2] = 0.0
    _, S, z = oracle_mod.gated(q, k, v, a, return_state=True)
    _, S1, z1 = oracle_mod.causal(q, k, v, return_state=True)
    fk9 = phi_np(k[9])
    assert rel_err(S[2], fk9[2] * v[9].astype(np.float64)) < 1e-15
    assert abs(z[2] - fk9[2]) <= 1e-15 * abs(fk9[2])
    for d in (0, 1, 3):
        assert rel_err(S[d], S1[d]) < 1e-14 and abs(z[d] - z1[d]) <= 1e-14 * abs(z1[d])


def test_gated_final_state_matches_the_unrolled_sum(oracle_mod):
    """The state after the last token, unrolled from the gated recurrence:
    S[d, :] = sum_s (prod_(u = s+1..N-1) a_u[d]) phi(k_s)[d] v_s and z[d]
    the same without v_s, with random gates in [0, 1)."""
    for N, D, Dv, lo in ((1, 3, 2, 0.0), (13, 5, 4, 0.0), (30, 4, 6, 0.7)):
        q, k, v = rng_inputs(500 + N, N, D, Dv)
        a = gate_inputs(600 + N, N, D, lo, 1.0)
        _, S, z = oracle_mod.gated(q, k, v, a, return_state=True)
        fk = phi_np(k)
        vv = v.astype(np.float64)
        S_ref = np.zeros((D, Dv))
        z_ref = np.zeros(D)
        for s in range(N):
            w = np.ones(D)
            for u in range(s + 1, N):
                w = w * a[u]
            S_ref += np.outer(w * fk[s], vv[s])
            z_ref += w * fk[s]
        assert rel_err(S, S_ref) < 1e-13 and rel_err(z, z_ref) < 1e-13
