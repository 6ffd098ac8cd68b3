"""fp64 oracle of the Performer random-feature map and of linear attention
over given features.

TEST INFRASTRUCTURE ONLY: nothing in the library's compute path may import
or call this module; only the test suite, the smoke check and the benchmark's
CPU-baseline leg do.  It shares no code with the CUDA path.

Feature map ("Linear Attention Mechanisms" (dileepadev.github.io),
"Choosing the Feature Map", Random Fourier Features (Performer) and positive
orthogonal random features (FAVOR+); "Attention-Free / Sub-Quadratic
Architectures", "Feature maps"): with r random directions w_1..w_r (the rows
of W, drawn by the caller and passed in)

    phi(x) = r^(-1/2) [exp(w_1.x - |x|^2/2), ..., exp(w_r.x - |x|^2/2)]

Reading of the pages: the printed map omits the -|x|^2/2 term, but the same
passage states that E[phi(q).phi(k)] = exp(q.k); with w ~ N(0, I),
E[exp(w.(q + k))] = exp(|q + k|^2 / 2), so that statement holds only with
exp(-|q|^2/2 - |k|^2/2) folded in.  That is the positive random feature the
FAVOR+ paragraph names, and the oracle takes it.  The kernel approximated is
exp(q.k) exactly as the pages write it (no 1/sqrt(D) temperature).

Attention over features fq, fk (the pages' o_i = phi(q_i)^T S_i /
(phi(q_i)^T z_i + eps) with phi replaced by the given features):
  causal      S_i = gamma S_(i-1) + fk_i v_i^T, z_i = gamma z_(i-1) + fk_i
              ("Recurrent Reformulation"; decay from "Gating and Selective
              State Updates"), token by token;
  non-causal  S = sum_j fk_j v_j^T, z = sum_j fk_j ("The Kernel Trick for
              Attention").
"""
from __future__ import annotations

import numpy as np


def favor_features(x, W):
    """phi(x) for x [..., D] and W [r, D] (fp32 values, widened): [..., r] fp64."""
    x = np.asarray(x, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    r = W.shape[0]
    proj = x @ W.T                                  # w_j . x
    half_sq = 0.5 * np.sum(x * x, axis=-1, keepdims=True)
    return np.exp(proj - half_sq) / np.sqrt(r)


def causal_features(fq, fk, v, gamma=None, eps=1e-6, return_state=False):
    """Causal linear attention over given features, the recurrence token by
    token.  fq, fk [U..., N, r]; v [U..., N, Dv]; gamma None, a float, or one
    value per leading unit (broadcast over the leading dims)."""
    fq = np.asarray(fq, dtype=np.float64)
    fk = np.asarray(fk, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    lead = fq.shape[:-2]
    N, r = fq.shape[-2:]
    Dv = v.shape[-1]
    g = np.ones(lead) if gamma is None else np.broadcast_to(
        np.asarray(gamma, dtype=np.float64), lead)
    S = np.zeros(lead + (r, Dv))
    z = np.zeros(lead + (r,))
    o = np.empty(lead + (N, Dv))
    gs, gz = g[..., None, None], g[..., None]
    for i in range(N):
        S = gs * S + fk[..., i, :, None] * v[..., i, None, :]
        z = gz * z + fk[..., i, :]
        num = np.einsum("...r,...re->...e", fq[..., i, :], S)
        den = np.einsum("...r,...r->...", fq[..., i, :], z) + eps
        o[..., i, :] = num / den[..., None]
    return (o, S, z) if return_state else o


def noncausal_features(fq, fk, v, eps=1e-6):
    """Non-causal linear attention over given features: one (S, z) per unit
    shared by every query."""
    fq = np.asarray(fq, dtype=np.float64)
    fk = np.asarray(fk, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    S = np.einsum("...nr,...ne->...re", fk, v)
    z = fk.sum(axis=-2)
    num = np.einsum("...nr,...re->...ne", fq, S)
    den = np.einsum("...nr,...r->...n", fq, z) + eps
    return num / den[..., None]


def favor(q, k, v, W, causal=True, gamma=None, eps=1e-6):
    """Performer attention: the random-feature map of q and k with the rows of
    W, then linear attention over those features."""
    fq, fk = favor_features(q, W), favor_features(k, W)
    if causal:
        return causal_features(fq, fk, v, gamma=gamma, eps=eps)
    if gamma is not None and np.any(np.asarray(gamma) != 1.0):
        raise ValueError("a decay needs the causal form")
    return noncausal_features(fq, fk, v, eps=eps)
