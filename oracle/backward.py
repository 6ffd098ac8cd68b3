"""fp64 oracle of the gradient of causal linear attention.

TEST INFRASTRUCTURE ONLY: nothing in the library's compute path may import
or call this module; only the test suite and the benchmark's CPU-baseline leg
do.  It shares no code with the CUDA path.

The forward is the pages' causal form ("Linear Attention Mechanisms"
(dileepadev.github.io), "Recurrent Reformulation", with the decay of "Gating
and Selective State Updates"), unrolled over the prefix:

    w_ij = gamma^(i-j) phi(q_i) . phi(k_j)        (j <= i)
    n_i  = sum_j w_ij v_j,   d_i = sum_j w_ij + eps,   o_i = n_i / d_i

and, for an upstream gradient g_i = dL/do_i, the chain rule through that
quotient gives, with gt_i = g_i / d_i and c_i = gt_i . o_i,

    dL/dw_ij   = gt_i . v_j - c_i                 (j <= i)
    dL/dv_j    = sum_(i>=j) w_ij gt_i
    dL/dphiq_i = sum_(j<=i) gamma^(i-j) (dL/dw_ij) phi(k_j)
    dL/dphik_j = sum_(i>=j) gamma^(i-j) (dL/dw_ij) phi(q_i)
    dL/dq = dL/dphiq * phi'(q),   phi'(x) = 1 (x > 0), exp(x) (x <= 0),

and the same for k.  The "parallel" view of the pages (the masked n x n
weight matrix) is used as it stands: quadratic in N, for the test sizes.
"""
from __future__ import annotations

import numpy as np


def _phi(x):
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def _dphi(x):
    return np.where(x > 0, 1.0, np.exp(np.minimum(x, 0.0)))


def _decay_mask(N, gamma):
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    if gamma is None or gamma == 1.0:
        return (j <= i).astype(np.float64)
    e = np.where(j <= i, i - j, 0).astype(np.float64)
    # gamma is an fp32 value (one per head), widened exactly
    g = float(np.float32(gamma))
    return np.where(j <= i, np.power(g, e), 0.0)


def causal_forward(q, k, v, gamma=None, eps=1e-6):
    """o [N, Dv] of one unit from the masked weight matrix (fp64)."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    Wm = (_phi(q) @ _phi(k).T) * _decay_mask(q.shape[0], gamma)
    return (Wm @ v) / (Wm.sum(1) + eps)[:, None]


def causal_backward(q, k, v, do, gamma=None, eps=1e-6):
    """(dq, dk, dv) of one unit: q, k [N, D]; v, do [N, Dv]; gamma a float
    or None.  fp64."""
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    fq, fk = _phi(q), _phi(k)
    G = _decay_mask(q.shape[0], gamma)
    Wm = (fq @ fk.T) * G                   # w_ij, zero above the diagonal
    d = Wm.sum(1) + eps
    o = (Wm @ v) / d[:, None]
    gt = do / d[:, None]
    c = np.sum(gt * o, axis=1)
    dW = (gt @ v.T - c[:, None]) * (G > 0)  # dL/dw_ij on j <= i
    dv = Wm.T @ gt
    dfq = (dW * G) @ fk
    dfk = (dW * G).T @ fq
    return dfq * _dphi(q), dfk * _dphi(k), dv


def causal_backward_units(q, k, v, do, gamma=None, eps=1e-6):
    """The same over leading unit dims: q, k [U..., N, D]; gamma None, a
    float, or one value per leading unit."""
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    lead = q.shape[:-2]
    g = np.broadcast_to(np.asarray(1.0 if gamma is None else gamma, dtype=np.float64), lead)
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    for idx in np.ndindex(*lead):
        dq[idx], dk[idx], dv[idx] = causal_backward(q[idx], k[idx], v[idx], do[idx],
                                                    float(g[idx]), eps)
    return dq, dk, dv
