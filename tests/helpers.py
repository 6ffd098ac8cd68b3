"""Shared helpers of the test suite: error metrics and tolerances."""
import numpy as np
import torch

# Per-row normwise relative error bars: max over rows i of
# max_e |o_ie - r_ie| / max_e |r_ie|.  Element-wise relative error is
# ill-posed here (outputs are signed weighted means of zero-mean values, some
# of them near zero), so each row is measured against its own largest entry.
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def to_np(t):
    return t.detach().to("cpu", torch.float32).numpy()


def row_errors(out, ref):
    """out, ref: [..., Dv] arrays; returns per-row normwise errors."""
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.max(np.abs(out - ref), axis=-1)
    den = np.maximum(np.max(np.abs(ref), axis=-1), 1e-30)
    return num / den


def max_row_error(out, ref):
    e = row_errors(out, ref)
    return float(e.max()) if e.size else 0.0


def state_error(S, S_ref):
    """Normwise error of a state per unit: max |S - S_ref| / max |S_ref|."""
    S = np.asarray(S, dtype=np.float64)
    S_ref = np.asarray(S_ref, dtype=np.float64)
    ax = tuple(range(S.ndim - 2, S.ndim)) if S.ndim >= 2 else (S.ndim - 1,)
    num = np.max(np.abs(S - S_ref), axis=ax)
    den = np.maximum(np.max(np.abs(S_ref), axis=ax), 1e-30)
    return float((num / den).max())


# Worst error per checked quantity, {name: (error, tolerance)}; printed at the
# end of the run (tests/conftest.py) so that the margin to each tolerance is
# visible without -s.
MARGINS = {}


def record(name, err, tol):
    """Keep the worst error of one checked quantity for the end-of-run report."""
    err = float(err)
    if name not in MARGINS or err > MARGINS[name][0]:
        MARGINS[name] = (err, float(tol))
    return err
