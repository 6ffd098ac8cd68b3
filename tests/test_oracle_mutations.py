"""The oracle's pins catch plausible mistakes planted in the oracle (CPU only).

Each case copies one oracle source (``oracle/linattn_oracle.c``,
``oracle/favor.py`` or ``oracle/backward.py``) to a temporary directory,
plants one mistake (a dropped term, a misplaced decay, a transposed operand,
a wrong index, another reading of a formula), loads it (the C file built with
the oracle's own gcc command, through a fresh instance of its wrapper), and
runs every pin of that oracle's test module against it: at least one pin
must fail.  Each unmodified source goes through the same steps and must pass
every pin, so that a failure of the harness itself cannot pass for a caught
mutant.

Every planted mistake keeps the oracle's memory accesses inside its buffers
(no stride or bound is changed), so a mutant can only compute wrong values.
Nothing here touches the library or a GPU.
"""
import importlib.util
import inspect
import itertools
import os

import pytest

import oracle
import test_oracle
import test_oracle_backward
import test_oracle_favor

ORACLE_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")
ORACLE_C = os.path.join(ORACLE_DIR, "linattn_oracle.c")
ORACLE_PY = os.path.join(ORACLE_DIR, "__init__.py")
FAVOR_PY = os.path.join(ORACLE_DIR, "favor.py")
BACKWARD_PY = os.path.join(ORACLE_DIR, "backward.py")

C_MUTANTS = [
    ("z_not_decayed", "z[d] = gamma * z[d] + fk[d];", "z[d] = z[d] + fk[d];", 0),
    ("S_decayed_after_update",
     "Sd[e] = gamma * Sd[e] + fk[d] * (double)vi[e];",
     "Sd[e] = gamma * (Sd[e] + fk[d] * (double)vi[e]);", 0),
    ("S_decay_squared",
     "Sd[e] = gamma * Sd[e] + fk[d] * (double)vi[e];",
     "Sd[e] = gamma * gamma * Sd[e] + fk[d] * (double)vi[e];", 0),
    ("causal_eps_dropped", "den += eps;", "den += 0.0 * eps;", 0),
    ("causal_eps_as_floor", "den += eps;", "den = den > eps ? den : eps;", 0),
    ("phi_plain_elu", "return x > 0.0 ? x + 1.0 : exp(x);",
     "return x > 0.0 ? x : exp(x) - 1.0;", 0),
    ("phi_linear_below_zero", "return x > 0.0 ? x + 1.0 : exp(x);",
     "return x > 0.0 ? x + 1.0 : 1.0 + x;", 0),
    ("causal_state_read_transposed",
     "num += fq[d] * S[(int64_t)d * Dv + e];",
     "num += fq[d] * S[(int64_t)e * D + d];", 0),
    ("keys_mapped_from_queries",
     "for (int d = 0; d < D; ++d) fk[d] = oracle_phi((double)ki[d]);",
     "for (int d = 0; d < D; ++d) fk[d] = oracle_phi((double)(q ? q[i * D + d] : ki[d]));", 0),
    ("causal_read_out_with_phi_of_k",
     "for (int d = 0; d < D; ++d) fq[d] = oracle_phi((double)qi[d]);",
     "for (int d = 0; d < D; ++d) fq[d] = fk[d] + 0.0 * qi[d];", 0),
    ("decode_ignores_decay",
     "causal_unit(J->q + u * D, J->k + u * D, J->v + u * Dv, g, J->eps, 1, D,",
     "causal_unit(J->q + u * D, J->k + u * D, J->v + u * Dv, 1.0, J->eps, 1, D,", 0),
    ("continued_sequence_restarts", "if (!J->have_state_in) {", "if (1) {", 0),
    ("gate_not_applied_to_z", "z[d] = g * z[d] + fk[d];", "z[d] = z[d] + fk[d];", 0),
    ("gate_applied_after_update",
     "Sd[e] = g * Sd[e] + fk[d] * (double)vi[e];",
     "Sd[e] = g * (Sd[e] + fk[d] * (double)vi[e]);", 0),
    ("gate_of_previous_token",
     "*ai = a + i * D;", "*ai = a + (i > 0 ? i - 1 : 0) * D;", 0),
    ("gate_complement", "const double g = (double)ai[d];",
     "const double g = 1.0 - (double)ai[d];", 0),
    ("gated_eps_dropped", "den += eps;", "den += 0.0 * eps;", 1),
    ("gated_state_read_transposed",
     "num += fq[d] * S[(int64_t)d * Dv + e];",
     "num += fq[d] * S[(int64_t)e * D + d];", 1),
    ("noncausal_z_of_squares", "z[d] += fk[d];", "z[d] += fk[d] * fk[d];", 0),
    ("noncausal_eps_dropped", "den += eps;", "den += 0.0 * eps;", 2),
    ("noncausal_state_read_transposed",
     "num += fq[d] * S[(int64_t)d * Dv + e];",
     "num += fq[d] * S[(int64_t)e * D + d];", 2),
]


FAVOR_MUTANTS = [
    ("norm_term_dropped", "np.exp(proj - half_sq)", "np.exp(proj)", 0),
    ("full_square_norm", "half_sq = 0.5 * np.sum(", "half_sq = 1.0 * np.sum(", 0),
    ("scaled_by_r_not_sqrt_r", "/ np.sqrt(r)", "/ r", 0),
    ("directions_transposed", "proj = x @ W.T", "proj = x @ W", 0),
    ("features_out_of_order", "proj = x @ W.T", "proj = x @ W.T[:, ::-1]", 0),
    ("causal_z_not_decayed", "z = gz * z + fk[..., i, :]", "z = z + fk[..., i, :]", 0),
    ("causal_eps_dropped", "fq[..., i, :], z) + eps", "fq[..., i, :], z) + 0.0 * eps", 0),
    ("causal_read_out_with_key_features",
     'num = np.einsum("...r,...re->...e", fq[..., i, :], S)',
     'num = np.einsum("...r,...re->...e", fk[..., i, :], S)', 0),
    ("noncausal_z_averaged", "z = fk.sum(axis=-2)", "z = fk.mean(axis=-2)", 0),
    ("noncausal_eps_dropped", '"...nr,...r->...n", fq, z) + eps', '"...nr,...r->...n", fq, z) + 0.0 * eps', 0),
]

BACKWARD_MUTANTS = [
    ("dphi_is_phi", "return np.where(x > 0, 1.0, np.exp(", "return np.where(x > 0, x + 1.0, np.exp(", 0),
    ("c_term_dropped", "dW = (gt @ v.T - c[:, None]) * (G > 0)", "dW = (gt @ v.T) * (G > 0)", 0),
    ("dv_weights_not_transposed", "dv = Wm.T @ gt", "dv = Wm @ gt", 0),
    ("dk_from_key_features", "dfk = (dW * G).T @ fq", "dfk = (dW * G).T @ fk", 0),
    ("dq_decay_dropped", "dfq = (dW * G) @ fk", "dfq = (dW * (G > 0)) @ fk", 0),
    ("upstream_not_divided_by_d", "gt = do / d[:, None]", "gt = do", 0),
    ("eps_dropped_in_d", "d = Wm.sum(1) + eps", "d = Wm.sum(1) + 0.0 * eps", 0),
    ("strict_causal_mask", "return (j <= i).astype(np.float64)", "return (j < i).astype(np.float64)", 0),
    ("per_head_decay_ignored", "float(g[idx]), eps)", "float(g.flat[0]), eps)", 0),
]


def plant(src, old, new, nth):
    """``src`` with occurrence ``nth`` of ``old`` replaced by ``new``."""
    at = -1
    for _ in range(nth + 1):
        at = src.find(old, at + 1)
        assert at >= 0, f"occurrence {nth} of {old!r} not in the oracle source"
    return src[:at] + new + src[at + len(old):]


def oracle_from_source(text, tmp_path, tag):
    """A fresh instance of the oracle wrapper bound to a build of ``text``."""
    src = tmp_path / f"oracle_{tag}.c"
    src.write_text(text)
    spec = importlib.util.spec_from_file_location(f"oracle_variant_{tag}", ORACLE_PY)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC = str(src)
    mod._LIB_PATH = str(tmp_path / f"liboracle_{tag}.so")
    mod._load()
    return mod


def module_from_source(text, tmp_path, tag):
    """A Python oracle module executed from ``text``."""
    src = tmp_path / f"{tag}.py"
    src.write_text(text)
    spec = importlib.util.spec_from_file_location(f"oracle_py_variant_{tag}", str(src))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def pins(test_module):
    """Every (id, function, parameters) of the pins in ``test_module``: its
    test functions, each over its parametrize grid."""
    out = []
    for name, fn in inspect.getmembers(test_module, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        grids = []
        for mark in getattr(fn, "pytestmark", []):
            if mark.name != "parametrize":
                continue
            argnames, argvalues = mark.args[0], mark.args[1]
            names = [a.strip() for a in argnames.split(",")] if isinstance(argnames, str) else list(argnames)
            rows = []
            for val in argvalues:
                vals = val if len(names) > 1 else (val,)
                rows.append(dict(zip(names, vals)))
            grids.append(rows)
        params = set(inspect.signature(fn).parameters)
        covered = {n for g in grids for row in g[:1] for n in row}
        assert params - covered <= {"oracle_mod"}, f"{name} takes an unknown fixture"
        for combo in itertools.product(*grids) if grids else [()]:
            kw = {}
            for part in combo:
                kw.update(part)
            out.append((f"{name}{sorted(kw.items()) if kw else ''}", fn, kw))
    return out


def failing_pins(test_module, oracle_mod, stop_at_first):
    failed = []
    for pid, fn, kw in pins(test_module):
        if "oracle_mod" in inspect.signature(fn).parameters:
            kw = dict(kw, oracle_mod=oracle_mod)
        try:
            fn(**kw)
        except Exception as e:  # a failed assertion, or an error the mistake causes
            failed.append((pid, type(e).__name__))
            if stop_at_first:
                break
    return failed


def read(path):
    with open(path) as f:
        return f.read()


# ---------------------------------------------------------------------------
# the C oracle: forms, decode step, gated form

def test_unmodified_c_oracle_passes_every_pin(tmp_path):
    assert len(pins(test_oracle)) >= 40
    mod = oracle_from_source(read(ORACLE_C), tmp_path, "clean")
    assert failing_pins(test_oracle, mod, False) == []


@pytest.mark.parametrize("mutant", C_MUTANTS, ids=[m[0] for m in C_MUTANTS])
def test_mistake_in_c_oracle_fails_a_pin(tmp_path, mutant):
    name, old, new, nth = mutant
    text = read(ORACLE_C)
    planted = plant(text, old, new, nth)
    assert planted != text
    caught = failing_pins(test_oracle, oracle_from_source(planted, tmp_path, name), True)
    assert caught, f"no pin fails with the mistake {name!r} planted in the oracle"


# ---------------------------------------------------------------------------
# the Python oracles: Performer features and attention, the gradient

PY_ORACLES = {
    "favor": (FAVOR_PY, test_oracle_favor, "fv", FAVOR_MUTANTS),
    "backward": (BACKWARD_PY, test_oracle_backward, "bw", BACKWARD_MUTANTS),
}


@pytest.mark.parametrize("which", sorted(PY_ORACLES))
def test_unmodified_python_oracle_passes_every_pin(tmp_path, monkeypatch, which):
    path, tests, attr, _ = PY_ORACLES[which]
    oracle.build()
    monkeypatch.setattr(tests, attr, module_from_source(read(path), tmp_path, which))
    assert len(pins(tests)) >= 5
    assert failing_pins(tests, oracle, False) == []


@pytest.mark.parametrize("which,mutant",
                         [(w, m) for w in sorted(PY_ORACLES) for m in PY_ORACLES[w][3]],
                         ids=[f"{w}-{m[0]}" for w in sorted(PY_ORACLES) for m in PY_ORACLES[w][3]])
def test_mistake_in_python_oracle_fails_a_pin(tmp_path, monkeypatch, which, mutant):
    path, tests, attr, _ = PY_ORACLES[which]
    name, old, new, nth = mutant
    text = read(path)
    planted = plant(text, old, new, nth)
    assert planted != text
    oracle.build()
    monkeypatch.setattr(tests, attr, module_from_source(planted, tmp_path, f"{which}_{name}"))
    caught = failing_pins(tests, oracle, True)
    assert caught, f"no pin fails with the mistake {name!r} planted in oracle/{which}.py"
