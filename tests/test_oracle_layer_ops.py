"""The oracle's layer steps (RMSNorm, SiLU(gate) * up, residual add) pinned to
closed forms and invariants, and shown strong enough: each plausible slip
planted in a copy of the oracle's source fails at least one pin (no GPU)."""
import importlib.util
import math
import os

import numpy as np
import pytest

from oracle import layer_ops

SRC = layer_ops.__file__


# ---- pins: each takes the module under test and asserts -------------------

def pin_rmsnorm_three_four(m):
    # mean of squares of (3, 4) is 12.5; 1/sqrt(12.5) = sqrt(2)/5
    out = m.rmsnorm(np.array([3.0, 4.0]), np.ones(2), 0.0)
    r2 = math.sqrt(2.0)
    assert np.allclose(out, [3 * r2 / 5, 4 * r2 / 5], rtol=1e-15, atol=0)


def pin_rmsnorm_unit_mean_square(m):
    # with unit weights and eps = 0 the output's mean square is exactly 1
    x = np.random.default_rng(1).normal(size=(3, 257)) * np.array([[1e-3], [1.0], [1e4]])
    out = m.rmsnorm(x, np.ones(257), 0.0)
    assert np.allclose(np.mean(out * out, axis=1), 1.0, rtol=1e-13, atol=0)


def pin_rmsnorm_scale_invariant(m):
    x = np.random.default_rng(2).normal(size=(2, 64))
    w = np.random.default_rng(3).normal(size=64)
    assert np.allclose(m.rmsnorm(7.0 * x, w, 0.0), m.rmsnorm(x, w, 0.0), rtol=1e-13, atol=1e-15)


def pin_rmsnorm_weights_elementwise(m):
    # (3, 4) scaled by weights (2, 0.5): each output is its own weight times the unit-weight one
    r2 = math.sqrt(2.0)
    out = m.rmsnorm(np.array([[3.0, 4.0]]), np.array([2.0, 0.5]), 0.0)
    assert np.allclose(out, [[6 * r2 / 5, 2 * r2 / 5]], rtol=1e-15, atol=0)


def pin_rmsnorm_epsilon(m):
    # all-zero input: eps keeps it finite (0); a constant input c: c / sqrt(c^2 + eps)
    assert np.array_equal(m.rmsnorm(np.zeros(8), np.ones(8), 1e-6), np.zeros(8))
    out = m.rmsnorm(np.full(4, 0.5), np.ones(4), 0.75)   # 0.5 / sqrt(0.25 + 0.75) = 0.5
    assert np.allclose(out, 0.5, rtol=1e-15, atol=0)


def pin_rmsnorm_rows_independent(m):
    x = np.random.default_rng(4).normal(size=(3, 32))
    w = np.random.default_rng(5).normal(size=32)
    whole = m.rmsnorm(x, w, 1e-5)
    for i in range(3):
        assert np.allclose(whole[i], m.rmsnorm(x[i], w, 1e-5), rtol=1e-15, atol=0)


def pin_silu_values(m):
    # SiLU(0) = 0; SiLU(1) = logistic(1) = e / (1 + e); SiLU(v) -> v for large v, -> 0 for very negative v
    assert m.silu(np.array([0.0]))[0] == 0.0
    assert math.isclose(m.silu(np.array([1.0]))[0], math.e / (1.0 + math.e), rel_tol=1e-15)
    assert math.isclose(m.silu(np.array([60.0]))[0], 60.0, rel_tol=1e-15)
    assert abs(m.silu(np.array([-800.0]))[0]) < 1e-300


def pin_silu_reflection(m):
    # v * s(v) - v = -v * s(-v) with s the logistic function: SiLU(-v) = SiLU(v) - v
    v = np.linspace(-20, 20, 81)
    assert np.allclose(m.silu(-v), m.silu(v) - v, rtol=1e-12, atol=1e-12)


def pin_silu_mul_up(m):
    g = np.random.default_rng(6).normal(size=40)
    u = np.random.default_rng(7).normal(size=40)
    assert np.allclose(m.silu_mul(g, u), m.silu(g) * u, rtol=0, atol=0)
    assert np.allclose(m.silu_mul(g, 3.0 * u), 3.0 * m.silu_mul(g, u), rtol=1e-15, atol=0)
    assert np.array_equal(m.silu_mul(g, np.zeros(40)), np.zeros(40))


def pin_add(m):
    a = np.random.default_rng(8).normal(size=(2, 9))
    assert np.array_equal(m.add(a, np.zeros((2, 9))), a)
    assert np.array_equal(m.add(a, -a), np.zeros((2, 9)))
    assert np.array_equal(m.add(np.array([1.5]), np.array([2.25])), np.array([3.75]))


PINS = [pin_rmsnorm_three_four, pin_rmsnorm_unit_mean_square, pin_rmsnorm_scale_invariant,
        pin_rmsnorm_weights_elementwise, pin_rmsnorm_epsilon, pin_rmsnorm_rows_independent, pin_silu_values,
        pin_silu_reflection, pin_silu_mul_up, pin_add]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_layer_ops_pin(pin):
    pin(layer_ops)


# ---- mutants: a plausible slip planted in a copy of the source ------------

MUTANTS = {
    "rms_mean_not_squared": ("np.mean(x2 * x2, axis=1", "np.mean(x2, axis=1"),
    "rms_sum_not_mean": ("np.mean(x2 * x2, axis=1, keepdims=True)", "np.sum(x2 * x2, axis=1, keepdims=True)"),
    "rms_no_sqrt": ("/ np.sqrt(ms + float(eps))", "/ (ms + float(eps))"),
    "rms_eps_outside": ("np.sqrt(ms + float(eps))", "(np.sqrt(ms) + float(eps))"),
    "rms_weights_divide": ("out = w[None, :] * x2 /", "out = x2 / w[None, :] /"),
    "rms_column_mean": ("axis=1, keepdims=True", "axis=0, keepdims=True"),
    "silu_sign": ("np.exp(-v)", "np.exp(v)"),
    "silu_is_sigmoid": ("return v / (1.0 + np.exp(-v))", "return 1.0 / (1.0 + np.exp(-v))"),
    "silu_mul_no_up": ("return silu(gate) * np.asarray(up, dtype=np.float64)", "return silu(gate)"),
    "silu_mul_on_up": ("return silu(gate) * np.asarray(up, dtype=np.float64)",
                       "return np.asarray(gate, dtype=np.float64) * silu(up)"),
    "add_subtracts": ("np.asarray(a, dtype=np.float64) + np.asarray(b", "np.asarray(a, dtype=np.float64) - np.asarray(b"),
}


def _load_mutant(tmp_path, name):
    before, after = MUTANTS[name]
    with open(SRC) as f:
        src = f.read()
    assert src.count(before) == 1, name
    path = os.path.join(tmp_path, f"layer_ops_{name}.py")
    with open(path, "w") as f:
        f.write(src.replace(before, after))
    spec = importlib.util.spec_from_file_location(f"layer_ops_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_layer_ops_mutant_is_caught(name, tmp_path):
    mod = _load_mutant(str(tmp_path), name)
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mod)
        except (AssertionError, FloatingPointError, ValueError, ZeroDivisionError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passes every pin"
