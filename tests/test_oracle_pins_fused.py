"""Pins of the fused residual + modulated RMS normalisation oracle
(oracle/fused_ops_oracle.py) against facts independent of its formulas: pure-Python loops
on tiny rows, the unit RMS of a normalised row, scale invariance, the identities of the
modulation and of the gate, the per-sample expansion of the modulation vectors, and planted
mistakes that must each make a pin fail. CPU only."""

import importlib.util
import math
import os

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_FILE = os.path.join(ROOT, "oracle", "fused_ops_oracle.py")


def _load():
    spec = importlib.util.spec_from_file_location("fused_oracle_pinned", ORACLE_FILE)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


F = _load()
ident = lambda v: np.asarray(v, np.float64)


def pin_python_loops(o):
    """Tiny rows evaluated element by element with math.sqrt."""
    r = np.random.default_rng(2)
    rows, D, rps, eps = 4, 5, 2, 1e-3
    h, u = r.standard_normal((rows, D)), r.standard_normal((rows, D))
    gate, scale, shift = (r.standard_normal((2, D)) for _ in range(3))
    h2, y = o.residual_modnorm(h, u, gate, scale, shift, eps, rps, ident)
    for i in range(rows):
        b = i // rps
        hh = [h[i][d] + gate[b][d] * u[i][d] for d in range(D)]
        ms = sum(v * v for v in hh) / D
        for d in range(D):
            assert abs(h2[i][d] - hh[d]) <= 1e-14
            ref = hh[d] / math.sqrt(ms + eps) * (1 + scale[b][d]) + shift[b][d]
            assert abs(y[i][d] - ref) <= 1e-12 * (1 + abs(ref))


def pin_unit_rms_and_scale_invariance(o):
    """Without modulation, mean(y^2) = ms / (ms + eps), and normalising c x gives the
    same rows as x when eps is negligible."""
    r = np.random.default_rng(3)
    x = r.standard_normal((6, 256)) * np.exp(r.uniform(-3, 3, (6, 1)))
    _, y = o.residual_modnorm(x, None, None, None, None, 0.0, 6, ident)
    np.testing.assert_allclose(np.mean(y * y, axis=1), 1.0, rtol=1e-12)
    _, y2 = o.residual_modnorm(7.5 * x, None, None, None, None, 0.0, 6, ident)
    np.testing.assert_allclose(y2, y, rtol=1e-12)
    eps = 0.5
    _, ye = o.residual_modnorm(x, None, None, None, None, eps, 6, ident)
    ms = np.mean(x * x, axis=1)
    np.testing.assert_allclose(np.mean(ye * ye, axis=1), ms / (ms + eps), rtol=1e-12)


def pin_modulation_and_gate_identities(o):
    """scale = shift = 0 is the plain normalisation; a shift only adds; scale = -1 gives
    the shift; gate 0 leaves h, gate 1 adds u."""
    r = np.random.default_rng(4)
    h, u = r.standard_normal((4, 64)), r.standard_normal((4, 64))
    z = np.zeros((1, 64))
    _, y0 = o.residual_modnorm(h, None, None, None, None, 1e-6, 4, ident)
    _, yz = o.residual_modnorm(h, None, None, z, z, 1e-6, 4, ident)
    np.testing.assert_allclose(yz, y0, rtol=0, atol=0)
    sh = r.standard_normal((1, 64))
    _, ys = o.residual_modnorm(h, None, None, None, sh, 1e-6, 4, ident)
    np.testing.assert_allclose(ys - y0, np.repeat(sh, 4, axis=0), rtol=1e-13, atol=1e-13)
    _, ym = o.residual_modnorm(h, None, None, -np.ones((1, 64)), sh, 1e-6, 4, ident)
    np.testing.assert_allclose(ym, np.repeat(sh, 4, axis=0), rtol=0, atol=1e-15)
    h2, _ = o.residual_modnorm(h, u, np.zeros((1, 64)), None, None, 1e-6, 4, ident)
    np.testing.assert_allclose(h2, h, rtol=0, atol=0)
    h2, _ = o.residual_modnorm(h, u, np.ones((1, 64)), None, None, 1e-6, 4, ident)
    np.testing.assert_allclose(h2, h + u, rtol=0, atol=1e-15)


def pin_per_sample_vectors(o):
    """Rows r and r' of one sample share its vectors; rows of different samples do not:
    with shifts only, y - y_plain is the row's sample vector."""
    r = np.random.default_rng(5)
    rows, rps, D = 6, 3, 16
    h = r.standard_normal((rows, D))
    sh = np.stack([np.full(D, 1.0), np.full(D, -2.0)])
    _, y0 = o.residual_modnorm(h, None, None, None, None, 1e-6, rps, ident)
    _, y = o.residual_modnorm(h, None, None, None, sh, 1e-6, rps, ident)
    assert np.allclose(y[:3] - y0[:3], 1.0) and np.allclose(y[3:] - y0[3:], -2.0)


def pin_norm_reads_stored_residual(o):
    """The normalisation reads h' as stored: with a rounding that keeps one decimal, the
    output is the normalisation of the rounded h'."""
    h = np.array([[0.04, 1.0, -2.0, 0.0]])
    u = np.array([[0.02, 0.0, 0.0, 1.0]])
    rnd = lambda v: np.round(np.asarray(v, np.float64), 1)
    h2, y = o.residual_modnorm(h, u, None, None, None, 1e-9, 1, rnd)
    np.testing.assert_allclose(h2, [[0.1, 1.0, -2.0, 1.0]], atol=1e-15)
    ref = np.array([0.1, 1.0, -2.0, 1.0]) / math.sqrt((0.01 + 1 + 4 + 1) / 4 + 1e-9)
    np.testing.assert_allclose(y[0], ref, rtol=1e-12)


PINS = [pin_python_loops, pin_unit_rms_and_scale_invariance, pin_modulation_and_gate_identities,
        pin_per_sample_vectors, pin_norm_reads_stored_residual]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_fused_oracle_pin(pin):
    pin(F)


def _mut_eps_outside(m):
    m.rms_norm = lambda x, eps: np.asarray(x, np.float64) / (np.sqrt(np.mean(np.asarray(x, np.float64) ** 2, axis=-1, keepdims=True)) + eps)


def _mut_sum_not_mean(m):
    m.rms_norm = lambda x, eps: np.asarray(x, np.float64) / np.sqrt(np.sum(np.asarray(x, np.float64) ** 2, axis=-1, keepdims=True) + eps)


def _mut_scale_not_one_plus(m):
    orig = m.modulate
    m.modulate = lambda x, scale, shift: orig(x, None if scale is None else np.asarray(scale) - 1.0, shift)


def _mut_norm_before_residual(m):
    orig = m.residual_modnorm

    def f(h, u, gate, scale, shift, eps, rps, round_to):
        h2, _ = orig(h, u, gate, scale, shift, eps, rps, round_to)
        _, y = orig(h, None, gate, scale, shift, eps, rps, round_to)
        return h2, y
    m.residual_modnorm = f


def _mut_norm_unrounded(m):
    orig = m.residual_modnorm

    def f(h, u, gate, scale, shift, eps, rps, round_to):
        h2, _ = orig(h, u, gate, scale, shift, eps, rps, round_to)
        _, y = orig(h, u, gate, scale, shift, eps, rps, lambda v: np.asarray(v, np.float64))
        return h2, y
    m.residual_modnorm = f


def _mut_sample_index(m):
    m.per_row = lambda vec, rows, rps: None if vec is None else np.asarray(vec, np.float64)[np.arange(rows) % np.asarray(vec).shape[0]]


MUTANTS = {"eps_outside_sqrt": _mut_eps_outside, "sum_not_mean": _mut_sum_not_mean,
           "scale_not_one_plus": _mut_scale_not_one_plus, "norm_before_residual": _mut_norm_before_residual,
           "norm_of_unrounded_residual": _mut_norm_unrounded, "wrong_sample_index": _mut_sample_index}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_fused_pins_catch_planted_mistakes(name):
    mod = _load()
    MUTANTS[name](mod)
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mod)
        except (AssertionError, ValueError, FloatingPointError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"planted mistake {name} was not caught"
